// Shared host helpers and hand-written sm_103a PTX wrappers (mbarrier, TMA,
// tcgen05) used by the kernels of this library.  Written from the PTX ISA
// descriptions of these instructions.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "iha.h"

namespace iha {

// Every wait in these kernels gives up after this long and reports
// DEV_ERR_WAIT_TIMEOUT instead of spinning forever.
constexpr uint64_t kWaitLimitNs = 4000000000ull;

// ---------------------------------------------------------------- host side
// Records a formatted detail for iha_last_error() and returns `s`.
iha_status fail(iha_status s, const char* fmt, ...);
// Maps the last launch error to IHA_ERR_CUDA (with detail) or IHA_OK.
iha_status check_launch(const char* what);
// 16-byte alignment of a device pointer.
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
// SM count of the current device (cached per device).
int sm_count();
// cuTensorMapEncodeTiled through the runtime's driver entry point (no -lcuda).
CUresult encode_tiled(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t rank,
                      void* base, const uint64_t* dims, const uint64_t* strides_bytes,
                      const uint32_t* box, CUtensorMapSwizzle swizzle);

// Wait limit and withheld-load flag for the next kernel launch on this host
// thread: kWaitLimitNs and false unless iha_test_fail_next_wait() armed a
// one-shot test of the failure path (consumed by the read).
uint64_t wait_limit_for_next_launch();
bool withhold_for_this_launch();

// Device error codes (see iha_device_error in iha.h).
enum : unsigned { DEV_ERR_KEEP_INDEX = 1u, DEV_ERR_WAIT_TIMEOUT = 2u, DEV_ERR_SMEM_ALIGN = 4u };

// Each translation unit owns one device error word (no relocatable device
// code); its reader is registered here and iha_device_error() ORs them all.
typedef int (*dev_error_reader)(int clear);
int register_dev_error_reader(dev_error_reader r);

// Dynamic work distribution for persistent kernels.  Each translation unit
// that uses it owns a table of kWorkSlots counter pairs {next, done}; every
// launch takes the next slot (round robin on the host), CTA b starts on item
// b and takes each further item from the slot's `next` counter (offset by the
// grid), so a CTA that finishes early takes more of the remaining items.  The
// last CTA to leave resets the pair for the next launch that takes the slot
// (launches sharing a slot would need kWorkSlots launches in flight at once).
constexpr int kWorkSlots = 256;
#define IHA_WORK_QUEUE(tag)                                                     \
  static __device__ unsigned int g_work[::iha::kWorkSlots][2];                  \
  static unsigned int tag##_work_slot() {                                       \
    static std::atomic<unsigned int> seq{0};                                    \
    return seq.fetch_add(1u, std::memory_order_relaxed) % ::iha::kWorkSlots;    \
  }

// A kernel's dynamic shared-memory limit, raised on each device the first
// time the kernel is launched there: the attribute belongs to the kernel's
// instance in that device's context, so one call per process would leave a
// second device of the same process at the default limit.  The first caller
// on a device sets it under the lock; later callers see the device's bit.
class SmemLimit {
 public:
  template <typename F>
  cudaError_t ensure(F* kernel, int bytes) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
    if (bit != 0 && (done_.load(std::memory_order_acquire) & bit) != 0) return cudaSuccess;
    std::lock_guard<std::mutex> lk(mu_);
    if (bit != 0 && (done_.load(std::memory_order_relaxed) & bit) != 0) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done_.fetch_or(bit, std::memory_order_release);
    return e;
  }

 private:
  std::atomic<uint64_t> done_{0};  // bit d: set on device d
  std::mutex mu_;
};

#define IHA_DEVICE_ERROR_WORD(tag)                                              \
  static __device__ unsigned int g_dev_error;                                   \
  static int tag##_read_dev_error(int clear) {                                  \
    unsigned int v = 0;                                                         \
    if (cudaMemcpyFromSymbol(&v, g_dev_error, sizeof(v)) != cudaSuccess)        \
      return -1;                                                                \
    if (clear && v) {                                                           \
      unsigned int z = 0;                                                       \
      if (cudaMemcpyToSymbol(g_dev_error, &z, sizeof(z)) != cudaSuccess)        \
        return -1;                                                              \
    }                                                                           \
    return (int)v;                                                              \
  }                                                                             \
  static int tag##_reg_ = ::iha::register_dev_error_reader(tag##_read_dev_error);

// ---------------------------------------------------------------- device side
#if defined(__CUDACC__)

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
// Ends the barrier's life: required before its memory is used for anything
// else, including another barrier.
__device__ __forceinline__ void mbar_inval(uint32_t bar) {
  asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for phase `parity` of the barrier.  Returns false if the wait
// gave up (after limit_ns) or if `abort_flag` (shared) was raised by another
// thread of the block; the caller then unwinds.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          volatile int* abort_flag,
                                          uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
}

// The same wait for a whole warp that goes on to warp-collective tcgen05
// loads or stores: every lane gets the same answer, so a wait that gives up
// on one lane while the barrier completes on another cannot split the warp.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity,
                                               volatile int* abort_flag,
                                               uint64_t limit_ns = kWaitLimitNs) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, limit_ns));
}

// ---- TMA (tiled bulk tensor copies)
__device__ __forceinline__ void tma_prefetch_desc(const void* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* map, uint32_t bar, int c0,
                                            int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const void* map, uint32_t bar, int c0,
                                            int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}
__device__ __forceinline__ void tma_load_5d(uint32_t dst, const void* map, uint32_t bar, int c0,
                                            int c1, int c2, int c3, int c4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
      "r"(c4)
      : "memory");
}

// Untiled bulk copies (addresses 16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_load(uint32_t dst_smem, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst_smem),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void bulk_store(void* dst, uint32_t src_smem, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(
                   reinterpret_cast<uint64_t>(dst)),
               "r"(src_smem), "r"(bytes)
               : "memory");
}

// TMA store from shared memory (bulk-group completion).
__device__ __forceinline__ void tma_store_3d(const void* map, uint32_t src, int c0, int c1,
                                             int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(src), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void tma_store_5d(const void* map, uint32_t src, int c0, int c1,
                                             int c2, int c3, int c4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.global.shared::cta.tile.bulk_group"
      " [%0, {%2, %3, %4, %5, %6}], [%1];" ::"l"(reinterpret_cast<uint64_t>(map)),
      "r"(src), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
      : "memory");
}
// Tiled bulk reduce-add from shared memory into global (element type of the
// tensor map; fp32 here), bulk-group completion like a store.
__device__ __forceinline__ void tma_reduce_add_4d(const void* map, uint32_t src, int c0, int c1,
                                                  int c2, int c3) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.4d.global.shared::cta.add.tile.bulk_group"
      " [%0, {%2, %3, %4, %5}], [%1];" ::"l"(reinterpret_cast<uint64_t>(map)),
      "r"(src), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until at most N committed bulk groups are still reading shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Wait until at most N committed bulk groups are still in flight (writes done).
template <int N>
__device__ __forceinline__ void bulk_wait() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}
// Make generic-proxy shared-memory writes visible to the async proxy (TMA,
// tcgen05.mma operands).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Named barrier over `nthreads` threads (warp multiples).
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---- tcgen05: tensor memory
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ---- tcgen05: MMA (kind::f16, one CTA), operands from shared memory
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// A operand from tensor memory (K-major, two 16-bit elements per column).
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Issue-only variants for tight MMA loops: no "memory" clobber, so the
// compiler keeps descriptors in registers across back-to-back issues.  The
// ordering against shared-memory producers and TMEM consumers comes from the
// mbarrier waits and tcgen05.commit (volatile asm with memory clobbers)
// around the loop; volatile asm statements keep their relative order.
__device__ __forceinline__ void mma_ss_nm(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate));
}
__device__ __forceinline__ void mma_ts_nm(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate));
}
// Arrive once on `bar` when every tcgen05 operation issued so far by this
// thread has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// Instruction descriptor, kind::f16, bf16 x bf16 -> f32, dense.
//   bits 4-5 D format (1 = f32), 7-9 A format (1 = bf16), 10-12 B format,
//   15 A major (0 = K), 16 B major (1 = MN), 17-22 N >> 3, 24-28 M >> 4.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn_major,
                                                      bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) |
         ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

// Shared-memory matrix descriptor (tcgen05 format): start address >> 4 in
// bits 0-13, leading byte offset >> 4 in 16-29, stride byte offset >> 4 in
// 32-45, version 1 in bits 46-47, swizzle mode in 61-63 (2 = 128-byte).
//   K-major, 128B swizzle: rows of 128 bytes, 8-row atoms; SBO = atom-row
//     stride (1024 for dense rows); LBO unused (1).
//   MN-major, 128B swizzle: 64 contiguous MN elements per 128-byte row, one
//     row per K index, 8 K rows per atom; LBO = stride between 64-element MN
//     blocks, SBO = stride between 8-row K groups.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo_bytes,
                                                    uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1u << 46;
  d |= (uint64_t)2u << 61;
  return d;
}

// ---- tcgen05: tensor memory <-> registers (32 lanes x 32 bits, 32 columns)
#define IHA_R32(p)                                                                         \
  "=r"(p[0]), "=r"(p[1]), "=r"(p[2]), "=r"(p[3]), "=r"(p[4]), "=r"(p[5]), "=r"(p[6]),      \
      "=r"(p[7]), "=r"(p[8]), "=r"(p[9]), "=r"(p[10]), "=r"(p[11]), "=r"(p[12]),           \
      "=r"(p[13]), "=r"(p[14]), "=r"(p[15]), "=r"(p[16]), "=r"(p[17]), "=r"(p[18]),        \
      "=r"(p[19]), "=r"(p[20]), "=r"(p[21]), "=r"(p[22]), "=r"(p[23]), "=r"(p[24]),        \
      "=r"(p[25]), "=r"(p[26]), "=r"(p[27]), "=r"(p[28]), "=r"(p[29]), "=r"(p[30]),        \
      "=r"(p[31])
#define IHA_W32(p)                                                                          \
  "r"(p[0]), "r"(p[1]), "r"(p[2]), "r"(p[3]), "r"(p[4]), "r"(p[5]), "r"(p[6]), "r"(p[7]),  \
      "r"(p[8]), "r"(p[9]), "r"(p[10]), "r"(p[11]), "r"(p[12]), "r"(p[13]), "r"(p[14]),    \
      "r"(p[15]), "r"(p[16]), "r"(p[17]), "r"(p[18]), "r"(p[19]), "r"(p[20]), "r"(p[21]),  \
      "r"(p[22]), "r"(p[23]), "r"(p[24]), "r"(p[25]), "r"(p[26]), "r"(p[27]), "r"(p[28]),  \
      "r"(p[29]), "r"(p[30]), "r"(p[31])

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%32];"
      : IHA_R32(r)
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31, %32};" ::"r"(taddr),
      IHA_W32(r)
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Waits (bounded) until every tcgen05 operation this thread issued has
// completed: a commit to the single-use barrier `bar` (count 1, phase 0).
// Used before tensor memory is released on every exit path.
// Whole-warp issue of tcgen05 work.  When one lane of a warp issues MMAs
// inside a lane-divergent branch while the SM's other warps keep the issue
// slots busy, each MMA waits for its descriptor operands to be moved into
// uniform registers; measured, a 128 x 128 x 16 MMA then costs ~110 cycles
// instead of ~65.  So the issuing warp runs its whole schedule in step (every
// value stays warp-uniform) and one elected lane executes each tcgen05
// instruction.
__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n\t.reg .pred P;\n\telect.sync _|P, 0xffffffff;\n\tselp.b32 %0, 1, 0, P;\n\t}"
      : "=r"(pred));
  return pred != 0;
}
__device__ __forceinline__ void mma_commit_warp(uint32_t bar) {
  if (elect_one()) mma_commit(bar);
  __syncwarp();
}

__device__ __forceinline__ void mma_drain(uint32_t bar) {
  mma_commit(bar);
  volatile int no_abort = 0;
  mbar_wait(bar, 0, &no_abort);
}
// The same for a warp that issues MMAs with elect_one().
__device__ __forceinline__ void mma_drain_warp(uint32_t bar) {
  mma_commit_warp(bar);
  volatile int no_abort = 0;
  mbar_wait(bar, 0, &no_abort);
}

// ---- dynamic work distribution (see IHA_WORK_QUEUE)
// The item after this CTA's current one (one lane asks; items >= the item
// count mean "no more").
__device__ __forceinline__ int work_next(unsigned int* slot) {
  return (int)(atomicAdd(slot, 1u) + gridDim.x);
}
// Called by one thread of the CTA after every work_next of the CTA: the last
// CTA to leave resets the slot for a later launch.
__device__ __forceinline__ void work_leave(unsigned int* slot) {
  __threadfence();
  if (atomicAdd(slot + 1, 1u) == gridDim.x - 1) {
    atomicExch(slot, 0u);
    atomicExch(slot + 1, 0u);
  }
}

// ---- misc
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// 2^x for a pair, on the FMA and integer pipes instead of the MUFU unit.
// Method: Cody-Waite style range reduction x = j + f with j = round(x) (the
// 1.5 * 2^23 shifter leaves j in the low mantissa bits) and f in [-1/2, 1/2],
// then 2^f by a degree-3 polynomial fitted for minimax relative error on
// [-1/2, 1/2] with the Remez exchange algorithm (max relative error 7.5e-5,
// far below the 2^-9 of the bf16 probabilities it feeds), and 2^j added
// into the exponent field.  x is clamped to >= -125 so the exponent stays
// normal; -inf (masked scores) gives 2^-125 ~ 2e-38 instead of 0.
__device__ __forceinline__ float2 exp2_poly3_x2(float2 x) {
  constexpr float kShift = 12582912.0f;  // 1.5 * 2^23
  x.x = fmaxf(x.x, -125.f);
  x.y = fmaxf(x.y, -125.f);
  const float2 t = __fadd2_rn(x, make_float2(kShift, kShift));
  const float2 r = __fadd2_rn(t, make_float2(-kShift, -kShift));
  const float2 f = __fadd2_rn(x, make_float2(-r.x, -r.y));
  float2 q = __ffma2_rn(make_float2(0.0551716685f, 0.0551716685f), f,
                        make_float2(0.242611125f, 0.242611125f));
  q = __ffma2_rn(q, f, make_float2(0.693260968f, 0.693260968f));
  q = __ffma2_rn(q, f, make_float2(0.999928057f, 0.999928057f));
  return make_float2(
      __uint_as_float(__float_as_uint(q.x) + (__float_as_uint(t.x) << 23)),
      __uint_as_float(__float_as_uint(q.y) + (__float_as_uint(t.y) << 23)));
}

// c ? a : b without a branch (one selp; a per-lane condition on a register
// array element must not become a divergent branch per element).
__device__ __forceinline__ uint32_t sel_u32(bool c, uint32_t a, uint32_t b) {
  uint32_t r;
  asm("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %1, 0;\n\tselp.b32 %0, %2, %3, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)c), "r"(a), "r"(b));
  return r;
}

// max(a, b, c) in one instruction (three-input max.f32, sm_100 family).
__device__ __forceinline__ float fmax3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// Elementwise maximum of two bf16 pairs (a maximum returns one of its inputs).
__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ float bf16lo_to_f32(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t v) {
  return __uint_as_float(v & 0xFFFF0000u);
}

#endif  // __CUDACC__

}  // namespace iha
