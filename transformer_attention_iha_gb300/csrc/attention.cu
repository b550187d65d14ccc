// Multi-head softmax attention forward over pseudo-heads / mask units.
//
// "IHA-CUDA: Interleaved Head Attention Kernels for Hopper GPUs", sections
// "Kernel Design" (attention over the H*P pseudo-heads after the premix,
// sliding window) and "FLOP Matching" (window W = WSL + 1, 128-token tiles);
// "hiera-optim 0.1.0", hiera_optim/attention/mask_unit.py,
// MaskUnitAttentionFast.forward (unmasked attention inside each mask unit,
// scale head_dim ** -0.5, tokens laid out (T outer, units inner)).
//
// bf16 path (sm_103a tensor cores), persistent:
//   One CTA per SM walks a list of work items; an item is two adjacent
//   128-row query tiles of one head.  Items are grouped by heads (a group's
//   K / V stays in L2 while its items run) and, inside a group, ordered
//   heaviest first (longest key range).  CTA b starts on item b and takes
//   each further item from a global counter when it reaches it (the
//   producer warp asks one item ahead and passes the index to the other
//   warps through a four-entry ring in shared memory), so CTAs that draw
//   short items take more of them.
//   10 warps:
//     warps 0-3  softmax + epilogue of query tile 0 (thread = row = TMEM lane)
//     warps 4-7  softmax + epilogue of query tile 1
//     warp  8    TMA producer: Q tiles per item, K and V tiles into separate
//                two-slot rings (a K slot frees after its QK^T, a V slot
//                after its P.V, so K runs ahead of V)
//     warp  9    tcgen05.mma issuer (one thread) and TMEM owner
//   TMEM (512 columns): S0 | S1 | O0 | O1, 128 fp32 columns each.  P (bf16)
//   overwrites the first 64 columns of S and feeds the P.V MMA as the
//   A operand straight from tensor memory.
//   Each query tile visits only its own key-tile range (causal / window
//   block skipping); the two tiles of an item share the K / V stream.
//   Online softmax in the log2 domain with conditional rescaling: O and l
//   are rescaled only when a row maximum grows by more than 8 (a factor of
//   256), which keeps every exponent <= 2^8 and is exact in real arithmetic.
//   A quarter of the exponentials run as a polynomial on the FMA pipe so the
//   MUFU unit does not bound the softmax.
// f32 path: CUDA-core kernel in fp32 throughout (no TF32), for fp32 tensors.
#include <math.h>

#include <mutex>

#include "common.cuh"
#include "mu_attention.h"

namespace iha {
namespace {

IHA_DEVICE_ERROR_WORD(attention)
IHA_WORK_QUEUE(attention)

constexpr int kBM = 128;             // query rows per tile
constexpr int kBN = 128;             // keys per tile
constexpr int kChunk = 64;           // head-dim elements per 128-byte swizzle row
constexpr int kTileChunkBytes = kBM * 128;  // 16 KB: 128 rows x 64 bf16
constexpr int kThreads = 320;
constexpr int kKSlots = 2;           // K ring depth (V ring: 2)
constexpr int kStgBytes = 32 * 128;  // per softmax warp: 32 rows x 64 bf16 of O
// Q 2x2, K 2x2, V 2x2 chunks | O staging of the 8 softmax warps
constexpr int kSmemTiles = (4 + 2 * kKSlots + 4) * kTileChunkBytes + 8 * kStgBytes;
constexpr int kSmemBytes = kSmemTiles + 512 + 1024;  // + barriers + alignment slack
static_assert(kSmemBytes <= 227 * 1024, "attention forward: over the per-block shared memory limit");
constexpr float kRescaleLog2 = 8.0f;
// L2 budget for the K / V of one head group.
constexpr int64_t kGroupKVBytes = 48ll << 20;

struct AttnParams {
  int Bo, Bi, Hh, Nq, Nk, d, nD;
  int mask, window;
  int n_qt, n_qpairs, n_hb, group, n_items;
  float scale_log2;
  int64_t so_bo, so_bi, so_seq, so_h;
  __nv_bfloat16* o;
  float* lse;
  uint64_t wait_limit_ns;
  int withhold;  // failure-path test: CTA 0 never loads its first V tile
  int work_slot;  // counter pair of this launch (dynamic item distribution)
};

struct Item {
  int h, bo, bi, bz;
  int qt0;          // query tiles qt0 and qt0 + 1 (the second only if act1)
  bool act1;
  int lo0, hi0;     // key-tile range of query tile qt0 (inclusive)
  int lo1, hi1;     // ... of query tile qt0 + 1 (empty unless act1)
  int jlo, jhi;     // union
};

// KV tile range [lo, hi] (inclusive) of query tile qt.
__device__ __forceinline__ void kv_tile_range(const AttnParams& p, int qt, int& lo, int& hi) {
  const int n_kt = (p.Nk + kBN - 1) / kBN;
  if (p.mask == IHA_MASK_NONE) {
    lo = 0;
    hi = n_kt - 1;
    return;
  }
  const int q_lo = qt * kBM, q_hi = min(q_lo + kBM - 1, p.Nq - 1);
  hi = min(q_hi / kBN, n_kt - 1);
  lo = (p.mask == IHA_MASK_CAUSAL_WINDOW) ? max(0, q_lo - (p.window - 1)) / kBN : 0;
}

// Work item idx: head groups of p.group heads (hb = bz * Hh + h); inside a
// group, query-tile pairs from the heaviest (latest) down, heads innermost.
__device__ __forceinline__ Item decode_item(const AttnParams& p, int idx) {
  const int per_group = p.group * p.n_qpairs;
  const int n_groups = (p.n_hb + p.group - 1) / p.group;
  const int g = min(idx / per_group, n_groups - 1);
  const int hb0 = g * p.group;
  const int gs = min(p.group, p.n_hb - hb0);
  const int r = idx - g * per_group;
  const int rank = r / gs;
  const int hb = hb0 + (r - rank * gs);
  Item it;
  it.h = hb % p.Hh;
  it.bz = hb / p.Hh;
  it.bo = it.bz / p.Bi;
  it.bi = it.bz - it.bo * p.Bi;
  const int pair = p.n_qpairs - 1 - rank;
  it.qt0 = 2 * pair;
  it.act1 = it.qt0 + 1 < p.n_qt;
  kv_tile_range(p, it.qt0, it.lo0, it.hi0);
  if (it.act1) {
    kv_tile_range(p, it.qt0 + 1, it.lo1, it.hi1);
  } else {
    it.lo1 = it.lo0;
    it.hi1 = it.lo0 - 1;  // empty
  }
  it.jlo = it.lo0;  // lo1 >= lo0 and hi1 >= hi0: tile 1 is the later one
  it.jhi = it.act1 ? max(it.hi0, it.hi1) : it.hi0;
  return it;
}

// -inf outside the visible columns [c_lo, c_hi] of a row, for NC chunks of 32
// scores starting at column c0.  A row's visible columns form one interval
// and a warp holds 32 consecutive rows, so most chunks are visible (or
// hidden) for the whole warp: those take a warp-uniform shortcut, and only
// the chunks the interval edge crosses pay a select per score.
template <int NC>
__device__ __forceinline__ void mask_cols(uint32_t* s, int c0, int c_lo, int c_hi) {
#pragma unroll
  for (int cc = 0; cc < NC; ++cc) {
    const int a = c0 + 32 * cc;
    // visible columns of this chunk, bits lo .. hi - 1
    const int lo = min(max(c_lo - a, 0), 32), hi = min(max(c_hi - a + 1, 0), 32);
    const uint32_t vis = (hi >= 32 ? 0xFFFFFFFFu : ((1u << hi) - 1u)) &
                         ~(lo >= 32 ? 0xFFFFFFFFu : ((1u << lo) - 1u));
    if (__any_sync(0xffffffffu, vis != 0xFFFFFFFFu)) {
#pragma unroll
      for (int e = 0; e < 32; ++e)
        s[32 * cc + e] = (vis >> e) & 1u ? s[32 * cc + e] : 0xFF800000u;
    }
  }
}

__device__ __forceinline__ void raise_error(volatile int* abort_flag) {
  *abort_flag = 1;
  atomicOr(&g_dev_error, DEV_ERR_WAIT_TIMEOUT);
}

// NCH = head-dim chunks of 64 (d <= 64: 1, d <= 128: 2).
template <int NCH>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                       const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV,
                       const __grid_constant__ CUtensorMap tmO, const AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sQ = smem_u32(smem);                       // [tile][chunk]
  const uint32_t sK = sQ + 4 * kTileChunkBytes;             // [slot][chunk], 2 slots
  const uint32_t sV = sK + 2 * kKSlots * kTileChunkBytes;   // [slot][chunk], 2 slots
  const uint32_t sStg = sV + 4 * kTileChunkBytes;          // [softmax warp][32 rows][128 B]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kSmemTiles);
  const uint32_t bar0 = smem_u32(bars);
  auto b_qfull = [&](int t) { return bar0 + 8u * (0 + t); };
  auto b_qempty = [&](int t) { return bar0 + 8u * (2 + t); };
  auto b_kfull = [&](int s) { return bar0 + 8u * (4 + s); };    // 3 slots
  auto b_kempty = [&](int s) { return bar0 + 8u * (7 + s); };   // 3 slots
  auto b_vfull = [&](int s) { return bar0 + 8u * (10 + s); };
  auto b_vempty = [&](int s) { return bar0 + 8u * (12 + s); };
  auto b_sfull = [&](int t) { return bar0 + 8u * (14 + t); };
  auto b_pfull = [&](int t) { return bar0 + 8u * (16 + t); };
  auto b_ofull = [&](int t) { return bar0 + 8u * (18 + t); };
  const uint32_t b_drain = bar0 + 8u * 20;
  auto b_ifull = [&](int s) { return bar0 + 8u * (22 + s); };   // item ring, 4 entries
  auto b_iempty = [&](int s) { return bar0 + 8u * (26 + s); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 30);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* item_ring = reinterpret_cast<volatile int*>(tmem_slot + 2);
  // 30 barriers, then the TMEM address, the abort flag and the 4-entry ring
  static_assert(30 * 8 + 4 + 4 + 4 * 4 <= 512, "attention forward: barrier region");
  unsigned int* work = g_work[p.work_slot];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint64_t lim = p.wait_limit_ns;
  constexpr uint32_t kChunkBytes = (uint32_t)NCH * kTileChunkBytes;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kKSlots; ++s) {
      mbar_init(b_kfull(s), 1);
      mbar_init(b_kempty(s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(b_qfull(s), 1);
      mbar_init(b_qempty(s), 1);
      mbar_init(b_vfull(s), 1);
      mbar_init(b_vempty(s), 1);
      mbar_init(b_sfull(s), 1);
      mbar_init(b_pfull(s), 128);
      mbar_init(b_ofull(s), 1);
    }
    mbar_init(b_drain, 1);
    for (int s = 0; s < 4; ++s) {
      mbar_init(b_ifull(s), 1);
      mbar_init(b_iempty(s), 9);  // the MMA warp and the 8 softmax warps
    }
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Next item index for a consumer warp (whole warp; false once the wait
  // gave up).  Item indices >= n_items end the walk.
  uint32_t in_c = 0;  // ring entries consumed by this warp
  auto next_item = [&](int& idx) -> bool {
    const int s = (int)(in_c & 3u);
    if (!mbar_wait_warp(b_ifull(s), (in_c >> 2) & 1u, abort_flag, p.wait_limit_ns)) return false;
    idx = item_ring[s];
    __syncwarp();
    if (elect_one()) mbar_arrive(b_iempty(s));
    __syncwarp();
    ++in_c;
    return true;
  };

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    // The whole warp runs the schedule; one elected lane issues (see elect_one).
    {
      if (elect_one()) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
      }
      __syncwarp();
      uint32_t kc = 0, vc = 0, qn0 = 0, qn1 = 0;  // loads issued per ring / Q tile
      bool ok = true;
      // Q tile t of item `it` (qn: loads of that tile so far); returns the new count
      auto load_q = [&](const Item& it, int t, uint32_t qn) -> uint32_t {
        if (qn > 0 && !(ok = mbar_wait_warp(b_qempty(t), (qn - 1) & 1, abort_flag, lim)))
          return qn;
        if (elect_one()) {
          mbar_arrive_expect_tx(b_qfull(t), kChunkBytes);
#pragma unroll
          for (int c = 0; c < NCH; ++c)
            tma_load_5d(sQ + (2 * t + c) * kTileChunkBytes, &tmQ, b_qfull(t), c * kChunk,
                        (it.qt0 + t) * kBM, it.h, it.bi, it.bo);
        }
        __syncwarp();
        return qn + 1;
      };
      // load number n of the K (is_v = false) or V ring; returns the new count
      auto load_kv = [&](const Item& it, int j, bool is_v, uint32_t n) -> uint32_t {
        const uint32_t depth = is_v ? 2u : (uint32_t)kKSlots;
        const int s = (int)(n % depth);
        if (is_v && n == 0 && p.withhold && blockIdx.x == 0)
          return n + 1;  // withheld: its consumer's wait runs out (failure-path test)
        if (n >= depth && !(ok = mbar_wait_warp(is_v ? b_vempty(s) : b_kempty(s),
                                                ((n / depth) - 1) & 1, abort_flag, lim)))
          return n;
        const uint32_t full = is_v ? b_vfull(s) : b_kfull(s);
        const uint32_t dst = (is_v ? sV : sK) + (uint32_t)(2 * s) * kTileChunkBytes;
        if (elect_one()) {
          mbar_arrive_expect_tx(full, kChunkBytes);
#pragma unroll
          for (int c = 0; c < NCH; ++c)
            tma_load_5d(dst + c * kTileChunkBytes, is_v ? &tmV : &tmK, full, c * kChunk, j * kBN,
                        it.h, it.bi, it.bo);
        }
        __syncwarp();
        return n + 1;
      };
      int idx = blockIdx.x;
      for (uint32_t in = 0; ok; ++in) {
        // publish the item to the other warps
        const int s = (int)(in & 3u);
        if (in >= 4 && !(ok = mbar_wait_warp(b_iempty(s), ((in >> 2) - 1) & 1u, abort_flag, lim)))
          break;
        if (elect_one()) {
          item_ring[s] = idx;
          mbar_arrive(b_ifull(s));
        }
        __syncwarp();
        if (idx >= p.n_items) break;
        unsigned int nxt = 0;
        if (lane == 0) nxt = (unsigned int)work_next(work);  // used after the loads
        const Item it = decode_item(p, idx);
        qn0 = load_q(it, 0, qn0);
        for (int j = it.jlo; ok && j <= it.jhi; ++j) {
          kc = load_kv(it, j, false, kc);
          if (ok && j == it.jlo && it.act1) qn1 = load_q(it, 1, qn1);
          if (ok) vc = load_kv(it, j, true, vc);
        }
        idx = (int)__shfl_sync(0xffffffffu, nxt, 0);
      }
      if (!ok) raise_error(abort_flag);
      // Whoever aborted, no copy may still be landing when the CTA exits: wait
      // for the last load issued into every slot (in a normal run each has
      // completed already and the wait returns at once).
      volatile int no_abort = 0;
      for (uint32_t n = kc > (uint32_t)kKSlots ? kc - kKSlots : 0; n < kc; ++n)
        mbar_wait(b_kfull(n % kKSlots), (n / kKSlots) & 1, &no_abort, lim);
      for (uint32_t n = vc > 2u ? vc - 2u : 0; n < vc; ++n)
        mbar_wait(b_vfull(n & 1), (n >> 1) & 1, &no_abort, lim);
      if (qn0 > 0) mbar_wait(b_qfull(0), (qn0 - 1) & 1, &no_abort, lim);
      if (qn1 > 0) mbar_wait(b_qfull(1), (qn1 - 1) & 1, &no_abort, lim);
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the schedule; one elected lane issues (see elect_one).
    {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(kBM, kBN, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(kBM, NCH * kChunk, false, true);
      const uint32_t tS0 = tmem, tS1 = tmem + 128u, tO0 = tmem + 256u, tO1 = tmem + 384u;
      // descriptors of the chunk-0 / K-step-0 positions; K-step kk of a
      // 128-byte-swizzled tile adds (kk / 4) * 16 KB + (kk % 4) * 32 B to the
      // start address, i.e. that >> 4 to the descriptor's low field
      const uint64_t dQ0 = smem_desc_sw128(sQ, 16, 1024);
      const uint64_t dQ1 = smem_desc_sw128(sQ + 2 * kTileChunkBytes, 16, 1024);
      const uint64_t dK0 = smem_desc_sw128(sK, 16, 1024);
      constexpr uint64_t kKSlotDesc = (uint64_t)((2 * kTileChunkBytes) >> 4);  // one K slot
      const uint64_t dV0 = smem_desc_sw128(sV, kTileChunkBytes, 1024);
      const uint64_t dV1 = smem_desc_sw128(sV + 2 * kTileChunkBytes, kTileChunkBytes, 1024);
      uint32_t kc = 0, vc = 0, qn0 = 0, qn1 = 0, pn0 = 0, pn1 = 0;
      bool ok = true;
      auto issue_qk = [&](uint32_t dS, uint64_t dq, uint32_t kslot) {
        const uint64_t dk = dK0 + kKSlotDesc * kslot;
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < 4 * NCH; ++kk) {
            const uint64_t off = (uint64_t)(((kk >> 2) * kTileChunkBytes + (kk & 3) * 32) >> 4);
            mma_ss_nm(dS, dq + off, dk + off, idesc_qk, kk > 0 ? 1u : 0u);
          }
        }
        __syncwarp();
      };
      auto issue_pv = [&](uint32_t dO, uint32_t aP, uint32_t vslot, uint32_t first) {
        const uint64_t dv = vslot ? dV1 : dV0;
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk)
            mma_ts_nm(dO, aP + (uint32_t)(kk * 8), dv + (uint64_t)(kk * 128), idesc_pv,
                      (kk > 0 || !first) ? 1u : 0u);
        }
        __syncwarp();
      };
      // When query tile 0 of an item ends a key step before tile 1 (causal and
      // window masks), the next item is taken from the ring at that step and
      // its first QK^T for tile 0 is issued there (`early0`), so that S is
      // ready when tile 0's softmax warps finish their epilogue instead of
      // after tile 1's last softmax step.
      int idx = 0, idx_next = 0;
      bool have_next = false, early0 = false;
      while (ok) {
        if (have_next) {
          idx = idx_next;
          have_next = false;
        } else if (!(ok = next_item(idx))) {
          break;
        }
        if (idx >= p.n_items) break;
        const Item it = decode_item(p, idx);
        const uint32_t kbase = kc, vbase = vc;
        uint32_t k_ready = early0 ? 1u : 0u;  // K tiles of this item known to be loaded
        auto wait_k = [&](int j) {
          const uint32_t q = (uint32_t)(j - it.jlo);
          while (ok && k_ready <= q) {
            const uint32_t n = kbase + k_ready;
            ok = mbar_wait_warp(b_kfull(n % kKSlots), (n / kKSlots) & 1, abort_flag, lim);
            ++k_ready;
          }
          return ok;
        };
        // prologue: first QK^T of each tile
        if (early0) {
          early0 = false;
        } else if ((ok = mbar_wait_warp(b_qfull(0), qn0 & 1, abort_flag, lim)) && wait_k(it.lo0)) {
          ++qn0;
          tc_fence_after();
          issue_qk(tS0, dQ0, (kbase + (uint32_t)(it.lo0 - it.jlo)) % kKSlots);
          mma_commit_warp(b_sfull(0));
          if (it.lo0 == it.hi0) mma_commit_warp(b_qempty(0));
        }
        if (ok && it.act1) {
          if ((ok = mbar_wait_warp(b_qfull(1), qn1 & 1, abort_flag, lim)) && wait_k(it.lo1)) {
            ++qn1;
            tc_fence_after();
            issue_qk(tS1, dQ1, (kbase + (uint32_t)(it.lo1 - it.jlo)) % kKSlots);
            mma_commit_warp(b_sfull(1));
            if (it.lo1 == it.hi1) mma_commit_warp(b_qempty(1));
          }
        }
        for (int j = it.jlo; ok && j <= it.jhi; ++j) {
          const uint32_t nk = kbase + (uint32_t)(j - it.jlo), nv = vbase + (uint32_t)(j - it.jlo);
          // every QK^T reading K(j) has been issued: release its slot when they finish
          mma_commit_warp(b_kempty(nk % kKSlots));
          if (!(ok = mbar_wait_warp(b_vfull(nv & 1), (nv >> 1) & 1, abort_flag, lim))) break;
          const uint32_t knext = (nk + 1) % kKSlots;
          // tile 0
          if (j >= it.lo0 && j <= it.hi0) {
            if (!(ok = mbar_wait_warp(b_pfull(0), pn0 & 1, abort_flag, lim))) break;
            ++pn0;
            tc_fence_after();
            issue_pv(tO0, tS0, nv & 1, j == it.lo0);
            if (j == it.hi0) {
              mma_commit_warp(b_ofull(0));
            } else {
              if (!wait_k(j + 1)) break;
              tc_fence_after();
              issue_qk(tS0, dQ0, knext);
              mma_commit_warp(b_sfull(0));
              if (j + 1 == it.hi0) mma_commit_warp(b_qempty(0));  // last use of Q tile 0
            }
          }
          // tile 1
          if (it.act1 && j >= it.lo1 && j <= it.hi1) {
            if (!(ok = mbar_wait_warp(b_pfull(1), pn1 & 1, abort_flag, lim))) break;
            ++pn1;
            tc_fence_after();
            issue_pv(tO1, tS1, nv & 1, j == it.lo1);
            if (j == it.hi1) {
              mma_commit_warp(b_ofull(1));
            } else {
              if (!wait_k(j + 1)) break;
              tc_fence_after();
              issue_qk(tS1, dQ1, knext);
              mma_commit_warp(b_sfull(1));
              if (j + 1 == it.hi1) mma_commit_warp(b_qempty(1));
            }
          }
          mma_commit_warp(b_vempty(nv & 1));
          if (ok && j == it.hi0 && it.hi1 > it.hi0) {
            // tile 0 is done with this item: start the next item's tile 0
            if (!(ok = next_item(idx_next))) break;
            have_next = true;
            if (idx_next < p.n_items) {
              const Item nx = decode_item(p, idx_next);
              const uint32_t nk0 = kbase + (uint32_t)(it.jhi - it.jlo + 1);  // its first K load
              if (!(ok = mbar_wait_warp(b_qfull(0), qn0 & 1, abort_flag, lim))) break;
              if (!(ok = mbar_wait_warp(b_kfull(nk0 % kKSlots), (nk0 / kKSlots) & 1, abort_flag,
                                        lim)))
                break;
              ++qn0;
              tc_fence_after();
              issue_qk(tS0, dQ0, nk0 % kKSlots);
              mma_commit_warp(b_sfull(0));
              if (nx.lo0 == nx.hi0) mma_commit_warp(b_qempty(0));
              early0 = true;
            }
          }
        }
        kc = kbase + (uint32_t)(it.jhi - it.jlo + 1);
        vc = vbase + (uint32_t)(it.jhi - it.jlo + 1);
      }
      if (!ok) raise_error(abort_flag);
      mma_drain_warp(b_drain);  // no MMA in flight when TMEM is released
    }
  } else {
    // ------------------------------------------------------------ softmax warps
    const int t = warp >> 2;                 // query tile of this warpgroup
    const int row = (warp & 3) * 32 + lane;  // TMEM lane
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + (uint32_t)(t * 128);
    const uint32_t tO = tmem + lane_base + (uint32_t)(256 + t * 128);
    const float sl2 = p.scale_log2;
    uint32_t sn = 0, on = 0;  // S tiles consumed, O tiles consumed
    bool ok = true;
    int idx = 0;
    while (ok && (ok = next_item(idx)) && idx < p.n_items) {
      const Item it = decode_item(p, idx);
      if (t == 1 && !it.act1) continue;
      const int qt = it.qt0 + t;
      const int lo_t = t ? it.lo1 : it.lo0, hi_t = t ? it.hi1 : it.hi0;
      const int i = qt * kBM + row;  // query index
      const int tq_lo = qt * kBM, tq_hi = min(tq_lo + kBM - 1, p.Nq - 1);
      // keys this row may see: [key_lo, key_hi]
      const int key_hi = p.mask == IHA_MASK_NONE ? p.Nk - 1 : min(i, p.Nk - 1);
      const int key_lo = p.mask == IHA_MASK_CAUSAL_WINDOW ? i - (p.window - 1) : 0;
      float m_used = -INFINITY;  // running row maximum, log2 units (scale included)
      float l = 0.f;             // running row sum relative to m_used
      for (int j = lo_t; j <= hi_t; ++j) {
        const int k0 = j * kBN;
        if (!(ok = mbar_wait(b_sfull(t), sn & 1, abort_flag, lim))) break;
        ++sn;
        tc_fence_after();
        const bool full_tile =
            (k0 + kBN <= p.Nk) &&
            (p.mask == IHA_MASK_NONE ||
             (k0 + kBN - 1 <= tq_lo && (p.mask == IHA_MASK_CAUSAL || tq_hi - k0 < p.window)));
        // visible columns of this tile for this row: [c_lo, c_hi]
        const int c_lo = max(key_lo - k0, 0), c_hi = min(key_hi - k0, kBN - 1);
        // pass 1: row maximum (the whole row, four independent max chains)
        float mt;
        {
          uint32_t s[128];
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld32(tS + 32u * c, s + 32 * c);
          tmem_wait_ld();
          if (!full_tile) mask_cols<4>(s, 0, c_lo, c_hi);
          // chain q takes columns q, q + 4, ...: 0-3 to start, two more
          // per step over 4-123, and 124-127 last
          float mx[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) mx[q] = __uint_as_float(s[q]);
#pragma unroll
          for (int e = 4; e < 124; e += 8)
#pragma unroll
            for (int q = 0; q < 4; ++q)
              mx[q] = fmax3f(mx[q], __uint_as_float(s[e + q]), __uint_as_float(s[e + 4 + q]));
#pragma unroll
          for (int q = 0; q < 4; ++q) mx[q] = fmaxf(mx[q], __uint_as_float(s[124 + q]));
          mt = fmaxf(fmax3f(mx[0], mx[1], mx[2]), mx[3]);
        }
        const float m_new = fmaxf(m_used, mt * sl2);
        bool rescale = false;
        float factor = 1.f;
        if (j == lo_t) {
          m_used = m_new;
        } else if (__any_sync(0xffffffffu, m_new > m_used + kRescaleLog2)) {
          factor = (m_new == -INFINITY) ? 1.f : fast_exp2(m_used - m_new);
          l *= factor;
          m_used = m_new;
          rescale = true;
        }
        const float base = (m_used == -INFINITY) ? 0.f : m_used;
        // pass 2, by halves of 64 columns: P = 2^(s * scale_log2 - base),
        // packed to bf16 pairs over the S columns (P half h lands in columns
        // 32h .. 32h+31, below every S column still to be read); pairs 3, 7,
        // 11, 15 of every 16 use the FMA-pipe polynomial.
        const float2 sc2 = make_float2(sl2, sl2), nb2 = make_float2(-base, -base);
        float2 sum2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t s[64];
          tmem_ld32(tS + 64u * h, s);
          tmem_ld32(tS + 64u * h + 32u, s + 32);
          tmem_wait_ld();
          if (!full_tile) mask_cols<2>(s, 64 * h, c_lo, c_hi);
          uint32_t pk[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const float2 xx = __ffma2_rn(
                make_float2(__uint_as_float(s[2 * e]), __uint_as_float(s[2 * e + 1])), sc2, nb2);
            float2 pp;
            if ((e & 3) == 3) {
              pp = exp2_poly3_x2(xx);
            } else {
              pp.x = fast_exp2(xx.x);
              pp.y = fast_exp2(xx.y);
            }
            sum2[e & 1] = __fadd2_rn(sum2[e & 1], pp);
            pk[e] = pack_bf16x2(pp.x, pp.y);
          }
          tmem_st32(tS + 32u * h, pk);
        }
        const float2 st = __fadd2_rn(sum2[0], sum2[1]);
        l += st.x + st.y;
        if (rescale) {
          // O <- O * factor before this tile's P.V is issued (P.V of the
          // previous tile is complete: the S commit waited on above tracks it)
#pragma unroll
          for (int c = 0; c < 2 * NCH; ++c) {
            uint32_t r[32];
            tmem_ld32(tO + 32u * c, r);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * factor);
            tmem_st32(tO + 32u * c, r);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(b_pfull(t));
      }
      if (!ok) break;
      // ---------------------------------------------------------- epilogue
      if (!(ok = mbar_wait(b_ofull(t), on & 1, abort_flag, lim))) break;
      ++on;
      tc_fence_after();
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
      // O rows of this warp (32 queries) go out by TMA: normalised, packed
      // to bf16 into the warp's 128-byte-swizzled staging, one store per 64
      // columns (rows past Nq and columns past d are clipped by the store)
      const int i0 = qt * kBM + (warp & 3) * 32;
      const uint32_t stg = sStg + (uint32_t)warp * kStgBytes;
      uint8_t* stg_p = smem + (stg - sQ);
#pragma unroll
      for (int c = 0; c < NCH; ++c) {  // 64 columns of O at a time
        uint32_t r[64];
        tmem_ld32(tO + 64u * c, r);
        tmem_ld32(tO + 64u * c + 32u, r + 32);
        tmem_wait_ld();
        if (lane == 0) bulk_wait_read<0>();  // the previous store has read the staging
        __syncwarp();
#pragma unroll
        for (int g8 = 0; g8 < 8; ++g8) {
          uint4 v;
          v.x = pack_bf16x2(__uint_as_float(r[8 * g8 + 0]) * inv_l, __uint_as_float(r[8 * g8 + 1]) * inv_l);
          v.y = pack_bf16x2(__uint_as_float(r[8 * g8 + 2]) * inv_l, __uint_as_float(r[8 * g8 + 3]) * inv_l);
          v.z = pack_bf16x2(__uint_as_float(r[8 * g8 + 4]) * inv_l, __uint_as_float(r[8 * g8 + 5]) * inv_l);
          v.w = pack_bf16x2(__uint_as_float(r[8 * g8 + 6]) * inv_l, __uint_as_float(r[8 * g8 + 7]) * inv_l);
          *reinterpret_cast<uint4*>(stg_p + lane * 128 + ((g8 ^ (lane & 7)) << 4)) = v;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && i0 < p.Nq) {
          tma_store_5d(&tmO, stg, c * kChunk, i0, it.h, it.bi, it.bo);
          bulk_commit();
        }
      }
      tc_fence_before();  // O may be overwritten once the next P of this tile is published
      if (i < p.Nq && p.lse) {
        const float base = (m_used == -INFINITY) ? 0.f : m_used;
        p.lse[((int64_t)it.bz * p.Hh + it.h) * p.Nq + i] =
            l > 0.f ? (base + log2f(l)) * 0.6931471805599453f : -INFINITY;
      }
    }
    if (lane == 0) bulk_wait<0>();  // O stores complete before the CTA exits
    if (!ok) raise_error(abort_flag);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0) work_leave(work);
}

// ---------------------------------------------------------------- fp32 path
// Thread quad per query row (each thread owns d/4 features), 32 rows per
// block, keys staged 32 at a time in shared memory; online softmax in fp32
// with expf.
struct AttnF32Params {
  int Bo, Bi, Hh, Nq, Nk, d;
  int mask, window;
  float scale;
  iha_strides sq, sk, sv, so;
  const float *q, *k, *v;
  float *o, *lse;
};

constexpr int kF32Rows = 32, kF32Keys = 32;

// DQ: a bound on the features per thread (d / 4), so that the per-thread
// query and accumulator arrays are indexed by unrolled loops and stay in
// registers (a runtime-bounded loop over them puts them in local memory).
template <int DQ>
__global__ void __launch_bounds__(128) attn_fwd_f32_kernel(const AttnF32Params p) {
  __shared__ float ks[kF32Keys][128 + 1];
  __shared__ float vs[kF32Keys][128 + 1];
  const int quad = threadIdx.x >> 2, qi = threadIdx.x & 3;
  const int dq = p.d >> 2;  // features per thread (<= DQ)
  const int h = blockIdx.y;
  const int bz = blockIdx.z, bo = bz / p.Bi, bi = bz - bo * p.Bi;
  const int i = blockIdx.x * kF32Rows + quad;
  const bool valid = i < p.Nq;
  float qv[DQ], acc[DQ];
  const float* qrow = p.q + bo * p.sq.b_outer + bi * p.sq.b_inner + (int64_t)min(i, p.Nq - 1) * p.sq.seq + h * p.sq.head;
#pragma unroll
  for (int e = 0; e < DQ; ++e) {
    qv[e] = (e < dq) ? qrow[qi * dq + e] : 0.f;
    acc[e] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  int k_hi = p.Nk - 1;
  if (p.mask != IHA_MASK_NONE) k_hi = min(k_hi, blockIdx.x * kF32Rows + kF32Rows - 1);
  int k_lo = 0;
  if (p.mask == IHA_MASK_CAUSAL_WINDOW) k_lo = max(0, (int)(blockIdx.x * kF32Rows) - (p.window - 1));
  for (int kb = k_lo; kb <= k_hi; kb += kF32Keys) {
    __syncthreads();
    for (int e = threadIdx.x; e < kF32Keys * p.d; e += blockDim.x) {
      const int kr = e / p.d, f = e - kr * p.d;
      const int kj = kb + kr;
      float kvv = 0.f, vvv = 0.f;
      if (kj < p.Nk) {
        kvv = p.k[bo * p.sk.b_outer + bi * p.sk.b_inner + (int64_t)kj * p.sk.seq + h * p.sk.head + f];
        vvv = p.v[bo * p.sv.b_outer + bi * p.sv.b_inner + (int64_t)kj * p.sv.seq + h * p.sv.head + f];
      }
      ks[kr][f] = kvv;
      vs[kr][f] = vvv;
    }
    __syncthreads();
    // the chunk's 32 scores first (independent, so their dot products and
    // shuffles overlap), then one rescale and the chunk's P.V
    float sc[kF32Keys];
#pragma unroll
    for (int kr = 0; kr < kF32Keys; ++kr) {
      const int kj = kb + kr;
      float dot = 0.f;
#pragma unroll
      for (int e = 0; e < DQ; ++e)
        if (e < dq) dot = fmaf(qv[e], ks[kr][qi * dq + e], dot);
      dot += __shfl_xor_sync(0xffffffffu, dot, 1);
      dot += __shfl_xor_sync(0xffffffffu, dot, 2);
      bool vis = kj < p.Nk;
      if (p.mask != IHA_MASK_NONE) {
        vis = vis && kj <= i;
        if (p.mask == IHA_MASK_CAUSAL_WINDOW) vis = vis && (i - kj < p.window);
      }
      sc[kr] = vis ? dot * p.scale : -INFINITY;
    }
    float mc = sc[0];
#pragma unroll
    for (int kr = 1; kr < kF32Keys; ++kr) mc = fmaxf(mc, sc[kr]);
    if (mc == -INFINITY) continue;  // no visible key in this chunk for this row
    const float m_new = fmaxf(m, mc);
    const float corr = expf(m - m_new);
    l *= corr;
#pragma unroll
    for (int e = 0; e < DQ; ++e) acc[e] *= corr;
#pragma unroll
    for (int kr = 0; kr < kF32Keys; ++kr) {
      const float pe = expf(sc[kr] - m_new);  // 0 for a hidden key
      l += pe;
#pragma unroll
      for (int e = 0; e < DQ; ++e)
        if (e < dq) acc[e] = fmaf(pe, vs[kr][qi * dq + e], acc[e]);
    }
    m = m_new;
  }
  if (valid) {
    float* orow = p.o + bo * p.so.b_outer + bi * p.so.b_inner + (int64_t)i * p.so.seq + h * p.so.head;
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
    for (int e = 0; e < DQ; ++e)
      if (e < dq) orow[qi * dq + e] = acc[e] * inv;
    if (p.lse && qi == 0) p.lse[((int64_t)bz * p.Hh + h) * p.Nq + i] = l > 0.f ? m + logf(l) : -INFINITY;
  }
}

// ---------------------------------------------------------------- host side
bool stride_ok(const iha_strides& s, int64_t elem) {
  return (s.b_outer * elem) % 16 == 0 && (s.b_inner * elem) % 16 == 0 && (s.seq * elem) % 16 == 0 &&
         (s.head * elem) % 16 == 0;
}

// 5-D tensor map over a [Bo, Bi, N, Hh, d] bf16 view, box 64 x 128 rows,
// 128-byte swizzle.  Strides of size-1 dimensions are replaced by a harmless
// aligned value.
CUresult make_map(CUtensorMap* m, const void* base, int Bo, int Bi, int N, int Hh, int d,
                  const iha_strides& s, int box_rows = kBM) {
  uint64_t dims[5] = {(uint64_t)d, (uint64_t)N, (uint64_t)Hh, (uint64_t)Bi, (uint64_t)Bo};
  uint64_t st[4] = {(uint64_t)s.seq * 2, (uint64_t)s.head * 2, (uint64_t)s.b_inner * 2,
                    (uint64_t)s.b_outer * 2};
  if (N == 1) st[0] = 16;
  if (Hh == 1) st[1] = 16;
  if (Bi == 1) st[2] = 16;
  if (Bo == 1) st[3] = 16;
  uint32_t box[5] = {(uint32_t)kChunk, (uint32_t)box_rows, 1, 1, 1};
  return encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, st, box,
                      CU_TENSOR_MAP_SWIZZLE_128B);
}

SmemLimit g_tc_limit[2];

// Dynamic shared memory limit of both instantiations on the current device
// (set on the device's first launch, thread-safe).
cudaError_t set_tc_attributes() {
  cudaError_t e = g_tc_limit[0].ensure(attn_fwd_tc_kernel<1>, kSmemBytes);
  if (e == cudaSuccess) e = g_tc_limit[1].ensure(attn_fwd_tc_kernel<2>, kSmemBytes);
  return e;
}

iha_status launch_tc(const void* q, const void* k, const void* v, void* o, float* lse, int Bo,
                     int Bi, int Hh, int Nq, int Nk, int d, const iha_strides& sq,
                     const iha_strides& sk, const iha_strides& sv, const iha_strides& so,
                     float scale, int mask, int window, cudaStream_t stream) {
  CUtensorMap mq, mk, mv;
  CUtensorMap mo;
  if (make_map(&mq, q, Bo, Bi, Nq, Hh, d, sq) != CUDA_SUCCESS ||
      make_map(&mk, k, Bo, Bi, Nk, Hh, d, sk) != CUDA_SUCCESS ||
      make_map(&mv, v, Bo, Bi, Nk, Hh, d, sv) != CUDA_SUCCESS ||
      make_map(&mo, o, Bo, Bi, Nq, Hh, d, so, 32) != CUDA_SUCCESS)
    return fail(IHA_ERR_CUDA, "mha_fwd: tensor map encoding failed");
  AttnParams p;
  p.Bo = Bo;
  p.Bi = Bi;
  p.Hh = Hh;
  p.Nq = Nq;
  p.Nk = Nk;
  p.d = d;
  p.nD = (d + kChunk - 1) / kChunk;
  p.mask = mask;
  p.window = window;
  p.n_qt = (Nq + kBM - 1) / kBM;
  p.n_qpairs = (p.n_qt + 1) / 2;
  p.n_hb = Bo * Bi * Hh;
  const int64_t kv_bytes = 2ll * Nk * d * 2;  // K and V of one head
  int64_t g = kGroupKVBytes / (kv_bytes > 0 ? kv_bytes : 1);
  if (g < 1) g = 1;
  if (g > p.n_hb) g = p.n_hb;
  p.group = (int)g;
  p.n_items = p.n_hb * p.n_qpairs;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.so_bo = so.b_outer;
  p.so_bi = so.b_inner;
  p.so_seq = so.seq;
  p.so_h = so.head;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.wait_limit_ns = wait_limit_for_next_launch();
  p.withhold = withhold_for_this_launch() ? 1 : 0;
  p.work_slot = (int)attention_work_slot();
  const cudaError_t ae = set_tc_attributes();
  if (ae != cudaSuccess)
    return fail(IHA_ERR_CUDA, "mha_fwd (smem attribute): %s", cudaGetErrorString(ae));
  int grid = sm_count();
  if (grid > p.n_items) grid = p.n_items;
  if (p.nD == 1)
    attn_fwd_tc_kernel<1><<<grid, kThreads, kSmemBytes, stream>>>(mq, mk, mv, mo, p);
  else
    attn_fwd_tc_kernel<2><<<grid, kThreads, kSmemBytes, stream>>>(mq, mk, mv, mo, p);
  return check_launch("mha_fwd");
}

}  // namespace
}  // namespace iha

extern "C" iha_status mha_fwd(const void* q, const void* k, const void* v, void* o,
                              float* lse_out, int B_outer, int B_inner, int Hh, int Nq, int Nk,
                              int d, iha_strides sq, iha_strides sk, iha_strides sv,
                              iha_strides so, float scale, iha_mask mask_mode, int window,
                              iha_dtype dt, void* stream) {
  using namespace iha;
  if (!q || !k || !v || !o) return fail(IHA_ERR_INVALID_ARG, "mha_fwd: null pointer");
  if (B_outer <= 0 || B_inner <= 0 || Hh <= 0 || Nq <= 0 || Nk <= 0 || d <= 0)
    return fail(IHA_ERR_INVALID_ARG, "mha_fwd: sizes must be positive");
  if (dt != IHA_BF16 && dt != IHA_F32) return fail(IHA_ERR_INVALID_ARG, "mha_fwd: bad dtype");
  if (mask_mode != IHA_MASK_NONE && mask_mode != IHA_MASK_CAUSAL &&
      mask_mode != IHA_MASK_CAUSAL_WINDOW)
    return fail(IHA_ERR_INVALID_ARG, "mha_fwd: bad mask_mode %d", (int)mask_mode);
  if (mask_mode == IHA_MASK_CAUSAL_WINDOW && window < 1)
    return fail(IHA_ERR_INVALID_ARG, "mha_fwd: window must be >= 1");
  if (mask_mode != IHA_MASK_NONE && Nq != Nk)
    return fail(IHA_ERR_UNSUPPORTED, "mha_fwd: causal masks need Nq == Nk");
  if (d > 128) return fail(IHA_ERR_UNSUPPORTED, "mha_fwd: d = %d > 128", d);
  if ((int64_t)B_outer * B_inner * Hh * (((int64_t)Nq + 255) / 256) > INT32_MAX ||
      (int64_t)B_outer * B_inner > 65535 || Hh > 65535)
    return fail(IHA_ERR_UNSUPPORTED, "mha_fwd: too many heads, batches or rows for one launch");
  if (mask_mode != IHA_MASK_CAUSAL_WINDOW) window = 0;
  if (!(scale > 0.f)) scale = 1.f / sqrtf((float)d);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (dt == IHA_BF16) {
    if (d % 8) return fail(IHA_ERR_UNSUPPORTED, "mha_fwd: bf16 needs d %% 8 == 0");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o))
      return fail(IHA_ERR_ALIGNMENT, "mha_fwd: base pointers must be 16-byte aligned");
    if (!stride_ok(sq, 2) || !stride_ok(sk, 2) || !stride_ok(sv, 2) || !stride_ok(so, 2))
      return fail(IHA_ERR_ALIGNMENT, "mha_fwd: strides must be multiples of 8 elements");
    if (lse_out && (reinterpret_cast<uintptr_t>(lse_out) & 3))
      return fail(IHA_ERR_ALIGNMENT, "mha_fwd: lse_out must be 4-byte aligned");
    if (mu_attention_supported(Nq, Nk, d, mask_mode))
      return mu_attention_fwd(q, k, v, o, lse_out, B_outer, B_inner, Hh, Nq, d, sq, sk, sv, so,
                              scale, s);
    return launch_tc(q, k, v, o, lse_out, B_outer, B_inner, Hh, Nq, Nk, d, sq, sk, sv, so, scale,
                     mask_mode, window, s);
  }
  if (d % 4) return fail(IHA_ERR_UNSUPPORTED, "mha_fwd: f32 needs d %% 4 == 0");
  AttnF32Params p;
  p.Bo = B_outer;
  p.Bi = B_inner;
  p.Hh = Hh;
  p.Nq = Nq;
  p.Nk = Nk;
  p.d = d;
  p.mask = mask_mode;
  p.window = window;
  p.scale = scale;
  p.sq = sq;
  p.sk = sk;
  p.sv = sv;
  p.so = so;
  p.q = static_cast<const float*>(q);
  p.k = static_cast<const float*>(k);
  p.v = static_cast<const float*>(v);
  p.o = static_cast<float*>(o);
  p.lse = lse_out;
  dim3 grid((Nq + kF32Rows - 1) / kF32Rows, Hh, B_outer * B_inner);
  const int dq = d / 4;
  if (dq <= 2)
    attn_fwd_f32_kernel<2><<<grid, 128, 0, s>>>(p);
  else if (dq <= 4)
    attn_fwd_f32_kernel<4><<<grid, 128, 0, s>>>(p);
  else if (dq <= 8)
    attn_fwd_f32_kernel<8><<<grid, 128, 0, s>>>(p);
  else if (dq <= 16)
    attn_fwd_f32_kernel<16><<<grid, 128, 0, s>>>(p);
  else
    attn_fwd_f32_kernel<32><<<grid, 128, 0, s>>>(p);
  return check_launch("mha_fwd");
}

extern "C" iha_status mha_fwd_qpool(const void* q, const void* k, const void* v, void* o,
                                    float* lse_out, int B_outer, int B_inner, int Hh, int T,
                                    int d, int q_stride, iha_strides sq, iha_strides sk,
                                    iha_strides sv, iha_strides so, float scale, iha_dtype dt,
                                    void* stream) {
  using namespace iha;
  if (!q || !k || !v || !o) return fail(IHA_ERR_INVALID_ARG, "mha_fwd_qpool: null pointer");
  if (B_outer <= 0 || B_inner <= 0 || Hh <= 0 || T <= 0 || d <= 0 || q_stride <= 0)
    return fail(IHA_ERR_INVALID_ARG, "mha_fwd_qpool: sizes must be positive");
  if (T % q_stride)
    return fail(IHA_ERR_INVALID_ARG, "mha_fwd_qpool: q_stride %d does not divide T %d", q_stride,
                T);
  if (dt != IHA_BF16) return fail(IHA_ERR_UNSUPPORTED, "mha_fwd_qpool: bf16 only");
  if (!mu_attention_supported(T, T, d, IHA_MASK_NONE) || d % 8)
    return fail(IHA_ERR_UNSUPPORTED, "mha_fwd_qpool: needs T <= 64, d <= 128, d %% 8 == 0");
  if ((int64_t)B_outer * B_inner * Hh > INT32_MAX / 2)
    return fail(IHA_ERR_UNSUPPORTED, "mha_fwd_qpool: too many units for one launch");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o))
    return fail(IHA_ERR_ALIGNMENT, "mha_fwd_qpool: base pointers must be 16-byte aligned");
  if (!stride_ok(sq, 2) || !stride_ok(sk, 2) || !stride_ok(sv, 2) || !stride_ok(so, 2))
    return fail(IHA_ERR_ALIGNMENT, "mha_fwd_qpool: strides must be multiples of 8 elements");
  if (lse_out && (reinterpret_cast<uintptr_t>(lse_out) & 3))
    return fail(IHA_ERR_ALIGNMENT, "mha_fwd_qpool: lse_out must be 4-byte aligned");
  if (!(scale > 0.f)) scale = 1.f / sqrtf((float)d);
  return mu_attention_fwd(q, k, v, o, lse_out, B_outer, B_inner, Hh, T, d, sq, sk, sv, so, scale,
                          reinterpret_cast<cudaStream_t>(stream), q_stride);
}
