// Mask-unit gather / scatter ("hiera-optim 0.1.0", README, item 2 of what
// optimize(model) does: boolean indexing of kept mask units replaced by an
// explicit gather and scatter).
//
// HBM-bound byte copies.  A kept unit is mu_h row segments of mu_w tokens of
// the grid (each segment contiguous: 1536 bytes for 8 tokens x 96 bf16), and
// a contiguous block of mu_h * mu_w tokens in the unit layout.  When rows and
// pointers are 16-byte aligned and a unit fits a stage, the copy runs on the
// bulk-copy engine: one thread per CTA loads units into a ring of shared-
// memory stages (segments for gather, one block for scatter) and writes
// each stage back out (one block, or segments), several units in flight.
// Otherwise threads move 16-, 4- or 1-byte chunks.  The kept-unit id is
// checked on the GPU; an out-of-range id skips the unit and raises the
// device error word.
#include <mutex>

#include "common.cuh"
#include "mu_attention.h"

namespace iha {
namespace {

IHA_DEVICE_ERROR_WORD(mask_unit)

struct MuGeom {
  int64_t total;        // B * n_keep * T * chunks
  int32_t chunks;       // chunks per token row
  int32_t T;            // tokens per unit (mu_h * mu_w)
  int32_t n_keep;
  int32_t n_units;
  int32_t units_per_row;
  int32_t mu_h, mu_w, grid_w;
  int64_t G;            // tokens per sample (grid_h * grid_w)
};

// Token index of unit u, in-unit token t, on the row-major grid.
__device__ __forceinline__ int64_t unit_token(const MuGeom& g, int u, int t) {
  const int uy = u / g.units_per_row, ux = u - uy * g.units_per_row;
  const int ty = t / g.mu_w, tx = t - ty * g.mu_w;
  return (int64_t)(uy * g.mu_h + ty) * g.grid_w + ux * g.mu_w + tx;
}

// One block per kept unit (grid-stride over units); its threads walk the
// unit's T * chunks chunks, so the kept-unit id is read once per block and
// the per-chunk index math stays 32-bit.
// GATHER = true : out[b,k,t,:] = x[b, tok, :]
// GATHER = false: x[b, tok, :] = src[b,k,t,:]
template <typename V, bool GATHER>
__global__ void __launch_bounds__(256) mu_copy_kernel(const V* __restrict__ from,
                                                      const int32_t* __restrict__ keep,
                                                      V* __restrict__ to, MuGeom g) {
  const int per_unit = g.T * g.chunks;
  const int64_t n_bk = g.total / per_unit;
  for (int64_t bk = blockIdx.x; bk < n_bk; bk += gridDim.x) {
    const int u = __ldg(keep + bk);
    if (u < 0 || u >= g.n_units) {
      if (threadIdx.x == 0) atomicOr(&g_dev_error, DEV_ERR_KEEP_INDEX);
      continue;
    }
    const int64_t b = bk / g.n_keep;
    const int64_t unit_base = bk * per_unit;
    const int64_t grid_base = b * g.G;
    for (int e = threadIdx.x; e < per_unit; e += blockDim.x) {
      const int t = e / g.chunks, c = e - t * g.chunks;
      const int64_t grid_row = (grid_base + unit_token(g, u, t)) * g.chunks + c;
      const int64_t unit_row = unit_base + e;
      if (GATHER)
        to[unit_row] = __ldg(from + grid_row);
      else
        to[grid_row] = __ldg(from + unit_row);
    }
  }
}

// Bulk-copy path.  One thread per CTA drives a ring of kStages stages; unit
// i is loaded into stage i % kStages (its mbarrier counts the bytes), stored
// when it has landed, and the stage is reloaded only after the store that
// read it has finished reading.  Loads run kStages - 1 units ahead.
constexpr int kStages = 8;
constexpr int kStageMax = 12288;  // bytes per stage (one 8x8 unit of 96 bf16 channels)

struct MuBulkGeom {
  int n_bk;           // B * n_keep units
  int n_keep, n_units, units_per_row, mu_h, mu_w, grid_w;
  int64_t G;          // tokens per sample
  uint32_t row_bytes, seg_bytes, unit_bytes;
};

template <bool GATHER>
__global__ void __launch_bounds__(32) mu_bulk_kernel(const uint8_t* __restrict__ from,
                                                     const int32_t* __restrict__ keep,
                                                     uint8_t* __restrict__ to, MuBulkGeom g) {
  extern __shared__ __align__(128) uint8_t stage_mem[];
  __shared__ __align__(8) uint64_t full[kStages];
  __shared__ int skip[kStages];
  if (threadIdx.x != 0) return;
  const uint32_t s0 = smem_u32(stage_mem);
  for (int s = 0; s < kStages; ++s) mbar_init(smem_u32(&full[s]), 1);
  mbar_init_fence();
  const int n_my = (g.n_bk - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
  auto seg_ptr = [&](int bk, int u, int ty) {  // grid row segment ty of unit u of sample bk / n_keep
    const int64_t b = bk / g.n_keep;
    const int uy = u / g.units_per_row, ux = u - uy * g.units_per_row;
    const int64_t tok = b * g.G + (int64_t)(uy * g.mu_h + ty) * g.grid_w + ux * g.mu_w;
    return tok * g.row_bytes;
  };
  auto issue_load = [&](int i) {
    const int s = i % kStages, bk = blockIdx.x + i * gridDim.x;
    const uint32_t st = s0 + (uint32_t)s * g.unit_bytes, bar = smem_u32(&full[s]);
    const int u = __ldg(keep + bk);
    if (u < 0 || u >= g.n_units) {
      atomicOr(&g_dev_error, DEV_ERR_KEEP_INDEX);
      skip[s] = 1;
      mbar_arrive(bar);  // completes the phase without bytes
      return;
    }
    skip[s] = 0;
    mbar_arrive_expect_tx(bar, g.unit_bytes);
    if (GATHER) {
      for (int ty = 0; ty < g.mu_h; ++ty)
        bulk_load(st + (uint32_t)ty * g.seg_bytes, from + seg_ptr(bk, u, ty), g.seg_bytes, bar);
    } else {
      bulk_load(st, from + (int64_t)bk * g.unit_bytes, g.unit_bytes, bar);
    }
  };
  int issued = 0;
  for (; issued < kStages - 1 && issued < n_my; ++issued) issue_load(issued);
  volatile int no_abort = 0;
  bool ok = true;
  for (int i = 0; i < n_my; ++i) {
    const int s = i % kStages, bk = blockIdx.x + i * gridDim.x;
    if (!mbar_wait(smem_u32(&full[s]), (i / kStages) & 1, &no_abort)) {
      atomicOr(&g_dev_error, DEV_ERR_WAIT_TIMEOUT);
      ok = false;
      break;
    }
    if (!skip[s]) {
      const uint32_t st = s0 + (uint32_t)s * g.unit_bytes;
      if (GATHER) {
        bulk_store(to + (int64_t)bk * g.unit_bytes, st, g.unit_bytes);
      } else {
        const int u = __ldg(keep + bk);
        for (int ty = 0; ty < g.mu_h; ++ty)
          bulk_store(to + seg_ptr(bk, u, ty), st + (uint32_t)ty * g.seg_bytes, g.seg_bytes);
      }
    }
    bulk_commit();
    // the stage of unit i - 1 is free once its store has read it
    bulk_wait_read<1>();
    if (issued < n_my) issue_load(issued++);
  }
  if (!ok) {
    // let every load issued land before the CTA exits (the newest one of each stage)
    for (int i = issued - kStages > 0 ? issued - kStages : 0; i < issued; ++i)
      mbar_wait(smem_u32(&full[i % kStages]), (i / kStages) & 1, &no_abort);
  }
  bulk_wait<0>();  // stores complete before exit
}

template <bool GATHER>
iha_status mu_launch(const void* from, const int32_t* keep, void* to, int B, int grid_h,
                     int grid_w, int mu_h, int mu_w, int n_keep, int C, int elem_bytes,
                     void* stream, const char* name) {
  if (!from || !keep || !to) return fail(IHA_ERR_INVALID_ARG, "%s: null pointer", name);
  if (B <= 0 || grid_h <= 0 || grid_w <= 0 || mu_h <= 0 || mu_w <= 0 || n_keep <= 0 || C <= 0 ||
      elem_bytes <= 0)
    return fail(IHA_ERR_INVALID_ARG, "%s: sizes must be positive", name);
  if (grid_h % mu_h || grid_w % mu_w)
    return fail(IHA_ERR_INVALID_ARG, "%s: grid %dx%d not divisible by unit %dx%d", name, grid_h,
                grid_w, mu_h, mu_w);
  const int n_units = (grid_h / mu_h) * (grid_w / mu_w);
  if (n_keep > n_units)
    return fail(IHA_ERR_INVALID_ARG, "%s: n_keep %d > units %d", name, n_keep, n_units);
  if (from == to) return fail(IHA_ERR_INVALID_ARG, "%s: source and destination alias", name);

  const int64_t row = (int64_t)C * elem_bytes;
  MuGeom g;
  g.T = mu_h * mu_w;
  g.n_keep = n_keep;
  g.n_units = n_units;
  g.units_per_row = grid_w / mu_w;
  g.mu_h = mu_h;
  g.mu_w = mu_w;
  g.grid_w = grid_w;
  g.G = (int64_t)grid_h * grid_w;
  const uintptr_t align = reinterpret_cast<uintptr_t>(from) | reinterpret_cast<uintptr_t>(to);
  int vec;
  if (row % 16 == 0 && (align & 15) == 0) vec = 16;
  else if (row % 4 == 0 && (align & 3) == 0) vec = 4;
  else vec = 1;
  g.chunks = (int32_t)(row / vec);
  g.total = (int64_t)B * n_keep * g.T * g.chunks;

  if ((int64_t)g.T * g.chunks > (int64_t)INT32_MAX)
    return fail(IHA_ERR_UNSUPPORTED, "%s: mask unit of %lld bytes too large", name,
                (long long)(g.T * row));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int64_t unit_bytes = (int64_t)g.T * row;
  if (vec == 16 && unit_bytes <= kStageMax && (int64_t)B * n_keep <= INT32_MAX) {
    MuBulkGeom bg;
    bg.n_bk = B * n_keep;
    bg.n_keep = n_keep;
    bg.n_units = n_units;
    bg.units_per_row = grid_w / mu_w;
    bg.mu_h = mu_h;
    bg.mu_w = mu_w;
    bg.grid_w = grid_w;
    bg.G = g.G;
    bg.row_bytes = (uint32_t)row;
    bg.seg_bytes = (uint32_t)(mu_w * row);
    bg.unit_bytes = (uint32_t)unit_bytes;
    int blocks = sm_count() * 2;
    if (blocks > bg.n_bk) blocks = bg.n_bk;
    const size_t smem = (size_t)kStages * unit_bytes;
    auto kern = mu_bulk_kernel<GATHER>;
    // the ring's largest size, set on each device's first launch (thread-safe)
    static SmemLimit limit;
    const cudaError_t attr_err = limit.ensure(kern, kStages * kStageMax);
    if (attr_err != cudaSuccess)
      return fail(IHA_ERR_CUDA, "%s (smem attribute): %s", name, cudaGetErrorString(attr_err));
    kern<<<blocks, 32, smem, s>>>(static_cast<const uint8_t*>(from), keep,
                                  static_cast<uint8_t*>(to), bg);
    return check_launch(name);
  }
  const int threads = 256;
  int64_t blocks = (int64_t)B * n_keep;
  const int64_t cap = (int64_t)sm_count() * 64;
  if (blocks > cap) blocks = cap;
  if (vec == 16)
    mu_copy_kernel<uint4, GATHER><<<(unsigned)blocks, threads, 0, s>>>(
        static_cast<const uint4*>(from), keep, static_cast<uint4*>(to), g);
  else if (vec == 4)
    mu_copy_kernel<uint32_t, GATHER><<<(unsigned)blocks, threads, 0, s>>>(
        static_cast<const uint32_t*>(from), keep, static_cast<uint32_t*>(to), g);
  else
    mu_copy_kernel<uint8_t, GATHER><<<(unsigned)blocks, threads, 0, s>>>(
        static_cast<const uint8_t*>(from), keep, static_cast<uint8_t*>(to), g);
  return check_launch(name);
}

}  // namespace
}  // namespace iha

extern "C" {

iha_status mu_gather(const void* x, const int32_t* keep, void* out, int B, int grid_h,
                     int grid_w, int mu_h, int mu_w, int n_keep, int C, int elem_bytes,
                     void* stream) {
  return iha::mu_launch<true>(x, keep, out, B, grid_h, grid_w, mu_h, mu_w, n_keep, C,
                              elem_bytes, stream, "mu_gather");
}

iha_status mu_scatter(const void* src, const int32_t* keep, void* x, int B, int grid_h,
                      int grid_w, int mu_h, int mu_w, int n_keep, int C, int elem_bytes,
                      void* stream) {
  return iha::mu_launch<false>(src, keep, x, B, grid_h, grid_w, mu_h, mu_w, n_keep, C,
                               elem_bytes, stream, "mu_scatter");
}

iha_status mu_attention_fused(const void* x, const int32_t* keep, void* canvas, int B, int grid_h,
                              int grid_w, int mu_h, int mu_w, int n_keep, int C, float scale,
                              iha_dtype dt, void* stream) {
  using namespace iha;
  const char* name = "mu_attention_fused";
  if (!x || !keep || !canvas) return fail(IHA_ERR_INVALID_ARG, "%s: null pointer", name);
  if (B <= 0 || grid_h <= 0 || grid_w <= 0 || mu_h <= 0 || mu_w <= 0 || n_keep <= 0 || C <= 0)
    return fail(IHA_ERR_INVALID_ARG, "%s: sizes must be positive", name);
  if (grid_h % mu_h || grid_w % mu_w)
    return fail(IHA_ERR_INVALID_ARG, "%s: grid not divisible by the mask unit", name);
  const int64_t units = (int64_t)(grid_h / mu_h) * (grid_w / mu_w);
  if (n_keep > units) return fail(IHA_ERR_INVALID_ARG, "%s: n_keep > units", name);
  if (dt != IHA_BF16) return fail(IHA_ERR_UNSUPPORTED, "%s: bf16 only", name);
  if (mu_h * mu_w > 64 || C % 8 || C > 128 || mu_w > 256 || mu_h > 256)
    return fail(IHA_ERR_UNSUPPORTED, "%s: needs mu_h*mu_w <= 64, C %% 8 == 0, C <= 128", name);
  if ((int64_t)B * n_keep > INT32_MAX || (int64_t)B * grid_h * grid_w * C > (1ll << 40))
    return fail(IHA_ERR_UNSUPPORTED, "%s: problem too large", name);
  if (!aligned16(x) || !aligned16(canvas) || (reinterpret_cast<uintptr_t>(keep) & 3))
    return fail(IHA_ERR_ALIGNMENT, "%s: x and canvas must be 16-byte aligned, keep 4", name);
  const size_t nb = (size_t)B * grid_h * grid_w * C * 2, nk = (size_t)B * n_keep * 4;
  auto overlaps = [](const void* a, size_t na, const void* b, size_t nbb) {
    const uintptr_t p0 = reinterpret_cast<uintptr_t>(a), p1 = reinterpret_cast<uintptr_t>(b);
    return p0 < p1 + nbb && p1 < p0 + na;
  };
  if (overlaps(canvas, nb, x, nb) || overlaps(canvas, nb, keep, nk))
    return fail(IHA_ERR_INVALID_ARG, "%s: canvas overlaps an input", name);
  if (!(scale > 0.f)) scale = 1.f / sqrtf((float)C);
  return iha::mu_attention_fused(x, keep, canvas, B, grid_h, grid_w, mu_h, mu_w, n_keep, C, scale,
                                 reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
