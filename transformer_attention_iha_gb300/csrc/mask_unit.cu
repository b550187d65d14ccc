// Mask-unit gather / scatter ("hiera-optim 0.1.0", README, item 2 of what
// optimize(model) does: boolean indexing of kept mask units replaced by an
// explicit gather and scatter).
//
// HBM-bound byte copies.  A thread moves 16-byte chunks (4-byte / 1-byte
// when rows or pointers are not 16-byte aligned); consecutive threads move
// consecutive chunks of a token row, so a warp reads and writes whole
// 128-byte lines of each row.  The kept-unit id is checked on the GPU; an
// out-of-range id skips the copy and raises the device error word.
#include "common.cuh"

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
  const int threads = 256;
  int64_t blocks = (int64_t)B * n_keep;
  const int64_t cap = (int64_t)sm_count() * 64;
  if (blocks > cap) blocks = cap;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
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

}  // extern "C"
