// IHA premix: forward mix, input gradient and weight gradient.
//
// "IHA-CUDA: Interleaved Head Attention Kernels for Hopper GPUs", section
// "Pseudo-Token Mixing (Triton Premix Kernels)":
//   forward   Y[b,n,h*P+p,f] = sum_s W[h,p,s] X[b,n,s,f]  (+ optional RoPE)
//   backward  dX = W^T dY,  dW = sum over (b, n, f) of dY X^T.
// The page describes the op as memory-bound with a tiny weight tensor; the
// kernels here stream X / dY once with 8- or 16-byte vector accesses, keep W
// in shared memory (read as float4 broadcasts), unroll the source-head loop
// at compile time and keep one token's H x 4 input features in registers.
//
// RoPE reading (the page names "optional fused RoPE rotation" only):
// HF-LLaMA rotate-half at position n, inv_freq_i = base^(-2i/d); it is
// applied to each pseudo-head vector after the mix.  The mix acts on heads
// and the rotation on features, so they commute: the input gradient applies
// the inverse rotation after the transposed mix and the weight gradient
// rotates X instead of dY (<R^T a, b> = <a, R b>).
#include "common.cuh"
#include "premix_tc.h"

namespace iha {
namespace {

IHA_DEVICE_ERROR_WORD(premix)

struct PremixGeom {
  int64_t ntok;  // B * N
  int N, H, P, HP, d;
  float rope_base;
};

// ---------------------------------------------------------------- vector I/O
template <typename T>
struct Vec4;
template <>
struct Vec4<__nv_bfloat16> {
  static __device__ __forceinline__ void load(const __nv_bfloat16* p, float (&v)[4]) {
    const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
    v[0] = bf16lo_to_f32(u.x);
    v[1] = bf16hi_to_f32(u.x);
    v[2] = bf16lo_to_f32(u.y);
    v[3] = bf16hi_to_f32(u.y);
  }
  static __device__ __forceinline__ void store(__nv_bfloat16* p, const float (&v)[4]) {
    uint2 u;
    u.x = pack_bf16x2(v[0], v[1]);
    u.y = pack_bf16x2(v[2], v[3]);
    *reinterpret_cast<uint2*>(p) = u;
  }
};
template <>
struct Vec4<float> {
  static __device__ __forceinline__ void load(const float* p, float (&v)[4]) {
    const float4 u = __ldg(reinterpret_cast<const float4*>(p));
    v[0] = u.x;
    v[1] = u.y;
    v[2] = u.z;
    v[3] = u.w;
  }
  static __device__ __forceinline__ void store(float* p, const float (&v)[4]) {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  }
};

// ---------------------------------------------------------------- RoPE helpers
// inv_freq of rotation pair i (i < d/2), in double.
__device__ __forceinline__ double rope_inv_freq(int i, int d, float base) {
  return pow((double)base, -2.0 * (double)i / (double)d);
}
// cos / sin of n * inv_freq, reduced modulo 2*pi in double first so that
// large positions keep full fp32 accuracy.
__device__ __forceinline__ void rope_cs(int n, double inv_freq, float& c, float& s) {
  const double a = (double)n * inv_freq;
  const double k = rint(a * 0.15915494309189535);  // 1 / (2 pi)
  const float r = (float)fma(-k, 6.283185307179586, a);
  sincosf(r, &s, &c);
}

// Stage W[HP][H] fp32 into shared memory as [HP][HC], zero for s >= H.
template <int HC>
__device__ __forceinline__ void stage_w(float* wsm, const float* __restrict__ w,
                                        const PremixGeom& g) {
  for (int i = threadIdx.x; i < g.HP * HC; i += blockDim.x) {
    const int hp = i / HC, s = i - hp * HC;
    wsm[i] = s < g.H ? __ldg(w + hp * g.H + s) : 0.f;
  }
  __syncthreads();
}

// ---------------------------------------------------------------- forward
// Thread = (token, 4 consecutive features).  Threads of one token are
// consecutive lanes of one warp when d/4 divides 32 (always for RoPE), so
// the RoPE partner (feature f +- d/2) is lane ^ (d/8).  blockIdx.y picks one
// of up to three tensors (Q, K, V) of the launch, each with its own X, W, Y.
template <typename T>
struct FwdTensors {
  const T* x[3];
  const float* w[3];
  T* y[3];
};

template <typename T, int HC, bool ROPE>
__global__ void __launch_bounds__(256) premix_fwd_kernel(const FwdTensors<T> ts, PremixGeom g) {
  extern __shared__ float4 smem_f4[];
  float* wsm = reinterpret_cast<float*>(smem_f4);
  const T* __restrict__ x = ts.x[blockIdx.y];
  T* __restrict__ y = ts.y[blockIdx.y];
  stage_w<HC>(wsm, ts.w[blockIdx.y], g);

  const int tpt = g.d >> 2;
  const int64_t total = g.ntok * tpt;
  const int64_t total_r = (total + 31) & ~(int64_t)31;  // warp-uniform trip count
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t g0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int slot = (int)(g0 % tpt);  // fixed: stride % tpt == 0 is ensured by the launcher
  const int f0 = slot * 4;
  const int half = g.d >> 1;
  double inv_freq[4];
  float sign = 1.f;
  if (ROPE) {
    const int i0 = f0 % half;
#pragma unroll
    for (int j = 0; j < 4; ++j) inv_freq[j] = rope_inv_freq(i0 + j, g.d, g.rope_base);
    sign = f0 < half ? -1.f : 1.f;  // first half: x c - x' s ; second half: x c + x' s
  }

  for (int64_t gi = g0; gi < total_r; gi += stride) {
    const bool valid = gi < total;
    const int64_t tok = valid ? gi / tpt : 0;
    float xv[HC][4];
    const T* xrow = x + tok * (int64_t)g.H * g.d + f0;
#pragma unroll
    for (int s = 0; s < HC; ++s) {
      if (valid && s < g.H) {
        Vec4<T>::load(xrow + (int64_t)s * g.d, xv[s]);
      } else {
        xv[s][0] = xv[s][1] = xv[s][2] = xv[s][3] = 0.f;
      }
    }
    float cs[4], sn[4];
    if (ROPE) {
      const int n = (int)(tok % g.N);
#pragma unroll
      for (int j = 0; j < 4; ++j) rope_cs(n, inv_freq[j], cs[j], sn[j]);
    }
    T* yrow = y + tok * (int64_t)g.HP * g.d + f0;
#pragma unroll 2
    for (int hp = 0; hp < g.HP; ++hp) {
      const float* wr = wsm + hp * HC;
      float2 a01 = make_float2(0.f, 0.f), a23 = make_float2(0.f, 0.f);
#pragma unroll
      for (int s = 0; s < HC; s += 4) {
        const float4 w4 = *reinterpret_cast<const float4*>(wr + s);
        const float wv[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 ww = make_float2(wv[j], wv[j]);
          a01 = __ffma2_rn(ww, make_float2(xv[s + j][0], xv[s + j][1]), a01);
          a23 = __ffma2_rn(ww, make_float2(xv[s + j][2], xv[s + j][3]), a23);
        }
      }
      float o[4] = {a01.x, a01.y, a23.x, a23.y};
      if (ROPE) {
        const int lane_mask = tpt >> 1;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float other = __shfl_xor_sync(0xffffffffu, o[j], lane_mask);
          o[j] = fmaf(o[j], cs[j], sign * other * sn[j]);
        }
      }
      if (valid) Vec4<T>::store(yrow + (int64_t)hp * g.d, o);
    }
  }
}

// ---------------------------------------------------------------- input gradient
// dX[s, f] = sum_hp W[hp, s] dY[hp, f]; thread = (token, 4 features) with an
// H x 4 accumulator block; dY rows are streamed once.
template <typename T, int HC, bool ROPE>
__global__ void __launch_bounds__(256) premix_dx_kernel(const T* __restrict__ dy,
                                                        const float* __restrict__ w,
                                                        T* __restrict__ dx, PremixGeom g) {
  extern __shared__ float4 smem_f4[];
  float* wsm = reinterpret_cast<float*>(smem_f4);
  stage_w<HC>(wsm, w, g);

  const int tpt = g.d >> 2;
  const int64_t total = g.ntok * tpt;
  const int64_t total_r = (total + 31) & ~(int64_t)31;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t g0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int slot = (int)(g0 % tpt);
  const int f0 = slot * 4;
  const int half = g.d >> 1;
  double inv_freq[4];
  float sign = 1.f;
  if (ROPE) {
    const int i0 = f0 % half;
#pragma unroll
    for (int j = 0; j < 4; ++j) inv_freq[j] = rope_inv_freq(i0 + j, g.d, g.rope_base);
    sign = f0 < half ? 1.f : -1.f;  // inverse rotation: first half x c + x' s
  }

  for (int64_t gi = g0; gi < total_r; gi += stride) {
    const bool valid = gi < total;
    const int64_t tok = valid ? gi / tpt : 0;
    float2 acc[HC][2];
#pragma unroll
    for (int s = 0; s < HC; ++s) acc[s][0] = acc[s][1] = make_float2(0.f, 0.f);
    const T* grow = dy + tok * (int64_t)g.HP * g.d + f0;
#pragma unroll 4
    for (int hp = 0; hp < g.HP; ++hp) {
      float gv[4] = {0.f, 0.f, 0.f, 0.f};
      if (valid) Vec4<T>::load(grow + (int64_t)hp * g.d, gv);
      const float2 g01 = make_float2(gv[0], gv[1]), g23 = make_float2(gv[2], gv[3]);
      const float* wr = wsm + hp * HC;
#pragma unroll
      for (int s = 0; s < HC; s += 4) {
        const float4 w4 = *reinterpret_cast<const float4*>(wr + s);
        const float wv[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 ww = make_float2(wv[j], wv[j]);
          acc[s + j][0] = __ffma2_rn(ww, g01, acc[s + j][0]);
          acc[s + j][1] = __ffma2_rn(ww, g23, acc[s + j][1]);
        }
      }
    }
    float cs[4], sn[4];
    if (ROPE) {
      const int n = (int)(tok % g.N);
#pragma unroll
      for (int j = 0; j < 4; ++j) rope_cs(n, inv_freq[j], cs[j], sn[j]);
    }
    T* xrow = dx + tok * (int64_t)g.H * g.d + f0;
#pragma unroll
    for (int s = 0; s < HC; ++s) {
      float o[4] = {acc[s][0].x, acc[s][0].y, acc[s][1].x, acc[s][1].y};
      if (ROPE) {
        const int lane_mask = tpt >> 1;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float other = __shfl_xor_sync(0xffffffffu, o[j], lane_mask);
          o[j] = fmaf(o[j], cs[j], sign * other * sn[j]);
        }
      }
      if (valid && s < g.H) Vec4<T>::store(xrow + (int64_t)s * g.d, o);
    }
  }
}

// ---------------------------------------------------------------- weight gradient (bf16)
// dW[hp, s] = sum_{t, f} dY[t, hp, f] X'[t, s, f] with X' = R X (RoPE) or X,
// a GEMM with M = HP, N = H and a reduction K = B*N*d.  bf16 products are
// exact in fp32, so it runs on mma.sync m16n8k16 (bf16 in, fp32 accumulate).
// When RoPE rotates X, X' is no longer bf16: it is split into hi + lo bf16
// parts and both are multiplied (relative error ~2^-17).
// Block = MT warps, warp w owns hp rows [16w, 16w+16) and all s; a block
// walks a contiguous slab of tokens in chunks of DW_TT tokens staged in
// shared memory (X' hi / lo, rows padded to SP = 8 * NT, row stride d + 8 to
// spread banks).  Each block then adds its partial with one atomic per
// element.
constexpr int DW_TT = 4;

__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <int NT, bool ROPE>
__global__ void __launch_bounds__(256) premix_dw_mma_kernel(const __nv_bfloat16* __restrict__ dy,
                                                            const __nv_bfloat16* __restrict__ x,
                                                            float* __restrict__ dw, PremixGeom g,
                                                            int64_t tok_per_block) {
  constexpr int SP = 8 * NT;
  extern __shared__ float4 smem_f4[];
  const int ld = g.d + 8;  // row stride (elements)
  const int half = g.d >> 1;
  // layout: inv_freq[64] (double) | cos[DW_TT][64] | sin[DW_TT][64] | X' hi | X' lo
  double* s_invf = reinterpret_cast<double*>(smem_f4);
  float* s_cos = reinterpret_cast<float*>(s_invf + 64);
  float* s_sin = s_cos + DW_TT * 64;
  __nv_bfloat16* xhi = reinterpret_cast<__nv_bfloat16*>(s_sin + DW_TT * 64);
  __nv_bfloat16* xlo = xhi + DW_TT * SP * ld;
  if (ROPE) {
    for (int i = threadIdx.x; i < half; i += blockDim.x) s_invf[i] = rope_inv_freq(i, g.d, g.rope_base);
    __syncthreads();
  }

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, cq = lane & 3;
  const int hp0 = warp * 16;
  const int64_t t_begin = blockIdx.x * tok_per_block;
  int64_t t_end = t_begin + tok_per_block;
  if (t_end > g.ntok) t_end = g.ntok;

  float acc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;

  const int vec_per_row = g.d >> 3;  // 16-byte vectors per row
  for (int64_t tc = t_begin; tc < t_end; tc += DW_TT) {
    if (ROPE) {  // cos / sin of the chunk's positions
      for (int idx = threadIdx.x; idx < DW_TT * half; idx += blockDim.x) {
        const int tt = idx / half, i = idx - tt * half;
        rope_cs((int)((tc + tt) % g.N), s_invf[i], s_cos[tt * 64 + i], s_sin[tt * 64 + i]);
      }
      __syncthreads();
    }
    // ---- stage X' for DW_TT tokens (zero rows s >= H and tokens >= t_end)
    const int nvec = DW_TT * SP * vec_per_row;
    for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
      const int fv = v % vec_per_row;
      const int s = (v / vec_per_row) % SP;
      const int tt = v / (vec_per_row * SP);
      const int64_t tok = tc + tt;
      uint4 hi = make_uint4(0, 0, 0, 0), lo = make_uint4(0, 0, 0, 0);
      if (tok < t_end && s < g.H) {
        const __nv_bfloat16* row = x + (tok * g.H + s) * (int64_t)g.d;
        hi = __ldg(reinterpret_cast<const uint4*>(row) + fv);
        if (ROPE) {
          // partner features f +- d/2 of the same row
          const int f0 = fv * 8;
          const bool first = f0 < half;
          const uint4 pv = __ldg(reinterpret_cast<const uint4*>(row + (first ? f0 + half : f0 - half)));
          const uint32_t hw[4] = {hi.x, hi.y, hi.z, hi.w}, pw[4] = {pv.x, pv.y, pv.z, pv.w};
          uint32_t ho[4], lw[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            float r[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const float mine = e ? bf16hi_to_f32(hw[j]) : bf16lo_to_f32(hw[j]);
              const float other = e ? bf16hi_to_f32(pw[j]) : bf16lo_to_f32(pw[j]);
              const int i = (f0 + 2 * j + e) % half;
              const float c = s_cos[tt * 64 + i], sn = s_sin[tt * 64 + i];
              r[e] = first ? fmaf(mine, c, -other * sn) : fmaf(mine, c, other * sn);
            }
            ho[j] = pack_bf16x2(r[0], r[1]);
            lw[j] = pack_bf16x2(r[0] - bf16lo_to_f32(ho[j]), r[1] - bf16hi_to_f32(ho[j]));
          }
          hi = make_uint4(ho[0], ho[1], ho[2], ho[3]);
          lo = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
      }
      const int off = (tt * SP + s) * ld + fv * 8;
      *reinterpret_cast<uint4*>(xhi + off) = hi;
      if (ROPE) *reinterpret_cast<uint4*>(xlo + off) = lo;
    }
    __syncthreads();

    // ---- MMAs: A = dY rows from global, B = X' from shared memory
    const int ntt = (int)(t_end - tc < DW_TT ? t_end - tc : DW_TT);
    for (int tt = 0; tt < ntt; ++tt) {
      const int64_t tok = tc + tt;
      const __nv_bfloat16* arow0 = dy + (tok * g.HP + hp0 + gq) * (int64_t)g.d;
      const __nv_bfloat16* arow1 = arow0 + 8 * (int64_t)g.d;
      const bool r0 = hp0 + gq < g.HP, r1 = hp0 + gq + 8 < g.HP;
      for (int k0 = 0; k0 < g.d; k0 += 16) {
        // d % 8 == 0: the upper 8 columns of the last k-step may lie past d
        const bool hi8 = k0 + 8 < g.d;
        uint32_t a[4];
        a[0] = r0 ? __ldg(reinterpret_cast<const uint32_t*>(arow0 + k0 + 2 * cq)) : 0u;
        a[1] = r1 ? __ldg(reinterpret_cast<const uint32_t*>(arow1 + k0 + 2 * cq)) : 0u;
        a[2] = (r0 && hi8) ? __ldg(reinterpret_cast<const uint32_t*>(arow0 + k0 + 8 + 2 * cq)) : 0u;
        a[3] = (r1 && hi8) ? __ldg(reinterpret_cast<const uint32_t*>(arow1 + k0 + 8 + 2 * cq)) : 0u;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const int off = (tt * SP + nt * 8 + gq) * ld + k0 + 2 * cq;
          const uint32_t b0 = *reinterpret_cast<const uint32_t*>(xhi + off);
          const uint32_t b1 = hi8 ? *reinterpret_cast<const uint32_t*>(xhi + off + 8) : 0u;
          mma_bf16_16816(acc[nt], a, b0, b1);
          if (ROPE) {
            const uint32_t l0 = *reinterpret_cast<const uint32_t*>(xlo + off);
            const uint32_t l1 = hi8 ? *reinterpret_cast<const uint32_t*>(xlo + off + 8) : 0u;
            mma_bf16_16816(acc[nt], a, l0, l1);
          }
        }
      }
    }
    __syncthreads();
  }

  // ---- one atomic per element per block
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int s0 = nt * 8 + 2 * cq;
    const int h0 = hp0 + gq, h1 = hp0 + gq + 8;
    if (h0 < g.HP) {
      if (s0 < g.H) atomicAdd(dw + h0 * g.H + s0, acc[nt][0]);
      if (s0 + 1 < g.H) atomicAdd(dw + h0 * g.H + s0 + 1, acc[nt][1]);
    }
    if (h1 < g.HP) {
      if (s0 < g.H) atomicAdd(dw + h1 * g.H + s0, acc[nt][2]);
      if (s0 + 1 < g.H) atomicAdd(dw + h1 * g.H + s0 + 1, acc[nt][3]);
    }
  }
}

// ---------------------------------------------------------------- weight gradient (fp32)
// Plain CUDA-core reduction for fp32 tensors: one block per dW element,
// threads stride over (token, feature), block tree reduction, plain store.
template <bool ROPE>
__global__ void __launch_bounds__(256) premix_dw_f32_kernel(const float* __restrict__ dy,
                                                            const float* __restrict__ x,
                                                            float* __restrict__ dw, PremixGeom g) {
  const int hp = blockIdx.x / g.H, s = blockIdx.x % g.H;
  const int64_t total = g.ntok * g.d;
  const int half = g.d >> 1;
  float acc = 0.f;
  for (int64_t e = threadIdx.x; e < total; e += blockDim.x) {
    const int64_t tok = e / g.d;
    const int f = (int)(e % g.d);
    const float gv = dy[(tok * g.HP + hp) * g.d + f];
    float xv = x[(tok * g.H + s) * g.d + f];
    if (ROPE) {
      const int i = f % half;
      const float other = x[(tok * g.H + s) * g.d + (f < half ? f + half : f - half)];
      float c, sn;
      rope_cs((int)(tok % g.N), rope_inv_freq(i, g.d, g.rope_base), c, sn);
      xv = f < half ? fmaf(xv, c, -other * sn) : fmaf(xv, c, other * sn);
    }
    acc = fmaf(gv, xv, acc);
  }
  __shared__ float red[256];
  red[threadIdx.x] = acc;
  __syncthreads();
  for (int w = blockDim.x >> 1; w > 0; w >>= 1) {
    if ((int)threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) dw[hp * g.H + s] = red[0];
}

__global__ void zero_f32_kernel(float* p, int n) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) p[i] = 0.f;
}
// Three buffers of n floats, one block each.
__global__ void zero3_f32_kernel(float* a, float* b, float* c, int n) {
  float* p = blockIdx.x == 0 ? a : (blockIdx.x == 1 ? b : c);
  for (int i = threadIdx.x; i < n; i += blockDim.x) p[i] = 0.f;
}

// ---------------------------------------------------------------- host side
iha_status check_common(const char* name, const void* a, const void* b, const void* out, int B,
                        int N, int H, int P, int d, iha_dtype dt, int rope, float rope_base) {
  if (!a || !b || !out) return fail(IHA_ERR_INVALID_ARG, "%s: null pointer", name);
  if (B <= 0 || N <= 0 || H <= 0 || P <= 0 || d <= 0)
    return fail(IHA_ERR_INVALID_ARG, "%s: sizes must be positive", name);
  if (dt != IHA_BF16 && dt != IHA_F32) return fail(IHA_ERR_INVALID_ARG, "%s: bad dtype", name);
  if (H > 32) return fail(IHA_ERR_UNSUPPORTED, "%s: H = %d > 32", name, H);
  if (H * P > 128) return fail(IHA_ERR_UNSUPPORTED, "%s: H*P = %d > 128", name, H * P);
  if (dt == IHA_BF16 && d % 8) return fail(IHA_ERR_UNSUPPORTED, "%s: bf16 needs d %% 8 == 0", name);
  if (dt == IHA_F32 && d % 4) return fail(IHA_ERR_UNSUPPORTED, "%s: f32 needs d %% 4 == 0", name);
  if (rope && (d < 16 || d > 128 || (d & (d - 1))))
    return fail(IHA_ERR_UNSUPPORTED, "%s: RoPE needs d a power of two in [16, 128]", name);
  if (rope && !(rope_base > 0.f)) return fail(IHA_ERR_INVALID_ARG, "%s: rope_base <= 0", name);
  if (!aligned16(a) || !aligned16(b) || !aligned16(out))
    return fail(IHA_ERR_ALIGNMENT, "%s: pointers must be 16-byte aligned", name);
  return IHA_OK;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

int pick_hc(int H) {
  if (H <= 4) return 4;
  if (H <= 8) return 8;
  if (H <= 16) return 16;
  if (H <= 20) return 20;
  if (H <= 24) return 24;
  return 32;
}

// Grid for the (token, 4-feature) kernels: a multiple of the threads per
// token so each thread keeps its feature slot across the grid-stride loop.
unsigned slot_grid(const PremixGeom& g, int threads) {
  const int tpt = g.d / 4;
  const int64_t total = g.ntok * tpt;
  int64_t blocks = (total + threads - 1) / threads;
  const int64_t cap = (int64_t)sm_count() * 8;
  if (blocks > cap) blocks = cap;
  // stride = blocks * threads must be a multiple of tpt
  while (((int64_t)blocks * threads) % tpt) ++blocks;
  return (unsigned)blocks;
}

#define IHA_HC_SWITCH(HC, ...)            \
  switch (HC) {                           \
    case 4: { constexpr int kHC = 4; __VA_ARGS__; } break;   \
    case 8: { constexpr int kHC = 8; __VA_ARGS__; } break;   \
    case 16: { constexpr int kHC = 16; __VA_ARGS__; } break; \
    case 20: { constexpr int kHC = 20; __VA_ARGS__; } break; \
    case 24: { constexpr int kHC = 24; __VA_ARGS__; } break; \
    default: { constexpr int kHC = 32; __VA_ARGS__; } break; \
  }

template <typename T>
void launch_fwd_n(const PremixGeom& g, int ntens, const void* const* x, const float* const* w,
                  void* const* y, bool rope, cudaStream_t s) {
  const int threads = 256;
  const unsigned blocks = slot_grid(g, threads);
  const int hc = pick_hc(g.H);
  const size_t smem = (size_t)g.HP * hc * sizeof(float);
  FwdTensors<T> ts;
  for (int t = 0; t < 3; ++t) {
    const int u = t < ntens ? t : 0;
    ts.x[t] = static_cast<const T*>(x[u]);
    ts.w[t] = w[u];
    ts.y[t] = static_cast<T*>(y[u]);
  }
  const dim3 grid(blocks, ntens);
  IHA_HC_SWITCH(hc, {
    if (rope)
      premix_fwd_kernel<T, kHC, true><<<grid, threads, smem, s>>>(ts, g);
    else
      premix_fwd_kernel<T, kHC, false><<<grid, threads, smem, s>>>(ts, g);
  })
}

template <typename T>
void launch_fwd(const PremixGeom& g, const void* x, const float* w, void* y, bool rope,
                cudaStream_t s) {
  launch_fwd_n<T>(g, 1, &x, &w, &y, rope, s);
}

template <typename T>
void launch_dx(const PremixGeom& g, const void* dy, const float* w, void* dx, bool rope,
               cudaStream_t s) {
  const int threads = 256;
  const unsigned blocks = slot_grid(g, threads);
  const int hc = pick_hc(g.H);
  const size_t smem = (size_t)g.HP * hc * sizeof(float);
  IHA_HC_SWITCH(hc, {
    if (rope)
      premix_dx_kernel<T, kHC, true><<<blocks, threads, smem, s>>>(
          static_cast<const T*>(dy), w, static_cast<T*>(dx), g);
    else
      premix_dx_kernel<T, kHC, false><<<blocks, threads, smem, s>>>(
          static_cast<const T*>(dy), w, static_cast<T*>(dx), g);
  })
}

template <int NT, bool ROPE>
iha_status launch_dw_mma_nt(const PremixGeom& g, const void* dy, const void* x, float* dw,
                            cudaStream_t s) {
  const int MT = (g.HP + 15) / 16;
  const int threads = MT * 32;
  const int ld = g.d + 8;
  const size_t smem = 64 * sizeof(double) + 2 * DW_TT * 64 * sizeof(float) +
                      (size_t)DW_TT * 8 * NT * ld * sizeof(__nv_bfloat16) * (ROPE ? 2 : 1);
  auto kern = premix_dw_mma_kernel<NT, ROPE>;
  if (smem > 48 * 1024) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
      return check_launch("iha_premix_bwd_dw (smem attribute)");
  }
  int64_t blocks = (int64_t)sm_count() * 4;
  int64_t per = (g.ntok + blocks - 1) / blocks;
  per = ((per + DW_TT - 1) / DW_TT) * DW_TT;
  blocks = (g.ntok + per - 1) / per;
  kern<<<(unsigned)blocks, threads, smem, s>>>(static_cast<const __nv_bfloat16*>(dy),
                                               static_cast<const __nv_bfloat16*>(x), dw, g, per);
  return IHA_OK;
}

iha_status launch_dw_mma(const PremixGeom& g, const void* dy, const void* x, float* dw, bool rope,
                         cudaStream_t s) {
  const int nt = (g.H + 7) / 8;
  switch (nt) {
    case 1: return rope ? launch_dw_mma_nt<1, true>(g, dy, x, dw, s) : launch_dw_mma_nt<1, false>(g, dy, x, dw, s);
    case 2: return rope ? launch_dw_mma_nt<2, true>(g, dy, x, dw, s) : launch_dw_mma_nt<2, false>(g, dy, x, dw, s);
    case 3: return rope ? launch_dw_mma_nt<3, true>(g, dy, x, dw, s) : launch_dw_mma_nt<3, false>(g, dy, x, dw, s);
    default: return rope ? launch_dw_mma_nt<4, true>(g, dy, x, dw, s) : launch_dw_mma_nt<4, false>(g, dy, x, dw, s);
  }
}

PremixGeom make_geom(int B, int N, int H, int P, int d, float rope_base) {
  PremixGeom g;
  g.ntok = (int64_t)B * N;
  g.N = N;
  g.H = H;
  g.P = P;
  g.HP = H * P;
  g.d = d;
  g.rope_base = rope_base;
  return g;
}

}  // namespace
}  // namespace iha

extern "C" {

iha_status iha_premix_fwd(const void* x, const float* w, void* y, int B, int N, int H, int P,
                          int d, iha_dtype dt, int rope, float rope_base, void* stream) {
  using namespace iha;
  iha_status st = check_common("iha_premix_fwd", x, w, y, B, N, H, P, d, dt, rope, rope_base);
  if (st != IHA_OK) return st;
  const PremixGeom g = make_geom(B, N, H, P, d, rope_base);
  const size_t es = dt == IHA_BF16 ? 2 : 4;
  if (overlaps(y, g.ntok * g.HP * d * es, x, g.ntok * H * d * es) ||
      overlaps(y, g.ntok * g.HP * d * es, w, (size_t)g.HP * H * 4))
    return fail(IHA_ERR_INVALID_ARG, "iha_premix_fwd: y overlaps an input");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (dt == IHA_BF16 && premix_tc_supported(H, P, d))
    return premix_fwd_tc(x, w, y, B, N, H, P, d, rope, rope_base, s);
  if (dt == IHA_BF16) launch_fwd<__nv_bfloat16>(g, x, w, y, rope != 0, s);
  else launch_fwd<float>(g, x, w, y, rope != 0, s);
  return check_launch("iha_premix_fwd");
}

iha_status iha_premix_fwd_qkv(const void* xq, const void* xk, const void* xv, const float* wq,
                              const float* wk, const float* wv, void* yq, void* yk, void* yv,
                              int B, int N, int H, int P, int d, iha_dtype dt, int rope,
                              float rope_base, void* stream) {
  using namespace iha;
  const void* x[3] = {xq, xk, xv};
  const float* w[3] = {wq, wk, wv};
  void* y[3] = {yq, yk, yv};
  for (int t = 0; t < 3; ++t) {
    iha_status st = check_common("iha_premix_fwd_qkv", x[t], w[t], y[t], B, N, H, P, d, dt,
                                 t < 2 ? rope : 0, rope_base);
    if (st != IHA_OK) return st;
  }
  const PremixGeom g = make_geom(B, N, H, P, d, rope_base);
  const size_t es = dt == IHA_BF16 ? 2 : 4;
  const size_t ny = g.ntok * g.HP * d * es, nx = g.ntok * H * d * es, nw = (size_t)g.HP * H * 4;
  for (int t = 0; t < 3; ++t)
    for (int u = 0; u < 3; ++u)
      if (overlaps(y[t], ny, x[u], nx) || overlaps(y[t], ny, w[u], nw) ||
          (u != t && overlaps(y[t], ny, y[u], ny)))
        return fail(IHA_ERR_INVALID_ARG, "iha_premix_fwd_qkv: an output overlaps another tensor");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (dt == IHA_BF16 && premix_tc_supported(H, P, d))
    return premix_fwd_tc_multi(3, x, w, y, B, N, H, P, d, rope ? 3 : 0, rope_base, s);
  // CUDA-core kernel: Q, K and V in one launch, or Q, K (rotated) in one and
  // V in another when RoPE is on
  const int n_first = rope ? 2 : 3;
  if (dt == IHA_BF16) launch_fwd_n<__nv_bfloat16>(g, n_first, x, w, y, rope != 0, s);
  else launch_fwd_n<float>(g, n_first, x, w, y, rope != 0, s);
  iha_status st = check_launch("iha_premix_fwd_qkv");
  if (st != IHA_OK || !rope) return st;
  if (dt == IHA_BF16) launch_fwd_n<__nv_bfloat16>(g, 1, x + 2, w + 2, y + 2, false, s);
  else launch_fwd_n<float>(g, 1, x + 2, w + 2, y + 2, false, s);
  return check_launch("iha_premix_fwd_qkv");
}

iha_status iha_premix_fwd_qkv_interleaved(const void* xq, const void* xk, const void* xv,
                                          const float* wq, const float* wk, const float* wv,
                                          void* yq, void* yk, void* yv, int B, int N, int H, int P,
                                          int d, iha_dtype dt, int rope, float rope_base,
                                          void* stream) {
  using namespace iha;
  const void* x[3] = {xq, xk, xv};
  const float* w[3] = {wq, wk, wv};
  void* y[3] = {yq, yk, yv};
  for (int t = 0; t < 3; ++t) {
    iha_status st = check_common("iha_premix_fwd_qkv_interleaved", x[t], w[t], y[t], B, N, H, P,
                                 d, dt, t < 2 ? rope : 0, rope_base);
    if (st != IHA_OK) return st;
  }
  if (dt != IHA_BF16 || !premix_tc_supported(H, P, d))
    return fail(IHA_ERR_UNSUPPORTED,
                "iha_premix_fwd_qkv_interleaved: bf16 with d in {64, 128}, H <= 32, H*P <= 128");
  const PremixGeom g = make_geom(B, N, H, P, d, rope_base);
  const size_t ny = g.ntok * g.HP * d * 2, nx = g.ntok * H * d * 2, nw = (size_t)g.HP * H * 4;
  for (int t = 0; t < 3; ++t)
    for (int u = 0; u < 3; ++u)
      if (overlaps(y[t], ny, x[u], nx) || overlaps(y[t], ny, w[u], nw) ||
          (u != t && overlaps(y[t], ny, y[u], ny)))
        return fail(IHA_ERR_INVALID_ARG,
                    "iha_premix_fwd_qkv_interleaved: an output overlaps another tensor");
  return premix_fwd_tc_multi(3, x, w, y, B, N, H, P, d, rope ? 3 : 0, rope_base,
                             reinterpret_cast<cudaStream_t>(stream), 1);
}

iha_status iha_premix_bwd_dx(const void* dy, const float* w, void* dx, int B, int N, int H,
                             int P, int d, iha_dtype dt, int rope, float rope_base,
                             void* stream) {
  using namespace iha;
  iha_status st = check_common("iha_premix_bwd_dx", dy, w, dx, B, N, H, P, d, dt, rope, rope_base);
  if (st != IHA_OK) return st;
  const PremixGeom g = make_geom(B, N, H, P, d, rope_base);
  const size_t es = dt == IHA_BF16 ? 2 : 4;
  if (overlaps(dx, g.ntok * H * d * es, dy, g.ntok * g.HP * d * es) ||
      overlaps(dx, g.ntok * H * d * es, w, (size_t)g.HP * H * 4))
    return fail(IHA_ERR_INVALID_ARG, "iha_premix_bwd_dx: dx overlaps an input");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (dt == IHA_BF16 && premix_bwd_tc_supported(H, P, d, true, false, rope != 0))
    return premix_bwd_tc(dy, nullptr, w, dx, nullptr, B, N, H, P, d, rope, rope_base, s);
  if (dt == IHA_BF16) launch_dx<__nv_bfloat16>(g, dy, w, dx, rope != 0, s);
  else launch_dx<float>(g, dy, w, dx, rope != 0, s);
  return check_launch("iha_premix_bwd_dx");
}

iha_status iha_premix_bwd_dw(const void* dy, const void* x, float* dw, int B, int N, int H,
                             int P, int d, iha_dtype dt, int rope, float rope_base,
                             void* stream) {
  using namespace iha;
  iha_status st = check_common("iha_premix_bwd_dw", dy, x, dw, B, N, H, P, d, dt, rope, rope_base);
  if (st != IHA_OK) return st;
  const PremixGeom g = make_geom(B, N, H, P, d, rope_base);
  const size_t es = dt == IHA_BF16 ? 2 : 4;
  if (overlaps(dw, (size_t)g.HP * H * 4, dy, g.ntok * g.HP * d * es) ||
      overlaps(dw, (size_t)g.HP * H * 4, x, g.ntok * H * d * es))
    return fail(IHA_ERR_INVALID_ARG, "iha_premix_bwd_dw: dw overlaps an input");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (dt == IHA_BF16) {
    zero_f32_kernel<<<1, 256, 0, s>>>(dw, g.HP * H);
    if (premix_bwd_tc_supported(H, P, d, false, true, rope != 0))
      return premix_bwd_tc(dy, x, nullptr, nullptr, dw, B, N, H, P, d, rope, rope_base, s);
    st = launch_dw_mma(g, dy, x, dw, rope != 0, s);
    if (st != IHA_OK) return st;
  } else {
    if (rope)
      premix_dw_f32_kernel<true><<<g.HP * H, 256, 0, s>>>(static_cast<const float*>(dy),
                                                          static_cast<const float*>(x), dw, g);
    else
      premix_dw_f32_kernel<false><<<g.HP * H, 256, 0, s>>>(static_cast<const float*>(dy),
                                                           static_cast<const float*>(x), dw, g);
  }
  return check_launch("iha_premix_bwd_dw");
}

iha_status iha_premix_bwd(const void* dy, const void* x, const float* w, void* dx, float* dw,
                          int B, int N, int H, int P, int d, iha_dtype dt, int rope,
                          float rope_base, void* stream) {
  using namespace iha;
  iha_status st = check_common("iha_premix_bwd", dy, x, dx, B, N, H, P, d, dt, rope, rope_base);
  if (st != IHA_OK) return st;
  if (!w || !dw) return fail(IHA_ERR_INVALID_ARG, "iha_premix_bwd: null pointer");
  if (!aligned16(dw)) return fail(IHA_ERR_ALIGNMENT, "iha_premix_bwd: dw must be 16-byte aligned");
  const PremixGeom g = make_geom(B, N, H, P, d, rope_base);
  const size_t es = dt == IHA_BF16 ? 2 : 4;
  const size_t nx = g.ntok * H * d * es, ny = g.ntok * g.HP * d * es, nw = (size_t)g.HP * H * 4;
  if (overlaps(dx, nx, dy, ny) || overlaps(dx, nx, x, nx) || overlaps(dx, nx, w, nw) ||
      overlaps(dw, nw, dy, ny) || overlaps(dw, nw, x, nx) || overlaps(dw, nw, w, nw) ||
      overlaps(dw, nw, dx, nx))
    return fail(IHA_ERR_INVALID_ARG, "iha_premix_bwd: an output overlaps another buffer");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (dt == IHA_BF16 && premix_bwd_tc_supported(H, P, d, true, true, rope != 0)) {
    zero_f32_kernel<<<1, 256, 0, s>>>(dw, g.HP * H);
    return premix_bwd_tc(dy, x, w, dx, dw, B, N, H, P, d, rope, rope_base, s);
  }
  st = iha_premix_bwd_dx(dy, w, dx, B, N, H, P, d, dt, rope, rope_base, stream);
  if (st != IHA_OK) return st;
  return iha_premix_bwd_dw(dy, x, dw, B, N, H, P, d, dt, rope, rope_base, stream);
}

iha_status iha_premix_bwd_qkv(const void* dyq, const void* dyk, const void* dyv,
                              const void* xq, const void* xk, const void* xv, const float* wq,
                              const float* wk, const float* wv, void* dxq, void* dxk,
                              void* dxv, float* dwq, float* dwk, float* dwv, int B, int N, int H,
                              int P, int d, iha_dtype dt, int rope, float rope_base,
                              void* stream) {
  using namespace iha;
  const void* dy[3] = {dyq, dyk, dyv};
  const void* x[3] = {xq, xk, xv};
  const float* w[3] = {wq, wk, wv};
  void* dx[3] = {dxq, dxk, dxv};
  float* dw[3] = {dwq, dwk, dwv};
  for (int t = 0; t < 3; ++t) {
    iha_status st = check_common("iha_premix_bwd_qkv", dy[t], x[t], dx[t], B, N, H, P, d, dt,
                                 t < 2 ? rope : 0, rope_base);
    if (st != IHA_OK) return st;
    if (!w[t] || !dw[t]) return fail(IHA_ERR_INVALID_ARG, "iha_premix_bwd_qkv: null pointer");
    if (!aligned16(dw[t]))
      return fail(IHA_ERR_ALIGNMENT, "iha_premix_bwd_qkv: dw must be 16-byte aligned");
  }
  const PremixGeom g = make_geom(B, N, H, P, d, rope_base);
  const size_t es = dt == IHA_BF16 ? 2 : 4;
  const size_t nx = g.ntok * H * d * es, ny = g.ntok * g.HP * d * es, nw = (size_t)g.HP * H * 4;
  for (int t = 0; t < 3; ++t)
    for (int u = 0; u < 3; ++u) {
      const bool clash =
          overlaps(dx[t], nx, dy[u], ny) || overlaps(dx[t], nx, x[u], nx) ||
          overlaps(dx[t], nx, w[u], nw) || overlaps(dw[t], nw, dy[u], ny) ||
          overlaps(dw[t], nw, x[u], nx) || overlaps(dw[t], nw, w[u], nw) ||
          overlaps(dw[t], nw, dx[u], nx) ||
          (u != t && (overlaps(dx[t], nx, dx[u], nx) || overlaps(dw[t], nw, dw[u], nw)));
      if (clash)
        return fail(IHA_ERR_INVALID_ARG, "iha_premix_bwd_qkv: an output overlaps another buffer");
    }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (dt == IHA_BF16 && premix_bwd_tc_supported(H, P, d, true, true, rope != 0)) {
    zero3_f32_kernel<<<3, 256, 0, s>>>(dw[0], dw[1], dw[2], g.HP * H);
    const iha_status st = check_launch("iha_premix_bwd_qkv (zero dw)");
    if (st != IHA_OK) return st;
    return premix_bwd_tc_multi(3, dy, x, w, dx, dw, B, N, H, P, d, rope ? 3 : 0, rope_base, s);
  }
  for (int t = 0; t < 3; ++t) {
    const iha_status st = iha_premix_bwd(dy[t], x[t], w[t], dx[t], dw[t], B, N, H, P, d, dt,
                                         t < 2 ? rope : 0, rope_base, stream);
    if (st != IHA_OK) return st;
  }
  return IHA_OK;
}

}  // extern "C"
