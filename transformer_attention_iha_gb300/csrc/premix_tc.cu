// Tensor-core premix for bf16 tensors: the forward (d in {64, 128}) here,
// the backward (d = 128) in the second half of the file.
//
// "IHA-CUDA: Interleaved Head Attention Kernels for Hopper GPUs", section
// "Pseudo-Token Mixing (Triton Premix Kernels)": Y[b,n,h*P+p,f] =
// sum_s W[h,p,s] X[b,n,s,f] at every token and feature, optional fused RoPE.
//
// The mix is a contraction over the source heads, so per pair of tokens it is
// one MMA  D[hp, (t, f)] = W[hp, s] . X[s, (t, f)]  with M = 128 pseudo-head
// rows (H*P <= 128 valid), N = 2 tokens x d features and K = source heads
// (padded to 16 / 32).  The fp32 weight is split into bf16 hi + lo parts
// (W ~ hi + lo to ~2^-17 relative), both multiplied by the exact bf16 X and
// accumulated in fp32 in tensor memory, so the result matches an fp32-weight
// mix to far below the bf16 output rounding.  At H = 20 this moves the 2*H
// flops per output off the fp32 pipe, which alone could not keep up with HBM.
//
// One launch can mix up to three tensors (Q, K, V: each its own X, W, Y and
// RoPE flag).  The CTA walks stages of the concatenated token-pair lists;
// the three bf16 hi | lo weight tiles sit side by side in shared memory,
// spaced by the rows they use (ceil(H*P / 8) groups of 8 rows), since the
// MMA rows beyond H*P only feed accumulator rows that are never stored.
// Roles (320 threads, one CTA per SM, persistent over token pairs):
//   warps 0-7  epilogue: warp e reads TMEM lanes 32*(e%4).. (pseudo-head rows)
//              of token e/4 of the pair: 128 fp32 columns per thread, RoPE in
//              registers (partners f and f + d/2 are in the same thread),
//              bf16 pack into the warp's own 128-byte-swizzled staging and
//              TMA stores of its [32 rows, 64 f] boxes (no cross-warp sync).
//   warp 8     TMA producer of X: one [64 f, 32 s, d/64, 2 tokens] box per
//              stage (rows s >= H arrive as zeros), 4-stage ring.
//   warp 9     MMA issuer (one elected lane) and TMEM owner (2 x 256 accumulator
//              columns, double-buffered against the epilogue).
// W (hi | lo) sits in shared memory as a 128 x 64 K-major, 128-byte-swizzled
// A operand, written once per CTA.
#include <math.h>

#include <mutex>

#include "common.cuh"
#include "premix_tc.h"

namespace iha {
namespace {

IHA_DEVICE_ERROR_WORD(premix_tc)

constexpr int kThreads = 320;
constexpr int kEpiThreads = 256;
constexpr int kXStages = 4;
constexpr int kTok = 2;  // tokens per stage

constexpr int kMaxTens = 3;

struct FwdParams {
  int ntok, N, H, HP, d, nch, n_stages;  // n_stages: token pairs per tensor
  int ntens, rope_mask;                  // tensors of the launch; bit t: RoPE on tensor t
  int interleave;                        // output rows p * H + h instead of h * P + p
  int x_stages;                          // depth of the X ring (<= kXStages)
  uint32_t stage_bytes;                  // X bytes per stage
  uint32_t w_spacing;                    // bytes between the weight tiles
  const float* w[kMaxTens];
  RopeTable rt;
};

struct FwdMaps {
  CUtensorMap x[kMaxTens], y[kMaxTens];
};

// cos / sin of n * inv_freq with inv_freq = hi + lo (fp32 pair).  The product
// is carried as p + c (p = fl(n*hi), c = exact error + n*lo) and reduced
// modulo 2*pi by an FMA-based Cody-Waite step (2*pi split into fp32 hi + lo),
// keeping the reduced angle accurate to ~3e-7 for positions up to 2^24.  On
// the reduced angle (|r| <= pi + 1e-6) the hardware sine / cosine is accurate
// to ~2^-21 absolute, far below the bf16 rounding of the rotated values.
__device__ __forceinline__ void rope_cos_sin(int n, float hi, float lo, float& c, float& s) {
  const float nf = (float)n;
  const float p = nf * hi;
  const float corr = fmaf(nf, lo, fmaf(nf, hi, -p));
  const float k = rintf(p * 0.15915494309189535f);
  float r = fmaf(-k, 6.2831854820251465f, p);
  r = fmaf(-k, -1.7484555314695172e-07f, r);
  r += corr;
  __sincosf(r, &s, &c);
}

// inv_freq (hi, lo) of pair i, read with static indices only: a lane-dependent
// index into the by-value parameter block would go through local memory.
__device__ __forceinline__ float2 rope_inv_freq(const RopeTable& rt, int i) {
  float2 r = make_float2(0.f, 0.f);
#pragma unroll
  for (int k = 0; k < 64; ++k)
    if (k == i) r = make_float2(rt.hi[k], rt.lo[k]);
  return r;
}

__device__ __forceinline__ void raise_error(volatile int* abort_flag) {
  *abort_flag = 1;
  atomicOr(&g_dev_error, DEV_ERR_WAIT_TIMEOUT);
}

// dX chain of the backward: NK K-steps of 16 pseudo-heads; A = dY (MN-major,
// 2 KB per K-step), B = W^T hi | lo (K-major, 4 K-steps per 8 KB block).
template <int NK>
__device__ __forceinline__ void issue_dx(uint32_t d, uint64_t a0, uint64_t b0, uint32_t idesc) {
#pragma unroll
  for (int kk = 0; kk < NK; ++kk)
    mma_ss_nm(d, a0 + (uint64_t)(kk * 128), b0 + (uint64_t)(((kk >> 2) * 8192 + (kk & 3) * 32) >> 4),
              idesc, kk > 0 ? 1u : 0u);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    premix_fwd_tc_kernel(const __grid_constant__ FwdMaps maps, const FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  constexpr int NCH = D / 64, HALF = D / 2;
  constexpr uint32_t kWarpStage = 2u * NCH * 4096u;  // per epilogue warp: 2 buffers x NCH x [32][64]
  const uint32_t sW = smem_u32(smem);                      // weight tiles
  const uint32_t sX = sW + (uint32_t)(p.ntens - 1) * p.w_spacing + 16384u;  // X ring
  const uint32_t sStage = sX + (uint32_t)p.x_stages * p.stage_bytes;  // 8 warps x kWarpStage
  // per epilogue warp: cos / sin of its token, [HALF / 2] x (c_2j, c_2j+1, s_2j, s_2j+1)
  float4* rope_tabs = reinterpret_cast<float4*>(smem + (sStage - sW) + 8 * kWarpStage);  // [8][32]
  float2* inv_tab = reinterpret_cast<float2*>(rope_tabs + 8 * 32);  // [64] inv_freq (hi, lo)
  uint64_t* bars = reinterpret_cast<uint64_t*>(inv_tab + 64);
  const uint32_t bar0 = smem_u32(bars);
  auto b_xfull = [&](int s) { return bar0 + 8u * s; };
  auto b_xempty = [&](int s) { return bar0 + 8u * (kXStages + s); };
  auto b_accfull = [&](int a) { return bar0 + 8u * (2 * kXStages + a); };
  auto b_accempty = [&](int a) { return bar0 + 8u * (2 * kXStages + 2 + a); };
  const uint32_t b_drain = bar0 + 8u * (2 * kXStages + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kXStages + 5);
  const int XS = p.x_stages;
  const int total_stages = p.ntens * p.n_stages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < XS; ++s) {
      mbar_init(b_xfull(s), 1);
      mbar_init(b_xempty(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(b_accfull(a), 1);
      mbar_init(b_accempty(a), kEpiThreads);
    }
    mbar_init(b_drain, 1);
    *abort_flag = 0;
    mbar_init_fence();
#pragma unroll
    for (int i = 0; i < 64; ++i) inv_tab[i] = make_float2(p.rt.hi[i], p.rt.lo[i]);
  }
  // W -> bf16 hi | lo, K-major rows of 64 (hi s0..31 | lo s0..31), 128B swizzle,
  // one tile per tensor; only rows < H*P are written (the next tile starts
  // there).  Rows of the last tile past H*P stay unwritten: they only reach
  // accumulator rows that are never read.
  if (tid < kEpiThreads) {
    const int rows8 = (p.HP + 7) & ~7;
    for (int idx = tid; idx < p.ntens * rows8 * 8; idx += kEpiThreads) {
      const int tns = idx / (rows8 * 8), r = idx - tns * rows8 * 8;
      const int row = r >> 3, j = r & 7;
      // weight row of output row `row`: (h, p) = (row / P, row % P), or
      // interleaved (row % H, row / H)
      const int wrow = p.interleave ? (row % p.H) * (p.HP / p.H) + row / p.H : row;
      const float* w = p.w[0];
      if (tns == 1) w = p.w[1];
      if (tns == 2) w = p.w[2];
      uint32_t v[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float part[2];
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const int k = 8 * j + 2 * e + h2;  // 0..63
          const int s = k & 31;
          const float wv = (row < p.HP && s < p.H) ? __ldg(w + wrow * p.H + s) : 0.f;
          const float hi = __bfloat162float(__float2bfloat16_rn(wv));
          part[h2] = (k < 32) ? hi : (wv - hi);
        }
        v[e] = pack_bf16x2(part[0], part[1]);
      }
      const uint32_t off = (uint32_t)tns * p.w_spacing +
                           (uint32_t)((row >> 3) * 1024 + (row & 7) * 128 + ((j ^ (row & 7)) << 4));
      *reinterpret_cast<uint4*>(smem + off) = make_uint4(v[0], v[1], v[2], v[3]);
    }
    fence_proxy_async_smem();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      for (int t = 0; t < p.ntens; ++t) tma_prefetch_desc(&maps.x[t]);
      int k = 0;
      for (int G = blockIdx.x; G < total_stages; G += gridDim.x, ++k) {
        const int tns = G / p.n_stages, g = G - tns * p.n_stages;
        const int xs = k % XS;
        if (!mbar_wait(b_xempty(xs), ((k / XS) & 1) ^ 1, abort_flag)) {
          raise_error(abort_flag);
          break;
        }
        mbar_arrive_expect_tx(b_xfull(xs), p.stage_bytes);
        tma_load_4d(sX + xs * p.stage_bytes, &maps.x[tns], b_xfull(xs), 0, 0, 0, g * kTok);
      }
      // Whoever aborted, no copy may still be landing when the CTA exits
      // (in a normal run the last loads have completed and this returns at once).
      volatile int no_abort = 0;
      for (int kk = k - XS > 0 ? k - XS : 0; kk < k; ++kk)
        mbar_wait(b_xfull(kk % XS), (kk / XS) & 1, &no_abort);
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the schedule; one elected lane issues (see elect_one).
    {
      const uint32_t idesc = idesc_bf16_f32(128, kTok * D, false, true);
      const int nks = (p.H + 15) >> 4;
      int k = 0;
      bool ok = true;
      for (int G = blockIdx.x; G < total_stages; G += gridDim.x, ++k) {
        const int tns = G / p.n_stages;
        const uint32_t wt = sW + (uint32_t)tns * p.w_spacing;
        const int xs = k % XS, a = k & 1;
        if (!(ok = mbar_wait_warp(b_xfull(xs), (k / XS) & 1, abort_flag))) break;
        if (!(ok = mbar_wait_warp(b_accempty(a), ((k >> 1) & 1) ^ 1, abort_flag))) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + (uint32_t)(a * 256);
        const uint32_t xbase = sX + xs * p.stage_bytes;
        const uint64_t dw0 = smem_desc_sw128(wt, 16, 1024);
        const uint64_t dx0 = smem_desc_sw128(xbase, 32 * 128, 1024);
        if (elect_one()) {
          int j = 0;
          for (int part = 0; part < 2; ++part)
            for (int ks = 0; ks < nks; ++ks, ++j)
              mma_ss_nm(d_tmem, dw0 + (uint64_t)((part * 64 + ks * 32) >> 4),
                        dx0 + (uint64_t)(ks * 128), idesc, j > 0 ? 1u : 0u);
        }
        __syncwarp();
        mma_commit_warp(b_xempty(xs));
        mma_commit_warp(b_accfull(a));
      }
      if (!ok) raise_error(abort_flag);
      mma_drain_warp(b_drain);  // no MMA in flight when TMEM is released
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // Warp e owns pseudo-head rows 32*(e%4).. of token e/4 of each pair and
    // stores them itself (its own staging buffers and bulk groups), so the
    // epilogue warps never wait on one another.
    const int q = warp & 3, tt = warp >> 2;
    const int row = q * 32 + lane;  // pseudo-head row
    const bool warp_active = q * 32 < p.HP;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    const uint32_t wstage = sStage + (uint32_t)warp * kWarpStage;
    float4* tab = rope_tabs + warp * 32;
    int k = 0;
    for (int G = blockIdx.x; G < total_stages; G += gridDim.x, ++k) {
      const int tns = G / p.n_stages, g = G - tns * p.n_stages;
      const bool rope = (p.rope_mask >> tns) & 1;
      const int a = k & 1, sb = k & 1;
      const int t = g * kTok + tt;
      if (rope && warp_active && 2 * lane < HALF) {
        float c0, s0, c1, s1;
        const float4 inv = reinterpret_cast<const float4*>(inv_tab)[lane];  // pairs 2 lane, 2 lane + 1
        rope_cos_sin(t % p.N, inv.x, inv.y, c0, s0);
        rope_cos_sin(t % p.N, inv.z, inv.w, c1, s1);
        tab[lane] = make_float4(c0, c1, s0, s1);
      }
      __syncwarp();
      // after an abort: no TMEM loads and no stores, only the arrivals
      const bool live = mbar_wait_warp(b_accfull(a), (k >> 1) & 1, abort_flag);
      if (!live) raise_error(abort_flag);
      tc_fence_after();
      // Two passes over the accumulator: pass hh holds columns 32 hh .. +31
      // and their RoPE partners HALF + 32 hh .. +31 (64 registers, not D).
      const uint32_t col = tmem + lane_base + (uint32_t)(a * 256 + tt * D);
      const bool work = warp_active && live && t < p.ntok;
      if (work) {
        if (lane == 0) bulk_wait_read<1>();  // this warp's buffer sb is free again
        __syncwarp();
      }
#pragma unroll
      for (int hh = 0; hh < HALF / 32; ++hh) {
        float v[64];
        if (work) {
          tmem_ld32(col + 32u * hh, reinterpret_cast<uint32_t*>(v));
          tmem_ld32(col + (uint32_t)HALF + 32u * hh, reinterpret_cast<uint32_t*>(v) + 32);
          tmem_wait_ld();
        }
        if (hh == HALF / 32 - 1) {  // every column has been read
          tc_fence_before();
          mbar_arrive(b_accempty(a));
        }
        if (work && row < p.HP) {
          if (rope) {
            // pairs (i, i + HALF) two at a time on the packed fp32 pipe
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float4 cs = tab[16 * hh + j];
              const float2 c2 = make_float2(cs.x, cs.y), s2 = make_float2(cs.z, cs.w);
              const float2 x0 = make_float2(v[2 * j], v[2 * j + 1]);
              const float2 x1 = make_float2(v[32 + 2 * j], v[32 + 2 * j + 1]);
              const float2 y0 = __ffma2_rn(x0, c2, __fmul2_rn(make_float2(-x1.x, -x1.y), s2));
              const float2 y1 = __ffma2_rn(x0, s2, __fmul2_rn(x1, c2));
              v[2 * j] = y0.x;
              v[2 * j + 1] = y0.y;
              v[32 + 2 * j] = y1.x;
              v[32 + 2 * j + 1] = y1.y;
            }
          }
#pragma unroll
          for (int part = 0; part < 2; ++part) {
            const int c0 = part ? HALF + 32 * hh : 32 * hh;  // first column of the part
            uint8_t* blk = smem + (wstage - sW) + (uint32_t)(sb * NCH + c0 / 64) * 4096u + lane * 128;
#pragma unroll
            for (int g = 0; g < 4; ++g) {
              const int j = (c0 % 64) / 8 + g;  // 16-byte granule of the 128-byte row
              const float* vv = v + 32 * part + 8 * g;
              uint4 u;
              u.x = pack_bf16x2(vv[0], vv[1]);
              u.y = pack_bf16x2(vv[2], vv[3]);
              u.z = pack_bf16x2(vv[4], vv[5]);
              u.w = pack_bf16x2(vv[6], vv[7]);
              *reinterpret_cast<uint4*>(blk + ((j ^ (lane & 7)) << 4)) = u;
            }
          }
        }
      }
      if (!live) break;
      if (work) {
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
#pragma unroll
          for (int c = 0; c < NCH; ++c)
            tma_store_3d(&maps.y[tns], wstage + (uint32_t)(sb * NCH + c) * 4096u, 64 * c, q * 32, t);
          bulk_commit();
        }
      }
      __syncwarp();
    }
    if (lane == 0 && warp_active) bulk_wait<0>();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

bool premix_tc_supported(int H, int P, int d) {
  return (d == 64 || d == 128) && H <= 32 && H * P <= 128;
}

void make_rope_table(RopeTable* rt, int d, float base) {
  for (int i = 0; i < 64; ++i) {
    if (i < d / 2) {
      const double inv = pow((double)base, -2.0 * (double)i / (double)d);
      rt->hi[i] = (float)inv;
      rt->lo[i] = (float)(inv - (double)rt->hi[i]);
    } else {
      rt->hi[i] = rt->lo[i] = 0.f;
    }
  }
}

iha_status premix_fwd_tc_multi(int ntens, const void* const* x, const float* const* w,
                               void* const* y, int B, int N, int H, int P, int d, int rope_mask,
                               float rope_base, cudaStream_t stream, int interleave) {
  FwdParams p;
  p.interleave = interleave;
  p.ntok = B * N;
  p.N = N;
  p.H = H;
  p.HP = H * P;
  p.d = d;
  p.nch = d / 64;
  p.ntens = ntens;
  p.rope_mask = rope_mask;
  p.n_stages = (p.ntok + kTok - 1) / kTok;
  p.stage_bytes = (uint32_t)(kTok * p.nch * 32 * 128);
  p.w_spacing = (uint32_t)((p.HP + 7) / 8) * 1024u;
  for (int t = 0; t < kMaxTens; ++t) p.w[t] = w[t < ntens ? t : 0];
  make_rope_table(&p.rt, d, rope_base);

  FwdMaps maps;
  for (int t = 0; t < kMaxTens; ++t) {
    const int u = t < ntens ? t : 0;
    {
      // X as [tokens][d/64][s][64]: box = 64 features x 32 heads x d/64 x 2 tokens
      uint64_t dims[4] = {64, (uint64_t)H, (uint64_t)p.nch, (uint64_t)p.ntok};
      uint64_t st[3] = {(uint64_t)d * 2, 128, (uint64_t)H * d * 2};
      uint32_t box[4] = {64, 32, (uint32_t)p.nch, (uint32_t)kTok};
      if (encode_tiled(&maps.x[t], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(x[u]),
                       dims, st, box, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
        return fail(IHA_ERR_CUDA, "premix forward: X tensor map encoding failed");
    }
    {
      uint64_t dims[3] = {(uint64_t)d, (uint64_t)p.HP, (uint64_t)p.ntok};
      uint64_t st[2] = {(uint64_t)d * 2, (uint64_t)p.HP * d * 2};
      uint32_t box[3] = {64, 32, 1};
      if (encode_tiled(&maps.y[t], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, y[u], dims, st, box,
                       CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
        return fail(IHA_ERR_CUDA, "premix forward: Y tensor map encoding failed");
    }
  }
  // shared memory: alignment slack | weight tiles | X ring | epilogue staging |
  // cos / sin tables | inv_freq table | barriers; the ring is 4 deep when it fits
  const size_t fixed = 1024 + (size_t)(ntens - 1) * p.w_spacing + 16384 +
                       8 * 2 * p.nch * 4096 + 8 * 32 * sizeof(float4) + 64 * sizeof(float2) + 256;
  p.x_stages = kXStages;
  while (p.x_stages > 2 && fixed + (size_t)p.x_stages * p.stage_bytes > 227 * 1024) --p.x_stages;
  const size_t smem = fixed + (size_t)p.x_stages * p.stage_bytes;
  if (smem > 227 * 1024) return fail(IHA_ERR_UNSUPPORTED, "premix forward: shared memory budget");
  auto kern = d == 128 ? premix_fwd_tc_kernel<128> : premix_fwd_tc_kernel<64>;
  static SmemLimit limit[2];  // <128>, <64>: set on each device's first launch
  const cudaError_t attr_err = limit[d == 128 ? 0 : 1].ensure(kern, 227 * 1024);
  if (attr_err != cudaSuccess)
    return fail(IHA_ERR_CUDA, "premix forward (smem attribute): %s", cudaGetErrorString(attr_err));
  int grid = sm_count();
  if (grid > ntens * p.n_stages) grid = ntens * p.n_stages;
  kern<<<grid, kThreads, smem, stream>>>(maps, p);
  return check_launch("premix forward");
}

iha_status premix_fwd_tc(const void* x, const float* w, void* y, int B, int N, int H, int P,
                         int d, int rope, float rope_base, cudaStream_t stream) {
  const void* xs[1] = {x};
  const float* ws[1] = {w};
  void* ys[1] = {y};
  return premix_fwd_tc_multi(1, xs, ws, ys, B, N, H, P, d, rope ? 1 : 0, rope_base, stream);
}

}  // namespace iha

namespace iha {

// ===========================================================================
// Tensor-core premix backward (bf16, d = 128): dX = W^T dY and/or
// dW = sum_{tokens, f} dY X^T in one pass over dY.
//
// "IHA-CUDA: Interleaved Head Attention Kernels for Hopper GPUs", section
// "Pseudo-Token Mixing", backward: dX = W^T dY (transpose of the forward map)
// and dW = sum over (b, n, d) of dY X^T (atomic reduction).
//
// Per token the dY tile [H*P rows][128 f] arrives once by TMA (two 64-feature
// boxes, 128-byte swizzle) and serves both contractions from the same bytes:
//   dX:  D[f, (part, s)] = dY^T[f, hp] . [W_hi | W_lo][hp, (part, s)]
//        A = dY as an MN-major operand (M = 128 features), B = W^T with the
//        bf16 hi rows (s 0..31) and lo rows (32..63) stacked along N = 64, so
//        dY is read once per K-step; the epilogue adds the two halves.
//   dW:  D[hp, s] += dY[hp, f] . X[s, f]     A = the same dY bytes as a
//        K-major operand (M = pseudo-head rows), B = X, accumulated over all
//        tokens of the CTA in TMEM, then added to dW with one atomic per
//        element.  With RoPE, B = R X split into bf16 hi (rows 0..31) and lo
//        (rows 32..63) stacked along N = 64, again one read of dY.
// The kernel is bound by shared-memory traffic (TMA writes and MMA operand
// reads), which is why every operand is read once per K-step.
// Inverse RoPE on dX pairs feature f with f ^ 64, held by warp e ^ 2 of the
// same group: the pair of warps swaps fp32 values through shared memory
// (double-buffered, one 64-thread named barrier per token).
// Roles (320 threads, persistent over tokens):
//   warps 0-7   token groups: group G = warps 4G..4G+3 takes the CTA's tokens
//               k with k % 2 == G.  Per token: with RoPE, the token's cos /
//               sin table (one entry per feature pair, shared by both uses)
//               and R X (hi / lo) for the dW MMA into the group's own R X
//               slot; then the dX epilogue: warp e reads features 32*(e%4)..
//               from TMEM, stages bf16 [H][32] and TMA-stores it itself.
//               At the start they also build the W^T tile (while the first
//               tiles load), and group 0 folds the dW partials.
//   warp  8     TMA producer (dY and X tiles, ring of up to 4 stages)
//   warp  9     MMA issuer and TMEM owner
// ===========================================================================
namespace {

constexpr int kBwdThreads = 320;
constexpr int kBwdNA = 6;  // dX accumulator slots of 64 TMEM columns
// dW partials: the tensor core accumulates at most this many tokens (d/16
// MMA K-steps each) into one of two 64-column TMEM buffers; the partial is
// then added into fp32 registers with round-to-nearest adds.  Long chains of
// tensor-core accumulation drift systematically (measured 3e-5 relative at
// 216 tokens per CTA); chunks of 8 tokens keep it near fp32 rounding.
constexpr int kDwChunk = 8;
// Largest dynamic shared memory of a backward launch: the per-block limit
// less room for the kernel's static shared words.
constexpr int kBwdSmemMax = 227 * 1024 - 64;

struct BwdParams {
  int ntok, N, H, HP, hp_pad, nkb, ns;
  int ntens, rope_mask;  // tensors of the launch; bit t: tensor t takes RoPE
  uint32_t chunk;        // one 64-feature dY box: hp_pad x 128 B
  uint32_t dy_bytes;     // dY bytes per stage (2 boxes)
  uint32_t x_bytes;      // X bytes per token (2 boxes of 64 x 32), 0 without dW
  uint32_t stage_bytes;
  uint32_t out_bytes;    // per warp and buffer: H rows x 64 B, 128-aligned
  uint32_t ex_bytes;     // per warp and buffer: H x 32 fp32 exchange, 128-aligned
  RopeTable rt;
};

// One tensor's backward by the whole CTA (every thread calls it): its own
// barriers, W^T tile and pipeline in the 1024-aligned dynamic shared memory
// `smem`, TMEM allocated by the caller; the barriers are invalidated at the
// end so that the next pass may reuse the memory.
template <bool DO_DX, bool DO_DW, bool ROPE>
__device__ __forceinline__ void premix_bwd_pass(const CUtensorMap& tmDY, const CUtensorMap& tmX,
                                                const CUtensorMap& tmDX,
                                                const float* __restrict__ w,
                                                float* __restrict__ dw, const BwdParams& p,
                                                uint8_t* smem, const uint32_t tmem,
                                                volatile int* abort_flag) {
  constexpr int D = 128;
  constexpr bool PREP = ROPE && DO_DW;   // R X (hi / lo) for the dW MMA
  constexpr bool EXCH = ROPE && DO_DX;   // warp-pair exchange for the inverse rotation
  constexpr int NDW = PREP ? 64 : 32;    // dW accumulator columns
  // layout: W^T (nkb blocks of 64 rows x 128 B) | stages | R X (2 slots x 2 boxes
  //         of 64 rows) | dX staging (8 warps x 2) | exchange (8 warps x 2) |
  //         rope table (64 float2) | barriers
  const uint32_t wt_bytes = DO_DX ? (uint32_t)p.nkb * 8192u : 0u;
  const uint32_t sWT = smem_u32(smem);
  const uint32_t sStages = sWT + wt_bytes;
  const uint32_t sXr = sStages + (uint32_t)p.ns * p.stage_bytes;
  const uint32_t xr_bytes = PREP ? 2u * 16384u : 0u;
  const uint32_t sOut = sXr + xr_bytes;
  const uint32_t out_total = DO_DX ? 16u * p.out_bytes : 0u;
  const uint32_t sEx = sOut + out_total;
  const uint32_t ex_total = EXCH ? 16u * p.ex_bytes : 0u;
  const uint32_t sRope = sEx + ex_total;
  // cos / sin tables: [group][buffer][32] float4
  const uint32_t rope_bytes = (PREP || EXCH) ? 2u * 2u * 32u * 16u : 0u;
  auto gen = [&](uint32_t a) { return smem + (a - sWT); };  // shared address -> pointer
  uint64_t* bars = reinterpret_cast<uint64_t*>(gen((sRope + rope_bytes + 7u) & ~7u));
  const uint32_t bar0 = smem_u32(bars);
  const int NS = p.ns;
  auto b_infull = [&](int s) { return bar0 + 8u * s; };
  auto b_inempty = [&](int s) { return bar0 + 8u * (NS + s); };
  auto b_accfull = [&](int a) { return bar0 + 8u * (2 * NS + a); };
  auto b_accempty = [&](int a) { return bar0 + 8u * (2 * NS + 8 + a); };
  auto b_xrfull = [&](int s) { return bar0 + 8u * (2 * NS + 16 + s); };
  auto b_xrempty = [&](int s) { return bar0 + 8u * (2 * NS + 18 + s); };
  auto b_dwfull = [&](int b) { return bar0 + 8u * (2 * NS + 20 + b); };
  auto b_dwempty = [&](int b) { return bar0 + 8u * (2 * NS + 22 + b); };
  const uint32_t b_drain = bar0 + 8u * (2 * NS + 24);
  const uint32_t b_wt = bar0 + 8u * (2 * NS + 25);  // W^T tile built (256 arrivals)

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_my = (p.ntok - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(b_infull(s), 1);
      mbar_init(b_inempty(s), 1 + (PREP ? 128 : 0));
    }
    for (int a = 0; a < kBwdNA; ++a) {
      mbar_init(b_accfull(a), 1);
      mbar_init(b_accempty(a), 128);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(b_xrfull(s), 128);
      mbar_init(b_xrempty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(b_dwfull(b), 1);
      mbar_init(b_dwempty(b), 128);
    }
    mbar_init(b_drain, 1);
    mbar_init(b_wt, 256);
    mbar_init_fence();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_dw = tmem + (uint32_t)(kBwdNA * 64);  // + 64 * buffer

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tmDY);
      if (DO_DW) tma_prefetch_desc(&tmX);
      int k = 0;
      for (; k < n_my; ++k) {
        const int tok = blockIdx.x + k * gridDim.x, s = k % NS;
        if (!mbar_wait(b_inempty(s), ((k / NS) & 1) ^ 1, abort_flag)) {
          raise_error(abort_flag);
          break;
        }
        const uint32_t st = sStages + (uint32_t)s * p.stage_bytes;
        mbar_arrive_expect_tx(b_infull(s), p.dy_bytes + p.x_bytes);
        tma_load_3d(st, &tmDY, b_infull(s), 0, 0, tok);
        tma_load_3d(st + p.chunk, &tmDY, b_infull(s), 64, 0, tok);
        if (DO_DW) {
          tma_load_3d(st + p.dy_bytes, &tmX, b_infull(s), 0, 0, tok);
          tma_load_3d(st + p.dy_bytes + 4096u, &tmX, b_infull(s), 64, 0, tok);
        }
      }
      // Whoever aborted, no copy may still be landing when the CTA exits.
      volatile int no_abort = 0;
      for (int kk = k - NS > 0 ? k - NS : 0; kk < k; ++kk)
        mbar_wait(b_infull(kk % NS), (kk / NS) & 1, &no_abort);
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the schedule; one elected lane issues (see elect_one).
    {
      const uint32_t idesc_dx = idesc_bf16_f32(128, 64, true, false);
      const uint32_t idesc_dw = idesc_bf16_f32(128, NDW, false, false);
      const int nk_hp = p.hp_pad >> 4;
      // Descriptors of stage 0 / K-step 0; a K-step or a stage adds its byte
      // offset >> 4 to the start-address field (no carry: every operand lies
      // in the first 256 KB of shared memory).
      const uint64_t d_dx_a = smem_desc_sw128(sStages, p.chunk, 1024);  // dY, MN-major
      const uint64_t d_dx_b = smem_desc_sw128(sWT, 16, 1024);           // W^T hi | lo
      const uint64_t d_dw_a = smem_desc_sw128(sStages, 16, 1024);       // dY, K-major
      const uint64_t d_dw_b = PREP ? smem_desc_sw128(sXr, 16, 1024)
                                   : smem_desc_sw128(sStages + p.dy_bytes, 16, 1024);
      const uint32_t xchunk = PREP ? 8192u : 4096u;
      const uint32_t chunk = p.chunk, stage_bytes = p.stage_bytes;
      bool ok = true;
      for (int k = 0; k < n_my; ++k) {
        const int s = k % NS;
        const uint64_t st16 = (uint64_t)(((uint32_t)s * stage_bytes) >> 4);
        if (!(ok = mbar_wait_warp(b_infull(s), (k / NS) & 1, abort_flag))) break;
        tc_fence_after();
        if (DO_DX) {
          const int a = k % kBwdNA;
          if (k == 0 && !(ok = mbar_wait_warp(b_wt, 0, abort_flag))) break;  // W^T built
          if (!(ok = mbar_wait_warp(b_accempty(a), ((k / kBwdNA) & 1) ^ 1, abort_flag))) break;
          tc_fence_after();
          const uint32_t dxd = tmem + (uint32_t)(a * 64);
          const uint64_t dxa = d_dx_a + st16;
          if (elect_one()) switch (nk_hp) {  // a fully unrolled chain
            case 1: issue_dx<1>(dxd, dxa, d_dx_b, idesc_dx); break;
            case 2: issue_dx<2>(dxd, dxa, d_dx_b, idesc_dx); break;
            case 3: issue_dx<3>(dxd, dxa, d_dx_b, idesc_dx); break;
            case 4: issue_dx<4>(dxd, dxa, d_dx_b, idesc_dx); break;
            case 5: issue_dx<5>(dxd, dxa, d_dx_b, idesc_dx); break;
            case 6: issue_dx<6>(dxd, dxa, d_dx_b, idesc_dx); break;
            case 7: issue_dx<7>(dxd, dxa, d_dx_b, idesc_dx); break;
            default: issue_dx<8>(dxd, dxa, d_dx_b, idesc_dx); break;
          }
          __syncwarp();
          mma_commit_warp(b_accfull(a));
        }
        if (DO_DW) {
          const int dwc = k / kDwChunk, dwb = dwc & 1;
          const bool dw_first = (k % kDwChunk) == 0;
          if (dw_first && dwc >= 2 &&
              !(ok = mbar_wait_warp(b_dwempty(dwb), ((dwc >> 1) - 1) & 1, abort_flag))) break;
          uint64_t xb = d_dw_b + st16;
          if (PREP) {
            if (!(ok = mbar_wait_warp(b_xrfull(k & 1), (k >> 1) & 1, abort_flag))) break;
            tc_fence_after();
            xb = d_dw_b + (uint64_t)((k & 1) * (16384 >> 4));
          }
          const uint32_t dwd = tmem_dw + (uint32_t)(64 * dwb);
          const uint64_t dwa0 = d_dw_a + st16, dwa1 = dwa0 + (uint64_t)(chunk >> 4);
          const uint64_t xb1 = xb + (uint64_t)(xchunk >> 4);
          const uint32_t acc0 = dw_first ? 0u : 1u;
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
              mma_ss_nm(dwd, (kk < 4 ? dwa0 : dwa1) + (uint64_t)((kk & 3) * 2),
                        (kk < 4 ? xb : xb1) + (uint64_t)((kk & 3) * 2), idesc_dw,
                        kk > 0 ? 1u : acc0);
          }
          __syncwarp();
          if (PREP) mma_commit_warp(b_xrempty(k & 1));
          if ((k % kDwChunk) == kDwChunk - 1 || k == n_my - 1) mma_commit_warp(b_dwfull(dwb));
        }
        mma_commit_warp(b_inempty(s));
      }
      if (!ok) raise_error(abort_flag);
      mma_drain_warp(b_drain);  // no MMA in flight when TMEM is released
    }
  } else {
    // ------------------------------------------------------------ token groups
    // Group G (warps 4G..4G+3) takes tokens k with k % 2 == G; warp e holds
    // features f = 32*(e%4) + lane of them (TMEM lanes of the dX tile).
    // Group 0 also folds each dW chunk (TMEM lanes = pseudo-head rows f) into
    // fp32 registers and adds them to dw at the end.
    const int G = warp >> 2, q = warp & 3, gt = tid & 127;
    const int f = q * 32 + lane;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    const uint32_t wout = sOut + (uint32_t)(warp * 2) * p.out_bytes;
    if (DO_DX) {
      // W^T, the B operand of dX, built while the first tiles load: W (fp32)
      // read once, coalesced, into the not yet used dX staging; then row
      // n = part * 32 + s (part 0 = bf16 hi, 1 = lo of W[hp][s]), K =
      // pseudo-head in blocks of 64, 128-byte swizzle.
      float* wst = reinterpret_cast<float*>(gen(sOut));
      for (int i = tid; i < p.HP * p.H; i += 256) wst[i] = __ldg(w + i);
      named_bar_sync(1, 256);
      const int nchunks = p.nkb * 64 * 8;
      for (int idx = tid; idx < nchunks; idx += 256) {
        const int j = idx & 7, n = (idx >> 3) & 63, blk = idx >> 9;
        const int part = n >> 5, sr = n & 31;
        const int hp0 = blk * 64 + 8 * j;
        uint32_t v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float two[2];
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            const int hp = hp0 + 2 * e + h2;
            const float wv = (hp < p.HP && sr < p.H) ? wst[hp * p.H + sr] : 0.f;
            const float hi = __bfloat162float(__float2bfloat16_rn(wv));
            two[h2] = part ? (wv - hi) : hi;
          }
          v[e] = pack_bf16x2(two[0], two[1]);
        }
        *reinterpret_cast<uint4*>(gen(sWT + (uint32_t)blk * 8192u + (uint32_t)n * 128u +
                                      (uint32_t)((j ^ (n & 7)) << 4))) =
            make_uint4(v[0], v[1], v[2], v[3]);
      }
      fence_proxy_async_smem();
      mbar_arrive(b_wt);
      named_bar_sync(1, 256);  // the staging is free again
    }
    const uint32_t xr = sXr + (uint32_t)G * 16384u;  // this group's R X slot
    if (PREP) {  // its rows s >= H stay zero
      for (int idx = gt; idx < 2 * 64 * 8; idx += 128) {
        const int j = idx & 7, n = (idx >> 3) & 63, c = idx >> 9;
        if ((n & 31) >= p.H)
          *reinterpret_cast<uint4*>(gen(xr + (uint32_t)c * 8192u + (uint32_t)n * 128u +
                                        (uint32_t)(j << 4))) = make_uint4(0, 0, 0, 0);
      }
    }
    float dwacc[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) dwacc[e] = 0.f;
    bool ok = true;
    // fold dW chunk c (all its tokens' MMAs are committed to dwfull(c & 1))
    auto fold_dw = [&](int c) {
      const int b = c & 1;
      if (!(ok = mbar_wait_warp(b_dwfull(b), (c >> 1) & 1, abort_flag))) return;
      tc_fence_after();
      uint32_t r[32];
      tmem_ld32(tmem_dw + lane_base + (uint32_t)(64 * b), r);
      if (PREP) {
        uint32_t r2[32];
        tmem_ld32(tmem_dw + lane_base + (uint32_t)(64 * b + 32), r2);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) dwacc[e] += __uint_as_float(r[e]) + __uint_as_float(r2[e]);
      } else {
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) dwacc[e] += __uint_as_float(r[e]);
      }
      tc_fence_before();
      mbar_arrive(b_dwempty(b));
    };
    // cos / sin tables [group][buffer]: 32 float4 (c_2m, c_2m+1, s_2m, s_2m+1)
    float* tabs = reinterpret_cast<float*>(gen(sRope));
    const float2 inv = ROPE ? rope_inv_freq(p.rt, gt & 63) : make_float2(0.f, 0.f);
    const int n_dwc = (n_my + kDwChunk - 1) / kDwChunk;
    int dwc_done = 0;
    int it = 0;
    if (DO_DX || PREP) {
      // After an abort the loop keeps stepping (TMEM, shared-memory work and
      // stores skipped) so that every warp still meets the group's and the
      // inverse-RoPE pair's named barriers; later waits return at once.
      for (int k = G; k < n_my; k += 2, ++it) {
        const int tok = blockIdx.x + k * gridDim.x, s = k % NS;
        const float* tw = tabs + (G * 2 + (it & 1)) * 128;
        if (ROPE) {
          if (gt < 64) {
            float c, sn;
            rope_cos_sin(tok % p.N, inv.x, inv.y, c, sn);
            float* twm = tabs + (G * 2 + (it & 1)) * 128;
            twm[4 * (gt >> 1) + (gt & 1)] = c;
            twm[4 * (gt >> 1) + 2 + (gt & 1)] = sn;
          }
          named_bar_sync(6 + G, 128);  // the table is complete
        }
        if (PREP) {
          // R X (hi / lo) for the dW MMA, from the token's X tile in the stage
          const bool rx = ok && mbar_wait(b_infull(s), (k / NS) & 1, abort_flag) &&
                          mbar_wait(b_xrempty(G), (it & 1) ^ 1, abort_flag);
          if (ok && !rx) {
            ok = false;
            raise_error(abort_flag);
          }
          if (rx) {
            const uint32_t xs = sStages + (uint32_t)s * p.stage_bytes + p.dy_bytes;
            const float4* t4 = reinterpret_cast<const float4*>(tw);
            for (int task = gt; task < p.H * 8; task += 128) {
              const int j = task / p.H, row = task - j * p.H;  // neighbours share j: table broadcast
              const uint32_t off = (uint32_t)row * 128u + (uint32_t)((j ^ (row & 7)) << 4);
              const uint32_t offl = (uint32_t)(row + 32) * 128u + (uint32_t)((j ^ (row & 7)) << 4);
              const uint4 xa = *reinterpret_cast<const uint4*>(gen(xs + off));
              const uint4 xb = *reinterpret_cast<const uint4*>(gen(xs + 4096u + off));
              const uint32_t av[4] = {xa.x, xa.y, xa.z, xa.w}, bv[4] = {xb.x, xb.y, xb.z, xb.w};
              uint32_t ah[4], al[4], bh[4], bl[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                // features 8j + 2e, +1 (x0) and their partners 64 + 8j + 2e, +1 (x1)
                const float4 cs = t4[4 * j + e];
                const float2 c2 = make_float2(cs.x, cs.y), s2 = make_float2(cs.z, cs.w);
                const float2 x0 = make_float2(bf16lo_to_f32(av[e]), bf16hi_to_f32(av[e]));
                const float2 x1 = make_float2(bf16lo_to_f32(bv[e]), bf16hi_to_f32(bv[e]));
                const float2 ra = __ffma2_rn(x0, c2, __fmul2_rn(make_float2(-x1.x, -x1.y), s2));
                const float2 rb = __ffma2_rn(x0, s2, __fmul2_rn(x1, c2));
                ah[e] = pack_bf16x2(ra.x, ra.y);
                bh[e] = pack_bf16x2(rb.x, rb.y);
                al[e] = pack_bf16x2(ra.x - bf16lo_to_f32(ah[e]), ra.y - bf16hi_to_f32(ah[e]));
                bl[e] = pack_bf16x2(rb.x - bf16lo_to_f32(bh[e]), rb.y - bf16hi_to_f32(bh[e]));
              }
              // box c of the slot: 64 rows (hi rows 0..31, lo rows 32..63) x 128 B
              *reinterpret_cast<uint4*>(gen(xr + off)) = make_uint4(ah[0], ah[1], ah[2], ah[3]);
              *reinterpret_cast<uint4*>(gen(xr + 8192u + off)) = make_uint4(bh[0], bh[1], bh[2], bh[3]);
              *reinterpret_cast<uint4*>(gen(xr + offl)) = make_uint4(al[0], al[1], al[2], al[3]);
              *reinterpret_cast<uint4*>(gen(xr + 8192u + offl)) = make_uint4(bl[0], bl[1], bl[2], bl[3]);
            }
          }
          fence_proxy_async_smem();
          mbar_arrive(b_xrfull(G));
          mbar_arrive(b_inempty(s));
        }
        if (DO_DX) {
          const int a = k % kBwdNA;
          float c = 1.f, sn = 0.f;
          if (ROPE) {
            const int u = f & 63;
            c = tw[4 * (u >> 1) + (u & 1)];
            sn = tw[4 * (u >> 1) + 2 + (u & 1)];
          }
          const bool live = ok && mbar_wait_warp(b_accfull(a), (k / kBwdNA) & 1, abort_flag);
          if (ok && !live) {
            ok = false;
            raise_error(abort_flag);
          }
          float v[32];
          if (live) {
            tc_fence_after();
            uint32_t r[32], r2[32];
            tmem_ld32(tmem + lane_base + (uint32_t)(a * 64), r);
            tmem_ld32(tmem + lane_base + (uint32_t)(a * 64 + 32), r2);
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(b_accempty(a));
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(r[e]) + __uint_as_float(r2[e]);
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = 0.f;
          }
          if (EXCH) {
            // inverse rotation: swap with the warp holding features f ^ 64
            float* mine = reinterpret_cast<float*>(gen(sEx + (uint32_t)(warp * 2 + (it & 1)) * p.ex_bytes));
            const float* theirs = reinterpret_cast<const float*>(
                gen(sEx + (uint32_t)((warp ^ 2) * 2 + (it & 1)) * p.ex_bytes));
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (e < p.H) mine[e * 32 + lane] = v[e];
            named_bar_sync(2 + G * 2 + (q & 1), 64);
            const float sg = f < 64 ? sn : -sn;
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (e < p.H) v[e] = fmaf(v[e], c, theirs[e * 32 + lane] * sg);
          }
          if (live) {
            if (lane == 0) bulk_wait_read<1>();  // buffer it & 1 is free again
            __syncwarp();
            __nv_bfloat16* out =
                reinterpret_cast<__nv_bfloat16*>(gen(wout + (uint32_t)(it & 1) * p.out_bytes));
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (e < p.H) out[e * 32 + lane] = __float2bfloat16_rn(v[e]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_3d(&tmDX, wout + (uint32_t)(it & 1) * p.out_bytes, q * 32, 0, tok);
              bulk_commit();
            }
          }
        }
        // a dW chunk is complete once the last even token of it has passed
        if (DO_DW && G == 0 && ok && (k + 2 >= n_my || (k + 2) / kDwChunk != k / kDwChunk)) {
          fold_dw(dwc_done);
          ++dwc_done;
          if (!ok) raise_error(abort_flag);
        }
      }
      if (DO_DX && lane == 0) bulk_wait<0>();
    }
    if (DO_DW && G == 0) {
      for (; ok && dwc_done < n_dwc; ++dwc_done) fold_dw(dwc_done);
      if (ok && f < p.HP && n_my > 0) {
#pragma unroll
        for (int e = 0; e < 32; ++e)
          if (e < p.H) atomicAdd(dw + f * p.H + e, dwacc[e]);
      }
    }
    if (!ok) raise_error(abort_flag);
  }

  tc_fence_before();
  __syncthreads();
  if (tid == 0) {  // this pass's barriers are dead; their memory may be reused
    for (int s = 0; s < NS; ++s) {
      mbar_inval(b_infull(s));
      mbar_inval(b_inempty(s));
    }
    for (int a = 0; a < kBwdNA; ++a) {
      mbar_inval(b_accfull(a));
      mbar_inval(b_accempty(a));
    }
    for (int s = 0; s < 2; ++s) {
      mbar_inval(b_xrfull(s));
      mbar_inval(b_xrempty(s));
      mbar_inval(b_dwfull(s));
      mbar_inval(b_dwempty(s));
    }
    mbar_inval(b_drain);
    mbar_inval(b_wt);
  }
  __syncthreads();
}

struct BwdMaps {
  CUtensorMap dy[kMaxTens], x[kMaxTens], dx[kMaxTens];
};
struct BwdPtrs {
  const float* w[kMaxTens];
  float* dw[kMaxTens];
};

// The backward of p.ntens tensors (Q, K, V: each its own dY, X, W, dX, dW)
// in one launch: every CTA runs one pass per tensor over its share of the
// tokens, the RoPE variant chosen per tensor (bit t of p.rope_mask).  TMEM
// is allocated once for all passes; a raised abort flag skips the rest.
template <bool DO_DX, bool DO_DW>
__global__ void __launch_bounds__(kBwdThreads, 1)
    premix_bwd_tc_kernel(const __grid_constant__ BwdMaps maps, const BwdPtrs ptrs,
                         const BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  volatile int* abort_flag = &s_abort;
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) *abort_flag = 0;
  if (warp == 9) {
    tmem_alloc(smem_u32(&s_tmem), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  for (int t = 0; t < p.ntens && *abort_flag == 0; ++t) {
    if ((p.rope_mask >> t) & 1)
      premix_bwd_pass<DO_DX, DO_DW, true>(maps.dy[t], maps.x[t], maps.dx[t], ptrs.w[t],
                                          ptrs.dw[t], p, smem, tmem, abort_flag);
    else
      premix_bwd_pass<DO_DX, DO_DW, false>(maps.dy[t], maps.x[t], maps.dx[t], ptrs.w[t],
                                           ptrs.dw[t], p, smem, tmem, abort_flag);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

namespace {

// Launch geometry of the backward kernel; returns false when even the
// two-stage ring does not fit in shared memory.
bool bwd_geometry(int H, int P, bool do_dx, bool do_dw, bool rope, BwdParams* p, size_t* smem) {
  const bool exch = rope && do_dx, prep = rope && do_dw;
  p->H = H;
  p->HP = H * P;
  p->hp_pad = (p->HP + 15) / 16 * 16;
  p->nkb = (p->hp_pad + 63) / 64;
  p->chunk = (uint32_t)p->hp_pad * 128u;
  p->dy_bytes = 2u * p->chunk;
  p->x_bytes = do_dw ? 2u * 32u * 128u : 0u;
  // The dW MMA reads each 64-feature dY box as an M = 128 row operand
  // (16 KB from the box start) whatever hp_pad is; rows >= H*P only feed
  // discarded accumulator rows, but the bytes must lie inside the stage.
  uint32_t need = p->dy_bytes + p->x_bytes;
  if (do_dw && need < p->chunk + 16384u) need = p->chunk + 16384u;
  p->stage_bytes = (need + 1023u) / 1024u * 1024u;
  p->out_bytes = ((uint32_t)H * 64u + 127u) / 128u * 128u;
  p->ex_bytes = ((uint32_t)H * 128u + 127u) / 128u * 128u;
  const size_t fixed = 1024 + (do_dx ? (size_t)p->nkb * 8192u : 0) + (prep ? 32768 : 0) +
                       (do_dx ? 16u * p->out_bytes : 0) + (exch ? 16u * p->ex_bytes : 0) +
                       (rope ? 2048 : 0) + 512;  // last: barriers (<= 2*4 + 26 slots)
  const size_t limit = kBwdSmemMax;
  p->ns = 4;
  while (p->ns > 2 && fixed + (size_t)p->ns * p->stage_bytes > limit) --p->ns;
  *smem = fixed + (size_t)p->ns * p->stage_bytes;
  return *smem <= limit;
}

}  // namespace

bool premix_bwd_tc_supported(int H, int P, int d, bool do_dx, bool do_dw, bool rope) {
  if (d != 128 || H > 32 || H * P > 128) return false;
  BwdParams p;
  size_t smem;
  return bwd_geometry(H, P, do_dx, do_dw, rope, &p, &smem);
}

namespace {

// Dynamic shared memory attribute of each backward instantiation, set once
// per process (thread-safe) to the largest size any launch asks for.
template <bool DX, bool DW>
cudaError_t bwd_smem_attribute() {
  static SmemLimit limit;  // per instantiation, set on each device's first launch
  return limit.ensure(premix_bwd_tc_kernel<DX, DW>, kBwdSmemMax);
}

}  // namespace

iha_status premix_bwd_tc_multi(int ntens, const void* const* dy, const void* const* x,
                               const float* const* w, void* const* dx, float* const* dw, int B,
                               int N, int H, int P, int d, int rope_mask, float rope_base,
                               cudaStream_t stream) {
  if (ntens < 1 || ntens > kMaxTens)
    return fail(IHA_ERR_INVALID_ARG, "premix backward: 1 to 3 tensors per launch");
  const bool do_dx = dx[0] != nullptr, do_dw = dw[0] != nullptr;
  for (int t = 1; t < ntens; ++t)
    if ((dx[t] != nullptr) != do_dx || (dw[t] != nullptr) != do_dw)
      return fail(IHA_ERR_INVALID_ARG, "premix backward: every tensor needs the same outputs");
  rope_mask &= (1 << ntens) - 1;
  BwdParams p;
  size_t smem;
  if (!bwd_geometry(H, P, do_dx, do_dw, rope_mask != 0, &p, &smem))
    return fail(IHA_ERR_UNSUPPORTED, "premix backward: shared memory budget");
  p.ntok = B * N;
  p.N = N;
  p.ntens = ntens;
  p.rope_mask = rope_mask;
  make_rope_table(&p.rt, d, rope_base);

  BwdMaps maps;
  BwdPtrs ptrs;
  for (int t = 0; t < ntens; ++t) {
    ptrs.w[t] = w[t];
    ptrs.dw[t] = dw[t];
    {
      uint64_t dims[3] = {(uint64_t)d, (uint64_t)p.HP, (uint64_t)p.ntok};
      uint64_t st[2] = {(uint64_t)d * 2, (uint64_t)p.HP * d * 2};
      uint32_t box[3] = {64, (uint32_t)p.hp_pad, 1};
      if (encode_tiled(&maps.dy[t], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(dy[t]),
                       dims, st, box, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
        return fail(IHA_ERR_CUDA, "premix backward: dY tensor map encoding failed");
    }
    maps.x[t] = maps.dy[t];
    if (do_dw) {
      uint64_t dims[3] = {(uint64_t)d, (uint64_t)H, (uint64_t)p.ntok};
      uint64_t st[2] = {(uint64_t)d * 2, (uint64_t)H * d * 2};
      uint32_t box[3] = {64, 32, 1};
      if (encode_tiled(&maps.x[t], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(x[t]),
                       dims, st, box, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
        return fail(IHA_ERR_CUDA, "premix backward: X tensor map encoding failed");
    }
    maps.dx[t] = maps.dy[t];
    if (do_dx) {
      uint64_t dims[3] = {(uint64_t)d, (uint64_t)H, (uint64_t)p.ntok};
      uint64_t st[2] = {(uint64_t)d * 2, (uint64_t)H * d * 2};
      uint32_t box[3] = {32, (uint32_t)H, 1};
      if (encode_tiled(&maps.dx[t], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, dx[t], dims, st, box,
                       CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS)
        return fail(IHA_ERR_CUDA, "premix backward: dX tensor map encoding failed");
    }
  }
  for (int t = ntens; t < kMaxTens; ++t) {  // unused slots: valid copies, never read
    maps.dy[t] = maps.dy[0];
    maps.x[t] = maps.x[0];
    maps.dx[t] = maps.dx[0];
    ptrs.w[t] = nullptr;
    ptrs.dw[t] = nullptr;
  }
  void (*kern)(const BwdMaps, const BwdPtrs, const BwdParams);
  cudaError_t ae;
  if (do_dx && do_dw) {
    kern = premix_bwd_tc_kernel<true, true>;
    ae = bwd_smem_attribute<true, true>();
  } else if (do_dx) {
    kern = premix_bwd_tc_kernel<true, false>;
    ae = bwd_smem_attribute<true, false>();
  } else {
    kern = premix_bwd_tc_kernel<false, true>;
    ae = bwd_smem_attribute<false, true>();
  }
  if (ae != cudaSuccess)
    return fail(IHA_ERR_CUDA, "premix backward (smem attribute): %s", cudaGetErrorString(ae));
  int grid = sm_count();
  if (grid > p.ntok) grid = p.ntok;
  kern<<<grid, kBwdThreads, smem, stream>>>(maps, ptrs, p);
  return check_launch("premix backward");
}

iha_status premix_bwd_tc(const void* dy, const void* x, const float* w, void* dx, float* dw,
                         int B, int N, int H, int P, int d, int rope, float rope_base,
                         cudaStream_t stream) {
  const void* dys[1] = {dy};
  const void* xs[1] = {x};
  const float* ws[1] = {w};
  void* dxs[1] = {dx};
  float* dws[1] = {dw};
  return premix_bwd_tc_multi(1, dys, xs, ws, dxs, dws, B, N, H, P, d, rope ? 1 : 0, rope_base,
                             stream);
}

}  // namespace iha
