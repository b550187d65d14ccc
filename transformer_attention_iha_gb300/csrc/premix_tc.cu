// Tensor-core premix forward for bf16 tensors with d in {64, 128}.
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
// Roles (320 threads, one CTA per SM, persistent over token pairs):
//   warps 0-7  epilogue: warp e reads TMEM lanes 32*(e%4).. (pseudo-head rows)
//              of token e/4 of the pair: 128 fp32 columns per thread, RoPE in
//              registers (partners f and f + d/2 are in the same thread),
//              bf16 pack, 128-byte-swizzled staging, TMA store of the
//              [H*P, 64] boxes.
//   warp 8     TMA producer of X: one [64 f, 32 s, d/64, 2 tokens] box per
//              stage (rows s >= H arrive as zeros), 4-stage ring.
//   warp 9     MMA issuer (lane 0) and TMEM owner (2 x 256 accumulator
//              columns, double-buffered against the epilogue).
// W (hi | lo) sits in shared memory as a 128 x 64 K-major, 128-byte-swizzled
// A operand, written once per CTA.
#include <math.h>

#include "common.cuh"
#include "premix_tc.h"

namespace iha {
namespace {

IHA_DEVICE_ERROR_WORD(premix_tc)

constexpr int kThreads = 320;
constexpr int kEpiThreads = 256;
constexpr int kXStages = 4;
constexpr int kTok = 2;  // tokens per stage

struct FwdParams {
  int ntok, N, H, HP, d, nch, rope, n_stages;
  uint32_t stage_bytes;  // X bytes per stage
  uint32_t blk;          // staging bytes per (token, 64-feature chunk), 1024-aligned
  RopeTable rt;
};

// cos / sin of n * inv_freq with inv_freq = hi + lo (fp32 pair).  The product
// is carried as p + c (p = fl(n*hi), c = exact error + n*lo) and reduced
// modulo 2*pi by an FMA-based Cody-Waite step (2*pi split into fp32 hi + lo),
// keeping the reduced angle accurate to ~3e-7 for positions up to 2^24.
__device__ __forceinline__ void rope_cos_sin(int n, float hi, float lo, float& c, float& s) {
  const float nf = (float)n;
  const float p = nf * hi;
  const float corr = fmaf(nf, lo, fmaf(nf, hi, -p));
  const float k = rintf(p * 0.15915494309189535f);
  float r = fmaf(-k, 6.2831854820251465f, p);
  r = fmaf(-k, -1.7484555314695172e-07f, r);
  r += corr;
  sincosf(r, &s, &c);
}

__device__ __forceinline__ void raise_error(volatile int* abort_flag) {
  *abort_flag = 1;
  atomicOr(&g_dev_error, DEV_ERR_WAIT_TIMEOUT);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    premix_fwd_tc_kernel(const __grid_constant__ CUtensorMap tmX,
                         const __grid_constant__ CUtensorMap tmY, const float* __restrict__ w,
                         const FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sW = smem_u32(smem);                   // 16 KB
  const uint32_t sX = sW + 16384;                       // kXStages x stage_bytes
  const uint32_t sStage = sX + kXStages * p.stage_bytes;  // 2 x kTok x nch x blk
  float* rope_tab = reinterpret_cast<float*>(smem + 16384 + kXStages * p.stage_bytes +
                                             2 * kTok * p.nch * p.blk);  // [2][kTok][64][2]
  uint64_t* bars = reinterpret_cast<uint64_t*>(rope_tab + 2 * kTok * 64 * 2);
  const uint32_t bar0 = smem_u32(bars);
  auto b_xfull = [&](int s) { return bar0 + 8u * s; };
  auto b_xempty = [&](int s) { return bar0 + 8u * (kXStages + s); };
  auto b_accfull = [&](int a) { return bar0 + 8u * (2 * kXStages + a); };
  auto b_accempty = [&](int a) { return bar0 + 8u * (2 * kXStages + 2 + a); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kXStages + 4);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < kXStages; ++s) {
      mbar_init(b_xfull(s), 1);
      mbar_init(b_xempty(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(b_accfull(a), 1);
      mbar_init(b_accempty(a), kEpiThreads);
    }
    *abort_flag = 0;
    mbar_init_fence();
  }
  // W -> bf16 hi | lo, K-major rows of 64 (hi s0..31 | lo s0..31), 128B swizzle
  if (tid < kEpiThreads) {
    for (int idx = tid; idx < 128 * 8; idx += kEpiThreads) {
      const int row = idx >> 3, j = idx & 7;
      uint32_t v[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float part[2];
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const int k = 8 * j + 2 * e + h2;  // 0..63
          const int s = k & 31;
          const float wv = (row < p.HP && s < p.H) ? __ldg(w + row * p.H + s) : 0.f;
          const float hi = __bfloat162float(__float2bfloat16_rn(wv));
          part[h2] = (k < 32) ? hi : (wv - hi);
        }
        v[e] = pack_bf16x2(part[0], part[1]);
      }
      const uint32_t off = (uint32_t)((row >> 3) * 1024 + (row & 7) * 128 + ((j ^ (row & 7)) << 4));
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
      tma_prefetch_desc(&tmX);
      int k = 0;
      for (int g = blockIdx.x; g < p.n_stages; g += gridDim.x, ++k) {
        const int xs = k % kXStages;
        if (!mbar_wait(b_xempty(xs), ((k / kXStages) & 1) ^ 1, abort_flag)) {
          raise_error(abort_flag);
          break;
        }
        mbar_arrive_expect_tx(b_xfull(xs), p.stage_bytes);
        tma_load_4d(sX + xs * p.stage_bytes, &tmX, b_xfull(xs), 0, 0, 0, g * kTok);
      }
      if (*abort_flag) {
        // let the copies still in flight land before the CTA exits
        volatile int no_abort = 0;
        for (int kk = k - kXStages > 0 ? k - kXStages : 0; kk < k; ++kk)
          mbar_wait(b_xfull(kk % kXStages), (kk / kXStages) & 1, &no_abort);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(128, kTok * D, false, true);
      const int nks = (p.H + 15) >> 4;
      int k = 0;
      bool ok = true;
      for (int g = blockIdx.x; g < p.n_stages; g += gridDim.x, ++k) {
        const int xs = k % kXStages, a = k & 1;
        if (!(ok = mbar_wait(b_xfull(xs), (k / kXStages) & 1, abort_flag))) break;
        if (!(ok = mbar_wait(b_accempty(a), ((k >> 1) & 1) ^ 1, abort_flag))) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + (uint32_t)(a * 256);
        const uint32_t xbase = sX + xs * p.stage_bytes;
        int j = 0;
        for (int part = 0; part < 2; ++part)
          for (int ks = 0; ks < nks; ++ks, ++j)
            mma_ss(d_tmem, smem_desc_sw128(sW + part * 64 + ks * 32, 16, 1024),
                   smem_desc_sw128(xbase + ks * 2048, 32 * 128, 1024), idesc, j > 0 ? 1u : 0u);
        mma_commit(b_xempty(xs));
        mma_commit(b_accfull(a));
      }
      if (!ok) raise_error(abort_flag);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // Every epilogue thread walks the same stages and named barriers even if
    // a wait gives up (no early exit), so the barriers cannot deadlock.
    constexpr int NCH = D / 64, HALF = D / 2;
    const int q = warp & 3, tt = warp >> 2;
    const int row = q * 32 + lane;  // pseudo-head row
    const bool warp_active = q * 32 < p.HP;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    int k = 0;
    for (int g = blockIdx.x; g < p.n_stages; g += gridDim.x, ++k) {
      const int a = k & 1, sb = k & 1;
      const int t = g * kTok + tt;
      if (tid == 0) bulk_wait_read<1>();  // staging buffer sb is free again
      if (p.rope && tid < kTok * 64) {
        const int t2 = g * kTok + (tid >> 6), i = tid & 63;
        if (i < HALF) {
          float c, s;
          rope_cos_sin(t2 % p.N, p.rt.hi[i], p.rt.lo[i], c, s);
          rope_tab[((sb * kTok + (tid >> 6)) * 64 + i) * 2 + 0] = c;
          rope_tab[((sb * kTok + (tid >> 6)) * 64 + i) * 2 + 1] = s;
        }
      }
      named_bar_sync(1, kEpiThreads);
      if (!mbar_wait(b_accfull(a), (k >> 1) & 1, abort_flag)) raise_error(abort_flag);
      tc_fence_after();
      float v[D];
      if (warp_active) {
        const uint32_t col = tmem + lane_base + (uint32_t)(a * 256 + tt * D);
        uint32_t r[32];
#pragma unroll
        for (int c = 0; c < 2 * NCH; ++c) {
          tmem_ld32(col + 32u * c, r);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) v[32 * c + e] = __uint_as_float(r[e]);
        }
      }
      tc_fence_before();
      mbar_arrive(b_accempty(a));
      if (warp_active && row < p.HP && t < p.ntok) {
        if (p.rope) {
          const float2* tab = reinterpret_cast<const float2*>(rope_tab) + (sb * kTok + tt) * 64;
#pragma unroll
          for (int i = 0; i < HALF; ++i) {
            const float2 cs = tab[i];
            const float x0 = v[i], x1 = v[i + HALF];
            v[i] = fmaf(x0, cs.x, -x1 * cs.y);
            v[i + HALF] = fmaf(x1, cs.x, x0 * cs.y);
          }
        }
        const uint32_t stage_base = (uint32_t)((sb * kTok + tt) * NCH) * p.blk;
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
          uint8_t* blk = smem + (sStage - sW) + stage_base + c * p.blk + row * 128;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int f = 64 * c + 8 * j;
            uint4 u;
            u.x = pack_bf16x2(v[f + 0], v[f + 1]);
            u.y = pack_bf16x2(v[f + 2], v[f + 3]);
            u.z = pack_bf16x2(v[f + 4], v[f + 5]);
            u.w = pack_bf16x2(v[f + 6], v[f + 7]);
            *reinterpret_cast<uint4*>(blk + ((j ^ (row & 7)) << 4)) = u;
          }
        }
      }
      fence_proxy_async_smem();
      named_bar_sync(1, kEpiThreads);
      if (tid == 0) {
        for (int t2 = 0; t2 < kTok; ++t2) {
          const int tok = g * kTok + t2;
          if (tok >= p.ntok) break;
          for (int c = 0; c < NCH; ++c)
            tma_store_3d(&tmY, sStage + (uint32_t)((sb * kTok + t2) * NCH + c) * p.blk,
                         64 * c, 0, tok);
        }
        bulk_commit();
      }
    }
    if (tid == 0) bulk_wait<0>();
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

iha_status premix_fwd_tc(const void* x, const float* w, void* y, int B, int N, int H, int P,
                         int d, int rope, float rope_base, cudaStream_t stream) {
  FwdParams p;
  p.ntok = B * N;
  p.N = N;
  p.H = H;
  p.HP = H * P;
  p.d = d;
  p.nch = d / 64;
  p.rope = rope;
  p.n_stages = (p.ntok + kTok - 1) / kTok;
  p.stage_bytes = (uint32_t)(kTok * p.nch * 32 * 128);
  p.blk = (uint32_t)(((p.HP * 128) + 1023) / 1024 * 1024);
  make_rope_table(&p.rt, d, rope_base);

  CUtensorMap mx, my;
  {
    // X as [tokens][d/64][s][64]: box = 64 features x 32 heads x d/64 x 2 tokens
    uint64_t dims[4] = {64, (uint64_t)H, (uint64_t)p.nch, (uint64_t)p.ntok};
    uint64_t st[3] = {(uint64_t)d * 2, 128, (uint64_t)H * d * 2};
    uint32_t box[4] = {64, 32, (uint32_t)p.nch, (uint32_t)kTok};
    if (encode_tiled(&mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(x), dims, st, box,
                     CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return fail(IHA_ERR_CUDA, "iha_premix_fwd: X tensor map encoding failed");
  }
  {
    uint64_t dims[3] = {(uint64_t)d, (uint64_t)p.HP, (uint64_t)p.ntok};
    uint64_t st[2] = {(uint64_t)d * 2, (uint64_t)p.HP * d * 2};
    uint32_t box[3] = {64, (uint32_t)p.HP, 1};
    if (encode_tiled(&my, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, y, dims, st, box,
                     CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return fail(IHA_ERR_CUDA, "iha_premix_fwd: Y tensor map encoding failed");
  }
  const size_t smem = 1024 + 16384 + kXStages * p.stage_bytes + 2 * kTok * p.nch * p.blk +
                      2 * kTok * 64 * 2 * sizeof(float) + 256;
  auto kern = d == 128 ? premix_fwd_tc_kernel<128> : premix_fwd_tc_kernel<64>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return check_launch("iha_premix_fwd (smem attribute)");
  int grid = sm_count();
  if (grid > p.n_stages) grid = p.n_stages;
  kern<<<grid, kThreads, smem, stream>>>(mx, my, w, p);
  return check_launch("iha_premix_fwd");
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
//   dX:  D[f, s]  = dY^T[f, hp] . W[hp, s]   A = dY as an MN-major operand
//        (M = 128 features), B = W^T (bf16 hi, then lo) K-major, N = 32 heads;
//        one 32-column TMEM accumulator per token, ring of 8.
//   dW:  D[hp, s] += dY[hp, f] . X[s, f]     A = the same dY bytes as a
//        K-major operand (M = pseudo-head rows), B = X (or R X split into
//        bf16 hi + lo when RoPE rotates it), accumulated over all tokens of
//        the CTA in one 32-column TMEM block, then added to dW with one
//        atomic per element.
// Roles (320 threads, persistent over tokens):
//   warps 0-3 / 4-7  two epilogue groups, even / odd tokens of the CTA:
//                    dX read-out (thread = feature lane), inverse RoPE through
//                    an fp32 exchange in shared memory, bf16 staging, TMA
//                    store; for RoPE + dW they also build R X (hi / lo).
//   warp 8           TMA producer (dY and X tiles, 4-stage ring)
//   warp 9           MMA issuer and TMEM owner
// ===========================================================================
namespace {

constexpr int kBwdNA = 8;  // dX accumulator slots (32 TMEM columns each)

struct BwdParams {
  int ntok, N, H, HP, hp_pad, nkb, ns;
  uint32_t dy_bytes;   // dY bytes per token (2 boxes of 64 x hp_pad)
  uint32_t x_bytes;    // X bytes per token (2 boxes of 64 x 32), 0 without dW
  uint32_t stage_bytes;
  uint32_t out_bytes;  // dX staging per buffer (H rows x 256 B), 1024-aligned
  RopeTable rt;
};

template <bool DO_DX, bool DO_DW, bool ROPE>
__global__ void __launch_bounds__(kThreads, 1)
    premix_bwd_tc_kernel(const __grid_constant__ CUtensorMap tmDY,
                         const __grid_constant__ CUtensorMap tmX,
                         const __grid_constant__ CUtensorMap tmDX, const float* __restrict__ w,
                         float* __restrict__ dw, const BwdParams p) {
  constexpr int D = 128;
  constexpr bool PREP = ROPE && DO_DW;  // epilogue builds R X for the dW MMA
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  // layout: W^T (32 rows x 2*nkb blocks x 128 B) | stages | X' (2 slots x hi,lo x 8 KB)
  //         | dX staging (2 groups x 2 bufs) | fp32 exchange (2 groups x 32 x 128 x 4)
  //         | rope tables (2 groups x 64 float2) | barriers
  const uint32_t wt_bytes = 32u * 2u * (uint32_t)p.nkb * 128u;
  const uint32_t sWT = smem_u32(smem);
  const uint32_t sStages = sWT + wt_bytes;
  const uint32_t sXr = sStages + (uint32_t)p.ns * p.stage_bytes;
  const uint32_t xr_bytes = PREP ? 2u * 2u * 8192u : 0u;
  const uint32_t sOut = sXr + xr_bytes;
  const uint32_t out_total = DO_DX ? 4u * p.out_bytes : 0u;
  const uint32_t sEx = sOut + out_total;
  const uint32_t ex_bytes = (DO_DX && ROPE) ? 2u * 32u * 128u * 4u : 0u;
  const uint32_t sRope = sEx + ex_bytes;
  const uint32_t rope_bytes = ROPE ? 2u * 64u * 8u : 0u;
  uint8_t* const base_ptr = smem;
  const uint32_t base_u32 = sWT;
  auto gen = [&](uint32_t a) { return base_ptr + (a - base_u32); };  // shared addr -> pointer
  uint64_t* bars = reinterpret_cast<uint64_t*>(gen(sRope + rope_bytes));
  const uint32_t bar0 = smem_u32(bars);
  const int NS = p.ns;
  auto b_infull = [&](int s) { return bar0 + 8u * s; };
  auto b_inempty = [&](int s) { return bar0 + 8u * (NS + s); };
  auto b_accfull = [&](int a) { return bar0 + 8u * (2 * NS + a); };
  auto b_accempty = [&](int a) { return bar0 + 8u * (2 * NS + kBwdNA + a); };
  auto b_xrfull = [&](int s) { return bar0 + 8u * (2 * NS + 2 * kBwdNA + s); };
  auto b_xrempty = [&](int s) { return bar0 + 8u * (2 * NS + 2 * kBwdNA + 2 + s); };
  const uint32_t b_dwfull = bar0 + 8u * (2 * NS + 2 * kBwdNA + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * NS + 2 * kBwdNA + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

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
    mbar_init(b_dwfull, 1);
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (DO_DX && tid < 256) {
    // W^T as the dX B operand: row s, K = pseudo-head; blocks of 64 along K
    // (hi blocks 0..nkb-1, lo blocks nkb..2nkb-1), 128-byte swizzle.
    const int nchunks = 32 * 2 * p.nkb * 8;
    for (int idx = tid; idx < nchunks; idx += 256) {
      const int j = idx & 7, s = (idx >> 3) & 31, blk = idx >> 8;
      const bool lo = blk >= p.nkb;
      const int hp0 = (blk - (lo ? p.nkb : 0)) * 64 + 8 * j;
      uint32_t v[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float part[2];
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const int hp = hp0 + 2 * e + h2;
          const float wv = (hp < p.HP && s < p.H) ? __ldg(w + hp * p.H + s) : 0.f;
          const float hi = __bfloat162float(__float2bfloat16_rn(wv));
          part[h2] = lo ? (wv - hi) : hi;
        }
        v[e] = pack_bf16x2(part[0], part[1]);
      }
      *reinterpret_cast<uint4*>(gen(sWT + (uint32_t)blk * 4096u + (uint32_t)s * 128u +
                                    (uint32_t)((j ^ (s & 7)) << 4))) =
          make_uint4(v[0], v[1], v[2], v[3]);
    }
  }
  if (PREP && tid < 256) {
    {  // rows s >= H of R X stay zero
      for (int idx = tid; idx < 2 * 2 * 32 * 8 * 2; idx += 256) {
        const int j = idx & 7, s = (idx >> 3) & 31, rest = idx >> 8;  // rest: slot*2*2 + part*2 + chunk
        if (s >= p.H)
          *reinterpret_cast<uint4*>(gen(sXr + (uint32_t)rest * 4096u + (uint32_t)s * 128u +
                                        (uint32_t)(j << 4))) = make_uint4(0, 0, 0, 0);
      }
    }
  }
  fence_proxy_async_smem();
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tmem_dw = tmem + (uint32_t)(kBwdNA * 32);

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
        tma_load_3d(st + p.dy_bytes / 2, &tmDY, b_infull(s), 64, 0, tok);
        if (DO_DW) {
          tma_load_3d(st + p.dy_bytes, &tmX, b_infull(s), 0, 0, tok);
          tma_load_3d(st + p.dy_bytes + 4096, &tmX, b_infull(s), 64, 0, tok);
        }
      }
      if (*abort_flag) {
        volatile int no_abort = 0;
        for (int kk = k - NS > 0 ? k - NS : 0; kk < k; ++kk)
          mbar_wait(b_infull(kk % NS), (kk / NS) & 1, &no_abort);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc_dx = idesc_bf16_f32(128, 32, true, false);
      const uint32_t idesc_dw = idesc_bf16_f32(128, 32, false, false);
      const int nk_hp = p.hp_pad >> 4;
      const uint32_t chunk_dy = p.dy_bytes / 2;  // one 64-feature box of dY
      bool ok = true;
      for (int k = 0; k < n_my; ++k) {
        const int s = k % NS;
        const uint32_t st = sStages + (uint32_t)s * p.stage_bytes;
        if (!(ok = mbar_wait(b_infull(s), (k / NS) & 1, abort_flag))) break;
        tc_fence_after();
        if (DO_DX) {
          const int a = k % kBwdNA;
          if (!(ok = mbar_wait(b_accempty(a), ((k / kBwdNA) & 1) ^ 1, abort_flag))) break;
          tc_fence_after();
          int j = 0;
          for (int part = 0; part < 2; ++part)
            for (int kk = 0; kk < nk_hp; ++kk, ++j) {
              const uint32_t bw = sWT + (uint32_t)(part * p.nkb + (kk >> 2)) * 4096u +
                                  (uint32_t)(kk & 3) * 32u;
              mma_ss(tmem + (uint32_t)(a * 32), smem_desc_sw128(st + (uint32_t)kk * 2048u, chunk_dy, 1024),
                     smem_desc_sw128(bw, 16, 1024), idesc_dx, j > 0 ? 1u : 0u);
            }
          mma_commit(b_accfull(a));
        }
        if (DO_DW) {
          uint32_t xsrc = st + p.dy_bytes;
          if (PREP) {
            if (!(ok = mbar_wait(b_xrfull(k & 1), (k >> 1) & 1, abort_flag))) break;
            tc_fence_after();
            xsrc = sXr + (uint32_t)(k & 1) * 16384u;
          }
          for (int part = 0; part < (PREP ? 2 : 1); ++part)
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t aoff = (uint32_t)(kk >> 2) * chunk_dy + (uint32_t)(kk & 3) * 32u;
              const uint32_t boff = (uint32_t)part * 8192u + (uint32_t)(kk >> 2) * 4096u +
                                    (uint32_t)(kk & 3) * 32u;
              mma_ss(tmem_dw, smem_desc_sw128(st + aoff, 16, 1024),
                     smem_desc_sw128(xsrc + boff, 16, 1024), idesc_dw,
                     (k > 0 || part > 0 || kk > 0) ? 1u : 0u);
            }
          if (PREP) mma_commit(b_xrempty(k & 1));
        }
        mma_commit(b_inempty(s));
      }
      if (!ok) raise_error(abort_flag);
      mma_commit(b_dwfull);
    }
  } else {
    // ------------------------------------------------------------ epilogue groups
    // Group G (warps 4G..4G+3) owns the CTA's tokens k with k % 2 == G.  The
    // groups never exit early, so their named barriers cannot deadlock.
    const int G = warp >> 2, gt = tid & 127;  // gt = TMEM lane = feature (dX)
    const int bar_id = 1 + G;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    float2* rope_tab = reinterpret_cast<float2*>(gen(sRope)) + G * 64;
    float* ex = reinterpret_cast<float*>(gen(sEx)) + G * 32 * 128;
    int it = 0;  // index among this group's tokens
    for (int k = G; k < n_my; k += 2, ++it) {
      const int tok = blockIdx.x + k * gridDim.x;
      const int s = k % NS;
      const uint32_t st = sStages + (uint32_t)s * p.stage_bytes;
      if (ROPE) {
        if (gt < 64) {
          float c, sn;
          rope_cos_sin(tok % p.N, p.rt.hi[gt], p.rt.lo[gt], c, sn);
          rope_tab[gt] = make_float2(c, sn);
        }
      }
      if (DO_DX && gt == 0) bulk_wait_read<1>();  // staging buffer (it & 1) is free
      named_bar_sync(bar_id, 128);
      if (PREP) {
        // R X (forward rotation) split into bf16 hi / lo, same swizzled layout as X
        if (!mbar_wait(b_infull(s), (k / NS) & 1, abort_flag)) raise_error(abort_flag);
        if (!mbar_wait(b_xrempty(k & 1), ((k >> 1) & 1) ^ 1, abort_flag)) raise_error(abort_flag);
        const uint32_t xs = st + p.dy_bytes;
        const uint32_t xr = sXr + (uint32_t)(k & 1) * 16384u;
        for (int task = gt; task < p.H * 8; task += 128) {
          const int row = task >> 3, j = task & 7;
          const uint32_t off = (uint32_t)row * 128u + (uint32_t)((j ^ (row & 7)) << 4);
          const uint4 a = *reinterpret_cast<const uint4*>(gen(xs + off));
          const uint4 b = *reinterpret_cast<const uint4*>(gen(xs + 4096u + off));
          const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
          uint32_t ah[4], al[4], bh[4], bl[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float ra[2], rb[2];
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              const float x0 = h2 ? bf16hi_to_f32(av[e]) : bf16lo_to_f32(av[e]);
              const float x1 = h2 ? bf16hi_to_f32(bv[e]) : bf16lo_to_f32(bv[e]);
              const float2 cs = rope_tab[8 * j + 2 * e + h2];
              ra[h2] = fmaf(x0, cs.x, -x1 * cs.y);
              rb[h2] = fmaf(x1, cs.x, x0 * cs.y);
            }
            ah[e] = pack_bf16x2(ra[0], ra[1]);
            bh[e] = pack_bf16x2(rb[0], rb[1]);
            al[e] = pack_bf16x2(ra[0] - bf16lo_to_f32(ah[e]), ra[1] - bf16hi_to_f32(ah[e]));
            bl[e] = pack_bf16x2(rb[0] - bf16lo_to_f32(bh[e]), rb[1] - bf16hi_to_f32(bh[e]));
          }
          *reinterpret_cast<uint4*>(gen(xr + off)) = make_uint4(ah[0], ah[1], ah[2], ah[3]);
          *reinterpret_cast<uint4*>(gen(xr + 4096u + off)) = make_uint4(bh[0], bh[1], bh[2], bh[3]);
          *reinterpret_cast<uint4*>(gen(xr + 8192u + off)) = make_uint4(al[0], al[1], al[2], al[3]);
          *reinterpret_cast<uint4*>(gen(xr + 12288u + off)) = make_uint4(bl[0], bl[1], bl[2], bl[3]);
        }
        fence_proxy_async_smem();
        mbar_arrive(b_xrfull(k & 1));
        mbar_arrive(b_inempty(s));
      }
      if (DO_DX) {
        const int a = k % kBwdNA;
        if (!mbar_wait(b_accfull(a), (k / kBwdNA) & 1, abort_flag)) raise_error(abort_flag);
        tc_fence_after();
        uint32_t r[32];
        tmem_ld32(tmem + lane_base + (uint32_t)(a * 32), r);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(b_accempty(a));
        float v[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(r[e]);
        if (ROPE) {
          // inverse rotation: partner feature gt ^ 64 lives in another warp
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (e < p.H) ex[e * 128 + gt] = v[e];
          named_bar_sync(bar_id, 128);
          const float2 cs = rope_tab[gt & 63];
          const float sg = gt < 64 ? 1.f : -1.f;
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (e < p.H) v[e] = fmaf(v[e], cs.x, sg * ex[e * 128 + (gt ^ 64)] * cs.y);
        }
        __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(
            gen(sOut + (uint32_t)(G * 2 + (it & 1)) * p.out_bytes));
#pragma unroll
        for (int e = 0; e < 32; ++e)
          if (e < p.H) out[e * 128 + gt] = __float2bfloat16_rn(v[e]);
        fence_proxy_async_smem();
        named_bar_sync(bar_id, 128);
        if (gt == 0) {
          tma_store_3d(&tmDX, sOut + (uint32_t)(G * 2 + (it & 1)) * p.out_bytes, 0, 0, tok);
          bulk_commit();
        }
      }
    }
    if (DO_DX && gt == 0) bulk_wait<0>();
    if (DO_DW && G == 0) {
      if (!mbar_wait(b_dwfull, 0, abort_flag)) raise_error(abort_flag);
      tc_fence_after();
      uint32_t r[32];
      tmem_ld32(tmem_dw + lane_base, r);
      tmem_wait_ld();
      if (gt < p.HP && n_my > 0) {
#pragma unroll
        for (int e = 0; e < 32; ++e)
          if (e < p.H) atomicAdd(dw + gt * p.H + e, __uint_as_float(r[e]));
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

bool premix_bwd_tc_supported(int H, int P, int d) { return d == 128 && H <= 32 && H * P <= 128; }

iha_status premix_bwd_tc(const void* dy, const void* x, const float* w, void* dx, float* dw,
                         int B, int N, int H, int P, int d, int rope, float rope_base,
                         cudaStream_t stream) {
  const bool do_dx = dx != nullptr, do_dw = dw != nullptr;
  BwdParams p;
  p.ntok = B * N;
  p.N = N;
  p.H = H;
  p.HP = H * P;
  p.hp_pad = (p.HP + 15) / 16 * 16;
  p.nkb = (p.hp_pad + 63) / 64;
  p.dy_bytes = 2u * (uint32_t)p.hp_pad * 128u;
  p.x_bytes = do_dw ? 2u * 32u * 128u : 0u;
  p.stage_bytes = (p.dy_bytes + p.x_bytes + 1023u) / 1024u * 1024u;
  p.out_bytes = ((uint32_t)H * 256u + 1023u) / 1024u * 1024u;
  make_rope_table(&p.rt, d, rope_base);
  const bool prep = rope && do_dw;
  const size_t fixed = 1024 + 32u * 2u * p.nkb * 128u + (prep ? 32768 : 0) +
                       (do_dx ? 4u * p.out_bytes : 0) + ((do_dx && rope) ? 32768 : 0) +
                       (rope ? 1024 : 0) + 512;
  const size_t limit = 227 * 1024;
  p.ns = 4;
  while (p.ns > 2 && fixed + (size_t)p.ns * p.stage_bytes > limit) --p.ns;
  const size_t smem = fixed + (size_t)p.ns * p.stage_bytes;
  if (smem > limit) return fail(IHA_ERR_UNSUPPORTED, "premix backward: shared memory budget");

  CUtensorMap mdy, mx, mdx;
  {
    uint64_t dims[3] = {(uint64_t)d, (uint64_t)p.HP, (uint64_t)p.ntok};
    uint64_t st[2] = {(uint64_t)d * 2, (uint64_t)p.HP * d * 2};
    uint32_t box[3] = {64, (uint32_t)p.hp_pad, 1};
    if (encode_tiled(&mdy, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(dy), dims, st,
                     box, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return fail(IHA_ERR_CUDA, "premix backward: dY tensor map encoding failed");
  }
  mx = mdy;
  if (do_dw) {
    uint64_t dims[3] = {(uint64_t)d, (uint64_t)H, (uint64_t)p.ntok};
    uint64_t st[2] = {(uint64_t)d * 2, (uint64_t)H * d * 2};
    uint32_t box[3] = {64, 32, 1};
    if (encode_tiled(&mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(x), dims, st, box,
                     CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return fail(IHA_ERR_CUDA, "premix backward: X tensor map encoding failed");
  }
  mdx = mdy;
  if (do_dx) {
    uint64_t dims[3] = {(uint64_t)d, (uint64_t)H, (uint64_t)p.ntok};
    uint64_t st[2] = {(uint64_t)d * 2, (uint64_t)H * d * 2};
    uint32_t box[3] = {128, (uint32_t)H, 1};
    if (encode_tiled(&mdx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, dx, dims, st, box,
                     CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS)
      return fail(IHA_ERR_CUDA, "premix backward: dX tensor map encoding failed");
  }
  void (*kern)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const float*, float*,
               const BwdParams);
  if (do_dx && do_dw)
    kern = rope ? premix_bwd_tc_kernel<true, true, true> : premix_bwd_tc_kernel<true, true, false>;
  else if (do_dx)
    kern = rope ? premix_bwd_tc_kernel<true, false, true> : premix_bwd_tc_kernel<true, false, false>;
  else
    kern = rope ? premix_bwd_tc_kernel<false, true, true> : premix_bwd_tc_kernel<false, true, false>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return check_launch("premix backward (smem attribute)");
  int grid = sm_count();
  if (grid > p.ntok) grid = p.ntok;
  kern<<<grid, kThreads, smem, stream>>>(mdy, mx, mdx, w, dw, p);
  return check_launch("premix backward");
}

}  // namespace iha
