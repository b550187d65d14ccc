// Multi-head softmax attention forward over pseudo-heads / mask units.
//
// "IHA-CUDA: Interleaved Head Attention Kernels for Hopper GPUs", sections
// "Kernel Design" (attention over the H*P pseudo-heads after the premix,
// sliding window) and "FLOP Matching" (window W = WSL + 1, 128-token tiles);
// "hiera-optim 0.1.0", hiera_optim/attention/mask_unit.py,
// MaskUnitAttentionFast.forward (unmasked attention inside each mask unit,
// scale head_dim ** -0.5, tokens laid out (T outer, units inner)).
//
// bf16 path (sm_103a tensor cores):
//   CTA = two 128-row query tiles of one head (256 rows), 10 warps:
//     warps 0-3  softmax of query tile 0 (thread = row = TMEM lane)
//     warps 4-7  softmax of query tile 1
//     warp  8    TMA producer: Q once, then K / V tiles into a 2-stage ring
//     warp  9    tcgen05.mma issuer (one thread) and TMEM owner
//   TMEM (512 columns): S0 | S1 | O0 | O1, 128 fp32 columns each.  P (bf16)
//   overwrites the first 64 columns of S and feeds the P.V MMA as the
//   A operand straight from tensor memory.
//   Online softmax in the log2 domain with conditional rescaling: O and l
//   are rescaled only when a row maximum grows by more than 8 (a factor of
//   256), which keeps every exponent <= 2^8 and is exact in real arithmetic.
//   KV tiles outside the causal / window band of the query-tile pair are
//   never loaded (block skipping); tiles crossing a band edge or the key
//   tail are masked element-wise.
// f32 path: CUDA-core kernel in fp32 throughout (no TF32), for fp32 tensors.
#include <math.h>

#include "common.cuh"

namespace iha {
namespace {

IHA_DEVICE_ERROR_WORD(attention)

constexpr int kBM = 128;             // query rows per tile
constexpr int kBN = 128;             // keys per tile
constexpr int kChunk = 64;           // head-dim elements per 128-byte swizzle row
constexpr int kTileChunkBytes = kBM * 128;  // 16 KB: 128 rows x 64 bf16
constexpr int kThreads = 320;
constexpr int kSmemTiles = 12 * kTileChunkBytes;  // Q 2x2, K 2x2, V 2x2 chunks
constexpr int kSmemBytes = kSmemTiles + 256 + 1024;  // + barriers + alignment slack
constexpr float kRescaleLog2 = 8.0f;

struct AttnParams {
  int Bo, Bi, Hh, Nq, Nk, d, nD;
  int mask, window;
  int n_qpairs;
  float scale_log2;
  int64_t so_bo, so_bi, so_seq, so_h;
  __nv_bfloat16* o;
  float* lse;
};

// KV tile range [lo, hi] (inclusive) visited by query rows [q_lo, q_hi].
__device__ __forceinline__ void kv_tile_range(const AttnParams& p, int q_lo, int q_hi, int& lo,
                                              int& hi) {
  const int n_kt = (p.Nk + kBN - 1) / kBN;
  if (p.mask == IHA_MASK_NONE) {
    lo = 0;
    hi = n_kt - 1;
    return;
  }
  hi = min(q_hi / kBN, n_kt - 1);
  lo = (p.mask == IHA_MASK_CAUSAL_WINDOW) ? max(0, q_lo - (p.window - 1)) / kBN : 0;
}

__device__ __forceinline__ void raise_error(volatile int* abort_flag) {
  *abort_flag = 1;
  atomicOr(&g_dev_error, DEV_ERR_WAIT_TIMEOUT);
}

__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                       const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sQ = smem_u32(smem);                       // [tile][chunk]
  const uint32_t sK = sQ + 4 * kTileChunkBytes;             // [stage][chunk]
  const uint32_t sV = sK + 4 * kTileChunkBytes;             // [stage][chunk]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kSmemTiles);
  const uint32_t bar0 = smem_u32(bars);
  // barrier slots
  const uint32_t b_q = bar0;
  auto b_kfull = [&](int s) { return bar0 + 8u * (1 + s); };
  auto b_vfull = [&](int s) { return bar0 + 8u * (3 + s); };
  auto b_kvempty = [&](int s) { return bar0 + 8u * (5 + s); };
  auto b_sfull = [&](int t) { return bar0 + 8u * (7 + t); };
  auto b_pfull = [&](int t) { return bar0 + 8u * (9 + t); };
  auto b_ofull = [&](int t) { return bar0 + 8u * (11 + t); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 16);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x;
  const int bz = blockIdx.y;
  const int bo = bz / p.Bi, bi = bz - bo * p.Bi;
  const int pair = p.n_qpairs - 1 - (int)blockIdx.z;  // heaviest (latest) pairs first
  const int n_qt = (p.Nq + kBM - 1) / kBM;
  const int qt0 = 2 * pair, qt1 = 2 * pair + 1;
  const bool act1 = qt1 < n_qt;
  const int q_lo = qt0 * kBM;
  const int q_hi = min((act1 ? qt1 : qt0) * kBM + kBM - 1, p.Nq - 1);
  int j_lo, j_hi;
  kv_tile_range(p, q_lo, q_hi, j_lo, j_hi);
  const int n_kv = j_hi - j_lo + 1;

  if (threadIdx.x == 0) {
    mbar_init(b_q, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(b_kfull(s), 1);
      mbar_init(b_vfull(s), 1);
      mbar_init(b_kvempty(s), 1);
      mbar_init(b_sfull(s), 1);
      mbar_init(b_pfull(s), 128);
      mbar_init(b_ofull(s), 1);
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
  const uint32_t chunk_bytes = (uint32_t)p.nD * kTileChunkBytes;

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      mbar_arrive_expect_tx(b_q, (act1 ? 2u : 1u) * chunk_bytes);
      for (int c = 0; c < p.nD; ++c) {
        tma_load_5d(sQ + c * kTileChunkBytes, &tmQ, b_q, c * kChunk, qt0 * kBM, h, bi, bo);
        if (act1)
          tma_load_5d(sQ + (2 + c) * kTileChunkBytes, &tmQ, b_q, c * kChunk, qt1 * kBM, h, bi, bo);
      }
      int issued = 0;
      for (int it = 0; it < n_kv; ++it) {
        const int s = it & 1, j = j_lo + it;
        if (it >= 2 && !mbar_wait(b_kvempty(s), ((it >> 1) - 1) & 1, abort_flag)) {
          raise_error(abort_flag);
          break;
        }
        mbar_arrive_expect_tx(b_kfull(s), chunk_bytes);
        for (int c = 0; c < p.nD; ++c)
          tma_load_5d(sK + (2 * s + c) * kTileChunkBytes, &tmK, b_kfull(s), c * kChunk, j * kBN, h,
                      bi, bo);
        mbar_arrive_expect_tx(b_vfull(s), chunk_bytes);
        for (int c = 0; c < p.nD; ++c)
          tma_load_5d(sV + (2 * s + c) * kTileChunkBytes, &tmV, b_vfull(s), c * kChunk, j * kBN, h,
                      bi, bo);
        issued = it + 1;
      }
      if (*abort_flag) {
        // drain: let the copies already in flight land before the CTA exits
        for (int it = max(0, issued - 2); it < issued; ++it) {
          const int s = it & 1;
          volatile int no_abort = 0;
          mbar_wait(b_kfull(s), (it >> 1) & 1, &no_abort);
          mbar_wait(b_vfull(s), (it >> 1) & 1, &no_abort);
        }
        volatile int no_abort = 0;
        mbar_wait(b_q, 0, &no_abort);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc_qk = idesc_bf16_f32(kBM, kBN, false, false);
      const uint32_t idesc_pv = idesc_bf16_f32(kBM, p.nD * kChunk, false, true);
      auto tS = [&](int t) { return tmem + (uint32_t)(t * 128); };
      auto tO = [&](int t) { return tmem + (uint32_t)(256 + t * 128); };
      auto issue_qk = [&](int t, int s) {
        const uint32_t qa = sQ + (uint32_t)(2 * t) * kTileChunkBytes;
        const uint32_t ka = sK + (uint32_t)(2 * s) * kTileChunkBytes;
        for (int kk = 0; kk < 4 * p.nD; ++kk) {
          const uint32_t off = (uint32_t)(kk >> 2) * kTileChunkBytes + (uint32_t)(kk & 3) * 32u;
          mma_ss(tS(t), smem_desc_sw128(qa + off, 16, 1024), smem_desc_sw128(ka + off, 16, 1024),
                 idesc_qk, kk > 0 ? 1u : 0u);
        }
      };
      auto issue_pv = [&](int t, int s, bool acc) {
        const uint32_t va = sV + (uint32_t)(2 * s) * kTileChunkBytes;
        for (int kk = 0; kk < kBN / 16; ++kk)
          mma_ts(tO(t), tS(t) + (uint32_t)(kk * 8), smem_desc_sw128(va + kk * 2048u, kTileChunkBytes, 1024),
                 idesc_pv, (acc || kk > 0) ? 1u : 0u);
      };
      bool ok = mbar_wait(b_q, 0, abort_flag) && mbar_wait(b_kfull(0), 0, abort_flag);
      if (ok) {
        tc_fence_after();
        issue_qk(0, 0);
        mma_commit(b_sfull(0));
        if (act1) {
          issue_qk(1, 0);
          mma_commit(b_sfull(1));
        }
      }
      for (int it = 0; ok && it < n_kv; ++it) {
        const int s = it & 1;
        const bool more = it + 1 < n_kv;
        const int s2 = (it + 1) & 1;
        if (!(ok = mbar_wait(b_vfull(s), (it >> 1) & 1, abort_flag))) break;
        if (!(ok = mbar_wait(b_pfull(0), it & 1, abort_flag))) break;
        tc_fence_after();
        issue_pv(0, s, it > 0);
        if (more) {
          if (!(ok = mbar_wait(b_kfull(s2), ((it + 1) >> 1) & 1, abort_flag))) break;
          tc_fence_after();
          issue_qk(0, s2);
          mma_commit(b_sfull(0));
        }
        if (act1) {
          if (!(ok = mbar_wait(b_pfull(1), it & 1, abort_flag))) break;
          tc_fence_after();
          issue_pv(1, s, it > 0);
        }
        mma_commit(b_kvempty(s));
        if (more && act1) {
          issue_qk(1, s2);
          mma_commit(b_sfull(1));
        }
      }
      if (!ok) raise_error(abort_flag);
      mma_commit(b_ofull(0));
      mma_commit(b_ofull(1));
    }
  } else {
    // ------------------------------------------------------------ softmax warps
    const int t = warp >> 2;                 // query tile of this warpgroup
    const int qt = t ? qt1 : qt0;
    const int row = (warp & 3) * 32 + lane;  // TMEM lane
    const int i = qt * kBM + row;            // query index
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + (uint32_t)(t * 128);
    const uint32_t tO = tmem + lane_base + (uint32_t)(256 + t * 128);
    const int tq_lo = qt * kBM, tq_hi = min(tq_lo + kBM - 1, p.Nq - 1);
    const float sl2 = p.scale_log2;
    float m_used = -INFINITY;  // running row maximum, log2 units (scale included)
    float l = 0.f;             // running row sum relative to m_used
    bool ok = (t == 0) || act1;
    for (int it = 0; ok && it < n_kv; ++it) {
      const int k0 = (j_lo + it) * kBN;
      if (!(ok = mbar_wait(b_sfull(t), it & 1, abort_flag))) break;
      tc_fence_after();
      uint32_t s[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tS + 32u * c, s + 32 * c);
      tmem_wait_ld();
      const bool full_tile =
          (k0 + kBN <= p.Nk) &&
          (p.mask == IHA_MASK_NONE ||
           (k0 + kBN - 1 <= tq_lo &&
            (p.mask == IHA_MASK_CAUSAL || tq_hi - k0 < p.window)));
      if (!full_tile) {
#pragma unroll
        for (int e = 0; e < 128; ++e) {
          const int kj = k0 + e;
          bool vis = kj < p.Nk;
          if (p.mask != IHA_MASK_NONE) {
            vis = vis && kj <= i;
            if (p.mask == IHA_MASK_CAUSAL_WINDOW) vis = vis && (i - kj < p.window);
          }
          if (!vis) s[e] = 0xFF800000u;  // -inf
        }
      }
      // row maximum: 8 independent three-input max chains, then a small tree
      float mx[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) mx[j] = __uint_as_float(s[j]);
#pragma unroll
      for (int e = 8; e < 128; e += 16)
#pragma unroll
        for (int j = 0; j < 8; ++j)
          mx[j] = fmax3f(mx[j], __uint_as_float(s[e + j]), __uint_as_float(s[e + 8 + j]));
      const float mt = fmaxf(fmax3f(mx[0], mx[1], mx[2]), fmax3f(mx[3], mx[4], fmax3f(mx[5], mx[6], mx[7])));
      const float m_new = fmaxf(m_used, mt * sl2);
      bool rescale = false;
      float factor = 1.f;
      if (it == 0) {
        m_used = m_new;
      } else if (__any_sync(0xffffffffu, m_new > m_used + kRescaleLog2)) {
        factor = (m_new == -INFINITY) ? 1.f : fast_exp2(m_used - m_new);
        l *= factor;
        m_used = m_new;
        rescale = true;
      }
      const float base = (m_used == -INFINITY) ? 0.f : m_used;
      // P = 2^(s * scale_log2 - base), packed to bf16 pairs over the S columns
      const float2 sc2 = make_float2(sl2, sl2), nb2 = make_float2(-base, -base);
      float2 sum2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                        make_float2(0.f, 0.f)};
      uint32_t pk[64];
#pragma unroll
      for (int e = 0; e < 64; ++e) {
        const float2 xx = __ffma2_rn(
            make_float2(__uint_as_float(s[2 * e]), __uint_as_float(s[2 * e + 1])), sc2, nb2);
        const float p0 = fast_exp2(xx.x), p1 = fast_exp2(xx.y);
        sum2[e & 3] = __fadd2_rn(sum2[e & 3], make_float2(p0, p1));
        pk[e] = pack_bf16x2(p0, p1);
      }
      tmem_st32(tS, pk);
      tmem_st32(tS + 32u, pk + 32);
      const float2 s01 = __fadd2_rn(sum2[0], sum2[1]), s23 = __fadd2_rn(sum2[2], sum2[3]);
      const float2 st = __fadd2_rn(s01, s23);
      l += st.x + st.y;
      if (rescale) {
        // O <- O * factor before this tile's P.V is issued (PV of the previous
        // tile is complete: the S commit waited on above tracks it)
        uint32_t r[32];
        for (int c = 0; c < 2 * p.nD; ++c) {
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
    if ((t == 0) || act1) {
      if (ok) ok = mbar_wait(b_ofull(t), 0, abort_flag);
      if (!ok) raise_error(abort_flag);
      tc_fence_after();
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
      __nv_bfloat16* orow = p.o + bo * p.so_bo + bi * p.so_bi + (int64_t)i * p.so_seq + h * p.so_h;
      uint32_t r[128];
      tmem_ld32(tO, r);
      tmem_ld32(tO + 32u, r + 32);
      if (p.nD == 2) {
        tmem_ld32(tO + 64u, r + 64);
        tmem_ld32(tO + 96u, r + 96);
      }
      tmem_wait_ld();
      if (ok && i < p.Nq) {
#pragma unroll
        for (int g8 = 0; g8 < 16; ++g8) {
          const int f = 8 * g8;
          if (f < p.d) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(r[f + 0]) * inv_l, __uint_as_float(r[f + 1]) * inv_l);
            v.y = pack_bf16x2(__uint_as_float(r[f + 2]) * inv_l, __uint_as_float(r[f + 3]) * inv_l);
            v.z = pack_bf16x2(__uint_as_float(r[f + 4]) * inv_l, __uint_as_float(r[f + 5]) * inv_l);
            v.w = pack_bf16x2(__uint_as_float(r[f + 6]) * inv_l, __uint_as_float(r[f + 7]) * inv_l);
            *reinterpret_cast<uint4*>(orow + f) = v;
          }
        }
      }
      if (ok && p.lse && i < p.Nq) {
        const float base = (m_used == -INFINITY) ? 0.f : m_used;
        p.lse[((int64_t)bz * p.Hh + h) * p.Nq + i] =
            l > 0.f ? (base + log2f(l)) * 0.6931471805599453f : -INFINITY;
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

__global__ void __launch_bounds__(128) attn_fwd_f32_kernel(const AttnF32Params p) {
  __shared__ float ks[kF32Keys][128 + 1];
  __shared__ float vs[kF32Keys][128 + 1];
  const int quad = threadIdx.x >> 2, qi = threadIdx.x & 3;
  const int dq = p.d >> 2;  // features per thread
  const int h = blockIdx.y;
  const int bz = blockIdx.z, bo = bz / p.Bi, bi = bz - bo * p.Bi;
  const int i = blockIdx.x * kF32Rows + quad;
  const bool valid = i < p.Nq;
  float qv[32], acc[32];
  const float* qrow = p.q + bo * p.sq.b_outer + bi * p.sq.b_inner + (int64_t)min(i, p.Nq - 1) * p.sq.seq + h * p.sq.head;
  for (int e = 0; e < 32; ++e) {
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
    for (int kr = 0; kr < kF32Keys; ++kr) {
      const int kj = kb + kr;
      float dot = 0.f;
      for (int e = 0; e < dq; ++e) dot = fmaf(qv[e], ks[kr][qi * dq + e], dot);
      dot += __shfl_xor_sync(0xffffffffu, dot, 1);
      dot += __shfl_xor_sync(0xffffffffu, dot, 2);
      bool vis = kj < p.Nk;
      if (p.mask != IHA_MASK_NONE) {
        vis = vis && kj <= i;
        if (p.mask == IHA_MASK_CAUSAL_WINDOW) vis = vis && (i - kj < p.window);
      }
      if (!vis) continue;
      const float s = dot * p.scale;
      const float m_new = fmaxf(m, s);
      const float corr = expf(m - m_new);
      const float pe = expf(s - m_new);
      l = l * corr + pe;
      for (int e = 0; e < dq; ++e) acc[e] = fmaf(pe, vs[kr][qi * dq + e], acc[e] * corr);
      m = m_new;
    }
  }
  if (valid) {
    float* orow = p.o + bo * p.so.b_outer + bi * p.so.b_inner + (int64_t)i * p.so.seq + h * p.so.head;
    const float inv = l > 0.f ? 1.f / l : 0.f;
    for (int e = 0; e < dq; ++e) orow[qi * dq + e] = acc[e] * inv;
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
                  const iha_strides& s) {
  uint64_t dims[5] = {(uint64_t)d, (uint64_t)N, (uint64_t)Hh, (uint64_t)Bi, (uint64_t)Bo};
  uint64_t st[4] = {(uint64_t)s.seq * 2, (uint64_t)s.head * 2, (uint64_t)s.b_inner * 2,
                    (uint64_t)s.b_outer * 2};
  if (N == 1) st[0] = 16;
  if (Hh == 1) st[1] = 16;
  if (Bi == 1) st[2] = 16;
  if (Bo == 1) st[3] = 16;
  uint32_t box[5] = {(uint32_t)kChunk, (uint32_t)kBM, 1, 1, 1};
  return encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, st, box,
                      CU_TENSOR_MAP_SWIZZLE_128B);
}

iha_status launch_tc(const void* q, const void* k, const void* v, void* o, float* lse, int Bo,
                     int Bi, int Hh, int Nq, int Nk, int d, const iha_strides& sq,
                     const iha_strides& sk, const iha_strides& sv, const iha_strides& so,
                     float scale, int mask, int window, cudaStream_t stream) {
  CUtensorMap mq, mk, mv;
  if (make_map(&mq, q, Bo, Bi, Nq, Hh, d, sq) != CUDA_SUCCESS ||
      make_map(&mk, k, Bo, Bi, Nk, Hh, d, sk) != CUDA_SUCCESS ||
      make_map(&mv, v, Bo, Bi, Nk, Hh, d, sv) != CUDA_SUCCESS)
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
  p.n_qpairs = ((Nq + kBM - 1) / kBM + 1) / 2;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.so_bo = so.b_outer;
  p.so_bi = so.b_inner;
  p.so_seq = so.seq;
  p.so_h = so.head;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    if (cudaFuncSetAttribute(attn_fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes) != cudaSuccess)
      return check_launch("mha_fwd (smem attribute)");
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  dim3 grid(Hh, Bo * Bi, p.n_qpairs);
  attn_fwd_tc_kernel<<<grid, kThreads, kSmemBytes, stream>>>(mq, mk, mv, p);
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
  if (Hh > 65535 || (int64_t)B_outer * B_inner > 65535)
    return fail(IHA_ERR_UNSUPPORTED, "mha_fwd: too many heads or batches for one launch");
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
  attn_fwd_f32_kernel<<<grid, 128, 0, s>>>(p);
  return check_launch("mha_fwd");
}
