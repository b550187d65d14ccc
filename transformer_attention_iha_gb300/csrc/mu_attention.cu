// Softmax attention over short independent sequences: Hiera mask units.
//
// "hiera-optim 0.1.0", hiera_optim/attention/mask_unit.py,
// MaskUnitAttentionFast.forward: unmasked softmax attention inside each mask
// unit (64 tokens of an 8x8 unit at stage 1), scale head_dim ** -0.5, one
// (unit, head) pair per independent attention problem.
//
// A unit has T <= 64 tokens, so two units share one 128-row tile:
//   S = Q K^T with M = 128 (rows 0-63: unit a, 64-127: unit b) and N = 128
//   keys (0-63: unit a, 64-127: unit b); each row reads only its own unit's
//   64 key columns from TMEM.  P is written block-diagonal (its own unit's
//   keys, zeros for the other unit's), so one P.V MMA over 128 keys gives
//   both units' O without mixing them.
// Persistent: one CTA per SM walks unit pairs; Q, K and V of a pair arrive
// by TMA into one of two shared-memory stages (64-row boxes, 128-byte
// swizzle), S and O are double-buffered in TMEM, and the softmax warps of
// the two buffers alternate, so loads, MMAs and softmax of consecutive pairs
// overlap.  The op is HBM-bound (32 flop per byte at d = 96).
//   warps 0-3  softmax + epilogue of even pairs (TMEM buffer 0)
//   warps 4-7  softmax + epilogue of odd pairs (TMEM buffer 1)
//   warp  8    TMA producer,  warp 9  MMA issuer and TMEM owner
//
// Pooled queries (q_stride > 1; "hiera-optim 0.1.0", mask_unit.py,
// MaskUnitAttentionFast.forward, the q_pool of a pooling block): a unit's T
// query rows are q_stride blocks of Tq = T / q_stride rows (the block index
// the slow axis), and the attention uses their elementwise maximum, Tq
// queries over all T keys.  The pooling runs in the Q tile as it arrives:
// the softmax warps of the pair's buffer take, for each pooled row t, the
// maximum of rows t, Tq + t, ... and write it over row t (rows above Tq are
// only read), then release the tile to the QK^T MMA; rows t >= Tq of S are
// never stored.
//
// Fused mode (FUSED = true): the Hiera stage-1 step gather -> attention ->
// scatter ("hiera-optim 0.1.0", README, item 2 of what optimize(model) does,
// and MaskUnitAttentionFast.forward) as one pass.  A kept unit is read
// straight from the token grid x [B, grid_h, grid_w, C] by one 4-D TMA box
// (C / 64 chunks x mu_w x mu_h x 1): the box's rows arrive in the in-unit
// order t = ty * mu_w + tx, the unit layout the gather would have written.
// The one tile serves as Q, K and V, and each output row goes to its token
// of the decoder canvas [B, grid_h * grid_w, C], as the scatter would have
// put it; the gathered units never exist in HBM.
#include <math.h>

#include <mutex>

#include "common.cuh"
#include "mu_attention.h"

namespace iha {
namespace {

IHA_DEVICE_ERROR_WORD(mu_attention)

constexpr int kRows = 64;                    // rows (and keys) per unit half
constexpr int kChunkBytes = 128 * 128;       // one 64-wide d chunk of a 128-row tile
constexpr int kHalfBytes = kRows * 128;      // one unit's rows of a chunk (8 KB)
constexpr int kTensorBytes = 2 * kChunkBytes;  // up to d = 128
constexpr int kStageBytes = 3 * kTensorBytes;  // Q, K, V
constexpr int kThreads = 320;
constexpr int kSmemBytes = 2 * kStageBytes + 256 + 1024;
static_assert(kSmemBytes <= 227 * 1024, "mask-unit attention: over the per-block shared memory limit");

struct MuParams {
  int Bo, Bi, Hh, T, d, nch, ksteps, npv;
  int q_stride, Tq;  // pooled queries: Tq = T / q_stride rows stored per unit
  int n_units, n_items;
  float scale_log2;
  int64_t so_bo, so_bi, so_seq, so_h;
  __nv_bfloat16* o;
  float* lse;
  // fused mode: unit U = (sample U / n_keep, kept unit keep[U]) of the grid
  const int32_t* keep;
  int n_keep, grid_units, units_per_row, mu_h, mu_w, grid_w, B;
  int64_t G;  // tokens per sample
};

// Grid coordinates of kept unit U (fused mode); valid = a unit of a sample
// whose kept-unit id is in range.
struct GridUnit {
  int b, x0, y0;
  bool exists, valid;
};
__device__ __forceinline__ GridUnit grid_unit(const MuParams& p, int U) {
  GridUnit g;
  g.exists = U < p.n_units;
  const int UU = g.exists ? U : 0;
  const int id = __ldg(p.keep + UU);
  g.valid = g.exists && id >= 0 && id < p.grid_units;
  const int uid = g.valid ? id : 0;
  const int uy = uid / p.units_per_row, ux = uid - uy * p.units_per_row;
  g.b = UU / p.n_keep;
  g.x0 = ux * p.mu_w;
  g.y0 = uy * p.mu_h;
  return g;
}

struct UnitRef {
  int h, bo, bi, bz;
  bool valid;
};

__device__ __forceinline__ UnitRef unit_ref(const MuParams& p, int u) {
  UnitRef r;
  r.valid = u < p.n_units;
  const int uu = r.valid ? u : 0;
  r.h = uu % p.Hh;
  r.bz = uu / p.Hh;
  r.bo = r.bz / p.Bi;
  r.bi = r.bz - r.bo * p.Bi;
  return r;
}

__device__ __forceinline__ void raise_error(volatile int* abort_flag) {
  *abort_flag = 1;
  atomicOr(&g_dev_error, DEV_ERR_WAIT_TIMEOUT);
}

template <bool FUSED>
__global__ void __launch_bounds__(kThreads, 1)
    mu_attn_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const MuParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  // load stages: Q, K, V of a pair each (2 stages); fused, one tile serves
  // all three, so the same memory holds 6 stages and loads run further ahead
  constexpr int NS = FUSED ? 6 : 2;
  constexpr uint32_t kSStride = FUSED ? (uint32_t)kTensorBytes : (uint32_t)kStageBytes;
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 2 * kStageBytes);
  const uint32_t bar0 = smem_u32(bars);
  auto b_qkfull = [&](int s) { return bar0 + 8u * (0 + s); };
  auto b_vfull = [&](int s) { return bar0 + 8u * (NS + s); };
  auto b_sempty = [&](int s) { return bar0 + 8u * (2 * NS + s); };
  auto b_sfull = [&](int b) { return bar0 + 8u * (3 * NS + b); };
  auto b_pfull = [&](int b) { return bar0 + 8u * (3 * NS + 2 + b); };
  auto b_ofull = [&](int b) { return bar0 + 8u * (3 * NS + 4 + b); };
  auto b_oempty = [&](int b) { return bar0 + 8u * (3 * NS + 6 + b); };
  const uint32_t b_drain = bar0 + 8u * (3 * NS + 8);
  auto b_qpool = [&](int s) { return bar0 + 8u * (3 * NS + 10 + s); };  // Q of stage s pooled
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 3 * NS + 10 + (FUSED ? 0 : NS));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // barriers, then the TMEM address and the abort flag, in the 256 bytes
  static_assert(8 * (3 * NS + 10 + (FUSED ? 0 : NS)) + 4 + 4 <= 256,
                "mask-unit attention: barrier region");

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_my = (p.n_items - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(b_qkfull(s), 1);
      mbar_init(b_vfull(s), 1);
      mbar_init(b_sempty(s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(b_sfull(s), 1);
      mbar_init(b_pfull(s), 128);
      mbar_init(b_ofull(s), 1);
      mbar_init(b_oempty(s), 128);
    }
    mbar_init(b_drain, 1);
    if (!FUSED)
      for (int s = 0; s < NS; ++s) mbar_init(b_qpool(s), 128);
    *abort_flag = 0;
    mbar_init_fence();
  }
  const bool pool = !FUSED && p.q_stride > 1;
  if (FUSED && p.T < kRows) {
    // a unit box fills rows 0 .. T-1 of its half; rows T .. 63 are V rows of
    // keys whose P is 0, so they must hold finite values: zero them once
    for (int i = threadIdx.x; i < NS * kTensorBytes / 16; i += kThreads)
      reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
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
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      const uint32_t box_bytes = (uint32_t)p.nch * 2u * kHalfBytes;  // one tensor, both units
      bool ok = true;
      int k = 0;
      // both units' rows of one tensor; a missing second unit is read from an
      // out-of-range batch coordinate, which TMA fills with zeros
      auto load_tensor = [&](const CUtensorMap* map, uint32_t dst, uint32_t bar, int item) {
        for (int u = 0; u < 2; ++u) {
          const UnitRef r = unit_ref(p, 2 * item + u);
          const int bo = r.valid ? r.bo : p.Bo;  // one past the last batch: zeros
          for (int c = 0; c < p.nch; ++c)
            tma_load_5d(dst + (uint32_t)c * kChunkBytes + (uint32_t)u * kHalfBytes, map, bar,
                        c * 64, 0, r.h, r.bi, bo);
        }
      };
      for (; k < n_my; ++k) {
        const int item = blockIdx.x + k * gridDim.x, s = k % NS;
        if (k >= NS && !(ok = mbar_wait(b_sempty(s), ((k / NS) - 1) & 1, abort_flag))) break;
        const uint32_t st = sbase + (uint32_t)s * kSStride;
        if constexpr (FUSED) {
          // one tile of both units is Q, K and V; a missing or invalid unit
          // is read from an out-of-range sample, which TMA fills with zeros
          mbar_arrive_expect_tx(b_qkfull(s), (uint32_t)p.nch * 2u * (uint32_t)p.T * 128u);
          for (int u = 0; u < 2; ++u) {
            const GridUnit g = grid_unit(p, 2 * item + u);
            for (int c = 0; c < p.nch; ++c)
              tma_load_4d(st + (uint32_t)c * kChunkBytes + (uint32_t)u * kHalfBytes, &tmQ,
                          b_qkfull(s), c * 64, g.x0, g.y0, g.valid ? g.b : p.B);
          }
          mbar_arrive(b_vfull(s));  // V is the same tile: ordered behind Q K^T
        } else {
          mbar_arrive_expect_tx(b_qkfull(s), 2 * box_bytes);
          load_tensor(&tmQ, st, b_qkfull(s), item);
          load_tensor(&tmK, st + kTensorBytes, b_qkfull(s), item);
          mbar_arrive_expect_tx(b_vfull(s), box_bytes);
          load_tensor(&tmV, st + 2 * kTensorBytes, b_vfull(s), item);
        }
      }
      if (!ok) raise_error(abort_flag);
      // no copy may still be landing when the CTA exits
      volatile int no_abort = 0;
      for (int kk = k - NS > 0 ? k - NS : 0; kk < k; ++kk) {
        mbar_wait(b_qkfull(kk % NS), (kk / NS) & 1, &no_abort);
        mbar_wait(b_vfull(kk % NS), (kk / NS) & 1, &no_abort);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the schedule; one elected lane issues (see elect_one).
    {
      const uint32_t idesc_qk = idesc_bf16_f32(128, 128, false, false);
      const uint32_t idesc_pv = idesc_bf16_f32(128, p.npv, false, true);
      bool ok = true;
      auto issue_qk = [&](int k) {
        const int s = k % NS, b = k & 1;
        const uint32_t st = sbase + (uint32_t)s * kSStride;
        const uint64_t dq = smem_desc_sw128(st, 16, 1024);
        const uint64_t dk = smem_desc_sw128(FUSED ? st : st + kTensorBytes, 16, 1024);
        if (elect_one())
          for (int kk = 0; kk < p.ksteps; ++kk) {
            const uint64_t off = (uint64_t)(((kk >> 2) * kChunkBytes + (kk & 3) * 32) >> 4);
            mma_ss_nm(tmem + (uint32_t)(256 * b), dq + off, dk + off, idesc_qk, kk > 0 ? 1u : 0u);
          }
        __syncwarp();
        mma_commit_warp(b_sfull(b));
      };
      auto ready_qk = [&](int k) {
        const int b = k & 1;
        if (!(ok = mbar_wait_warp(b_qkfull(k % NS), (k / NS) & 1, abort_flag))) return false;
        if (pool && !(ok = mbar_wait_warp(b_qpool(k % NS), (k / NS) & 1, abort_flag))) return false;
        // S / O of buffer b are free once the epilogue of pair k - 2 has read O
        if (k >= 2 && !(ok = mbar_wait_warp(b_oempty(b), ((k >> 1) - 1) & 1, abort_flag))) return false;
        tc_fence_after();
        return true;
      };
      if (n_my > 0 && ready_qk(0)) issue_qk(0);
      for (int k = 0; ok && k < n_my; ++k) {
        const int s = k % NS, b = k & 1;
        if (k + 1 < n_my) {
          if (!ready_qk(k + 1)) break;
          issue_qk(k + 1);
        }
        if (!(ok = mbar_wait_warp(b_vfull(s), (k / NS) & 1, abort_flag))) break;
        if (!(ok = mbar_wait_warp(b_pfull(b), (k >> 1) & 1, abort_flag))) break;
        tc_fence_after();
        const uint64_t dv = smem_desc_sw128(
            sbase + (uint32_t)s * kSStride + (FUSED ? 0u : 2u * kTensorBytes), kChunkBytes, 1024);
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ts_nm(tmem + (uint32_t)(256 * b + 128), tmem + (uint32_t)(256 * b + kk * 8),
                      dv + (uint64_t)(kk * 128), idesc_pv, kk > 0 ? 1u : 0u);
        }
        __syncwarp();
        mma_commit_warp(b_ofull(b));
        mma_commit_warp(b_sempty(s));
      }
      if (!ok) raise_error(abort_flag);
      mma_drain_warp(b_drain);
    }
  } else {
    // ------------------------------------------------------------ softmax warps
    const int b = warp >> 2, q = warp & 3;
    const int row = q * 32 + lane;  // TMEM lane
    const int u = q >> 1;           // unit half of this row
    const int r = row & (kRows - 1);
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    const uint32_t tS = tmem + lane_base + (uint32_t)(256 * b);
    const uint32_t tO = tS + 128u;
    const float sl2 = p.scale_log2;
    bool ok = true;
    int n = 0;  // pairs of this buffer so far
    for (int k = b; k < n_my; k += 2, ++n) {
      const int item = blockIdx.x + k * gridDim.x;
      if (pool) {
        // q_pool of both units' Q in the stage, 16 bytes (8 features) per step
        const int s = k % NS;
        if (!(ok = mbar_wait_warp(b_qkfull(s), (k / NS) & 1, abort_flag))) break;
        uint8_t* st = smem + (uint32_t)s * kSStride;
        const int n_work = 2 * p.Tq * p.nch * 8;
        for (int w = row; w < n_work; w += 128) {
          const int g = w & 7, c = (w >> 3) % p.nch, rest = (w >> 3) / p.nch;
          const int t = rest % p.Tq, uu = rest / p.Tq;
          uint8_t* base = st + c * kChunkBytes + uu * kHalfBytes + ((g ^ (t & 7)) << 4);
          uint4 acc = *reinterpret_cast<const uint4*>(base + t * 128);
          for (int i = 1; i < p.q_stride; ++i) {
            const int rr = i * p.Tq + t;
            const uint4 x = *reinterpret_cast<const uint4*>(
                st + c * kChunkBytes + uu * kHalfBytes + rr * 128 + ((g ^ (rr & 7)) << 4));
            acc.x = bf16x2_max(acc.x, x.x);
            acc.y = bf16x2_max(acc.y, x.y);
            acc.z = bf16x2_max(acc.z, x.z);
            acc.w = bf16x2_max(acc.w, x.w);
          }
          *reinterpret_cast<uint4*>(base + t * 128) = acc;
        }
        fence_proxy_async_smem();
        mbar_arrive(b_qpool(s));
      }
      const bool live = ok && mbar_wait_warp(b_sfull(b), n & 1, abort_flag);
      if (!live) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t s[64];
      tmem_ld32(tS + 64u * u, s);
      tmem_ld32(tS + 64u * u + 32u, s + 32);
      tmem_wait_ld();
      if (p.T < kRows) {
#pragma unroll
        for (int e = 0; e < 64; ++e) s[e] = sel_u32(e >= p.T, 0xFF800000u, s[e]);
      }
      // chain qq takes columns qq, qq + 4, ...: 0-3 to start, two more per
      // step over 4-59, and 60-63 last
      float mx[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) mx[e] = __uint_as_float(s[e]);
#pragma unroll
      for (int e = 4; e < 60; e += 8)
#pragma unroll
        for (int qq = 0; qq < 4; ++qq)
          mx[qq] = fmax3f(mx[qq], __uint_as_float(s[e + qq]), __uint_as_float(s[e + 4 + qq]));
#pragma unroll
      for (int qq = 0; qq < 4; ++qq) mx[qq] = fmaxf(mx[qq], __uint_as_float(s[60 + qq]));
      const float m = fmaxf(fmax3f(mx[0], mx[1], mx[2]), mx[3]) * sl2;
      const float2 sc2 = make_float2(sl2, sl2), nb2 = make_float2(-m, -m);
      float2 sum2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
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
      // own keys' P in columns 32u.., zeros for the other unit's keys
      tmem_st32(tS + 32u * u, pk);
#pragma unroll
      for (int e = 0; e < 32; ++e) pk[e] = 0u;
      tmem_st32(tS + 32u * (1 - u), pk);
      const float2 st = __fadd2_rn(sum2[0], sum2[1]);
      const float l = st.x + st.y;
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(b_pfull(b));
      // ---------------------------------------------------------- epilogue
      if (!(ok = mbar_wait_warp(b_ofull(b), n & 1, abort_flag))) break;
      tc_fence_after();
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
      bool store;
      __nv_bfloat16* orow;
      UnitRef ur;
      if constexpr (FUSED) {
        // row r of the unit goes to its token of the canvas
        const GridUnit g = grid_unit(p, 2 * item + u);
        if (g.exists && !g.valid && r == 0) atomicOr(&g_dev_error, DEV_ERR_KEEP_INDEX);
        store = g.valid && r < p.T;
        const int rr = min(r, p.T - 1), ty = rr / p.mu_w, tx = rr - ty * p.mu_w;
        const int64_t tok = (int64_t)g.b * p.G + (int64_t)(g.y0 + ty) * p.grid_w + g.x0 + tx;
        orow = p.o + tok * p.d;
        ur.valid = false;
      } else {
        ur = unit_ref(p, 2 * item + u);
        store = ur.valid && r < p.Tq;
        orow = p.o + ur.bo * p.so_bo + ur.bi * p.so_bi + (int64_t)min(r, p.Tq - 1) * p.so_seq +
               ur.h * p.so_h;
      }
      for (int c = 0; c < p.npv; c += 32) {
        uint32_t v[32];
        tmem_ld32(tO + (uint32_t)c, v);
        tmem_wait_ld();
        if (store) {
#pragma unroll
          for (int g8 = 0; g8 < 4; ++g8) {
            const int f = c + 8 * g8;
            if (f < p.d) {
              uint4 w;
              w.x = pack_bf16x2(__uint_as_float(v[8 * g8 + 0]) * inv_l, __uint_as_float(v[8 * g8 + 1]) * inv_l);
              w.y = pack_bf16x2(__uint_as_float(v[8 * g8 + 2]) * inv_l, __uint_as_float(v[8 * g8 + 3]) * inv_l);
              w.z = pack_bf16x2(__uint_as_float(v[8 * g8 + 4]) * inv_l, __uint_as_float(v[8 * g8 + 5]) * inv_l);
              w.w = pack_bf16x2(__uint_as_float(v[8 * g8 + 6]) * inv_l, __uint_as_float(v[8 * g8 + 7]) * inv_l);
              *reinterpret_cast<uint4*>(orow + f) = w;
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(b_oempty(b));
      if (!FUSED && store && p.lse)
        p.lse[((int64_t)ur.bz * p.Hh + ur.h) * p.Tq + r] =
            l > 0.f ? (m + log2f(l)) * 0.6931471805599453f : -INFINITY;
    }
    if (!ok) raise_error(abort_flag);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// 5-D tensor map over a [Bo, Bi, T, Hh, d] bf16 view, box 64 x 64 rows,
// 128-byte swizzle (size-1 dimensions get a harmless aligned stride).
CUresult make_unit_map(CUtensorMap* m, const void* base, int Bo, int Bi, int T, int Hh, int d,
                       const iha_strides& s) {
  uint64_t dims[5] = {(uint64_t)d, (uint64_t)T, (uint64_t)Hh, (uint64_t)Bi, (uint64_t)Bo};
  uint64_t st[4] = {(uint64_t)s.seq * 2, (uint64_t)s.head * 2, (uint64_t)s.b_inner * 2,
                    (uint64_t)s.b_outer * 2};
  if (T == 1) st[0] = 16;
  if (Hh == 1) st[1] = 16;
  if (Bi == 1) st[2] = 16;
  if (Bo == 1) st[3] = 16;
  uint32_t box[5] = {64, (uint32_t)kRows, 1, 1, 1};
  return encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, st,
                      box, CU_TENSOR_MAP_SWIZZLE_128B);
}

SmemLimit g_mu_limit[2];

// Dynamic shared memory limit of both instantiations on the current device
// (set on the device's first launch, thread-safe).
cudaError_t set_mu_attributes() {
  cudaError_t e = g_mu_limit[0].ensure(mu_attn_kernel<false>, kSmemBytes);
  if (e == cudaSuccess) e = g_mu_limit[1].ensure(mu_attn_kernel<true>, kSmemBytes);
  return e;
}

}  // namespace

bool mu_attention_supported(int Nq, int Nk, int d, int mask) {
  return mask == IHA_MASK_NONE && Nq == Nk && Nq <= kRows && d <= 128;
}

iha_status mu_attention_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                            int Bo, int Bi, int Hh, int T, int d, const iha_strides& sq,
                            const iha_strides& sk, const iha_strides& sv, const iha_strides& so,
                            float scale, cudaStream_t stream, int q_stride) {
  CUtensorMap mq, mk, mv;
  if (make_unit_map(&mq, q, Bo, Bi, T, Hh, d, sq) != CUDA_SUCCESS ||
      make_unit_map(&mk, k, Bo, Bi, T, Hh, d, sk) != CUDA_SUCCESS ||
      make_unit_map(&mv, v, Bo, Bi, T, Hh, d, sv) != CUDA_SUCCESS)
    return fail(IHA_ERR_CUDA, "mha_fwd: tensor map encoding failed");
  MuParams p;
  p.Bo = Bo;
  p.Bi = Bi;
  p.Hh = Hh;
  p.T = T;
  p.d = d;
  p.q_stride = q_stride;
  p.Tq = T / q_stride;
  p.nch = (d + 63) / 64;
  p.ksteps = (d + 15) / 16;
  p.npv = p.ksteps * 16;
  const int64_t units = (int64_t)Bo * Bi * Hh;
  p.n_units = (int)units;
  p.n_items = (int)((units + 1) / 2);
  p.scale_log2 = scale * 1.4426950408889634f;
  p.so_bo = so.b_outer;
  p.so_bi = so.b_inner;
  p.so_seq = so.seq;
  p.so_h = so.head;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  const cudaError_t attr_err = set_mu_attributes();
  if (attr_err != cudaSuccess)
    return fail(IHA_ERR_CUDA, "mha_fwd (smem attribute): %s", cudaGetErrorString(attr_err));
  int grid = sm_count();
  if (grid > p.n_items) grid = p.n_items;
  mu_attn_kernel<false><<<grid, kThreads, kSmemBytes, stream>>>(mq, mk, mv, p);
  return check_launch("mha_fwd");
}

iha_status mu_attention_fused(const void* x, const int32_t* keep, void* canvas, int B, int grid_h,
                              int grid_w, int mu_h, int mu_w, int n_keep, int C, float scale,
                              cudaStream_t stream) {
  // x as [B][grid_h][grid_w][C]: box = 64 channels x mu_w x mu_h x 1 sample
  CUtensorMap mx;
  {
    uint64_t dims[4] = {(uint64_t)C, (uint64_t)grid_w, (uint64_t)grid_h, (uint64_t)B};
    uint64_t st[3] = {(uint64_t)C * 2, (uint64_t)grid_w * C * 2, (uint64_t)grid_h * grid_w * C * 2};
    uint32_t box[4] = {64, (uint32_t)mu_w, (uint32_t)mu_h, 1};
    if (encode_tiled(&mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(x), dims, st,
                     box, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return fail(IHA_ERR_CUDA, "mu_attention_fused: tensor map encoding failed");
  }
  MuParams p;
  p.Bo = B;
  p.Bi = 1;
  p.Hh = 1;
  p.T = mu_h * mu_w;
  p.q_stride = 1;
  p.Tq = p.T;
  p.d = C;
  p.nch = (C + 63) / 64;
  p.ksteps = (C + 15) / 16;
  p.npv = p.ksteps * 16;
  p.n_units = B * n_keep;
  p.n_items = (p.n_units + 1) / 2;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.so_bo = p.so_bi = p.so_seq = p.so_h = 0;
  p.o = static_cast<__nv_bfloat16*>(canvas);
  p.lse = nullptr;
  p.keep = keep;
  p.n_keep = n_keep;
  p.units_per_row = grid_w / mu_w;
  p.grid_units = (grid_h / mu_h) * p.units_per_row;
  p.mu_h = mu_h;
  p.mu_w = mu_w;
  p.grid_w = grid_w;
  p.B = B;
  p.G = (int64_t)grid_h * grid_w;
  const cudaError_t attr_err = set_mu_attributes();
  if (attr_err != cudaSuccess)
    return fail(IHA_ERR_CUDA, "mu_attention_fused (smem attribute): %s",
                cudaGetErrorString(attr_err));
  int grid = sm_count();
  if (grid > p.n_items) grid = p.n_items;
  mu_attn_kernel<true><<<grid, kThreads, kSmemBytes, stream>>>(mx, mx, mx, p);
  return check_launch("mu_attention_fused");
}

}  // namespace iha
