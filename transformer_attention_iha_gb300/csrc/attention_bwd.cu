// Multi-head softmax attention backward over the pseudo-heads.
//
// "IHA-CUDA: Interleaved Head Attention Kernels for Hopper GPUs", section
// "Repository Structure" (a preprocess, the backward proper and a
// postprocess) and section "End-to-End Training Benchmark" (the training
// step these gradients belong to).  With P = softmax(scale Q K^T) under the
// causal / window / no mask and dO the gradient of O = P V:
//   D_i  = sum_f dO_if O_if            (= sum_j P_ij dP_ij)
//   dP   = dO V^T,   dS = P o (dP - D)
//   dV   = P^T dO,   dK = scale dS^T Q,   dQ = scale dS K.
// P is recomputed from the forward's LSE: P_ij = exp(scale q_i.k_j - lse_i).
//
// Three launches on the caller's stream, with a caller-owned workspace:
//   attn_bwd_pre_kernel   D and lse * log2(e) per query row (rows padded to
//                         128), and dQ_acc (fp32) zeroed;
//   attn_bwd_tc_kernel    persistent, one CTA per SM; a work item is one
//                         128-key tile of one head and loops over the query
//                         tiles that see it (causal / window block skipping);
//                         CTA b starts on item b and takes every further item
//                         from a global counter (longest items first):
//                           S^T  = K Q^T,  dP^T = V dO^T      (TMEM)
//                           P^T, dS^T by 4 compute warps (thread = key),
//                           fp32 P kept over S^T in TMEM for dS
//                           dV += P^T dO,  dK += dS^T Q        (TMEM)
//                           dQ^T = K^T dS^T -> TMA reduce-add into dQ_acc
//   attn_bwd_post_kernel  dQ = bf16(scale dQ_acc).
// Roles of the main kernel (320 threads):
//   warps 0-7  P^T and dS^T (thread = key row = TMEM lane; warps w and w + 4
//              share the lanes and take query columns 0-63 / 64-127), dK / dV
//              epilogue (feature columns split the same way)
//   warps 8-11 dQ^T drain (thread = feature = TMEM lane): staged in the tile's
//              Q / dO stage (queries 0-63 in the Q half, 64-127 in the dO
//              half), added into dQ_acc by two TMA reduce-adds a tile; each
//              half goes back to the producer once its reduction has read it
//   warp  12   TMA producer (K, V once per item; Q, dO per query tile, 2 stages,
//              Q and dO each with their own full / empty barriers)
//   warp  13   tcgen05.mma issuer and TMEM owner
// TMEM (512 columns): regions R0 | R1 rotate S^T / dP^T / dQ^T between query
// tiles; dK at 256, dV at 384.  One shared 128 x 128 bf16 tile holds P^T,
// then (in place, once dV has read it) dS^T: rows = keys, 64-query chunks,
// 128-byte swizzle, so it is both the K-major A operand of dV / dK and the
// MN-major B operand of dQ^T.
#include <math.h>

#include <mutex>

#include "common.cuh"

namespace iha {
namespace {

IHA_DEVICE_ERROR_WORD(attention_bwd)
IHA_WORK_QUEUE(attention_bwd)

constexpr int kB = 128;                      // keys (and queries) per tile
constexpr int kChunkB = kB * 128;            // one 64-wide chunk of a 128-row tile (16 KB)
constexpr int kTileB = 2 * kChunkB;          // a 128 x 128 bf16 tile (32 KB)
constexpr int kThreads = 448;
constexpr int kCompute = 256;  // threads of warps 0-7
// shared memory: K | V | Q[2] | dO[2] | P/dS tiles | lse2, D per Q stage |
// barriers.  No alignment slack fits: the dynamic shared memory must start
// 1024-byte aligned (it does when the kernel has no static shared memory);
// a kernel that finds otherwise reports DEV_ERR_SMEM_ALIGN and does nothing.
constexpr int kSmemTiles = 7 * kTileB;
constexpr int kLDBytes = 2 * 2 * kB * 4;  // 2 stages x (lse2, D) x 128 floats
constexpr int kSmemBytes = kSmemTiles + kLDBytes + 512;
static_assert(kSmemBytes <= 227 * 1024, "attention backward: over the per-block shared memory limit");

struct BwdParams {
  int B, Hh, N, d, Npad, ksteps, nch;
  int mask, window;
  int n_kt, n_qt, n_hb, group, n_items;
  float scale, scale_log2;
  const float* lse2;   // [B*Hh][Npad]  lse * log2(e)
  const float* Dv;     // [B*Hh][Npad]  rowsum(dO o O)
  float* dq_acc;       // [B, N, Hh, d] fp32
  __nv_bfloat16* dk;   // [B, N, Hh, d]
  __nv_bfloat16* dv;
  int work_slot;  // counter pair of this launch (dynamic item distribution)
};

struct Item {
  int h, b, hb, jt;
  int qlo, qhi;  // query tiles that see key tile jt
};

__device__ __forceinline__ Item decode_item(const BwdParams& p, int idx) {
  const int per_group = p.group * p.n_kt;
  const int n_groups = (p.n_hb + p.group - 1) / p.group;
  const int g = min(idx / per_group, n_groups - 1);
  const int hb0 = g * p.group;
  const int gs = min(p.group, p.n_hb - hb0);
  const int r = idx - g * per_group;
  const int rank = r / gs;
  Item it;
  it.hb = hb0 + (r - rank * gs);
  it.h = it.hb % p.Hh;
  it.b = it.hb / p.Hh;
  it.jt = rank;  // ascending: the longest query ranges (causal) first
  if (p.mask == IHA_MASK_NONE) {
    it.qlo = 0;
    it.qhi = p.n_qt - 1;
  } else {
    it.qlo = it.jt;
    it.qhi = p.n_qt - 1;
    if (p.mask == IHA_MASK_CAUSAL_WINDOW)
      it.qhi = min(it.qhi, (it.jt * kB + kB - 1 + p.window - 1) / kB);
  }
  return it;
}

__device__ __forceinline__ void raise_error(volatile int* abort_flag) {
  *abort_flag = 1;
  atomicOr(&g_dev_error, DEV_ERR_WAIT_TIMEOUT);
}

// byte offset of 16-byte granule g (8 bf16) of row r in chunk c of a
// 128-byte-swizzled 128-row tile
__device__ __forceinline__ uint32_t swz(int c, int r, int g) {
  return (uint32_t)(c * kChunkB + r * 128 + ((g ^ (r & 7)) << 4));
}

__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                       const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV,
                       const __grid_constant__ CUtensorMap tmDO,
                       const __grid_constant__ CUtensorMap tmDQ, const BwdParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if ((smem_u32(smem_raw) & 1023u) != 0) {  // uniform: every thread leaves here
    if (threadIdx.x == 0) atomicOr(&g_dev_error, DEV_ERR_SMEM_ALIGN);
    return;
  }
  uint8_t* smem = smem_raw;
  const uint32_t sK = smem_u32(smem);
  const uint32_t sV = sK + kTileB;
  // 2 stages of Q | dO, each stage 64 KB contiguous (the dQ^T staging area)
  const uint32_t sQ = sV + kTileB;           // Q of stage s at sQ + 2 s kTileB
  const uint32_t sDO = sQ + kTileB;          // dO of stage s at sDO + 2 s kTileB
  const uint32_t sPS = sQ + 4 * kTileB;      // P^T, then dS^T
  uint8_t* ps = smem + (sPS - sK);
  const uint32_t sLD = sK + kSmemTiles;      // [stage][lse2 | D][128] fp32
  const float* ld_f = reinterpret_cast<const float*>(smem + kSmemTiles);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kSmemTiles + kLDBytes);
  const uint32_t bar0 = smem_u32(bars);
  const uint32_t b_kvfull = bar0, b_kvempty = bar0 + 8u;
  auto b_qfull = [&](int s) { return bar0 + 8u * (2 + s); };
  auto b_qempty = [&](int s) { return bar0 + 8u * (4 + s); };
  const uint32_t b_sfull = bar0 + 8u * 6, b_dpfull = bar0 + 8u * 7, b_ptfull = bar0 + 8u * 8;
  const uint32_t b_dvdone = bar0 + 8u * 9, b_dsfull = bar0 + 8u * 10, b_psfree = bar0 + 8u * 11;
  auto b_dqfull = [&](int r) { return bar0 + 8u * (12 + r); };
  auto b_dqempty = [&](int r) { return bar0 + 8u * (14 + r); };
  const uint32_t b_kvout = bar0 + 8u * 16, b_kvoutempty = bar0 + 8u * 17;
  const uint32_t b_drain = bar0 + 8u * 18, b_stg = bar0 + 8u * 19;
  // item ring (4 entries): the producer publishes the index of each item it
  // starts; the MMA, compute and drain warps take them in order
  auto b_ifull = [&](int s) { return bar0 + 8u * (20 + s); };
  auto b_iempty = [&](int s) { return bar0 + 8u * (24 + s); };
  // dO has its own full / empty pair: the two halves of a stage are handed
  // back separately (Q once the first half of dQ^T has been reduced from it,
  // dO once the second half has)
  auto b_dofull = [&](int s) { return bar0 + 8u * (28 + s); };
  auto b_doempty = [&](int s) { return bar0 + 8u * (30 + s); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 32);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* item_ring = reinterpret_cast<volatile int*>(tmem_slot + 2);
  unsigned int* work = g_work[p.work_slot];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t tile_bytes = (uint32_t)p.nch * kChunkB;

  if (threadIdx.x == 0) {
    mbar_init(b_kvfull, 1);
    mbar_init(b_kvempty, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(b_qfull(s), 1);
      mbar_init(b_qempty(s), 1);  // the first dQ reduction has read the Q half
      mbar_init(b_dofull(s), 1);
      mbar_init(b_doempty(s), 1);  // the second one has read the dO half
      mbar_init(b_dqfull(s), 1);
      mbar_init(b_dqempty(s), 128);
    }
    mbar_init(b_sfull, 1);
    mbar_init(b_dpfull, 1);
    mbar_init(b_ptfull, kCompute);
    mbar_init(b_dvdone, 1);
    mbar_init(b_dsfull, kCompute);
    mbar_init(b_psfree, 1);
    mbar_init(b_kvout, 1);
    mbar_init(b_kvoutempty, kCompute);
    mbar_init(b_drain, 1);
    mbar_init(b_stg, 128);
    for (int s = 0; s < 4; ++s) {
      mbar_init(b_ifull(s), 1);
      mbar_init(b_iempty(s), 13);  // MMA warp, 8 compute warps, 4 drain warps
    }
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (warp == 13) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tDK = tmem + 256u, tDV = tmem + 384u;
  // Next item index for a consumer warp (whole warp; false once the wait
  // gave up).  Indices >= n_items end the walk.
  uint32_t in_c = 0;
  auto next_item = [&](int& idx) -> bool {
    const int s = (int)(in_c & 3u);
    if (!mbar_wait_warp(b_ifull(s), (in_c >> 2) & 1u, abort_flag)) return false;
    idx = item_ring[s];
    __syncwarp();
    if (elect_one()) mbar_arrive(b_iempty(s));
    __syncwarp();
    ++in_c;
    return true;
  };

  if (warp == 12) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmDO);
      bool ok = true;
      uint32_t ni = 0, nq = 0;  // items and query tiles loaded
      int idx = blockIdx.x;
      for (;; ++ni) {
        const int s = (int)(ni & 3u);
        if (ni >= 4 && !(ok = mbar_wait(b_iempty(s), ((ni >> 2) - 1) & 1u, abort_flag))) break;
        item_ring[s] = idx;
        mbar_arrive(b_ifull(s));
        if (idx >= p.n_items) break;
        const int nxt = work_next(work);  // used after this item's loads
        const Item it = decode_item(p, idx);
        if (ni > 0 && !(ok = mbar_wait(b_kvempty, (ni - 1) & 1, abort_flag))) break;
        mbar_arrive_expect_tx(b_kvfull, 2 * tile_bytes);
        for (int c = 0; c < p.nch; ++c) {
          tma_load_4d(sK + c * kChunkB, &tmK, b_kvfull, c * 64, it.jt * kB, it.h, it.b);
          tma_load_4d(sV + c * kChunkB, &tmV, b_kvfull, c * 64, it.jt * kB, it.h, it.b);
        }
        for (int qt = it.qlo; qt <= it.qhi; ++qt, ++nq) {
          const int s = nq & 1;
          if (nq >= 2 && !(ok = mbar_wait(b_qempty(s), ((nq >> 1) - 1) & 1, abort_flag))) break;
          mbar_arrive_expect_tx(b_qfull(s), tile_bytes + 2 * kB * 4);
          const int64_t row0 = (int64_t)it.hb * p.Npad + qt * kB;  // 512-byte aligned
          bulk_load(sLD + (uint32_t)s * 2 * kB * 4, p.lse2 + row0, kB * 4, b_qfull(s));
          bulk_load(sLD + (uint32_t)s * 2 * kB * 4 + kB * 4, p.Dv + row0, kB * 4, b_qfull(s));
          for (int c = 0; c < p.nch; ++c)
            tma_load_4d(sQ + 2 * s * kTileB + c * kChunkB, &tmQ, b_qfull(s), c * 64, qt * kB, it.h,
                        it.b);
          if (nq >= 2 && !(ok = mbar_wait(b_doempty(s), ((nq >> 1) - 1) & 1, abort_flag))) break;
          mbar_arrive_expect_tx(b_dofull(s), tile_bytes);
          for (int c = 0; c < p.nch; ++c)
            tma_load_4d(sDO + 2 * s * kTileB + c * kChunkB, &tmDO, b_dofull(s), c * 64, qt * kB,
                        it.h, it.b);
        }
        if (!ok) break;
        idx = nxt;
      }
      if (!ok) raise_error(abort_flag);
      // no copy may still be landing when the CTA exits
      volatile int no_abort = 0;
      if (ni > 0) mbar_wait(b_kvfull, (ni - 1) & 1, &no_abort);
      for (uint32_t n = nq > 2 ? nq - 2 : 0; n < nq; ++n) {
        mbar_wait(b_qfull(n & 1), (n >> 1) & 1, &no_abort);
        mbar_wait(b_dofull(n & 1), (n >> 1) & 1, &no_abort);
      }
    }
  } else if (warp == 13) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the schedule; one elected lane issues (see elect_one).
    {
      const uint32_t id_sq = idesc_bf16_f32(128, 128, false, false);      // S^T, dP^T
      const uint32_t id_acc = idesc_bf16_f32(128, p.ksteps * 16, false, true);  // dV, dK
      const uint32_t id_dq = idesc_bf16_f32(128, 128, true, true);        // dQ^T
      bool ok = true;
      uint32_t ni = 0, gt = 0;  // items, query tiles (global count)
      int idx = 0;
      for (; ok && (ok = next_item(idx)) && idx < p.n_items; ++ni) {
        const Item it = decode_item(p, idx);
        if (!(ok = mbar_wait_warp(b_kvfull, ni & 1, abort_flag))) break;
        // dK / dV of the previous item have been read out
        if (ni > 0 && !(ok = mbar_wait_warp(b_kvoutempty, (ni - 1) & 1, abort_flag))) break;
        for (int qt = it.qlo; ok && qt <= it.qhi; ++qt, ++gt) {
          const int s = gt & 1, r = gt & 1;
          const uint32_t tS = tmem + 128u * r, tP = tmem + 128u * (r ^ 1);
          const uint32_t q_s = sQ + 2 * s * kTileB, do_s = sDO + 2 * s * kTileB;
          if (!(ok = mbar_wait_warp(b_qfull(s), (gt >> 1) & 1, abort_flag))) break;
          tc_fence_after();
          // S^T = K Q^T  (M = keys, N = queries, K = d)
          {
            const uint64_t da = smem_desc_sw128(sK, 16, 1024), db = smem_desc_sw128(q_s, 16, 1024);
            if (elect_one())
              for (int kk = 0; kk < p.ksteps; ++kk) {
                const uint64_t off = (uint64_t)(((kk >> 2) * kChunkB + (kk & 3) * 32) >> 4);
                mma_ss_nm(tS, da + off, db + off, id_sq, kk > 0 ? 1u : 0u);
              }
            __syncwarp();
            mma_commit_warp(b_sfull);
          }
          // dP^T = V dO^T into the region dQ^T of the previous tile used
          if (gt >= 1 && !(ok = mbar_wait_warp(b_dqempty(r ^ 1), ((gt - 1) >> 1) & 1, abort_flag)))
            break;
          if (!(ok = mbar_wait_warp(b_dofull(s), (gt >> 1) & 1, abort_flag))) break;
          tc_fence_after();
          {
            const uint64_t da = smem_desc_sw128(sV, 16, 1024), db = smem_desc_sw128(do_s, 16, 1024);
            if (elect_one())
              for (int kk = 0; kk < p.ksteps; ++kk) {
                const uint64_t off = (uint64_t)(((kk >> 2) * kChunkB + (kk & 3) * 32) >> 4);
                mma_ss_nm(tP, da + off, db + off, id_sq, kk > 0 ? 1u : 0u);
              }
            __syncwarp();
            mma_commit_warp(b_dpfull);
          }
          const bool first = qt == it.qlo;
          // dV += P^T dO  (M = keys, N = d, K = queries)
          if (!(ok = mbar_wait_warp(b_ptfull, gt & 1, abort_flag))) break;
          tc_fence_after();
          {
            const uint64_t da = smem_desc_sw128(sPS, 16, 1024);
            const uint64_t db = smem_desc_sw128(do_s, kChunkB, 1024);
            if (elect_one()) {
#pragma unroll
              for (int kk = 0; kk < kB / 16; ++kk) {
                const uint64_t offa = (uint64_t)(((kk >> 2) * kChunkB + (kk & 3) * 32) >> 4);
                mma_ss_nm(tDV, da + offa, db + (uint64_t)(kk * 128), id_acc,
                          (!first || kk > 0) ? 1u : 0u);
              }
            }
            __syncwarp();
            mma_commit_warp(b_dvdone);
          }
          // dK += dS^T Q ;  dQ^T = K^T dS^T (M = features, N = queries, K = keys)
          if (!(ok = mbar_wait_warp(b_dsfull, gt & 1, abort_flag))) break;
          tc_fence_after();
          {
            const uint64_t da = smem_desc_sw128(sPS, 16, 1024);
            const uint64_t db = smem_desc_sw128(q_s, kChunkB, 1024);
            const uint64_t dka = smem_desc_sw128(sK, kChunkB, 1024);
            const uint64_t dsb = smem_desc_sw128(sPS, kChunkB, 1024);
            if (elect_one()) {
#pragma unroll
              for (int kk = 0; kk < kB / 16; ++kk) {
                const uint64_t offa = (uint64_t)(((kk >> 2) * kChunkB + (kk & 3) * 32) >> 4);
                mma_ss_nm(tDK, da + offa, db + (uint64_t)(kk * 128), id_acc,
                          (!first || kk > 0) ? 1u : 0u);
              }
#pragma unroll
              for (int kk = 0; kk < kB / 16; ++kk)
                mma_ss_nm(tS, dka + (uint64_t)(kk * 128), dsb + (uint64_t)(kk * 128), id_dq,
                          kk > 0 ? 1u : 0u);
            }
            __syncwarp();
            mma_commit_warp(b_dqfull(r));
            mma_commit_warp(b_psfree);  // dK and dQ^T have read dS^T
          }
        }
        if (!ok) break;
        mma_commit_warp(b_kvempty);  // K / V of this item are no longer read
        mma_commit_warp(b_kvout);    // dK / dV accumulators complete
      }
      if (!ok) raise_error(abort_flag);
      mma_drain_warp(b_drain);
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ P^T, dS^T, dK / dV out
    const int row = (warp & 3) * 32 + lane;  // key row of the tile = TMEM lane
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const int hf = warp >> 2;                // query columns 64 hf .. 64 hf + 63
    bool ok = true;
    uint32_t ni = 0, gt = 0;
    int idx = 0;
    for (; ok && (ok = next_item(idx)) && idx < p.n_items; ++ni) {
      const Item it = decode_item(p, idx);
      const int kj = it.jt * kB + row;  // key index
      // queries that see this key: [vis_lo, vis_hi]
      const int vis_lo = p.mask == IHA_MASK_NONE ? 0 : kj;
      int vis_hi = p.N - 1;
      if (p.mask == IHA_MASK_CAUSAL_WINDOW) vis_hi = min(vis_hi, kj + p.window - 1);
      const bool key_ok = kj < p.N;
      for (int qt = it.qlo; qt <= it.qhi; ++qt, ++gt) {
        const int r = gt & 1;
        const uint32_t tS = tmem + lane_base + 128u * r, tP = tmem + lane_base + 128u * (r ^ 1);
        const int q0 = qt * kB;
        const int c_lo = key_ok ? max(vis_lo - q0, 0) : kB, c_hi = min(vis_hi - q0, kB - 1);
        // ---- P^T = exp2(s * scale_log2 - lse2) on visible (key, query) pairs
        if (!(ok = mbar_wait_warp(b_sfull, gt & 1, abort_flag))) break;
        // this tile's lse2 and D have landed with its Q / dO stage
        if (!(ok = mbar_wait_warp(b_qfull(gt & 1), (gt >> 1) & 1, abort_flag))) break;
        tc_fence_after();
        const float* lse2_s = ld_f + (gt & 1) * 2 * kB;
        const float* d_s = lse2_s + kB;
        // the P / dS tile is free once the previous tile's dQ^T has read it
        if (gt >= 1 && !(ok = mbar_wait_warp(b_psfree, (gt - 1) & 1, abort_flag))) break;
#pragma unroll 1
        for (int c = 2 * hf; c < 2 * hf + 2; ++c) {
          uint32_t sv[32];
          tmem_ld32(tS + 32u * c, sv);
          tmem_wait_ld();
          const float4* l4 = reinterpret_cast<const float4*>(lse2_s + 32 * c);
          uint32_t pk[16];
#pragma unroll
          for (int e4 = 0; e4 < 8; ++e4) {
            const float4 lv = l4[e4];
            const float lz[4] = {lv.x, lv.y, lv.z, lv.w};
            float x[4], pe[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
              x[u] = fmaf(__uint_as_float(sv[4 * e4 + u]), p.scale_log2, -lz[u]);
            // a quarter of the exponentials on the FMA pipe
            const float2 pp = (e4 & 1) ? exp2_poly3_x2(make_float2(x[2], x[3]))
                                       : make_float2(fast_exp2(x[2]), fast_exp2(x[3]));
            const float pv[4] = {fast_exp2(x[0]), fast_exp2(x[1]), pp.x, pp.y};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int col = 32 * c + 4 * e4 + u;
              pe[u] = (col >= c_lo && col <= c_hi) ? pv[u] : 0.f;
              sv[4 * e4 + u] = __float_as_uint(pe[u]);  // fp32 P kept for dS
            }
            pk[2 * e4] = pack_bf16x2(pe[0], pe[1]);
            pk[2 * e4 + 1] = pack_bf16x2(pe[2], pe[3]);
          }
          tmem_st32(tS + 32u * c, sv);  // P over S^T in TMEM
          // columns 32c .. 32c+31: chunk c / 2, granules 4 (c % 2) .. +3
#pragma unroll
          for (int g = 0; g < 4; ++g)
            *reinterpret_cast<uint4*>(ps + swz(c >> 1, row, 4 * (c & 1) + g)) =
                make_uint4(pk[4 * g], pk[4 * g + 1], pk[4 * g + 2], pk[4 * g + 3]);
        }
        tmem_wait_st();
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(b_ptfull);
        // ---- dS^T = P o (dP - D), written over P once dV has read it
        if (!(ok = mbar_wait_warp(b_dpfull, gt & 1, abort_flag))) break;
        if (!(ok = mbar_wait_warp(b_dvdone, gt & 1, abort_flag))) break;
        tc_fence_after();
#pragma unroll 1
        for (int c = 2 * hf; c < 2 * hf + 2; ++c) {
          // fp32 P (phase A left it over S^T in TMEM; a bf16 P here would
          // double the rounding error of dS) and dP
          uint32_t pv[32], dp[32];
          tmem_ld32(tS + 32u * c, pv);
          tmem_ld32(tP + 32u * c, dp);
          tmem_wait_ld();
          const float4* d4 = reinterpret_cast<const float4*>(d_s + 32 * c);
          uint32_t pw[16];
#pragma unroll
          for (int e4 = 0; e4 < 8; ++e4) {
            const float4 dv4 = d4[e4];
            const float dz[4] = {dv4.x, dv4.y, dv4.z, dv4.w};
            float ds[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
              ds[u] = __uint_as_float(pv[4 * e4 + u]) * (__uint_as_float(dp[4 * e4 + u]) - dz[u]);
            pw[2 * e4] = pack_bf16x2(ds[0], ds[1]);
            pw[2 * e4 + 1] = pack_bf16x2(ds[2], ds[3]);
          }
#pragma unroll
          for (int g = 0; g < 4; ++g)
            *reinterpret_cast<uint4*>(ps + swz(c >> 1, row, 4 * (c & 1) + g)) =
                make_uint4(pw[4 * g], pw[4 * g + 1], pw[4 * g + 2], pw[4 * g + 3]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(b_dsfull);
      }
      if (!ok) break;
      // ---- dK = scale * acc, dV = acc for this tile's keys
      if (!(ok = mbar_wait_warp(b_kvout, ni & 1, abort_flag))) break;
      tc_fence_after();
      const int64_t orow = (((int64_t)it.b * p.N + min(kj, p.N - 1)) * p.Hh + it.h) * p.d;
      for (int c = 32 * hf; c < p.ksteps * 16; c += 64) {
        uint32_t a[32], bv[32];
        tmem_ld32(tDK + lane_base + (uint32_t)c, a);
        tmem_ld32(tDV + lane_base + (uint32_t)c, bv);
        tmem_wait_ld();
        if (key_ok) {
#pragma unroll
          for (int g8 = 0; g8 < 4; ++g8) {
            const int f = c + 8 * g8;
            if (f < p.d) {
              uint4 wk, wv;
              wk.x = pack_bf16x2(__uint_as_float(a[8 * g8 + 0]) * p.scale, __uint_as_float(a[8 * g8 + 1]) * p.scale);
              wk.y = pack_bf16x2(__uint_as_float(a[8 * g8 + 2]) * p.scale, __uint_as_float(a[8 * g8 + 3]) * p.scale);
              wk.z = pack_bf16x2(__uint_as_float(a[8 * g8 + 4]) * p.scale, __uint_as_float(a[8 * g8 + 5]) * p.scale);
              wk.w = pack_bf16x2(__uint_as_float(a[8 * g8 + 6]) * p.scale, __uint_as_float(a[8 * g8 + 7]) * p.scale);
              wv.x = pack_bf16x2(__uint_as_float(bv[8 * g8 + 0]), __uint_as_float(bv[8 * g8 + 1]));
              wv.y = pack_bf16x2(__uint_as_float(bv[8 * g8 + 2]), __uint_as_float(bv[8 * g8 + 3]));
              wv.z = pack_bf16x2(__uint_as_float(bv[8 * g8 + 4]), __uint_as_float(bv[8 * g8 + 5]));
              wv.w = pack_bf16x2(__uint_as_float(bv[8 * g8 + 6]), __uint_as_float(bv[8 * g8 + 7]));
              *reinterpret_cast<uint4*>(p.dk + orow + f) = wk;
              *reinterpret_cast<uint4*>(p.dv + orow + f) = wv;
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(b_kvoutempty);
    }
    if (!ok) raise_error(abort_flag);
  } else if (warp < 12) {
    // ------------------------------------------------------------ dQ^T drain (warps 8-11)
    // Once dQ^T(t) is complete, every MMA that reads tile t's Q / dO stage
    // has finished, so the stage becomes the staging area: queries 0-63 in
    // the Q half, 64-127 in the dO half, rows = queries of d fp32 features,
    // thread = feature writes its column.  When all 128 drain threads have
    // written (b_stg), one thread adds the tile into dQ_acc with two TMA
    // reduce-adds (boxes d x 64; the reduction runs in the bulk-copy engine,
    // not as element atomics) and hands each half back to the producer as
    // soon as its reduction has read it: the next Q tile can land while the
    // second half is still being reduced.
    const int wq = warp - 8;
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const int feat = wq * 32 + lane;
    const bool issuer = wq == 0 && lane == 0;
    bool ok = true;
    uint32_t gt = 0;
    int idx = 0;
    while (ok && (ok = next_item(idx)) && idx < p.n_items) {
      const Item it = decode_item(p, idx);
      for (int qt = it.qlo; qt <= it.qhi; ++qt, ++gt) {
        const int r = gt & 1, s = gt & 1;
        const uint32_t stage_s = sQ + 2u * (uint32_t)s * kTileB;
        if (!(ok = mbar_wait_warp(b_dqfull(r), (gt >> 1) & 1, abort_flag))) break;
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_base + 128u * r + 32u * c, v);
          tmem_wait_ld();
          if (feat < p.d) {
            float* half = reinterpret_cast<float*>(smem + (stage_s - sK) + (c >> 1) * kTileB);
#pragma unroll
            for (int e = 0; e < 32; ++e)
              half[(32 * (c & 1) + e) * p.d + feat] = __uint_as_float(v[e]);
          }
        }
        tc_fence_before();
        mbar_arrive(b_dqempty(r));  // this TMEM region has been read
        fence_proxy_async_smem();
        mbar_arrive(b_stg);
        if (issuer) {
          if ((ok = mbar_wait(b_stg, gt & 1, abort_flag))) {
            tma_reduce_add_4d(&tmDQ, stage_s, 0, qt * kB, it.h, it.b);
            bulk_commit();
            const bool second = qt * kB + 64 < p.N;  // rows past N: nothing to add
            if (second) {
              tma_reduce_add_4d(&tmDQ, stage_s + kTileB, 0, qt * kB + 64, it.h, it.b);
              bulk_commit();
              bulk_wait_read<1>();  // the first reduce has read the Q half
            } else {
              bulk_wait_read<0>();
            }
            mbar_arrive(b_qempty(s));   // the Q half is the producer's again
            bulk_wait_read<0>();        // the second has read the dO half
            mbar_arrive(b_doempty(s));
          }
        }
        if (wq == 0) ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;  // warp-uniform
        if (!ok) break;
      }
    }
    if (issuer) bulk_wait<0>();  // reductions complete before the CTA exits
    if (!ok) raise_error(abort_flag);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 13) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0) work_leave(work);
}

// D[hb][i] = sum_f dO o O, lse2[hb][i] = lse * log2(e) (zero in the padding),
// and the fp32 dQ accumulator zeroed.  One warp per (b, i, h) row.
__global__ void __launch_bounds__(256) attn_bwd_pre_kernel(
    const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dout,
    const float* __restrict__ lse, float* __restrict__ lse2, float* __restrict__ Dv,
    float* __restrict__ dq_acc, int B, int Hh, int N, int d, int Npad) {
  const int64_t rows = (int64_t)B * Hh * Npad;
  const int64_t wid = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t w = wid; w < rows; w += nw) {
    const int i = (int)(w % Npad);
    const int64_t hb = w / Npad;
    const int h = (int)(hb % Hh), b = (int)(hb / Hh);
    float acc = 0.f;
    if (i < N) {
      const int64_t base = (((int64_t)b * N + i) * Hh + h) * d;
      for (int f = 2 * lane; f < d; f += 64) {
        const uint32_t ov = *reinterpret_cast<const uint32_t*>(o + base + f);
        const uint32_t gv = *reinterpret_cast<const uint32_t*>(dout + base + f);
        acc = fmaf(bf16lo_to_f32(ov), bf16lo_to_f32(gv), acc);
        acc = fmaf(bf16hi_to_f32(ov), bf16hi_to_f32(gv), acc);
      }
      for (int f = lane; f < d; f += 32) dq_acc[base + f] = 0.f;
    }
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
    if (lane == 0) {
      Dv[w] = acc;
      lse2[w] = i < N ? lse[hb * N + i] * 1.4426950408889634f : 0.f;
    }
  }
}

// dQ = bf16(scale * dQ_acc), 4 elements per thread.
__global__ void __launch_bounds__(256) attn_bwd_post_kernel(const float* __restrict__ dq_acc,
                                                            __nv_bfloat16* __restrict__ dq,
                                                            int64_t n4, float scale) {
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n4;
       e += (int64_t)gridDim.x * blockDim.x) {
    const float4 a = reinterpret_cast<const float4*>(dq_acc)[e];
    uint2 w;
    w.x = pack_bf16x2(a.x * scale, a.y * scale);
    w.y = pack_bf16x2(a.z * scale, a.w * scale);
    reinterpret_cast<uint2*>(dq)[e] = w;
  }
}

// 4-D tensor map over a dense [B, N, Hh, d] bf16 tensor, box 64 x 128 rows,
// 128-byte swizzle.
CUresult make_map4(CUtensorMap* m, const void* base, int B, int N, int Hh, int d) {
  uint64_t dims[4] = {(uint64_t)d, (uint64_t)N, (uint64_t)Hh, (uint64_t)B};
  uint64_t st[3] = {(uint64_t)Hh * d * 2, (uint64_t)d * 2, (uint64_t)N * Hh * d * 2};
  uint32_t box[4] = {64, (uint32_t)kB, 1, 1};
  return encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, st,
                      box, CU_TENSOR_MAP_SWIZZLE_128B);
}

struct WsLayout {
  size_t dq_acc, lse2, Dv, total;
};

WsLayout ws_layout(int B, int Hh, int N, int d) {
  const int Npad = (N + kB - 1) / kB * kB;
  WsLayout w;
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  w.dq_acc = 0;
  w.lse2 = up((size_t)B * N * Hh * d * 4);
  w.Dv = w.lse2 + up((size_t)B * Hh * Npad * 4);
  w.total = w.Dv + up((size_t)B * Hh * Npad * 4);
  return w;
}

SmemLimit g_bwd_limit;  // dynamic shared memory limit of attn_bwd_tc_kernel, per device

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

}  // namespace

// Launch of the three backward kernels with the workspace at `ws` (already
// checked: size, alignment).  Shared by the public entry points.
iha_status mha_bwd_launch(const void* q, const void* k, const void* v, const void* o,
                          const void* dout, const float* lse, void* dq, void* dk, void* dv,
                          void* ws, int B, int Hh, int N, int d, float scale, int mask, int window,
                          cudaStream_t stream) {
  const WsLayout wl = ws_layout(B, Hh, N, d);
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  float* dq_acc = reinterpret_cast<float*>(wsb + wl.dq_acc);
  float* lse2 = reinterpret_cast<float*>(wsb + wl.lse2);
  float* Dv = reinterpret_cast<float*>(wsb + wl.Dv);
  const int Npad = (N + kB - 1) / kB * kB;
  {
    const int64_t rows = (int64_t)B * Hh * Npad;
    int64_t blocks = (rows * 32 + 255) / 256;
    const int64_t cap = (int64_t)sm_count() * 16;
    if (blocks > cap) blocks = cap;
    attn_bwd_pre_kernel<<<(unsigned)blocks, 256, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dout), lse, lse2,
        Dv, dq_acc, B, Hh, N, d, Npad);
    const iha_status st = check_launch("mha_bwd (preprocess)");
    if (st != IHA_OK) return st;
  }
  CUtensorMap mq, mk, mv, mdo, mdq;
  {
    // dQ_acc [B, N, Hh, d] fp32, box d features x 64 queries, no swizzle
    uint64_t dims[4] = {(uint64_t)d, (uint64_t)N, (uint64_t)Hh, (uint64_t)B};
    uint64_t st[3] = {(uint64_t)Hh * d * 4, (uint64_t)d * 4, (uint64_t)N * Hh * d * 4};
    uint32_t box[4] = {(uint32_t)d, 64, 1, 1};
    if (encode_tiled(&mdq, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, dq_acc, dims, st, box,
                     CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS)
      return fail(IHA_ERR_CUDA, "mha_bwd: dQ accumulator tensor map encoding failed");
  }
  if (make_map4(&mq, q, B, N, Hh, d) != CUDA_SUCCESS ||
      make_map4(&mk, k, B, N, Hh, d) != CUDA_SUCCESS ||
      make_map4(&mv, v, B, N, Hh, d) != CUDA_SUCCESS ||
      make_map4(&mdo, dout, B, N, Hh, d) != CUDA_SUCCESS)
    return fail(IHA_ERR_CUDA, "mha_bwd: tensor map encoding failed");
  BwdParams p;
  p.B = B;
  p.Hh = Hh;
  p.N = N;
  p.d = d;
  p.Npad = Npad;
  p.ksteps = d / 16;
  p.nch = (d + 63) / 64;
  p.mask = mask;
  p.window = window;
  p.n_kt = (N + kB - 1) / kB;
  p.n_qt = p.n_kt;
  p.n_hb = B * Hh;
  // heads per group: their Q and dO (read by every key tile) stay in L2
  int64_t g = (48ll << 20) / ((int64_t)N * d * 2 * 2 + 1);
  if (g < 1) g = 1;
  if (g > p.n_hb) g = p.n_hb;
  p.group = (int)g;
  p.n_items = p.n_hb * p.n_kt;
  p.work_slot = (int)attention_bwd_work_slot();
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.lse2 = lse2;
  p.Dv = Dv;
  p.dq_acc = dq_acc;
  p.dk = static_cast<__nv_bfloat16*>(dk);
  p.dv = static_cast<__nv_bfloat16*>(dv);
  const cudaError_t attr_err = g_bwd_limit.ensure(attn_bwd_tc_kernel, kSmemBytes);
  if (attr_err != cudaSuccess)
    return fail(IHA_ERR_CUDA, "mha_bwd (smem attribute): %s", cudaGetErrorString(attr_err));
  int grid = sm_count();
  if (grid > p.n_items) grid = p.n_items;
  attn_bwd_tc_kernel<<<grid, kThreads, kSmemBytes, stream>>>(mq, mk, mv, mdo, mdq, p);
  iha_status st = check_launch("mha_bwd");
  if (st != IHA_OK) return st;
  const int64_t n4 = (int64_t)B * N * Hh * d / 4;
  int64_t blocks = (n4 + 255) / 256;
  const int64_t cap = (int64_t)sm_count() * 8;
  if (blocks > cap) blocks = cap;
  attn_bwd_post_kernel<<<(unsigned)blocks, 256, 0, stream>>>(
      dq_acc, static_cast<__nv_bfloat16*>(dq), n4, scale);
  return check_launch("mha_bwd (postprocess)");
}

// Host-side checks shared by the backward entry points.
iha_status mha_bwd_check(const char* name, const void* q, const void* k, const void* v,
                         const void* o, const void* dout, const float* lse, const void* dq,
                         const void* dk, const void* dv, int B, int Hh, int N, int d,
                         iha_mask mask_mode, int window, iha_dtype dt) {
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv)
    return fail(IHA_ERR_INVALID_ARG, "%s: null pointer", name);
  if (B <= 0 || Hh <= 0 || N <= 0 || d <= 0)
    return fail(IHA_ERR_INVALID_ARG, "%s: sizes must be positive", name);
  if (mask_mode != IHA_MASK_NONE && mask_mode != IHA_MASK_CAUSAL &&
      mask_mode != IHA_MASK_CAUSAL_WINDOW)
    return fail(IHA_ERR_INVALID_ARG, "%s: bad mask_mode %d", name, (int)mask_mode);
  if (mask_mode == IHA_MASK_CAUSAL_WINDOW && window < 1)
    return fail(IHA_ERR_INVALID_ARG, "%s: window must be >= 1", name);
  if (dt != IHA_BF16) return fail(IHA_ERR_UNSUPPORTED, "%s: bf16 only", name);
  if (d % 16 || d > 128) return fail(IHA_ERR_UNSUPPORTED, "%s: needs d %% 16 == 0, d <= 128", name);
  if ((int64_t)B * Hh * ((N + kB - 1) / kB) > INT32_MAX || (int64_t)B * N * Hh * d > (1ll << 40))
    return fail(IHA_ERR_UNSUPPORTED, "%s: problem too large", name);
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(lse))
    return fail(IHA_ERR_ALIGNMENT, "%s: pointers must be 16-byte aligned", name);
  const size_t nb = (size_t)B * N * Hh * d * 2;
  const void* ins[6] = {q, k, v, o, dout, lse};
  const size_t ins_n[6] = {nb, nb, nb, nb, nb, (size_t)B * Hh * N * 4};
  const void* outs[3] = {dq, dk, dv};
  for (int a = 0; a < 3; ++a) {
    for (int b = 0; b < 6; ++b)
      if (overlaps(outs[a], nb, ins[b], ins_n[b]))
        return fail(IHA_ERR_INVALID_ARG, "%s: a gradient overlaps an input", name);
    for (int b = a + 1; b < 3; ++b)
      if (overlaps(outs[a], nb, outs[b], nb))
        return fail(IHA_ERR_INVALID_ARG, "%s: gradients overlap", name);
  }
  return IHA_OK;
}

}  // namespace iha

extern "C" {

size_t mha_bwd_workspace_bytes(int B, int Hh, int N, int d) {
  if (B <= 0 || Hh <= 0 || N <= 0 || d <= 0) return 0;
  return iha::ws_layout(B, Hh, N, d).total;
}

iha_status mha_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                   const float* lse, void* dq, void* dk, void* dv, void* workspace,
                   size_t workspace_bytes, int B, int Hh, int N, int d, float scale,
                   iha_mask mask_mode, int window, iha_dtype dt, void* stream) {
  using namespace iha;
  iha_status st = mha_bwd_check("mha_bwd", q, k, v, o, dout, lse, dq, dk, dv, B, Hh, N, d,
                                mask_mode, window, dt);
  if (st != IHA_OK) return st;
  const size_t need = ws_layout(B, Hh, N, d).total;
  if (!workspace) return fail(IHA_ERR_INVALID_ARG, "mha_bwd: null workspace");
  if (workspace_bytes < need)
    return fail(IHA_ERR_INVALID_ARG, "mha_bwd: workspace of %zu bytes, %zu needed",
                workspace_bytes, need);
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0)
    return fail(IHA_ERR_ALIGNMENT, "mha_bwd: workspace must be 256-byte aligned");
  const size_t nb = (size_t)B * N * Hh * d * 2;
  const void* all[9] = {q, k, v, o, dout, lse, dq, dk, dv};
  for (int a = 0; a < 9; ++a)
    if (overlaps(workspace, need, all[a], a == 5 ? (size_t)B * Hh * N * 4 : nb))
      return fail(IHA_ERR_INVALID_ARG, "mha_bwd: workspace overlaps a tensor");
  if (mask_mode != IHA_MASK_CAUSAL_WINDOW) window = 0;
  if (!(scale > 0.f)) scale = 1.f / sqrtf((float)d);
  return mha_bwd_launch(q, k, v, o, dout, lse, dq, dk, dv, workspace, B, Hh, N, d, scale,
                        mask_mode, window, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free backward: the same three launches with the scratch in a
// file-scope device array instead of a caller workspace.  The array is part
// of the library image, so every GPU that loads the library holds it until
// the process exits, and every call shares it.
namespace iha {
namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)32 << 20;
static __device__ __align__(256) uint8_t g_bwd_scratch[kNoAllocScratchBytes];

// Device address of g_bwd_scratch per device: in host code the symbol is a
// host-side stand-in, so it is looked up (once per device, with that device
// current) and only the looked-up address is handed to kernels.
constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {nullptr};

iha_status scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(IHA_ERR_CUDA, "mha_bwd_noalloc: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return fail(IHA_ERR_UNSUPPORTED, "mha_bwd_noalloc: device %d beyond %d", dev, kMaxDevices);
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_bwd_scratch);
    if (e != cudaSuccess || !ptr)
      return fail(IHA_ERR_CUDA, "mha_bwd_noalloc: scratch address: %s",
                  cudaGetErrorString(e));
    g_scratch_addr[dev] = ptr;
  }
  *out = g_scratch_addr[dev];
  return IHA_OK;
}

}  // namespace
}  // namespace iha

extern "C" iha_status mha_bwd_noalloc(const void* q, const void* k, const void* v,
                                      const void* o, const void* dout, const float* lse,
                                      void* dq, void* dk, void* dv, int B, int Hh, int N, int d,
                                      float scale, iha_mask mask_mode, int window, iha_dtype dt,
                                      void* stream) {
  using namespace iha;
  iha_status st = mha_bwd_check("mha_bwd_noalloc", q, k, v, o, dout, lse, dq, dk, dv, B, Hh, N,
                                d, mask_mode, window, dt);
  if (st != IHA_OK) return st;
  const size_t need = ws_layout(B, Hh, N, d).total;
  if (need > kNoAllocScratchBytes)
    return fail(IHA_ERR_UNSUPPORTED,
                "mha_bwd_noalloc: this problem needs %zu bytes of scratch but the built-in "
                "buffer holds %zu; call mha_bwd with a workspace instead",
                need, kNoAllocScratchBytes);
  void* scratch = nullptr;
  st = scratch_address(&scratch);
  if (st != IHA_OK) return st;
  if (mask_mode != IHA_MASK_CAUSAL_WINDOW) window = 0;
  if (!(scale > 0.f)) scale = 1.f / sqrtf((float)d);
  // the preprocess rewrites every scratch word this call reads (dQ
  // accumulator zeroed, D and lse * log2(e) written), so the previous call's
  // contents never leak into this one
  return mha_bwd_launch(q, k, v, o, dout, lse, dq, dk, dv, scratch, B, Hh, N, d, scale,
                        mask_mode, window, reinterpret_cast<cudaStream_t>(stream));
}
