/*
 * iha.h — C ABI of the GB300 (sm_103a) library for the Interleaved Head
 * Attention (IHA) attention-layer hot path and Hiera mask-unit attention.
 *
 * Operations and where they are defined:
 *   iha_premix_fwd / iha_premix_bwd_dx / iha_premix_bwd_dw
 *     "IHA-CUDA: Interleaved Head Attention Kernels for Hopper GPUs",
 *     section "Pseudo-Token Mixing (Triton Premix Kernels)": the mix
 *     Out[h,p] = sum_s W[h,p,s] * X[s] at every (batch, position, feature),
 *     its input gradient dX = W^T dY and its weight gradient
 *     dW = sum over (b, n, d) of dY * X^T, with optional fused RoPE.
 *   mha_fwd
 *     same page, sections "Kernel Design" and "FLOP Matching": softmax
 *     attention over the H*P pseudo-heads with a causal sliding window of
 *     W = WSL + 1 keys; "hiera-optim 0.1.0", file
 *     hiera_optim/attention/mask_unit.py (MaskUnitAttentionFast.forward):
 *     unmasked attention inside each mask unit, read in Hiera's
 *     (T outer, num_windows inner) token layout.
 *   mu_gather / mu_scatter
 *     "hiera-optim 0.1.0", README, "optimize(model) does two things", item 2:
 *     boolean mask indexing of the kept mask units replaced by gather and
 *     scatter.
 *
 * Conventions shared by every entry point:
 *   - Pointers named x, y, q, ... are DEVICE pointers owned by the caller.
 *     The library allocates nothing, keeps no pointer after return and never
 *     writes outside the output buffers named in each call.
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream).  All argument checks happen on the host before
 *     any launch; a failed check returns an error and launches nothing.
 *   - IHA_ERR_CUDA means a CUDA runtime call failed (details in
 *     iha_last_error()).  Errors that only the GPU can see (an out-of-range
 *     keep index, an internal wait that gave up) set a device error word
 *     that iha_device_error() reads; the offending accesses are skipped.
 *   - Tensors are dense in their last dimension; byte strides of 16-bit
 *     tensors must be multiples of 16 and base pointers 16-byte aligned
 *     (IHA_ERR_ALIGNMENT otherwise).
 */
#ifndef IHA_H_
#define IHA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  IHA_OK = 0,
  IHA_ERR_INVALID_ARG = 1,   /* null pointer, non-positive size, bad enum   */
  IHA_ERR_UNSUPPORTED = 2,   /* valid but outside what the kernels handle   */
  IHA_ERR_ALIGNMENT = 3,     /* base pointer or stride not 16-byte aligned  */
  IHA_ERR_CUDA = 4           /* a CUDA runtime call or launch failed        */
} iha_status;

typedef enum { IHA_F32 = 0, IHA_BF16 = 1 } iha_dtype;

typedef enum {
  IHA_MASK_NONE = 0,           /* every key visible                          */
  IHA_MASK_CAUSAL = 1,         /* key j visible to query i iff j <= i         */
  IHA_MASK_CAUSAL_WINDOW = 2   /* ... and i - j < window (window = WSL + 1)   */
} iha_mask;

/* Element strides of a [B_outer, B_inner, seq, head, d] view; d is dense. */
typedef struct {
  int64_t b_outer;
  int64_t b_inner;
  int64_t seq;
  int64_t head;
} iha_strides;

/*
 * Premix forward ("Pseudo-Token Mixing", forward):
 *   y[b,n,h*P+p,f] = sum_{s<H} w[h,p,s] * x[b,n,s,f]
 * then, if rope != 0, each pseudo-head vector y[b,n,j,:] is rotated by the
 * rotate-half RoPE of position n: for i < d/2, angle = n * rope_base^(-2i/d),
 *   (y_i, y_{i+d/2}) <- (y_i cos - y_{i+d/2} sin, y_{i+d/2} cos + y_i sin).
 *   x  [B, N, H, d]    dtype dt (IHA_BF16 or IHA_F32), dense
 *   w  [H, P, H]       float32, dense
 *   y  [B, N, H*P, d]  dtype dt, dense, must not overlap x or w
 * Accumulation is fp32; bf16 outputs are rounded to nearest even.
 * Requires d % 8 == 0 (bf16) or d % 4 == 0 (f32), H <= 32, H*P <= 128;
 * rope needs d a power of two in [16, 128].
 */
iha_status iha_premix_fwd(const void* x, const float* w, void* y, int B, int N,
                          int H, int P, int d, iha_dtype dt, int rope,
                          float rope_base, void* stream);

/*
 * Premix forward of Q, K and V in one launch ("Pseudo-Token Mixing": one
 * premix per Q, K and V, each with its own weight; the pages fuse the
 * backward's six launches into two, and this fuses the forward's three into
 * one).  Tensor t in (q, k, v) computes exactly what iha_premix_fwd computes
 * for (x_t, w_t, y_t); RoPE (when rope != 0) is applied to q and k only.
 * All nine buffers follow iha_premix_fwd's layout and limits; no output may
 * overlap any input or another output.  Shapes outside the tensor-core
 * kernel run on the CUDA-core kernel: Q, K and V in one launch (with RoPE,
 * Q and K in one and V in a second), on the same stream.
 */
iha_status iha_premix_fwd_qkv(const void* xq, const void* xk, const void* xv,
                              const float* wq, const float* wk, const float* wv,
                              void* yq, void* yk, void* yv, int B, int N, int H, int P,
                              int d, iha_dtype dt, int rope, float rope_base, void* stream);

/*
 * Premix forward of Q, K and V with the interleaved pseudo-token layout of
 * the joint-softmax reading of Interleaved Head Attention ("IHA-CUDA", the
 * "interleaved" head layout and the softmax "joint" across pseudo-heads):
 *   y_t[b, n, p, h, f] = sum_s w_t[h, p, s] * x_t[b, n, s, f]  (+ RoPE at n)
 * i.e. the values of iha_premix_fwd_qkv with rows ordered p * H + h instead
 * of h * P + p.  Viewed as [B, N*P, H, d] (sequence stride H*d, head stride
 * d), it is an H-head sequence of N*P pseudo-tokens, pseudo-token n*P + p,
 * which mha_fwd attends over in place (causal on n*P + p).
 * bf16 only, d in {64, 128}, H <= 32, H*P <= 128; other limits as
 * iha_premix_fwd_qkv.
 */
iha_status iha_premix_fwd_qkv_interleaved(const void* xq, const void* xk, const void* xv,
                                          const float* wq, const float* wk, const float* wv,
                                          void* yq, void* yk, void* yv, int B, int N, int H,
                                          int P, int d, iha_dtype dt, int rope,
                                          float rope_base, void* stream);

/*
 * Premix input gradient ("Pseudo-Token Mixing", backward, dX = W^T dY):
 *   dx[b,n,s,f] = sum_{h,p} w[h,p,s] * g[b,n,h*P+p,f]
 * with g = dy, or g = R_n^T dy (inverse rotation) when rope != 0.
 *   dy [B, N, H*P, d]  dtype dt;  w [H, P, H] float32;  dx [B, N, H, d] dtype dt.
 * Same shape limits as iha_premix_fwd.
 */
iha_status iha_premix_bwd_dx(const void* dy, const float* w, void* dx, int B,
                             int N, int H, int P, int d, iha_dtype dt,
                             int rope, float rope_base, void* stream);

/*
 * Premix weight gradient ("Pseudo-Token Mixing", backward, dW = sum dY X^T):
 *   dw[h,p,s] = sum_{b,n,f} g[b,n,h*P+p,f] * x[b,n,s,f]   (g as in dX)
 *   dy [B, N, H*P, d] dtype dt;  x [B, N, H, d] dtype dt;
 *   dw [H, P, H] float32, OVERWRITTEN (zeroed on `stream` first).
 * Partial sums are reduced inside each block, then added with one float
 * atomic per element per block, so the last bits depend on block order.
 */
iha_status iha_premix_bwd_dw(const void* dy, const void* x, float* dw, int B,
                             int N, int H, int P, int d, iha_dtype dt,
                             int rope, float rope_base, void* stream);

/*
 * Premix backward, both gradients in one pass over dY ("Pseudo-Token Mixing",
 * backward): dx as iha_premix_bwd_dx and dw as iha_premix_bwd_dw, from one
 * read of dy (and x).  Algorithmic traffic per token: dY + X + dX instead of
 * 2 dY + X + dX for the two separate calls.
 *   dy [B, N, H*P, d], x [B, N, H, d], dx [B, N, H, d] (dtype dt);
 *   w [H, P, H] float32;  dw [H, P, H] float32, OVERWRITTEN.
 * Same shape limits as iha_premix_fwd; outputs must not overlap any input.
 */
iha_status iha_premix_bwd(const void* dy, const void* x, const float* w, void* dx,
                          float* dw, int B, int N, int H, int P, int d,
                          iha_dtype dt, int rope, float rope_base, void* stream);

/*
 * Premix backward of Q, K and V in one launch ("Pseudo-Token Mixing":
 * "Backward ... all three Q/K/V in a single launch each", six launches to
 * two).  Tensor t in (q, k, v) computes exactly what iha_premix_bwd computes
 * for (dy_t, x_t, w_t) into (dx_t, dw_t); RoPE (when rope != 0) applies to q
 * and k only.  Every buffer follows iha_premix_bwd's layout and limits; the
 * three dw are OVERWRITTEN (one small zeroing launch precedes the backward
 * launch on `stream`); no output may overlap any input or another output.
 * Shapes outside the tensor-core kernel run as three iha_premix_bwd calls.
 */
iha_status iha_premix_bwd_qkv(const void* dyq, const void* dyk, const void* dyv,
                              const void* xq, const void* xk, const void* xv,
                              const float* wq, const float* wk, const float* wv,
                              void* dxq, void* dxk, void* dxv,
                              float* dwq, float* dwk, float* dwv, int B, int N,
                              int H, int P, int d, iha_dtype dt, int rope,
                              float rope_base, void* stream);

/*
 * Multi-head softmax attention forward over Hh heads ("Kernel Design",
 * "FLOP Matching"; MaskUnitAttentionFast.forward):
 *   o[i] = sum_j softmax_j(scale * <q_i, k_j> | visible(i, j)) * v_j
 *   lse[i] = ln sum_{visible j} exp(scale * <q_i, k_j>)
 * Views: q, o are [B_outer, B_inner, Nq, Hh, d]; k, v are
 * [B_outer, B_inner, Nk, Hh, d]; element strides in sq, sk, sv, so.  With
 * B_inner = num mask units and seq stride = num_units * row, Hiera's
 * (T outer, units inner) layout is read in place.
 *   scale     <= 0 selects 1/sqrt(d)
 *   mask_mode IHA_MASK_NONE | IHA_MASK_CAUSAL | IHA_MASK_CAUSAL_WINDOW
 *             (causal masks require Nq == Nk)
 *   window    keys per query including the diagonal (W = WSL + 1), >= 1 for
 *             IHA_MASK_CAUSAL_WINDOW, ignored otherwise
 *   lse_out   nullable; float32 [B_outer, B_inner, Hh, Nq] dense
 * bf16: tensor-core kernel (tcgen05, TMEM accumulators, TMA tiles), fp32
 * softmax; needs 8 <= d <= 128, d % 8 == 0.  f32: CUDA-core kernel, fp32
 * throughout, d <= 128.
 */
iha_status mha_fwd(const void* q, const void* k, const void* v, void* o,
                   float* lse_out, int B_outer, int B_inner, int Hh, int Nq,
                   int Nk, int d, iha_strides sq, iha_strides sk,
                   iha_strides sv, iha_strides so, float scale,
                   iha_mask mask_mode, int window, iha_dtype dt, void* stream);

/*
 * Mask-unit attention with pooled queries (Hiera's q_pool; "hiera-optim
 * 0.1.0", hiera_optim/attention/mask_unit.py, MaskUnitAttentionFast.forward
 * with q_stride > 1): per (b_outer, b_inner, head) unit of T tokens, the
 * query rows are max-pooled over q_stride blocks of Tq = T / q_stride rows
 * (the block index is the slow axis),
 *   qp[t] = max_i q[i * Tq + t]          (elementwise, i < q_stride)
 * and attend, unmasked, over all T keys:
 *   o[t] = sum_j softmax_j(scale * <qp_t, k_j>) v_j,  lse[t] as mha_fwd.
 * The pooling happens inside the kernel, on the Q tile as it arrives; the
 * pooled queries are never written to memory.
 *   q, k, v   bf16 [B_outer, B_inner, T, Hh, d] views (strides sq, sk, sv)
 *   o         bf16 [B_outer, B_inner, Tq, Hh, d] view (strides so)
 *   lse_out   nullable; float32 [B_outer, B_inner, Hh, Tq] dense
 *   scale     <= 0 selects 1/sqrt(d)
 * Needs T <= 64, q_stride dividing T, d <= 128 and d % 8 == 0; alignment as
 * mha_fwd.  q_stride = 1 is mha_fwd's unmasked short-sequence attention.
 */
iha_status mha_fwd_qpool(const void* q, const void* k, const void* v, void* o,
                         float* lse_out, int B_outer, int B_inner, int Hh, int T,
                         int d, int q_stride, iha_strides sq, iha_strides sk,
                         iha_strides sv, iha_strides so, float scale,
                         iha_dtype dt, void* stream);

/*
 * Attention backward over Hh heads ("Repository Structure": preprocess,
 * backward, postprocess; "End-to-End Training Benchmark": the training step):
 * with P = softmax(scale Q K^T | mask) recomputed from lse and dO the
 * gradient of O = P V,
 *   D_i = sum_f dO_if O_if,   dS = P o (dO V^T - D)
 *   dq = scale dS K,   dk = scale dS^T Q,   dv = P^T dO.
 *   q, k, v, o, dout   bf16 [B, N, Hh, d] dense (o, lse: the forward's outputs)
 *   lse                float32 [B, Hh, N] (natural log, scale included)
 *   dq, dk, dv         bf16 [B, N, Hh, d] dense, written; must not overlap
 *                      each other, the inputs or the workspace
 *   workspace          device scratch of at least mha_bwd_workspace_bytes()
 *                      bytes, 256-byte aligned, owned by the caller: an fp32
 *                      dQ accumulator and per-row D and lse * log2(e); its
 *                      contents on entry do not matter and on return are
 *                      unspecified
 *   scale <= 0 selects 1/sqrt(d); mask_mode / window as mha_fwd (Nq = Nk = N).
 * Needs bf16, d % 16 == 0, d <= 128.  Three launches on `stream`; dq gathers
 * contributions with fp32 atomics, so its last bits depend on their order.
 */
size_t mha_bwd_workspace_bytes(int B, int Hh, int N, int d);
iha_status mha_bwd(const void* q, const void* k, const void* v, const void* o,
                   const void* dout, const float* lse, void* dq, void* dk, void* dv,
                   void* workspace, size_t workspace_bytes, int B, int Hh, int N,
                   int d, float scale, iha_mask mask_mode, int window,
                   iha_dtype dt, void* stream);

/*
 * Attention backward without any allocation.  The pages have no counterpart:
 * this entry point exists for callers that cannot hand the library a device
 * buffer and cannot call cudaMalloc themselves, for example a plugin inside a
 * host program whose own allocator owns all device memory, or a code path
 * that must not call cudaMalloc because it can synchronize the device.
 * Same arguments and results as mha_bwd, minus the workspace: the scratch
 * (fp32 dQ accumulator, per-row D and lse * log2(e)) lives in a 32 MiB array
 * built into the library, which every GPU that loads the library keeps for
 * the life of the process.
 *   - Problems whose scratch exceeds 32 MiB (mha_bwd_workspace_bytes > 32 MiB,
 *     e.g. B = 1, N = 4096, Hh = 8, d = 128 fits) are rejected with
 *     IHA_ERR_UNSUPPORTED before anything is launched; use mha_bwd.
 *   - The first call on a device looks up the array's device address (once
 *     per device, with that device current); make that first call before
 *     any stream capture on the device.
 *   - Every call shares the one array and it keeps the last call's contents;
 *     each call rewrites all of it that it reads, but calls that overlap on
 *     the GPU (other streams, other host threads) race on it: serialize them.
 */
iha_status mha_bwd_noalloc(const void* q, const void* k, const void* v,
                           const void* o, const void* dout, const float* lse,
                           void* dq, void* dk, void* dv, int B, int Hh, int N,
                           int d, float scale, iha_mask mask_mode, int window,
                           iha_dtype dt, void* stream);

/*
 * Mask-unit gather (README item 2, x[mask] -> gather):
 *   out[b,k,t,:] = x[b, tok(keep[b,k], t), :]
 * where the grid is row-major [grid_h, grid_w], mask units are mu_h x mu_w
 * (unit u = (u / (grid_w/mu_w), u % (grid_w/mu_w))), t = ty*mu_w + tx, and
 *   tok(u, t) = (uy*mu_h + ty) * grid_w + ux*mu_w + tx.
 *   x    [B, grid_h*grid_w, C] elements of elem_bytes bytes, dense
 *   keep [B, n_keep] int32 unit ids in [0, units); out-of-range ids are
 *        skipped on the GPU and flagged in iha_device_error()
 *   out  [B, n_keep, mu_h*mu_w, C]
 * Bit-exact byte copy.  Requires grid_h % mu_h == 0, grid_w % mu_w == 0.
 */
iha_status mu_gather(const void* x, const int32_t* keep, void* out, int B,
                     int grid_h, int grid_w, int mu_h, int mu_w, int n_keep,
                     int C, int elem_bytes, void* stream);

/*
 * Mask-unit scatter (README item 2, x_dec[mask] = ... -> scatter), in place:
 *   x[b, tok(keep[b,k], t), :] = src[b,k,t,:]; other tokens untouched.
 * Same shapes and rules as mu_gather; duplicate ids within a sample race.
 */
iha_status mu_scatter(const void* src, const int32_t* keep, void* x, int B,
                      int grid_h, int grid_w, int mu_h, int mu_w, int n_keep,
                      int C, int elem_bytes, void* stream);

/*
 * Hiera stage-1 attention step in one pass: gather, mask-unit attention and
 * scatter ("hiera-optim 0.1.0": README item 2 and MaskUnitAttentionFast.forward;
 * the qkv and proj layers around the attention are not on this path, so
 * Q = K = V = the unit's tokens).  For every kept unit (b, keep[b,k]):
 *   canvas[b, tok(u, t), :] = sum_t' softmax_t'(scale x_t . x_t') x_t'
 * with x_t = x[b, tok(u, t), :], t, t' over the unit's mu_h*mu_w tokens, and
 * tok() as for mu_gather; every other canvas token is left untouched.  It
 * equals mu_gather -> mha_fwd (mask none) -> mu_scatter without the
 * gathered units ever being written to memory.
 *   x      [B, grid_h*grid_w, C] bf16, dense, 16-byte aligned
 *   keep   [B, n_keep] int32 unit ids (out-of-range ids: unit skipped,
 *          iha_device_error() flagged)
 *   canvas [B, grid_h*grid_w, C] bf16, must not overlap x or keep
 * Requires mu_h*mu_w <= 64, C % 8 == 0, C <= 128, grid_h % mu_h == 0,
 * grid_w % mu_w == 0, n_keep <= units; scale <= 0 means C^-1/2.
 */
iha_status mu_attention_fused(const void* x, const int32_t* keep, void* canvas, int B,
                              int grid_h, int grid_w, int mu_h, int mu_w, int n_keep,
                              int C, float scale, iha_dtype dt, void* stream);

/*
 * Test hook for the failure path; never needed in normal use.  Arms the next
 * bf16 mha_fwd launch made on the calling host thread (one shot) so that
 * CTA 0 withholds the load of its first V tile and every wait of that launch
 * gives up after limit_us microseconds (1 .. 1e6) instead of the normal 4 s.
 * The launch then takes its abort path: the waiting role raises the block's
 * abort flag, the others unwind, TMA copies in flight land, the MMAs drain,
 * tensor memory is released, and the kernel returns with device error 2
 * (iha_device_error); the rows of CTA 0's work are left unwritten.  The GPU
 * context stays usable and the next launch runs normally.
 * IHA_ERR_INVALID_ARG for a limit out of range.
 */
iha_status iha_test_fail_next_wait(int limit_us);

/* Static description of a status code. */
const char* iha_status_string(iha_status status);

/* Detail of the last error returned on the calling host thread ("" if none). */
const char* iha_last_error(void);

/*
 * Device error word of the current device: 0 if no kernel has flagged an
 * error, else a bitwise OR of codes (1 = out-of-range keep index, 2 = a
 * bounded internal wait gave up, 4 = a kernel found its dynamic shared memory
 * not 1024-byte aligned and did nothing).  Synchronises the device; clears the word if clear != 0.
 * Returns -1 if the word cannot be read.
 */
int iha_device_error(int clear);

#ifdef __cplusplus
}
#endif

#endif /* IHA_H_ */
