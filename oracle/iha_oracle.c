/*
 * Oracle for the IHA attention-layer hot path: plain, slow, obviously correct.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link or call this
 * file; only the tests, the smoke check and the CPU-baseline leg of the bench
 * use it.  It shares no code, header, table or constant with the CUDA library.
 *
 * Every routine accumulates in double, reads its inputs as the exact values of
 * their storage type (the caller widens bf16 to float losslessly) and writes
 * double results; rounding to the output storage type is the caller's job.
 *
 * Sources (page title, section):
 *   "IHA-CUDA: Interleaved Head Attention Kernels for Hopper GPUs",
 *     section "Pseudo-Token Mixing (Triton Premix Kernels)":
 *       forward mix Out[h,p] = sum_s W[h,p,s] X[s] at every (batch, position,
 *       feature); backward dX = W^T dY and dW = sum over (b, n, d) of dY X^T;
 *       "optional fused RoPE rotation" (no formula given: rotate-half reading).
 *     section "FLOP Matching": window W = WSL + 1, 128-token tiles, the
 *       tile-matched WSL table.
 *   "hiera-optim 0.1.0" (PyPI page) and its sdist file
 *     hiera_optim/attention/mask_unit.py, class MaskUnitAttentionFast.forward:
 *       softmax attention inside each mask unit, scale head_dim ** -0.5;
 *     README "optimize(model) does two things", item 2: boolean mask indexing
 *       replaced by gather / scatter of the kept mask units.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - pseudo-head index j = h*P + p (order of Out[h,p] and W[h,p,s]);
 *   - RoPE is HF-LLaMA rotate-half, base b, position n (0-based),
 *     inv_freq_i = b^(-2i/d) for i < d/2, applied to each pseudo-head vector
 *     after mixing;
 *   - softmax is per pseudo-head and per query row;
 *   - key j is visible to query i under the causal-window mask iff
 *     0 <= i - j < window, with window = WSL + 1;
 *   - a mask unit u of a grid_h x grid_w token grid split into mu_h x mu_w
 *     units is unit (u / units_per_row, u % units_per_row); token t of a unit
 *     is (t / mu_w, t % mu_w) inside it; the grid is row-major.
 */
#include <math.h>
#include <stdlib.h>
#include <stdint.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ------------------------------------------------------------------------ */
/* RoPE (rotate-half), applied in place-free form to vectors of length d.    */
/* v has `heads` vectors of length d per (b, n) token; out = R_n v (or R_n^T). */
/* ------------------------------------------------------------------------ */
static void rope_token(const double* in, double* out, long heads, long d,
                       long n, double base, int inverse) {
  long half = d / 2;
  for (long i = 0; i < half; ++i) {
    double inv_freq = pow(base, -2.0 * (double)i / (double)d);
    double angle = (double)n * inv_freq;
    double c = cos(angle), s = sin(angle);
    if (inverse) s = -s;
    for (long h = 0; h < heads; ++h) {
      double a = in[h * d + i];
      double b = in[h * d + i + half];
      out[h * d + i] = a * c - b * s;
      out[h * d + i + half] = b * c + a * s;
    }
  }
}

/* Standalone RoPE over x[B][N][heads][d] (double), for the commutation pins. */
void oracle_rope(const double* x, double* y, long B, long N, long heads,
                 long d, double base, int inverse) {
#pragma omp parallel for schedule(static)
  for (long bn = 0; bn < B * N; ++bn) {
    long n = bn % N;
    rope_token(x + bn * heads * d, y + bn * heads * d, heads, d, n, base,
               inverse);
  }
}

/* ------------------------------------------------------------------------ */
/* Premix forward: Y[b,n,h*P+p,f] = sum_s W[h,p,s] * X[b,n,s,f]              */
/* then, if rope != 0, each pseudo-head vector Y[b,n,j,:] is rotated by R_n.  */
/* The input may be a window of positions: row n of the input sits at        */
/* position pos0 + n (pos0 = 0 for whole sequences).                         */
/* ------------------------------------------------------------------------ */
void oracle_premix_fwd(const float* x, const float* w, double* y, long B,
                       long N, long H, long P, long d, int rope,
                       double rope_base, long pos0) {
  long HP = H * P;
#pragma omp parallel for schedule(static)
  for (long bn = 0; bn < B * N; ++bn) {
    const float* xt = x + bn * H * d;
    double* yt = y + bn * HP * d;
    for (long h = 0; h < H; ++h)
      for (long p = 0; p < P; ++p)
        for (long f = 0; f < d; ++f) {
          double acc = 0.0;
          for (long s = 0; s < H; ++s)
            acc += (double)w[(h * P + p) * H + s] * (double)xt[s * d + f];
          yt[(h * P + p) * d + f] = acc;
        }
    if (rope) {
      double tmp[HP * d];
      memcpy(tmp, yt, sizeof(double) * HP * d);
      rope_token(tmp, yt, HP, d, pos0 + bn % N, rope_base, 0);
    }
  }
}

/* ------------------------------------------------------------------------ */
/* Premix backward, input gradient: dX = W^T dY, i.e.                        */
/* dX[b,n,s,f] = sum_{h,p} W[h,p,s] * G[b,n,h*P+p,f], where G = dY, or       */
/* G = R_n^T dY when the forward applied RoPE (the chain rule through R_n).   */
/* ------------------------------------------------------------------------ */
void oracle_premix_bwd_dx(const float* dy, const float* w, double* dx, long B,
                          long N, long H, long P, long d, int rope,
                          double rope_base, long pos0) {
  long HP = H * P;
#pragma omp parallel for schedule(static)
  for (long bn = 0; bn < B * N; ++bn) {
    double g[HP * d];
    for (long e = 0; e < HP * d; ++e) g[e] = (double)dy[bn * HP * d + e];
    if (rope) {
      double tmp[HP * d];
      memcpy(tmp, g, sizeof(double) * HP * d);
      rope_token(tmp, g, HP, d, pos0 + bn % N, rope_base, 1);
    }
    double* out = dx + bn * H * d;
    for (long s = 0; s < H; ++s)
      for (long f = 0; f < d; ++f) {
        double acc = 0.0;
        for (long h = 0; h < H; ++h)
          for (long p = 0; p < P; ++p)
            acc += (double)w[(h * P + p) * H + s] * g[(h * P + p) * d + f];
        out[s * d + f] = acc;
      }
  }
}

/* ------------------------------------------------------------------------ */
/* Premix backward, weight gradient:                                         */
/* dW[h,p,s] = sum_{b,n,f} G[b,n,h*P+p,f] * X[b,n,s,f]  (G as in dX above).   */
/* Tokens are split into one slab per thread; slabs are summed in slab order  */
/* so the result does not depend on scheduling.                              */
/* ------------------------------------------------------------------------ */
void oracle_premix_bwd_dw(const float* dy, const float* x, double* dw, long B,
                          long N, long H, long P, long d, int rope,
                          double rope_base) {
  long HP = H * P;
  long T = B * N;
  int nslab = oracle_num_threads();
  if (nslab > T) nslab = (int)(T > 0 ? T : 1);
  double part[nslab][HP * H];
  memset(part, 0, sizeof(part));
#pragma omp parallel for schedule(static, 1)
  for (int sl = 0; sl < nslab; ++sl) {
    long t0 = T * sl / nslab, t1 = T * (sl + 1) / nslab;
    double g[HP * d];
    for (long bn = t0; bn < t1; ++bn) {
      for (long e = 0; e < HP * d; ++e) g[e] = (double)dy[bn * HP * d + e];
      if (rope) {
        double tmp[HP * d];
        memcpy(tmp, g, sizeof(double) * HP * d);
        rope_token(tmp, g, HP, d, bn % N, rope_base, 1);
      }
      const float* xt = x + bn * H * d;
      for (long j = 0; j < HP; ++j)
        for (long s = 0; s < H; ++s) {
          double acc = 0.0;
          for (long f = 0; f < d; ++f) acc += g[j * d + f] * (double)xt[s * d + f];
          part[sl][j * H + s] += acc;
        }
    }
  }
  for (long e = 0; e < HP * H; ++e) {
    double acc = 0.0;
    for (int sl = 0; sl < nslab; ++sl) acc += part[sl][e];
    dw[e] = acc;
  }
}

/* ------------------------------------------------------------------------ */
/* Attention forward, one query row, by the two-pass definition:             */
/*   visible set V(i); s_j = scale * <q_i, k_j>; m = max s_j;                */
/*   O_i = sum_j e^{s_j - m} v_j / sum_j e^{s_j - m};                        */
/*   lse_i = m + ln sum_j e^{s_j - m}  (natural log, scale included).         */
/* mask: 0 none, 1 causal (j <= i), 2 causal window (0 <= i - j < window).   */
/* A row with no visible key gets O = 0 and lse = -inf.                      */
/* Strides are in elements: [b_outer, b_inner, seq, head]; last dim dense.   */
/* ------------------------------------------------------------------------ */
static int visible(long i, long j, int mask, long window) {
  if (mask == 0) return 1;
  if (j > i) return 0;
  if (mask == 2 && i - j >= window) return 0;
  return 1;
}

static void attn_row(const float* q, const float* k, const float* v,
                     const long* sq, const long* sk, const long* sv, long bo,
                     long bi, long h, long i, long Nk, long d, double scale,
                     int mask, long window, double* o_row, double* lse,
                     double* sbuf) {
  const float* qi = q + bo * sq[0] + bi * sq[1] + i * sq[2] + h * sq[3];
  double m = -INFINITY;
  long nvis = 0;
  for (long j = 0; j < Nk; ++j) {
    if (!visible(i, j, mask, window)) { sbuf[j] = -INFINITY; continue; }
    const float* kj = k + bo * sk[0] + bi * sk[1] + j * sk[2] + h * sk[3];
    double dot = 0.0;
    for (long f = 0; f < d; ++f) dot += (double)qi[f] * (double)kj[f];
    sbuf[j] = scale * dot;
    if (sbuf[j] > m) m = sbuf[j];
    ++nvis;
  }
  for (long f = 0; f < d; ++f) o_row[f] = 0.0;
  if (nvis == 0) { *lse = -INFINITY; return; }
  double l = 0.0;
  for (long j = 0; j < Nk; ++j) {
    if (sbuf[j] == -INFINITY) continue;
    double e = exp(sbuf[j] - m);
    l += e;
    const float* vj = v + bo * sv[0] + bi * sv[1] + j * sv[2] + h * sv[3];
    for (long f = 0; f < d; ++f) o_row[f] += e * (double)vj[f];
  }
  for (long f = 0; f < d; ++f) o_row[f] /= l;
  *lse = m + log(l);
}

/* Full attention: o dense [Bo][Bi][Nq][Hh][d], lse dense [Bo][Bi][Hh][Nq]. */
void oracle_attention(const float* q, const float* k, const float* v,
                      double* o, double* lse, long Bo, long Bi, long Hh,
                      long Nq, long Nk, long d, const long* sq, const long* sk,
                      const long* sv, double scale, int mask, long window) {
  long rows = Bo * Bi * Hh * Nq;
#pragma omp parallel
  {
    double sbuf[Nk > 0 ? Nk : 1];
#pragma omp for schedule(dynamic, 16)
    for (long r = 0; r < rows; ++r) {
      long i = r % Nq, h = (r / Nq) % Hh, bi = (r / (Nq * Hh)) % Bi,
           bo = r / (Nq * Hh * Bi);
      double* orow = o + (((bo * Bi + bi) * Nq + i) * Hh + h) * d;
      attn_row(q, k, v, sq, sk, sv, bo, bi, h, i, Nk, d, scale, mask, window,
               orow, &lse[r], sbuf);
    }
  }
}

/* Selected rows only: rows[r] = (bo, bi, h, i); o_rows [n][d], lse_rows [n]. */
void oracle_attention_rows(const float* q, const float* k, const float* v,
                           const long* rows, long n_rows, double* o_rows,
                           double* lse_rows, long Nk, long d, const long* sq,
                           const long* sk, const long* sv, double scale,
                           int mask, long window) {
#pragma omp parallel
  {
    double sbuf[Nk > 0 ? Nk : 1];
#pragma omp for schedule(dynamic, 1)
    for (long r = 0; r < n_rows; ++r) {
      const long* rr = rows + 4 * r;
      attn_row(q, k, v, sq, sk, sv, rr[0], rr[1], rr[2], rr[3], Nk, d, scale,
               mask, window, o_rows + r * d, &lse_rows[r], sbuf);
    }
  }
}

/* ------------------------------------------------------------------------ */
/* Tile visits: number of (head, query tile, key tile) triples that hold at  */
/* least one visible (i, j) pair, with tile_q x tile_k tiles over N x N.     */
/* A tile pair holds differences i - j over the whole integer interval       */
/* [qi0 - kj1, qi1 - kj0]; it is visited iff that interval meets the visible */
/* differences (>= 0 for causal, [0, window) for causal window, all for none).*/
/* ------------------------------------------------------------------------ */
/* ------------------------------------------------------------------------ */
/* Attention backward (training step of the pseudo-head attention, the      */
/* gradient of the forward above).  Dense tensors [B][N][Hh][d] (query and  */
/* key sequences of one length N), dout as o.  Per (b, head) and query row i */
/* with visible keys j, by the plain definitions:                            */
/*   P_ij  = softmax_j(scale <q_i, k_j>)          (two-pass, max-shifted)     */
/*   dV_j += P_ij dO_i                                                        */
/*   dP_ij = <dO_i, v_j>                                                      */
/*   D_i   = sum_j P_ij dP_ij                                                 */
/*   dS_ij = P_ij (dP_ij - D_i)                                               */
/*   dQ_i  = scale sum_j dS_ij k_j,   dK_j += scale dS_ij q_i                 */
/* Heads are independent (parallel); inside a head the rows are summed in   */
/* row order, so the result does not depend on scheduling.                  */
/* With absolute != 0 the same sums are formed from absolute values of every */
/* term (sum |dS||k|, sum |dS||q|, sum P |dO|): the magnitudes that bound     */
/* rounding errors of an implementation that rounds dS and P.                */
/* ------------------------------------------------------------------------ */
void oracle_attention_bwd(const float* q, const float* k, const float* v,
                          const float* dout, double* dq, double* dk, double* dv,
                          long B, long Hh, long N, long d, double scale,
                          int mask, long window, int absolute) {
  const long row = Hh * d;  /* elements between consecutive tokens */
#pragma omp parallel for schedule(dynamic, 1) collapse(2)
  for (long b = 0; b < B; ++b)
    for (long h = 0; h < Hh; ++h) {
      const long base = b * N * row + h * d;
      double* P = (double*)malloc(sizeof(double) * (size_t)N);
      double* dP = (double*)malloc(sizeof(double) * (size_t)N);
      for (long j = 0; j < N; ++j)
        for (long f = 0; f < d; ++f) {
          dk[base + j * row + f] = 0.0;
          dv[base + j * row + f] = 0.0;
        }
      for (long i = 0; i < N; ++i) {
        const float* qi = q + base + i * row;
        const float* gi = dout + base + i * row;
        double m = -INFINITY;
        for (long j = 0; j < N; ++j) {
          if (!visible(i, j, mask, window)) { P[j] = -INFINITY; continue; }
          const float* kj = k + base + j * row;
          double dot = 0.0;
          for (long f = 0; f < d; ++f) dot += (double)qi[f] * (double)kj[f];
          P[j] = scale * dot;
          if (P[j] > m) m = P[j];
        }
        double l = 0.0;
        for (long j = 0; j < N; ++j) {
          if (P[j] == -INFINITY) { P[j] = 0.0; continue; }
          P[j] = exp(P[j] - m);
          l += P[j];
        }
        double D = 0.0;
        for (long j = 0; j < N; ++j) {
          if (l > 0.0) P[j] /= l;
          dP[j] = 0.0;
          if (P[j] == 0.0) continue;
          const float* vj = v + base + j * row;
          for (long f = 0; f < d; ++f) dP[j] += (double)gi[f] * (double)vj[f];
          D += P[j] * dP[j];
        }
        double* dqi = dq + base + i * row;
        for (long f = 0; f < d; ++f) dqi[f] = 0.0;
        for (long j = 0; j < N; ++j) {
          if (P[j] == 0.0) continue;
          const double ds = P[j] * (dP[j] - D);
          const float* kj = k + base + j * row;
          double* dkj = dk + base + j * row;
          double* dvj = dv + base + j * row;
          if (absolute) {
            for (long f = 0; f < d; ++f) {
              dqi[f] += scale * fabs(ds) * fabs((double)kj[f]);
              dkj[f] += scale * fabs(ds) * fabs((double)qi[f]);
              dvj[f] += P[j] * fabs((double)gi[f]);
            }
            continue;
          }
          for (long f = 0; f < d; ++f) {
            dqi[f] += scale * ds * (double)kj[f];
            dkj[f] += scale * ds * (double)qi[f];
            dvj[f] += P[j] * (double)gi[f];
          }
        }
      }
      free(P);
      free(dP);
    }
}

long oracle_tile_visits(long N, long heads, int mask, long window, long tile_q,
                        long tile_k) {
  long tq = (N + tile_q - 1) / tile_q, tk = (N + tile_k - 1) / tile_k;
  long count = 0;
  for (long a = 0; a < tq; ++a) {
    long qi0 = a * tile_q, qi1 = (a + 1) * tile_q - 1;
    if (qi1 > N - 1) qi1 = N - 1;
    for (long b = 0; b < tk; ++b) {
      long kj0 = b * tile_k, kj1 = (b + 1) * tile_k - 1;
      if (kj1 > N - 1) kj1 = N - 1;
      long dlo = qi0 - kj1, dhi = qi1 - kj0;
      long vlo, vhi;
      if (mask == 0) { ++count; continue; }
      vlo = 0;
      vhi = (mask == 2) ? window - 1 : N;
      if (dhi >= vlo && dlo <= vhi) ++count;
    }
  }
  return count * heads;
}

/* ------------------------------------------------------------------------ */
/* Mask-unit gather / scatter (byte copies of C * elem_bytes per token).     */
/* x is the row-major token grid [B][grid_h*grid_w][C]; keep [B][n_keep]     */
/* lists kept unit ids; out/src is [B][n_keep][mu_h*mu_w][C].                */
/* ------------------------------------------------------------------------ */
static long unit_token(long u, long t, long grid_w, long mu_h, long mu_w) {
  long units_per_row = grid_w / mu_w;
  long uy = u / units_per_row, ux = u % units_per_row;
  long ty = t / mu_w, tx = t % mu_w;
  return (uy * mu_h + ty) * grid_w + ux * mu_w + tx;
}

void oracle_mu_gather(const uint8_t* x, const int32_t* keep, uint8_t* out,
                      long B, long grid_h, long grid_w, long mu_h, long mu_w,
                      long n_keep, long C, long elem_bytes) {
  long T = mu_h * mu_w, G = grid_h * grid_w, row = C * elem_bytes;
  for (long b = 0; b < B; ++b)
    for (long kk = 0; kk < n_keep; ++kk)
      for (long t = 0; t < T; ++t) {
        long tok = unit_token(keep[b * n_keep + kk], t, grid_w, mu_h, mu_w);
        memcpy(out + ((b * n_keep + kk) * T + t) * row, x + (b * G + tok) * row,
               (size_t)row);
      }
}

void oracle_mu_scatter(const uint8_t* src, const int32_t* keep, uint8_t* x,
                       long B, long grid_h, long grid_w, long mu_h, long mu_w,
                       long n_keep, long C, long elem_bytes) {
  long T = mu_h * mu_w, G = grid_h * grid_w, row = C * elem_bytes;
  for (long b = 0; b < B; ++b)
    for (long kk = 0; kk < n_keep; ++kk)
      for (long t = 0; t < T; ++t) {
        long tok = unit_token(keep[b * n_keep + kk], t, grid_w, mu_h, mu_w);
        memcpy(x + (b * G + tok) * row, src + ((b * n_keep + kk) * T + t) * row,
               (size_t)row);
      }
}
