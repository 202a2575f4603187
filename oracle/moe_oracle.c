/*
 * CPU oracle of the MoE-layer forward pass -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg load
 * this library.  The product (the CUDA path behind include/moe.h) never calls
 * it, and the two share no code: not a header, a helper or a constant.
 *
 * What it computes is the plain definition of the layer described in
 *   Weave abstract (arXiv 2609.21483): routing, then the experts, then the
 *     weighted combine of the expert outputs;
 *   xxqk.cn/news/665650 section 1 (the MoE megakernel: router, top-k expert
 *     selection, the expert matrix products, weighted merge of the results);
 *   m.xxqk.cn/news/657744 section 2.1 (an expert's up projection precedes its
 *     down projection; permute/combine move tokens between experts).
 * The method on those pages changes only the scheduling of this computation
 * (xxqk.cn/news/665650 section 3.1: only the scheduling policy changes, not
 * the operators or the weights), so the oracle is the definition written out:
 *   1. decode the bf16 inputs exactly to double;
 *   2. L[t,e] = sum_i x[t,i] * Wr[e,i] + b[e]                  (fp64)
 *   3. p[t,:] = softmax(L[t,:]) over all E experts              (fp64, max-shifted)
 *   4. top-k: order experts by (p descending, expert ascending), keep k
 *   5. w_j = p_j / sum of the k kept p                          (renormalise)
 *   6. counts, offsets, perm, pos by the canonical permutation (experts
 *      ascending, tokens ascending inside an expert)
 *   7. per (t, j) with e = idx[t,j]:
 *        g = Wg[e] x_t, u = Wu[e] x_t                          (fp64)
 *        h = bf16(silu(g) * u), silu(z) = z / (1 + exp(-z))   (the one rounding
 *                                                              inside the layer)
 *        y = Wd[e] h                                          (fp64)
 *   8. out[t] = bf16( sum_{j=0..k-1} w_j y_j  +  y_shared )  (shared expert,
 *      index E, weight 1, same h rounding, added after the routed sum)
 *   9. (optional, orc_residual_rmsnorm) the residual add and the RMSNorm that
 *      end the megakernel of xxqk.cn/news/665650 section 1:
 *      out = bf16(residual + the step-8 sum), norm = bf16(out / rms(out) * gamma)
 *  10. (orc_movers) the spatial split of the Weave abstract: once routing is
 *      known, the CTAs are divided between data movement and the expert GEMMs
 *      in the ratio of the two sides' work (the formula is this project's
 *      reading; see orc_movers).
 * Layouts: x [T,d], Wr [E,d], Wg/Wu [E+S,f,d], Wd [E+S,d,f], row-major bf16.
 * Rounding to bf16 is round-to-nearest, ties-to-even, straight from double.
 *
 * Readings where the pages are silent: the router bias is added to the logits
 * and used both to select and to weight; ties in top-k go to the lower expert
 * index; the permutation order is experts ascending then tokens ascending.
 *
 * Parity pins (tests/test_oracle_pins.py): exhaustive bf16 round trip and
 * half-way cases; brute-force sorting for top-k; sum of weights = 1 and k = E
 * giving the full softmax; brute-force recount of the permutation; k = E
 * giving the dense mixture; identical experts giving one FFN; a hand-computed
 * layer; for step 9, a zero residual giving the plain output, a hand-computed
 * row, unit mean square and scale invariance, a constant row giving the
 * signed gamma; for step 10, the byte and FLOP totals recounted copy by copy
 * and row by row, the split against a brute-force minimiser of the slower
 * side's time, and its clamps.  Nothing here is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Scratch allocation: the oracle stops (abort) rather than compute on a NULL
 * buffer when the host is out of memory. */
static void* orc_alloc(size_t n, int zero) {
  void* q = zero ? calloc(n ? n : 1, 1) : malloc(n ? n : 1);
  if (!q) abort();
  return q;
}

/* ---- bf16 <-> double ------------------------------------------------------ */

double orc_bf16_to_f64(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* Round a double to the nearest bf16 value, ties to even.  The value is split
 * as m * 2^e (m in [0.5, 1)); bf16 keeps 8 significant bits, i.e. a quantum of
 * 2^(e-8), never finer than the subnormal quantum 2^-133.  nearbyint in the
 * default rounding mode rounds half to even. */
uint16_t orc_f64_to_bf16(double v) {
  if (isnan(v)) return (uint16_t)0x7FC0;
  if (isinf(v)) return v > 0 ? (uint16_t)0x7F80 : (uint16_t)0xFF80;
  if (v == 0.0) return signbit(v) ? (uint16_t)0x8000 : (uint16_t)0x0000;
  int e;
  (void)frexp(v, &e);
  int q = e - 8;
  if (q < -133) q = -133;
  double r = nearbyint(ldexp(v, -q));
  double rounded = ldexp(r, q);
  if (fabs(rounded) >= ldexp(1.0, 128))
    return v > 0 ? (uint16_t)0x7F80 : (uint16_t)0xFF80;
  float fr = (float)rounded; /* exact: at most 8 significant bits */
  uint32_t u;
  memcpy(&u, &fr, 4);
  if (rounded == 0.0) return signbit(v) ? (uint16_t)0x8000 : (uint16_t)0x0000;
  return (uint16_t)(u >> 16);
}

void orc_bf16_to_f64_array(int64_t n, const uint16_t* in, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_to_f64(in[i]);
}

void orc_f64_to_bf16_array(int64_t n, const double* in, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_f64_to_bf16(in[i]);
}

double orc_silu(double z) { return z / (1.0 + exp(-z)); }

/* ---- step 2: router logits -------------------------------------------------- */

void orc_router_logits(int T, int d, int E, const uint16_t* x, const uint16_t* wr,
                       const float* bias, double* L) {
  for (int t = 0; t < T; ++t) {
    const uint16_t* xr = x + (size_t)t * d;
    for (int e = 0; e < E; ++e) {
      const uint16_t* wrow = wr + (size_t)e * d;
      double acc = 0.0;
      for (int i = 0; i < d; ++i) acc += orc_bf16_to_f64(xr[i]) * orc_bf16_to_f64(wrow[i]);
      if (bias) acc += (double)bias[e];
      L[(size_t)t * E + e] = acc;
    }
  }
}

/* ---- steps 3-5: softmax over all E, top-k, renormalise ---------------------- */

/* For each token: p = softmax(L) over all E; idx = the k experts first in the
 * order (p descending, expert ascending); w_j = p_j / sum_kept p.  Also
 * returns the full softmax (p_full, optional) and the routing margin
 * gap[t] = L_(k) - L_(k+1), the distance between the k-th and (k+1)-th
 * largest logits (1e300 when k == E). */
void orc_topk(int T, int E, int k, const double* L, int32_t* idx, double* w, double* p_full,
              double* gap) {
  double* p = (double*)orc_alloc(sizeof(double) * (size_t)E, 0);
  char* taken = (char*)orc_alloc((size_t)E, 0);
  for (int t = 0; t < T; ++t) {
    const double* l = L + (size_t)t * E;
    double mx = l[0];
    for (int e = 1; e < E; ++e)
      if (l[e] > mx) mx = l[e];
    double z = 0.0;
    for (int e = 0; e < E; ++e) {
      p[e] = exp(l[e] - mx);
      z += p[e];
    }
    for (int e = 0; e < E; ++e) p[e] /= z;
    if (p_full)
      for (int e = 0; e < E; ++e) p_full[(size_t)t * E + e] = p[e];
    memset(taken, 0, (size_t)E);
    double kept = 0.0;
    for (int j = 0; j < k; ++j) {
      int best = -1;
      for (int e = 0; e < E; ++e) {
        if (taken[e]) continue;
        if (best < 0 || p[e] > p[best]) best = e; /* strict: lower e wins ties */
      }
      taken[best] = 1;
      idx[(size_t)t * k + j] = best;
      kept += p[best];
    }
    for (int j = 0; j < k; ++j) w[(size_t)t * k + j] = p[idx[(size_t)t * k + j]] / kept;
    if (gap) {
      if (k >= E) {
        gap[t] = 1e300;
      } else {
        double lowest_kept = 1e308, highest_left = -1e308;
        for (int e = 0; e < E; ++e) {
          if (taken[e] && l[e] < lowest_kept) lowest_kept = l[e];
          if (!taken[e] && l[e] > highest_left) highest_left = l[e];
        }
        gap[t] = lowest_kept - highest_left;
      }
    }
  }
  free(taken);
  free(p);
}

/* ---- step 6: counts, offsets, permutation ---------------------------------- */

/* counts[e] = number of (t, j) with idx[t,j] = e; offsets = exclusive prefix
 * sum (offsets[E] = T*k); perm[offsets[e] + r] = the r-th smallest token that
 * selected e; pos[t,j] = the row of (t, idx[t,j]) in that order.  Returns 0,
 * or -1 when an index is out of range or a token selects an expert twice. */
int orc_permute(int T, int E, int k, const int32_t* idx, int32_t* counts, int32_t* offsets,
                int32_t* perm, int32_t* pos) {
  for (int t = 0; t < T; ++t)
    for (int j = 0; j < k; ++j) {
      int e = idx[(size_t)t * k + j];
      if (e < 0 || e >= E) return -1;
      for (int j2 = 0; j2 < j; ++j2)
        if (idx[(size_t)t * k + j2] == e) return -1;
    }
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (int t = 0; t < T; ++t)
    for (int j = 0; j < k; ++j) counts[idx[(size_t)t * k + j]] += 1;
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  int row = 0;
  for (int e = 0; e < E; ++e)
    for (int t = 0; t < T; ++t)
      for (int j = 0; j < k; ++j)
        if (idx[(size_t)t * k + j] == e) {
          perm[row] = t;
          pos[(size_t)t * k + j] = row;
          ++row;
        }
  return 0;
}

/* ---- step 7: one expert on one token --------------------------------------- */

/* y[c] = sum_r Wd[c, r] * h[r], h[r] = bf16(silu(g_r) * u_r),
 * g_r = sum_i Wg[r, i] x[i], u_r = sum_i Wu[r, i] x[i].  wg/wu point at the
 * expert's [f, d] block, wd at its [d, f] block.  h_out (optional) gets h. */
void orc_expert_ffn(int d, int f, const uint16_t* x_row, const uint16_t* wg, const uint16_t* wu,
                    const uint16_t* wd, double* h_out, double* y) {
  double* h = (double*)orc_alloc(sizeof(double) * (size_t)f, 0);
  double* xd = (double*)orc_alloc(sizeof(double) * (size_t)d, 0);
  for (int i = 0; i < d; ++i) xd[i] = orc_bf16_to_f64(x_row[i]);
  for (int r = 0; r < f; ++r) {
    const uint16_t* gr = wg + (size_t)r * d;
    const uint16_t* ur = wu + (size_t)r * d;
    double g = 0.0, u = 0.0;
    for (int i = 0; i < d; ++i) {
      g += orc_bf16_to_f64(gr[i]) * xd[i];
      u += orc_bf16_to_f64(ur[i]) * xd[i];
    }
    h[r] = orc_bf16_to_f64(orc_f64_to_bf16(orc_silu(g) * u));
  }
  for (int c = 0; c < d; ++c) {
    const uint16_t* dr = wd + (size_t)c * f;
    double acc = 0.0;
    for (int r = 0; r < f; ++r) acc += orc_bf16_to_f64(dr[r]) * h[r];
    y[c] = acc;
  }
  if (h_out) memcpy(h_out, h, sizeof(double) * (size_t)f);
  free(xd);
  free(h);
}

/* ---- step 8: one output row ------------------------------------------------- */

/* out = bf16( sum_j w_j * FFN_{idx_j}(x) + FFN_E(x) [if S == 1] ), fp64 sum in
 * slot order j = 0..k-1, then the shared expert.  acc (optional) gets the
 * value before the final rounding. */
void orc_token_out(int d, int f, int E, int k, int S, const uint16_t* x_row, const int32_t* idx_row,
                   const double* w_row, const uint16_t* wg, const uint16_t* wu, const uint16_t* wd,
                   double* acc_out, uint16_t* out_row) {
  double* acc = (double*)orc_alloc(sizeof(double) * (size_t)d, 1);
  double* y = (double*)orc_alloc(sizeof(double) * (size_t)d, 0);
  size_t fd = (size_t)f * (size_t)d;
  for (int j = 0; j < k; ++j) {
    int e = idx_row[j];
    orc_expert_ffn(d, f, x_row, wg + (size_t)e * fd, wu + (size_t)e * fd, wd + (size_t)e * fd,
                   NULL, y);
    for (int c = 0; c < d; ++c) acc[c] += w_row[j] * y[c];
  }
  for (int s = 0; s < S; ++s) {
    int e = E + s;
    orc_expert_ffn(d, f, x_row, wg + (size_t)e * fd, wu + (size_t)e * fd, wd + (size_t)e * fd,
                   NULL, y);
    for (int c = 0; c < d; ++c) acc[c] += y[c];
  }
  for (int c = 0; c < d; ++c) out_row[c] = orc_f64_to_bf16(acc[c]);
  if (acc_out) memcpy(acc_out, acc, sizeof(double) * (size_t)d);
  free(y);
  free(acc);
}

/* ---- the layer on a list of tokens ------------------------------------------ */

/* For each listed token t: route it (steps 2-5) and compute its output row
 * (steps 7-8).  Each output row depends on its own token only, so a subset
 * of rows is exact for those rows.  out_rows is [n_tok, d]. */
void orc_layer_tokens(int T, int d, int f, int E, int k, int S, const uint16_t* x,
                      const uint16_t* wr, const float* bias, const uint16_t* wg,
                      const uint16_t* wu, const uint16_t* wd, int n_tok, const int32_t* tokens,
                      uint16_t* out_rows, double* acc_rows) {
  double* L = (double*)orc_alloc(sizeof(double) * (size_t)E, 0);
  int32_t* idx = (int32_t*)orc_alloc(sizeof(int32_t) * (size_t)k, 0);
  double* w = (double*)orc_alloc(sizeof(double) * (size_t)k, 0);
  for (int n = 0; n < n_tok; ++n) {
    int t = tokens ? tokens[n] : n;
    if (t < 0 || t >= T) continue;
    const uint16_t* xr = x + (size_t)t * d;
    orc_router_logits(1, d, E, xr, wr, bias, L);
    orc_topk(1, E, k, L, idx, w, NULL, NULL);
    orc_token_out(d, f, E, k, S, xr, idx, w, wg, wu, wd,
                  acc_rows ? acc_rows + (size_t)n * d : NULL, out_rows + (size_t)n * d);
  }
  free(w);
  free(idx);
  free(L);
}

/* ---- residual add and RMSNorm after the combine ------------------------------ */

/* The MoE megakernel of xxqk.cn/news/665650 section 1 ends with the residual
 * add and the normalisation.  The pages give neither form; the reading here is
 * the pre-norm block of the models they discuss: the layer's output is added
 * to the residual stream, and the sum, as stored in bf16, is RMS-normalised
 * for the next sublayer:
 *   out[c]      = bf16( residual[c] + acc[c] )       acc: the combine's value
 *                                                     before rounding (fp64)
 *   ms          = (1/d) sum_c out[c]^2                (out decoded exactly)
 *   norm_out[c] = bf16( out[c] / sqrt(ms + eps) * gamma[c] )
 * Rows are [n, d]; norm_f64 (optional) receives the values before rounding. */
void orc_residual_rmsnorm(int n, int d, const double* acc, const uint16_t* residual,
                          const uint16_t* gamma, double eps, uint16_t* out, uint16_t* norm_out,
                          double* norm_f64) {
  for (int r = 0; r < n; ++r) {
    const double* a = acc + (size_t)r * d;
    const uint16_t* res = residual + (size_t)r * d;
    uint16_t* o = out + (size_t)r * d;
    double ms = 0.0;
    for (int c = 0; c < d; ++c) {
      o[c] = orc_f64_to_bf16(orc_bf16_to_f64(res[c]) + a[c]);
      const double h = orc_bf16_to_f64(o[c]);
      ms += h * h;
    }
    ms /= (double)d;
    const double inv = 1.0 / sqrt(ms + eps);
    for (int c = 0; c < d; ++c) {
      const double v = orc_bf16_to_f64(o[c]) * inv * orc_bf16_to_f64(gamma[c]);
      norm_out[(size_t)r * d + c] = orc_f64_to_bf16(v);
      if (norm_f64) norm_f64[(size_t)r * d + c] = v;
    }
  }
}

/* ---- step 10: the spatial split of the CTAs --------------------------------
 * Weave abstract: once routing completes, the layer's communication and
 * computation volumes are known, and a cost model inside the megakernel
 * divides the SMs into communication and computation workers so that the two
 * sides' throughputs match.  The page gives no formula; this project reads it
 * as follows, with the work of each side in worker-seconds:
 *   a = B_move / beta                      bytes the movers copy, at beta B/s
 *       B_move = T*k rows gathered          (each read and written: 2 * d * 2 B)
 *              + T*(k+S) expert-output rows read by the combine (d * ybytes B
 *                each: every routed slot and the shared expert's row)
 *              + T rows written by the combine (d * 2 B each)
 *   b = max(F / phi, N * G_w / BW)         the GEMM side: its FLOPs at phi
 *       F   = 6 * d * f per routed or shared row (T*k + T*S rows)   FLOP/s per
 *       G_w = 3 * f * d bf16 weights per touched expert              worker,
 *             (routed experts with a token, plus S shared)           or the
 *                                                  weight stream at BW for N
 *   M* = clamp(round(N * a / (a + b)), 1, N - 1)   (N * a / (a + b) minimises
 *        max(a / M, b / (N - M)), the slower side's time, over real M)
 * ybytes is the size in bytes of one stored expert-output value, summed over
 * the pieces the combine reads for it: 2 when the outputs are kept as bf16,
 * 4 * ks when they are kept as ks fp32 partial sums of a K-split down
 * projection (the caller passes the size of the layout in use).
 * M* is an integer decided by floating point, so it is computed in fp32, the
 * precision the kernel decides in, rounding half to even; *m_cont receives
 * N * a / (a + b) before rounding. */
int orc_movers(int T, int d, int f, int k, int S, int touched_routed, int N, float ybytes,
               float beta, float phi, float bw, float* m_cont) {
  const float Tk = (float)T * (float)k;
  const float gather = Tk * (float)d * 2.0f * 2.0f;
  const float combine_read = ((float)T * (float)(k + S)) * (float)d * ybytes;
  const float combine_write = (float)T * (float)d * 2.0f;
  const float b_move = gather + combine_read + combine_write;
  const float flops = 6.0f * (Tk + (float)T * (float)S) * (float)d * (float)f;
  const float wbytes = (float)(touched_routed + S) * 3.0f * (float)f * (float)d * 2.0f;
  const float a = b_move / beta;
  const float b_flops = flops / phi;
  const float b_bytes = (float)N * wbytes / bw;
  const float b = b_flops > b_bytes ? b_flops : b_bytes;
  const float x = (float)N * a / (a + b);
  if (m_cont) *m_cont = x;
  int m = (int)nearbyintf(x);
  const int hi = N - 1 > 1 ? N - 1 : 1;
  if (m > hi) m = hi;
  if (m < 1) m = 1;
  return m;
}
