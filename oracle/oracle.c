/*
 * oracle.c - plain, slow CPU reference of the exact width-k verify pass.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the tests, the smoke check and the bench's CPU
 * baseline use it.  It shares no code, header, table or helper with the CUDA
 * library; the two meet only in the seeded input generator.
 *
 * Arithmetic is float64 throughout (inputs are bf16 / fp32 and widen exactly),
 * summed in ascending index order, with no blocking or fusion: each function
 * is the plain definition the pages give.  Pages are cited by title:
 *   [T] "Flash-Next optimization transfer to Ornith and Qwen 27B"
 *   [R] "Red Lite dev45 - speculative decoding with the Qwen3-Next MTP block"
 *   [F] "QWEN38FLASH.md - Plan for supporting Qwen/Qwen3.8-Flash-Next"
 * Readings taken where the pages are silent are marked READING.
 *
 * Pins (checked by the CPU tests against closed forms, brute force and
 * invariants, not against this file): q4 nibble order and group indexing,
 * exact integer products, top-k order/ties and softmax identities, the
 * single-expert special case, the delta-rule identities (zero state, unit
 * gates, beta = 0, decay 1/2), conv taps, norms, greedy acceptance
 * (hand-worked cases, numpy's argmax, the serial-decoding identity), the
 * attention verify (binary16 rounding against numpy's cast, one-key and
 * zero-query closed forms, RoPE of one-hot keys, relative-position
 * invariance, the two-key score gap, k rows against k single-row steps, the
 * query-head grouping).
 *
 * Timing only: compiled with -fopenmp (a second library beside the plain
 * one), the output rows of each Q4 product are spread over the host cores.
 * Every output is still the same sequential float64 sum, so that build gives
 * bit-identical results; the plain build is single-threaded.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Threads the products may use (1 in the plain build). */
int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

static int thread_index(void) {
#ifdef _OPENMP
  return omp_get_thread_num();
#else
  return 0;
#endif
}

/* ------------------------------------------------------------ bf16 helpers */

/* bf16 bit pattern -> value (exact). */
static double bf16_value(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* value -> nearest bf16 (ties to even), rounded once from float64. */
uint16_t oracle_round_bf16(double v) {
  if (v == 0.0 || !isfinite(v)) {
    float f = (float)v;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
  }
  int e;
  double m = frexp(v, &e);             /* v = m * 2^e, 0.5 <= |m| < 1 */
  double scaled = ldexp(m, 8);         /* 8 significant bits: 128 <= |scaled| < 256 */
  double r = nearbyint(scaled);        /* default rounding mode: ties to even */
  float f = (float)ldexp(r, e - 8);    /* exact: 8-bit significand */
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return (uint16_t)(u >> 16);
}

static double sigmoid(double t) { return 1.0 / (1.0 + exp(-t)); }
static double silu(double t) { return t / (1.0 + exp(-t)); }
static double softplus(double t) { return (t > 0 ? t : 0.0) + log1p(exp(-fabs(t))); }

/* ------------------------------------------------------------- q4 weights */

/*
 * Affine Q4, group size 64 ([T] table "Shared architecture and implemented
 * paths": "affine Q4, group size 64, and compatible BF16 tensors").
 * READING (layout; the pages give only the format name): packed uint32
 * [n_out, k_in/8] row-major with column c in bits 4*(c%8).., scales and
 * biases bf16 [n_out, k_in/64], w = scale * q + bias.
 */
static double q4_weight(const uint32_t* packed, const uint16_t* scales,
                        const uint16_t* biases, int k_in, int64_t n, int c) {
  uint32_t word = packed[n * (k_in / 8) + c / 8];
  int q = (int)((word >> (4 * (c % 8))) & 15u);
  double s = bf16_value(scales[n * (k_in / 64) + c / 64]);
  double b = bf16_value(biases[n * (k_in / 64) + c / 64]);
  return s * q + b;
}

/*
 * y[r][n] = sum_c w[n][c] * x[r][c]  for r < k, n < n_out (ascending c).
 * Width-k is k independent width-1 products by construction ([T] "Exact
 * verification kernels": agreement with serial QMV; [R] "What it is").
 * x: bf16 [k, k_in] (row r at x + r*ldx); y: float64 [k, n_out].
 */
int oracle_q4_qmv(const uint32_t* packed, const uint16_t* scales, const uint16_t* biases,
                  int n_out, int k_in, const uint16_t* x, int64_t ldx, int k, double* y) {
  if (k_in % 64 != 0 || n_out < 0 || k < 0) return 1;
  /* one dequantised row per thread */
  double* w_all = (double*)malloc(sizeof(double) * (size_t)k_in * (size_t)oracle_num_threads());
  if (!w_all) return 2;
#pragma omp parallel for schedule(static)
  for (int64_t n = 0; n < n_out; ++n) {
    double* w = w_all + (size_t)thread_index() * (size_t)k_in;
    for (int c = 0; c < k_in; ++c) w[c] = q4_weight(packed, scales, biases, k_in, n, c);
    for (int r = 0; r < k; ++r) {
      double acc = 0.0;
      for (int c = 0; c < k_in; ++c) acc += w[c] * bf16_value(x[r * ldx + c]);
      y[(int64_t)r * n_out + n] = acc;
    }
  }
  free(w_all);
  return 0;
}

/* ------------------------------------------------------------ router top-k */

/*
 * Top-T routing of one row ([T] "Exact verification kernels": top-eight of
 * 256; [F] 2.3: router over 512 logits, top-k).  READING (scoring function
 * left open by [F] 2.3): softmax over all E, keep the T largest, renormalise;
 * this equals the softmax of the T selected logits, which is what is
 * computed.  Order: descending logit; equal logits: lower expert index first
 * (READING, the pages are silent).
 */
int oracle_route_topk(const float* logits, int64_t ld, int k, int E, int T,
                      int32_t* idx, double* w) {
  if (T < 1 || T > E) return 1;
  char* taken = (char*)malloc((size_t)E);
  if (!taken) return 2;
  for (int r = 0; r < k; ++r) {
    const float* l = logits + r * ld;
    memset(taken, 0, (size_t)E);
    for (int j = 0; j < T; ++j) {
      int best = -1;
      for (int e = 0; e < E; ++e)
        if (!taken[e] && (best < 0 || l[e] > l[best])) best = e;
      taken[best] = 1;
      idx[r * T + j] = best;
    }
    double top = l[idx[r * T]];
    double sum = 0.0;
    for (int j = 0; j < T; ++j) sum += exp((double)l[idx[r * T + j]] - top);
    for (int j = 0; j < T; ++j) w[r * T + j] = exp((double)l[idx[r * T + j]] - top) / sum;
  }
  free(taken);
  return 0;
}

/* ---------------------------------------------------------- routed experts */

/*
 * One SwiGLU expert applied to one row: g = W_gu[0..I).x, u = W_gu[I..2I).x
 * ([F] 2.3: gate+up concatenated [2I, H], SwiGLU), h = bf16(silu(g)*u),
 * p = W_d.h.  READING: h is rounded to bf16 because the down projection, like
 * every Q4 product of [T], takes BF16 activation rows.
 */
static int expert_row(const uint32_t* gp, const uint16_t* gs, const uint16_t* gb,
                      const uint32_t* dp, const uint16_t* ds, const uint16_t* db,
                      int H, int I, const uint16_t* xrow, double* p, uint16_t* h_out) {
  double* gu = (double*)malloc(sizeof(double) * 2 * (size_t)I);
  uint16_t* h = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)I);
  if (!gu || !h) { free(gu); free(h); return 2; }
  oracle_q4_qmv(gp, gs, gb, 2 * I, H, xrow, H, 1, gu);
  for (int i = 0; i < I; ++i) h[i] = oracle_round_bf16(silu(gu[i]) * gu[I + i]);
  if (h_out) memcpy(h_out, h, sizeof(uint16_t) * (size_t)I);
  oracle_q4_qmv(dp, ds, db, H, I, h, I, 1, p);
  free(gu);
  free(h);
  return 0;
}

/*
 * Routed MoE for k rows ([T] "Exact verification kernels": gathered
 * affine-Q4 experts with fused gate/up; [R] "What it is": all (expert,row)
 * pairs in one dispatch, one tail).  y[r] = sum_{j<T} w[r][j] * p_{r,j},
 * ascending j ([F] 5.3 fused sum over the top-k), then, if a shared expert is
 * given, + sigmoid(sg[r]) * shared(x[r]) ([F] 2.3: 10 routed + 1 shared;
 * READING: the shared expert's sigmoid gate as in the Qwen3-Next lineage [F]
 * section 3 names, added after the routed sum).
 * Gate/up stack [E, 2I, H], down stack [E, H, I].  h_out (optional) receives
 * the bf16 SwiGLU rows [k, T(+1), I].
 */
int oracle_gather_experts(const uint32_t* gup, const uint16_t* gus, const uint16_t* gub,
                          const uint32_t* dnp, const uint16_t* dns, const uint16_t* dnb,
                          int E, int H, int I, const float* logits, int64_t ld, int T,
                          const uint16_t* x, int k, int32_t* idx, double* w, double* y,
                          const uint32_t* sgup, const uint16_t* sgus, const uint16_t* sgub,
                          const uint32_t* sdnp, const uint16_t* sdns, const uint16_t* sdnb,
                          const float* sg_logit, uint16_t* h_out) {
  if (H % 64 || I % 64) return 1;
  int rc = oracle_route_topk(logits, ld, k, E, T, idx, w);
  if (rc) return rc;
  int slots = T + (sgup ? 1 : 0);
  double* p = (double*)malloc(sizeof(double) * (size_t)H);
  if (!p) return 2;
  const int64_t gu_w = (int64_t)2 * I * (H / 8), gu_g = (int64_t)2 * I * (H / 64);
  const int64_t dn_w = (int64_t)H * (I / 8), dn_g = (int64_t)H * (I / 64);
  for (int r = 0; r < k; ++r) {
    double* yr = y + (int64_t)r * H;
    for (int n = 0; n < H; ++n) yr[n] = 0.0;
    for (int j = 0; j < T; ++j) {
      int64_t e = idx[r * T + j];
      rc = expert_row(gup + e * gu_w, gus + e * gu_g, gub + e * gu_g,
                      dnp + e * dn_w, dns + e * dn_g, dnb + e * dn_g, H, I,
                      x + (int64_t)r * H, p, h_out ? h_out + ((int64_t)r * slots + j) * I : NULL);
      if (rc) { free(p); return rc; }
      for (int n = 0; n < H; ++n) yr[n] += w[r * T + j] * p[n];
    }
    if (sgup) {
      rc = expert_row(sgup, sgus, sgub, sdnp, sdns, sdnb, H, I, x + (int64_t)r * H, p,
                      h_out ? h_out + ((int64_t)r * slots + T) * I : NULL);
      if (rc) { free(p); return rc; }
      double gate = sigmoid((double)sg_logit[r * ld]);
      for (int n = 0; n < H; ++n) yr[n] += gate * p[n];
    }
  }
  free(p);
  return 0;
}

/* ------------------------------------------------------- Gated DeltaNet */

/*
 * k-row Gated DeltaNet verify, one row after the other, every row starting
 * from the previous row's state ([R] "What it is": row 1 runs from row 0's
 * state; [F] 2.1 per-token pipeline):
 *   1. causal depthwise conv over the q|k|v channels: window = the last W
 *      input rows ending at the current one ([F] 3.1 table: 3-tap history +
 *      current, 4 weights per channel; tap W-1 = current row), then SiLU
 *      (READING: the conv activation is not named on the pages; SiLU as in
 *      the Qwen3-Next lineage [F] section 3 cites).
 *   2. q = conv[QK head hq], k = conv[Hk*dk + QK head hq], v = conv[2*Hk*dk +
 *      V head h]; V head h uses QK head h / (Hv/Hk) ([F] 3.1: each k head
 *      shared by 3 v heads; READING: contiguous grouping).
 *   3. L2 norm per QK head: q <- q / sqrt(|q|^2 + l2_eps) * q_scale,
 *      k <- k / sqrt(|k|^2 + l2_eps) ([F] 2.1; READING: eps inside the sqrt,
 *      q_scale = 1/sqrt(dk)).
 *   4. beta = sigmoid(b), g = exp(-exp(A_log) * softplus(a + dt_bias)) ([F]
 *      3.1: per-head scalar decay in the A_log/dt_bias softplus form, scalar
 *      sigmoid beta; READING: the plainest form using all three quantities,
 *      the formula itself is elided in [F] 5.1 item 5).
 *   5. delta rule, state S[h] in [Dv, Dk] ([F] 2.1 steps 1-5): S <- g S;
 *      m_i = sum_j S_ij k_j; delta_i = (v_i - m_i) beta; S_ij += delta_i k_j
 *      (the k (x) delta outer product laid out in S's [Dv, Dk] order);
 *      y_i = sum_j S_ij q_j.
 *   6. gated RMSNorm per V head ([F] 2.1 output; 2.4: the gated variant uses
 *      y*weight): o_i = y_i / sqrt(mean(y^2) + norm_eps) * norm_w_i * act(z_i),
 *      act = sigmoid ([F] 2.1: sigmoid gates) or silu (gate_act = 1).
 *   7. the state after row r (S and the conv window) is snapshot r+1
 *      ([R] "What it is": the state after row 0 is written to snapshot
 *      buffers); S_snap[r], tail_snap[r] hold it.
 * S0: float64 [Hv, Dv, Dk]; tail0: bf16 [W-1, C] oldest first.
 * o: float64 [k, Hv*Dv].  dbg (optional): per row q[Hk*dk] k[Hk*dk]
 * v[Hv*dv] g[Hv] beta[Hv] y[Hv*dv] (pre-norm).
 */
int oracle_gdn_verify(int Hk, int Hv, int dk, int dv, int W, double q_scale,
                      double l2_eps, double norm_eps, int gate_act,
                      const float* conv_w, const float* A_log, const float* dt_bias,
                      const float* norm_w, const double* S0, const uint16_t* tail0,
                      const uint16_t* qkv, int64_t ld_qkv, const uint16_t* z, int64_t ld_z,
                      const uint16_t* a, int64_t ld_a, const uint16_t* b, int64_t ld_b,
                      int k, double* o, double* S_snap, uint16_t* tail_snap, double* dbg) {
  if (Hv % Hk || W < 1) return 1;
  const int C = 2 * Hk * dk + Hv * dv;
  const int64_t nS = (int64_t)Hv * dv * dk;
  double* S = (double*)malloc(sizeof(double) * (size_t)nS);
  uint16_t* tail = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)((W - 1) * C + 1));
  double* c = (double*)malloc(sizeof(double) * (size_t)C);
  double* y = (double*)malloc(sizeof(double) * (size_t)dv);
  if (!S || !tail || !c || !y) { free(S); free(tail); free(c); free(y); return 2; }
  memcpy(S, S0, sizeof(double) * (size_t)nS);
  memcpy(tail, tail0, sizeof(uint16_t) * (size_t)((W - 1) * C));

  for (int r = 0; r < k; ++r) {
    const uint16_t* xr = qkv + r * ld_qkv;
    /* 1. conv + SiLU, then slide the window */
    for (int ch = 0; ch < C; ++ch) {
      double acc = 0.0;
      for (int t = 0; t < W; ++t) {
        double v = (t < W - 1) ? bf16_value(tail[t * C + ch]) : bf16_value(xr[ch]);
        acc += (double)conv_w[ch * W + t] * v;
      }
      c[ch] = silu(acc);
    }
    for (int t = 0; t + 1 < W - 1; ++t) memcpy(tail + t * C, tail + (t + 1) * C, sizeof(uint16_t) * C);
    if (W > 1) memcpy(tail + (W - 2) * C, xr, sizeof(uint16_t) * C);

    /* 3. L2 norms per QK head (in place on the conv output) */
    for (int hq = 0; hq < Hk; ++hq) {
      double* q = c + hq * dk;
      double* kk = c + Hk * dk + hq * dk;
      double sq = 0.0, sk = 0.0;
      for (int j = 0; j < dk; ++j) { sq += q[j] * q[j]; sk += kk[j] * kk[j]; }
      double nq = sqrt(sq + l2_eps), nk = sqrt(sk + l2_eps);
      for (int j = 0; j < dk; ++j) { q[j] = q[j] / nq * q_scale; kk[j] = kk[j] / nk; }
    }
    double* dbg_r = dbg ? dbg + (int64_t)r * (2 * Hk * dk + 2 * Hv * dv + 2 * Hv) : NULL;
    if (dbg_r) {
      memcpy(dbg_r, c, sizeof(double) * (size_t)(2 * Hk * dk));
      memcpy(dbg_r + 2 * Hk * dk, c + 2 * Hk * dk, sizeof(double) * (size_t)(Hv * dv));
    }

    for (int h = 0; h < Hv; ++h) {
      const int hq = h / (Hv / Hk);
      const double* q = c + hq * dk;
      const double* kk = c + Hk * dk + hq * dk;
      const double* v = c + 2 * Hk * dk + h * dv;
      /* 4. gates */
      double beta = sigmoid(bf16_value(b[r * ld_b + h]));
      double g = exp(-exp((double)A_log[h]) * softplus(bf16_value(a[r * ld_a + h]) + (double)dt_bias[h]));
      /* 5. delta rule on S[h] (row i = value index, column j = key index) */
      double* Sh = S + (int64_t)h * dv * dk;
      for (int64_t e = 0; e < (int64_t)dv * dk; ++e) Sh[e] *= g;
      for (int i = 0; i < dv; ++i) {
        double m = 0.0;
        for (int j = 0; j < dk; ++j) m += Sh[i * dk + j] * kk[j];
        double delta = (v[i] - m) * beta;
        for (int j = 0; j < dk; ++j) Sh[i * dk + j] += delta * kk[j];
      }
      for (int i = 0; i < dv; ++i) {
        double acc = 0.0;
        for (int j = 0; j < dk; ++j) acc += Sh[i * dk + j] * q[j];
        y[i] = acc;
      }
      /* 6. gated RMSNorm over the head's dv outputs */
      double ss = 0.0;
      for (int i = 0; i < dv; ++i) ss += y[i] * y[i];
      double inv = 1.0 / sqrt(ss / dv + norm_eps);
      for (int i = 0; i < dv; ++i) {
        double zz = bf16_value(z[r * ld_z + h * dv + i]);
        double act = gate_act == 1 ? silu(zz) : sigmoid(zz);
        o[(int64_t)r * Hv * dv + h * dv + i] = y[i] * inv * (double)norm_w[i] * act;
      }
      if (dbg_r) {
        dbg_r[2 * Hk * dk + Hv * dv + h] = g;
        dbg_r[2 * Hk * dk + Hv * dv + Hv + h] = beta;
        memcpy(dbg_r + 2 * Hk * dk + Hv * dv + 2 * Hv + h * dv, y, sizeof(double) * (size_t)dv);
      }
    }
    /* 7. snapshot r+1 */
    memcpy(S_snap + (int64_t)r * nS, S, sizeof(double) * (size_t)nS);
    memcpy(tail_snap + (int64_t)r * (W - 1) * C, tail, sizeof(uint16_t) * (size_t)((W - 1) * C));
  }
  free(S); free(tail); free(c); free(y);
  return 0;
}

/* ------------------------------------------------------------- layer glue */

/*
 * Row RMSNorm ([F] 2.4: non-gated norms are zero-centred, y*(1+weight); the
 * conventional form is y*weight): out = x / sqrt(mean(x^2) + eps) * wt,
 * wt = 1 + w (zero_centered) or w.  x, out: float64 [k, n].
 */
int oracle_rmsnorm(const double* x, const float* w, double eps, int zero_centered,
                   int n, int k, double* out) {
  for (int r = 0; r < k; ++r) {
    const double* xr = x + (int64_t)r * n;
    double ss = 0.0;
    for (int c = 0; c < n; ++c) ss += xr[c] * xr[c];
    double inv = 1.0 / sqrt(ss / n + eps);
    for (int c = 0; c < n; ++c) {
      double wt = zero_centered ? 1.0 + (double)w[c] : (double)w[c];
      out[(int64_t)r * n + c] = xr[c] * inv * wt;
    }
  }
  return 0;
}

/* ------------------------------------------------------ greedy acceptance */

/*
 * Greedy acceptance of one verify block ([R] "What it is": the block runs the
 * pending token and the drafts in one pass; "Acceptance": a draft stands when
 * the token chosen from the previous row's logits equals it, and in greedy
 * mode the output is token for token what serial decoding gives).
 *
 * Row 0 of the block is the pending token, rows 1..k-1 are the drafts
 * d_1..d_{k-1}, given as draft[0..k-2].  Greedy choice of row r:
 *   t_r = argmax_v logits[r][v]
 * READING (the pages are silent): among equal maxima the lowest index wins;
 * -0 and +0 are equal; a NaN ranks above every number (so the first NaN
 * wins), which is numpy's argmax.  Then
 *   m = number of leading drafts with d_{r+1} == t_r  (0 <= m <= k-1),
 *   a = m + 1 rows stand (the pending token's row always does),
 *   the next pending token is t_m.
 * out: int32 [2 + k] = { a, t_m, t_0, ..., t_{k-1} }.
 */
int oracle_accept_greedy(const float* logits, int64_t ld, int V, int k, const int32_t* draft,
                         int32_t* out) {
  if (V < 1 || k < 1 || (k > 1 && !draft)) return 1;
  for (int r = 0; r < k; ++r) {
    const float* l = logits + (int64_t)r * ld;
    int best = 0;
    for (int v = 1; v < V; ++v) {
      const int bn = isnan(l[best]), vn = isnan(l[v]);
      if (!bn && (vn || l[v] > l[best])) best = v;
    }
    out[2 + r] = best;
  }
  int m = 0;
  while (m < k - 1 && draft[m] == out[2 + m]) ++m;
  out[0] = m + 1;
  out[1] = out[2 + m];
  return 0;
}

/* ------------------------------------------------------- attention verify */

/* IEEE binary16 bit pattern -> value (exact). */
static double f16_decode(uint16_t h) {
  const int sign = h >> 15, ex = (h >> 10) & 31, frac = h & 1023;
  double v;
  if (ex == 0) v = ldexp((double)frac, -24);
  else if (ex == 31) v = frac ? NAN : INFINITY;
  else v = ldexp((double)(1024 + frac), ex - 25);
  return sign ? -v : v;
}

/* The same through a table of all 65536 patterns (long caches decode each
 * value many times). */
static double f16_table[65536];
static int f16_table_ready = 0;
static double f16_value(uint16_t h) {
  if (!f16_table_ready) {
    for (int i = 0; i < 65536; ++i) f16_table[i] = f16_decode((uint16_t)i);
    f16_table_ready = 1;
  }
  return f16_table[h];
}

/* value -> nearest binary16 (ties to even), rounded once from float64. */
uint16_t oracle_round_f16(double v) {
  if (isnan(v)) return 0x7E00;
  const uint16_t sign = signbit(v) ? 0x8000 : 0;
  const double a = fabs(v);
  if (a == 0.0) return sign;
  if (isinf(a) || a >= 65520.0) return sign | 0x7C00;  /* 65520: halfway past 65504 */
  int ex;
  frexp(a, &ex);
  int E = ex - 1;                                       /* 2^E <= a < 2^(E+1) */
  if (E < -14) return sign | (uint16_t)nearbyint(ldexp(a, 24));  /* subnormal, quantum 2^-24 */
  double r = nearbyint(ldexp(a, 10 - E));               /* 1024 <= r <= 2048 */
  if (r >= 2048.0) { r = 1024.0; ++E; }
  if (E > 15) return sign | 0x7C00;
  return sign | (uint16_t)(((E + 15) << 10) | ((int)r - 1024));
}

/*
 * Rotary position embedding of one head vector at position pos, on its first
 * rope_dim entries ([F] 2.2: partial RoPE, rope dim 64 of 256, theta 1e7).
 * READING (the pages name only the dims and the base): the rotate-half
 * pairing, entry i with entry i + rope_dim/2, at angle pos * theta^(-2i/rope_dim);
 * entries from rope_dim on pass through.
 */
static void rope(const double* x, double* y, int D, int rope_dim, double theta, double pos) {
  const int half = rope_dim / 2;
  for (int i = 0; i < D; ++i) y[i] = x[i];
  for (int i = 0; i < half; ++i) {
    const double ang = pos * pow(theta, -2.0 * i / rope_dim);
    const double c = cos(ang), s = sin(ang);
    y[i] = x[i] * c - x[i + half] * s;
    y[i + half] = x[i + half] * c + x[i] * s;
  }
}

/*
 * Width-k attention verify over a KV cache ([R] "What it is": attention runs
 * per row, row r seeing the earlier rows' keys and values, and rejected rows
 * are overwritten later; [T] "Exact verification kernels": each row keeps its
 * serial KV window; [F] 2.2: grouped-query attention, 24 query and 2 KV heads
 * of dim 256, partial RoPE, a sigmoid gate on the output, an F16 cache).
 *
 * Row r of the block is the token at absolute position P + r.  Its key and
 * value (kn, vn) are appended to the cache: the key after RoPE at P + r, both
 * rounded to binary16 (k_app, v_app).  Its query (after RoPE at P + r)
 * attends to cache positions 0 .. P-1 and the block's rows 0 .. r, with score
 * q.key / sqrt(D) and a softmax over that window; query head h reads KV head
 * h / (Hq / Hkv) (READING: contiguous groups).  Output:
 *   o[r][h][:] = (sum_j p_j value_j) * sigmoid(gate[r][h][:]).
 * READING: the per-head query/key norms of the lineage are applied before
 * this step (q and k arrive normalised); the sparse indexer of [F] 2.2 is not
 * modelled: below its 2048-token budget QSA is dense attention, which this is.
 *
 * q, gate: bf16 [k, Hq, D]; kn, vn: bf16 [k, Hkv, D]; Kc, Vc: binary16
 * [Hkv, cap, D] with positions 0 .. P-1 valid.  o: float64 [k, Hq, D];
 * k_app, v_app: binary16 [k, Hkv, D].
 */
int oracle_attn_verify(int Hq, int Hkv, int D, int rope_dim, double theta, int P, int k, int64_t cap,
                       const uint16_t* q, const uint16_t* kn, const uint16_t* vn, const uint16_t* gate,
                       const uint16_t* Kc, const uint16_t* Vc, double* o, uint16_t* k_app,
                       uint16_t* v_app) {
  if (Hq < 1 || Hkv < 1 || Hq % Hkv || D < 2 || rope_dim < 0 || rope_dim > D || rope_dim % 2 || P < 0 ||
      k < 1 || (int64_t)P > cap)
    return 1;
  const int G = Hq / Hkv;
  double* x = (double*)malloc(sizeof(double) * D);
  double* y = (double*)malloc(sizeof(double) * D);
  double* s = (double*)malloc(sizeof(double) * ((size_t)P + k));
  double* acc = (double*)malloc(sizeof(double) * D);
  if (!x || !y || !s || !acc) return 2;
  /* the block's keys and values, as the cache holds them */
  for (int r = 0; r < k; ++r)
    for (int h = 0; h < Hkv; ++h) {
      const int64_t off = ((int64_t)r * Hkv + h) * D;
      for (int i = 0; i < D; ++i) x[i] = bf16_value(kn[off + i]);
      rope(x, y, D, rope_dim, theta, (double)P + r);
      for (int i = 0; i < D; ++i) {
        k_app[off + i] = oracle_round_f16(y[i]);
        v_app[off + i] = oracle_round_f16(bf16_value(vn[off + i]));
      }
    }
  const double scale = 1.0 / sqrt((double)D);
  for (int r = 0; r < k; ++r)
    for (int h = 0; h < Hq; ++h) {
      const int hk = h / G;
      const int64_t qo = ((int64_t)r * Hq + h) * D;
      for (int i = 0; i < D; ++i) x[i] = bf16_value(q[qo + i]);
      rope(x, y, D, rope_dim, theta, (double)P + r);
      const int n = P + r + 1;  /* the row's window */
      double mx = -INFINITY;
      for (int j = 0; j < n; ++j) {
        const uint16_t* key = j < P ? Kc + ((int64_t)hk * cap + j) * D : k_app + ((int64_t)(j - P) * Hkv + hk) * D;
        double dot = 0.0;
        for (int i = 0; i < D; ++i) dot += y[i] * f16_value(key[i]);
        s[j] = dot * scale;
        if (s[j] > mx) mx = s[j];
      }
      double sum = 0.0;
      for (int i = 0; i < D; ++i) acc[i] = 0.0;
      for (int j = 0; j < n; ++j) {
        const double p = exp(s[j] - mx);
        sum += p;
        const uint16_t* val = j < P ? Vc + ((int64_t)hk * cap + j) * D : v_app + ((int64_t)(j - P) * Hkv + hk) * D;
        for (int i = 0; i < D; ++i) acc[i] += p * f16_value(val[i]);
      }
      for (int i = 0; i < D; ++i) o[qo + i] = acc[i] / sum * sigmoid(bf16_value(gate[qo + i]));
    }
  free(x);
  free(y);
  free(s);
  free(acc);
  return 0;
}
