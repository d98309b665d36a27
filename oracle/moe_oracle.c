/*
 * CPU oracle for the sparse-MoE feed-forward layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link,
 * load or call this file: only the test suite, the package's smoke check and
 * the benchmark's CPU-baseline leg use it.  It shares no code, header, table
 * or helper with the CUDA path.
 *
 * What it computes is the plain definition of the layer, in double precision,
 * from the exact values of the bf16/fp32 inputs.  Source: "Step3.5 Flash
 * 大模型技术深度解析：稀疏 MoE、混合注意力与 MTP 的高效推理革命" (jsqmd.com),
 *   §3.2.1  expert configuration: 288 routed experts + 1 always-on shared
 *           expert per MoE layer, each an independent FFN;
 *   §3.2.2  top-8 routing: a linear router followed by a softmax gives every
 *           expert a probability; the 8 most probable routed experts plus the
 *           shared expert run; their 9 outputs are summed with weights.
 * Readings taken where that page is silent (each also listed in the design
 * notes): the expert FFN is SiLU-gated, h = silu(x.Wg) * (x.Wu), o = h.Wd;
 * the combine weight of a routed expert is its softmax probability over all
 * routed experts, NOT renormalised over the top-k; the shared expert's weight
 * is 1; equal probabilities are ordered by the lower expert index.
 *
 * Layouts (row-major):
 *   x          [T][d]          bf16 bit patterns (uint16)
 *   w_router   [E][d]          fp32
 *   w_gate_up  [G][2F][d]      bf16; rows 0..F-1 = gate, F..2F-1 = up;
 *                              G = E + has_shared, group E = shared expert
 *   w_down     [G][d][F]       bf16
 * FP8 expert weights (§8.1 of the same page: FP8/FP16 mixed-precision
 * inference; the page gives no format, so the reading is): codes of the OCP
 * FP8 E4M3 format, one byte per weight, with one fp32 scale per weight row
 * (see oracle_quantize_e4m3):
 *   w_gate_up  [G][2F][d] codes, s_gate_up [G][2F];  w_down [G][d][F] codes,
 *   s_down [G][d]; the weight value is decode(code) * scale of its row.
 * No function here keeps state; every buffer is owned by the caller.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 bit pattern -> exact double (bf16 is the top half of an fp32). */
static double bf16_to_double(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/*
 * OCP FP8 E4M3 ("E4M3FN"): sign bit, 4 exponent bits (bias 7), 3 mantissa
 * bits; exponent field 0 holds the subnormals m * 2^-9; no infinities; the
 * code with all exponent and mantissa bits set is NaN, so the largest finite
 * magnitude is 1.75 * 2^8 = 448.  Decoding straight from that definition.
 */
static double e4m3_to_double(uint8_t c) {
  const int sign = (c >> 7) & 1, ef = (c >> 3) & 15, m = c & 7;
  double v;
  if (ef == 15 && m == 7) return NAN;
  if (ef == 0)
    v = ldexp((double)m, -9);
  else
    v = ldexp(1.0 + m / 8.0, ef - 7);
  return sign ? -v : v;
}

/*
 * Nearest E4M3 value of a finite float, ties to the even code, magnitudes
 * beyond 448 saturated to 448 (saturating conversion).  Computed in double,
 * where every step below is exact: r is an fp32 value, scaling by powers of
 * two is exact and rint() rounds half to even.
 */
static uint8_t e4m3_from_float(float r) {
  const uint8_t sign = (r < 0.0f || (r == 0.0f && signbit(r))) ? 0x80 : 0x00;
  double a = fabs((double)r);
  if (a >= 448.0) return sign | 0x7e;
  if (a < ldexp(1.0, -6)) {  /* subnormal range: multiples of 2^-9 */
    const double m = rint(ldexp(a, 9));  /* 0..8; 8 is the smallest normal */
    return sign | (uint8_t)m;
  }
  int e;
  frexp(a, &e);  /* a = f * 2^e, f in [0.5, 1) */
  e -= 1;        /* a = (1 + frac) * 2^e */
  double m = rint((ldexp(a, -e) - 1.0) * 8.0);  /* 0..8 */
  if (m == 8.0) {
    m = 0.0;
    e += 1;
  }
  if (e + 7 > 15 || (e + 7 == 15 && m > 6.0)) return sign | 0x7e;  /* rounds past 448 */
  return sign | (uint8_t)(((e + 7) << 3) | (int)m);
}

static void set_threads(int n_threads) {
#ifdef _OPENMP
  if (n_threads > 0) omp_set_num_threads(n_threads);
#else
  (void)n_threads;
#endif
}

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/*
 * Router of §3.2.2 for one token: z_e = sum_i x_i * Wr[e][i] (summed in i
 * order), p = softmax(z) computed with the maximum subtracted first.
 * Writes p[0..E).
 */
static void route_token(const uint16_t* x_t, const float* w_router, int d, int E, double* p) {
  double zmax = -INFINITY;
  for (int e = 0; e < E; ++e) {
    const float* wr = w_router + (size_t)e * d;
    double z = 0.0;
    for (int i = 0; i < d; ++i) z += bf16_to_double(x_t[i]) * (double)wr[i];
    p[e] = z;
    if (z > zmax) zmax = z;
  }
  double s = 0.0;
  for (int e = 0; e < E; ++e) {
    p[e] = exp(p[e] - zmax);
    s += p[e];
  }
  for (int e = 0; e < E; ++e) p[e] /= s;
}

/*
 * Top-k of §3.2.2: the k experts with the highest probability, in
 * descending order of probability, equal probabilities taken lower index
 * first.  Done as k rounds of "pick the best expert not yet picked".
 * gap = p(k-th) - p((k+1)-th), +inf when every expert is picked.
 */
static void topk_token(const double* p, int E, int k, int* idx, double* w, double* gap) {
  unsigned char* taken = (unsigned char*)calloc((size_t)E, 1);
  for (int j = 0; j < k; ++j) {
    int best = -1;
    for (int e = 0; e < E; ++e) {
      if (taken[e]) continue;
      if (best < 0 || p[e] > p[best]) best = e; /* strict '>' keeps the lower index on ties */
    }
    taken[best] = 1;
    idx[j] = best;
    w[j] = p[best];
  }
  if (gap) {
    int next = -1;
    for (int e = 0; e < E; ++e) {
      if (taken[e]) continue;
      if (next < 0 || p[e] > p[next]) next = e;
    }
    *gap = (next < 0) ? INFINITY : (w[k - 1] - p[next]);
  }
  free(taken);
}

/*
 * Routing for T tokens.  Any of p_out / w_out / gap_out may be NULL.
 * Returns 0, or -1 on bad arguments.
 */
int oracle_route(const uint16_t* x, const float* w_router, int T, int d, int E, int k,
                 double* p_out, int* idx_out, double* w_out, double* gap_out, int n_threads) {
  if (T < 0 || d <= 0 || E <= 0 || k <= 0 || k > E || !x || !w_router || !idx_out) return -1;
  set_threads(n_threads);
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 4) reduction(| : bad)
  for (int t = 0; t < T; ++t) {
    double* p = (double*)malloc(sizeof(double) * (size_t)E);
    double* w = (double*)malloc(sizeof(double) * (size_t)k);
    if (!p || !w) { bad = 1; free(p); free(w); continue; }
    route_token(x + (size_t)t * d, w_router, d, E, p);
    topk_token(p, E, k, idx_out + (size_t)t * k, w, gap_out ? gap_out + t : NULL);
    if (p_out) memcpy(p_out + (size_t)t * E, p, sizeof(double) * (size_t)E);
    if (w_out) memcpy(w_out + (size_t)t * k, w, sizeof(double) * (size_t)k);
    free(p);
    free(w);
  }
  return bad ? -1 : 0;
}

/*
 * Dispatch implied by §3.2.2 (each token's rows go to its chosen experts):
 *   counts[e]   = number of (t, j) with idx[t][j] == e
 *   offsets[e]  = counts[0] + ... + counts[e-1], e = 0..E;
 *   offsets[E+1]= offsets[E] + T  (the shared expert's T rows, token order)
 *   perm[pos]   = assignment id a = t*k + j, listed expert by expert and,
 *                 inside one expert, by increasing token index.
 * Built by visiting experts in order and, for each, tokens in order.
 */
int oracle_dispatch(const int* idx, int T, int E, int k, int* counts, int* offsets, int* perm) {
  if (T < 0 || E <= 0 || k <= 0 || !idx || !counts || !offsets) return -1;
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (long a = 0; a < (long)T * k; ++a) {
    int e = idx[a];
    if (e < 0 || e >= E) return -1;
    counts[e]++;
  }
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  offsets[E + 1] = offsets[E] + T;
  if (perm) {
    long pos = 0;
    for (int e = 0; e < E; ++e)
      for (int t = 0; t < T; ++t)
        for (int j = 0; j < k; ++j)
          if (idx[(size_t)t * k + j] == e) perm[pos++] = t * k + j;
  }
  return 0;
}

/*
 * One expert FFN (§3.2.1: each expert is an independent FFN; SiLU-gated
 * reading): g = Wg.x, u = Wu.x, h = g * sigmoid(g) * u, o = Wd.h, all in
 * double, no intermediate rounding.  scale multiplies o into acc.
 */
typedef struct {
  int fp8;               /* 0: bf16 bit patterns; 1: E4M3 codes with per-row scales */
  const void* gate_up;   /* one group: [2F][d] */
  const float* s_gu;     /* one group: [2F] (fp8) */
  const void* down;      /* one group: [d][F] */
  const float* s_d;      /* one group: [d] (fp8) */
} group_w;

/* Value of element i of weight row `row` (row length n) of a group matrix. */
static double wval(int fp8, const void* base, const float* scale, size_t row, int n, int i) {
  if (fp8) return e4m3_to_double(((const uint8_t*)base)[row * (size_t)n + i]) * (double)scale[row];
  return bf16_to_double(((const uint16_t*)base)[row * (size_t)n + i]);
}

static void expert_ffn_acc_w(const uint16_t* x_t, group_w w, int d, int F, double scale, double* h, double* acc) {
  for (int f = 0; f < F; ++f) {
    double g = 0.0, u = 0.0;
    for (int i = 0; i < d; ++i) {
      double xi = bf16_to_double(x_t[i]);
      g += wval(w.fp8, w.gate_up, w.s_gu, (size_t)f, d, i) * xi;
      u += wval(w.fp8, w.gate_up, w.s_gu, (size_t)(F + f), d, i) * xi;
    }
    h[f] = g * (1.0 / (1.0 + exp(-g))) * u;
  }
  for (int o = 0; o < d; ++o) {
    double s = 0.0;
    for (int f = 0; f < F; ++f) s += wval(w.fp8, w.down, w.s_d, (size_t)o, F, f) * h[f];
    acc[o] += scale * s;
  }
}

static void expert_ffn_acc(const uint16_t* x_t, const uint16_t* w_gu, const uint16_t* w_d, int d, int F,
                           double scale, double* h, double* acc) {
  group_w w = {0, w_gu, NULL, w_d, NULL};
  expert_ffn_acc_w(x_t, w, d, F, scale, h, acc);
}

/* Group g of a weight set of either format. */
static group_w group_of(int fp8, const void* gate_up, const float* s_gu, const void* down, const float* s_d,
                        int d, int F, int g) {
  const size_t esz = fp8 ? 1 : 2;
  group_w w;
  w.fp8 = fp8;
  w.gate_up = (const char*)gate_up + (size_t)g * 2 * F * d * esz;
  w.down = (const char*)down + (size_t)g * d * F * esz;
  w.s_gu = fp8 ? s_gu + (size_t)g * 2 * F : NULL;
  w.s_d = fp8 ? s_d + (size_t)g * d : NULL;
  return w;
}

/*
 * FP8 weight quantisation, one scale per row: s = max_i |w_i| / 448 (an fp32
 * division), code_i = nearest E4M3 of the fp32 quotient w_i / s (ties to
 * even, saturating).  A row of zeros gets s = 0 and codes 0.  w holds bf16
 * bit patterns [rows][cols].
 */
int oracle_quantize_e4m3(const uint16_t* w, long rows, int cols, uint8_t* q, float* s) {
  if (rows < 0 || cols <= 0 || !w || !q || !s) return -1;
  for (long r = 0; r < rows; ++r) {
    const uint16_t* wr = w + (size_t)r * cols;
    float amax = 0.0f;
    for (int i = 0; i < cols; ++i) {
      const float v = (float)fabs(bf16_to_double(wr[i]));
      if (v > amax) amax = v;
    }
    const float sc = amax / 448.0f;
    s[r] = sc;
    for (int i = 0; i < cols; ++i) {
      const float v = (float)bf16_to_double(wr[i]);
      q[(size_t)r * cols + i] = sc > 0.0f ? e4m3_from_float(v / sc) : 0;
    }
  }
  return 0;
}

/*
 * Layer output (§3.2.2 step 3) for the tokens listed in `tokens`:
 *   y[t] = sum_{j<k} p[t, idx[t][j]] * FFN_{idx[t][j]}(x_t) + FFN_shared(x_t)
 * summed in slot order, then the shared expert.  If sel is non-NULL it gives
 * the k experts per listed token ([n_tokens][k]) instead of the oracle's own
 * top-k; the weights are still the oracle's probabilities of those experts.
 * w_gate_up / w_down hold E + has_shared groups.  y is [n_tokens][d].
 * renormalize != 0 (the per-call variant of §8.2 with a renormalised
 * top-k): the k weights are divided by their sum, summed in slot order.
 */
static int forward_any(const uint16_t* x, const float* w_router, int fp8, const void* w_gate_up, const float* s_gu,
                       const void* w_down, const float* s_d, int T, int d, int E, int k, int F, int has_shared,
                       const int* tokens, int n_tokens, const int* sel, int renormalize, double* y,
                       int n_threads) {
  if (T < 0 || d <= 0 || E <= 0 || k <= 0 || k > E || F <= 0 || n_tokens < 0) return -1;
  if (!x || !w_router || !w_gate_up || !w_down || !tokens || !y) return -1;
  if (fp8 && (!s_gu || !s_d)) return -1;
  for (int i = 0; i < n_tokens; ++i)
    if (tokens[i] < 0 || tokens[i] >= T) return -1;
  if (sel)
    for (long i = 0; i < (long)n_tokens * k; ++i)
      if (sel[i] < 0 || sel[i] >= E) return -1;
  set_threads(n_threads);
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (int i = 0; i < n_tokens; ++i) {
    const int t = tokens[i];
    const uint16_t* x_t = x + (size_t)t * d;
    double* p = (double*)malloc(sizeof(double) * (size_t)E);
    double* h = (double*)malloc(sizeof(double) * (size_t)F);
    int* ids = (int*)malloc(sizeof(int) * (size_t)k);
    double* w = (double*)malloc(sizeof(double) * (size_t)k);
    if (!p || !h || !ids || !w) { bad = 1; free(p); free(h); free(ids); free(w); continue; }
    route_token(x_t, w_router, d, E, p);
    if (sel) {
      for (int j = 0; j < k; ++j) { ids[j] = sel[(size_t)i * k + j]; w[j] = p[ids[j]]; }
    } else {
      topk_token(p, E, k, ids, w, NULL);
    }
    if (renormalize) {
      double sum = 0.0;
      for (int j = 0; j < k; ++j) sum += w[j];
      for (int j = 0; j < k; ++j) w[j] /= sum;
    }
    double* acc = y + (size_t)i * d;
    for (int o = 0; o < d; ++o) acc[o] = 0.0;
    for (int j = 0; j < k; ++j)
      expert_ffn_acc_w(x_t, group_of(fp8, w_gate_up, s_gu, w_down, s_d, d, F, ids[j]), d, F, w[j], h, acc);
    if (has_shared)
      expert_ffn_acc_w(x_t, group_of(fp8, w_gate_up, s_gu, w_down, s_d, d, F, E), d, F, 1.0, h, acc);
    free(p); free(h); free(ids); free(w);
  }
  return bad ? -1 : 0;
}

int oracle_forward_ex(const uint16_t* x, const float* w_router, const uint16_t* w_gate_up, const uint16_t* w_down,
                      int T, int d, int E, int k, int F, int has_shared, const int* tokens, int n_tokens,
                      const int* sel, int renormalize, double* y, int n_threads) {
  return forward_any(x, w_router, 0, w_gate_up, NULL, w_down, NULL, T, d, E, k, F, has_shared, tokens, n_tokens,
                     sel, renormalize, y, n_threads);
}

/* oracle_forward_ex with E4M3 expert weights and per-row scales. */
int oracle_forward_fp8(const uint16_t* x, const float* w_router, const uint8_t* q_gate_up, const float* s_gate_up,
                       const uint8_t* q_down, const float* s_down, int T, int d, int E, int k, int F, int has_shared,
                       const int* tokens, int n_tokens, const int* sel, int renormalize, double* y,
                       int n_threads) {
  return forward_any(x, w_router, 1, q_gate_up, s_gate_up, q_down, s_down, T, d, E, k, F, has_shared, tokens,
                     n_tokens, sel, renormalize, y, n_threads);
}

/* Decode E4M3 codes to double (for pins of the codec). */
int oracle_e4m3_decode(const uint8_t* q, long n, double* out) {
  if (n < 0 || !q || !out) return -1;
  for (long i = 0; i < n; ++i) out[i] = e4m3_to_double(q[i]);
  return 0;
}

/* Encode fp32 values to E4M3 codes (nearest, ties to even, saturating). */
int oracle_e4m3_encode(const float* v, long n, uint8_t* q) {
  if (n < 0 || !v || !q) return -1;
  for (long i = 0; i < n; ++i) q[i] = e4m3_from_float(v[i]);
  return 0;
}

/* oracle_forward_ex with the raw softmax weights (the §3.2.2 reading). */
int oracle_forward(const uint16_t* x, const float* w_router, const uint16_t* w_gate_up, const uint16_t* w_down,
                   int T, int d, int E, int k, int F, int has_shared, const int* tokens, int n_tokens,
                   const int* sel, double* y, int n_threads) {
  return oracle_forward_ex(x, w_router, w_gate_up, w_down, T, d, E, k, F, has_shared, tokens, n_tokens, sel, 0, y,
                           n_threads);
}

/*
 * Routing statistics of §3.2.3 (EP group-balanced routing): the E experts
 * form G groups of E/G consecutive indices.  From the oracle's own routing:
 *   counts[e]  rows routed to expert e (top-k selections)
 *   f[g]       share of the T*k selections that fall in group g
 *   pg[g]      mean over tokens of sum_{e in g} p_e
 *   summary    [0] L_EP = G * sum_g f[g] * pg[g]; [1] max_e counts / (T*k/E);
 *              [2] mean over tokens of -sum_e p_e ln p_e; [3] experts with no row
 */
int oracle_route_stats(const uint16_t* x, const float* w_router, int T, int d, int E, int k, int G, int* counts,
                       double* f, double* pg, double* summary, int n_threads) {
  if (T <= 0 || d <= 0 || E <= 0 || k <= 0 || k > E || G <= 0 || E % G != 0) return -1;
  if (!x || !w_router || !counts || !f || !pg || !summary) return -1;
  double* p = (double*)malloc(sizeof(double) * (size_t)T * E);
  int* idx = (int*)malloc(sizeof(int) * (size_t)T * k);
  if (!p || !idx) { free(p); free(idx); return -1; }
  if (oracle_route(x, w_router, T, d, E, k, p, idx, NULL, NULL, n_threads) != 0) { free(p); free(idx); return -1; }
  const int per = E / G;
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (long a = 0; a < (long)T * k; ++a) counts[idx[a]]++;
  double entropy = 0.0;
  for (int g = 0; g < G; ++g) pg[g] = 0.0;
  for (int t = 0; t < T; ++t) {
    const double* pt = p + (size_t)t * E;
    for (int e = 0; e < E; ++e) {
      pg[e / per] += pt[e];
      if (pt[e] > 0.0) entropy -= pt[e] * log(pt[e]);
    }
  }
  double lep = 0.0;
  int max_c = 0, empty = 0;
  for (int e = 0; e < E; ++e) {
    if (counts[e] > max_c) max_c = counts[e];
    if (counts[e] == 0) ++empty;
  }
  for (int g = 0; g < G; ++g) {
    long cg = 0;
    for (int e = g * per; e < (g + 1) * per; ++e) cg += counts[e];
    f[g] = (double)cg / ((double)T * k);
    pg[g] /= T;
    lep += f[g] * pg[g];
  }
  summary[0] = G * lep;
  summary[1] = max_c / ((double)T * k / E);
  summary[2] = entropy / T;
  summary[3] = empty;
  free(p);
  free(idx);
  return 0;
}

/*
 * One expert FFN over a batch of rows, exposed so that tests can pin the
 * FFN against a library matmul: out[r] = FFN_g(x[rows[r]]) with scale 1.
 */
int oracle_expert_ffn(const uint16_t* x, const uint16_t* w_gate_up, const uint16_t* w_down, int d, int F,
                      int group, const int* rows, int n_rows, double* out, int n_threads) {
  if (d <= 0 || F <= 0 || group < 0 || n_rows < 0 || !x || !w_gate_up || !w_down || !rows || !out) return -1;
  set_threads(n_threads);
  const uint16_t* gu = w_gate_up + (size_t)group * 2 * F * d;
  const uint16_t* dn = w_down + (size_t)group * d * F;
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (int r = 0; r < n_rows; ++r) {
    double* h = (double*)malloc(sizeof(double) * (size_t)F);
    if (!h) { bad = 1; continue; }
    double* acc = out + (size_t)r * d;
    for (int o = 0; o < d; ++o) acc[o] = 0.0;
    expert_ffn_acc(x + (size_t)rows[r] * d, gu, dn, d, F, 1.0, h, acc);
    free(h);
  }
  return bad ? -1 : 0;
}
