/*
 * flint_moe_ref.c — plain fp64 CPU oracle of the Flint decode MoE layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or helper with the CUDA path.
 *
 * What it computes, written out as the plain definition, only for the experts
 * that routing selects (every bf16 / fp32 input is decoded exactly to fp64 and
 * nothing is rounded afterwards):
 *   1. logits   R[t,e] = sum_h x[t,h] * Wr[e,h]; ranking key L = R + bias[e]
 *      (bias 0 if absent) -- the router scores every expert: [vLLM Day-0
 *      Support for Recursive's Flint, "Flint Model Architecture", "MoE
 *      Structure"].
 *   2. selection: rank experts by (L descending, index ascending) and keep the
 *      first top_k; score s = 1 / (1 + exp(-L)), or 1 / (1 + exp(-R)) when
 *      offset_mode is 1 (offsets steer the selection only); weight w_j = s_j /
 *      sum of the kept s.  "sigmoid top-6 selection": same section; the
 *      renormalisation, the lower-index tie rule and both offset readings are
 *      this library's (the pages are silent on all of them).
 *   3. expert FFN (SwiGLU, "Qwen3-MoE-style" and "SiLU-and-mul":
 *      [Flint on Intel Arc Pro B70, "Setup"; "norm.py: Triton kernels that
 *      assumed CUDA"]):  g = Wg v, u = Wu v, a = g / (1 + exp(-g)) * u,
 *      y = Wd a.
 *   4. out[t] = residual[t] + sum_s y_shared_s + sum_j w_j * y_{e_j}
 *      (shared experts added with weight 1: "plus one shared expert",
 *      [Flint on Intel Arc Pro B70, "Setup"]).
 * NVFP4 (weight-only W4A16, [vLLM Day-0 Support for Recursive's Flint,
 * "Flint Model Overview and Capabilities"]): W[r,k] = e2m1(q) * e4m3(sf) * ts,
 * decoded from the OCP Microscaling / OCP 8-bit floating point format
 * definitions; exact in fp64.
 *
 * Parity pins live in the tests: a separately written NumPy brute force over
 * all experts, invariants, closed forms (x = 0, identical experts, identity-
 * embedded weights, planted router ties) and exhaustive code decoding.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
  int32_t hidden, n_experts, top_k, inter, n_shared;
  int32_t offset_mode; /* 0: offsets move ranking and weights; 1: ranking only */
} ref_dims;

/* ---- exact decoders ------------------------------------------------------ */

static double bf16_value(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* OCP FP4 E2M1: bit 3 sign, bits 2..1 exponent (bias 1), bit 0 mantissa;
 * exponent 0 is subnormal (0.m x 2^0). */
double ref_e2m1(uint8_t code) {
  int sign = (code >> 3) & 1, exp = (code >> 1) & 3, man = code & 1;
  double mag = exp == 0 ? 0.5 * man : ldexp(1.0 + 0.5 * man, exp - 1);
  return sign ? -mag : mag;
}

/* OCP FP8 E4M3 ("FN": no infinities): bit 7 sign, bits 6..3 exponent (bias 7),
 * bits 2..0 mantissa; exponent 0 is subnormal (0.mmm x 2^-6); S.1111.111 is
 * NaN; the largest finite value is 448. */
double ref_e4m3(uint8_t code) {
  int sign = (code >> 7) & 1, exp = (code >> 3) & 15, man = code & 7;
  double mag;
  if (exp == 15 && man == 7) return NAN;
  if (exp == 0) mag = ldexp(man / 8.0, -6);
  else mag = ldexp(1.0 + man / 8.0, exp - 7);
  return sign ? -mag : mag;
}

/* ---- weight matrices ----------------------------------------------------- */

/* One projection matrix [rows, K], bf16 or NVFP4 (q/sf with a tensor scale
 * that may differ between rows below and at/after split_row). */
typedef struct {
  int fmt; /* 0 = bf16, 1 = nvfp4 */
  int K;
  const uint16_t* bf16;
  const uint8_t* q;
  const uint8_t* sf;
  double ts_lo, ts_hi;
  int split_row;
} ref_mat;

static double mat_at(const ref_mat* m, int r, int k) {
  if (m->fmt == 0) return bf16_value(m->bf16[(size_t)r * m->K + k]);
  uint8_t byte = m->q[(size_t)r * (m->K / 2) + k / 2];
  uint8_t code = (k & 1) ? (byte >> 4) : (byte & 15);
  double scale = ref_e4m3(m->sf[(size_t)r * (m->K / 16) + k / 16]);
  double ts = r < m->split_row ? m->ts_lo : m->ts_hi;
  return ref_e2m1(code) * scale * ts;
}

/* Weights of one layer.  Routed expert e, shared expert s. */
typedef struct {
  int fmt;
  /* bf16 */
  const uint16_t *w13, *w2, *ws13, *ws2;
  /* nvfp4 */
  const uint8_t *w13_q, *w13_sf, *w2_q, *w2_sf;
  const float *w13_ts, *w2_ts;
  const uint8_t *ws13_q, *ws13_sf, *ws2_q, *ws2_sf;
  const float *ws13_ts, *ws2_ts;
} ref_layer;

static void expert_mats(const ref_dims* d, const ref_layer* L, int shared, int e,
                        ref_mat* m13, ref_mat* m2) {
  const int H = d->hidden, I = d->inter;
  memset(m13, 0, sizeof *m13);
  memset(m2, 0, sizeof *m2);
  m13->fmt = m2->fmt = L->fmt;
  m13->K = H;
  m2->K = I;
  m13->split_row = I;
  m2->split_row = H;
  if (L->fmt == 0) {
    m13->bf16 = (shared ? L->ws13 : L->w13) + (size_t)e * 2 * I * H;
    m2->bf16 = (shared ? L->ws2 : L->w2) + (size_t)e * H * I;
  } else {
    m13->q = (shared ? L->ws13_q : L->w13_q) + (size_t)e * 2 * I * (H / 2);
    m13->sf = (shared ? L->ws13_sf : L->w13_sf) + (size_t)e * 2 * I * (H / 16);
    const float* ts13 = (shared ? L->ws13_ts : L->w13_ts) + (size_t)e * 2;
    m13->ts_lo = ts13[0];
    m13->ts_hi = ts13[1];
    m2->q = (shared ? L->ws2_q : L->w2_q) + (size_t)e * H * (I / 2);
    m2->sf = (shared ? L->ws2_sf : L->w2_sf) + (size_t)e * H * (I / 16);
    m2->ts_lo = m2->ts_hi = (shared ? L->ws2_ts : L->w2_ts)[e];
  }
}

/* y[H] = Wd ( silu(Wg v) * (Wu v) ), act[I] is scratch. */
static void expert_ffn(const ref_dims* d, const ref_mat* m13, const ref_mat* m2,
                       const double* v, double* act, double* y) {
  const int H = d->hidden, I = d->inter;
  for (int i = 0; i < I; ++i) {
    double g = 0.0, u = 0.0;
    for (int h = 0; h < H; ++h) {
      g += mat_at(m13, i, h) * v[h];
      u += mat_at(m13, I + i, h) * v[h];
    }
    act[i] = g / (1.0 + exp(-g)) * u;
  }
  for (int r = 0; r < H; ++r) {
    double acc = 0.0;
    for (int i = 0; i < I; ++i) acc += mat_at(m2, r, i) * act[i];
    y[r] = acc;
  }
}

/* ---- routing ------------------------------------------------------------- */

static void route_token(const ref_dims* d, const uint16_t* x, const uint16_t* wr,
                        const float* bias, double* logits, int32_t* idx, double* w) {
  const int H = d->hidden, E = d->n_experts, k = d->top_k;
  double* raw = (double*)malloc(sizeof(double) * (size_t)E);
  for (int e = 0; e < E; ++e) {
    double acc = 0.0;
    for (int h = 0; h < H; ++h)
      acc += bf16_value(x[h]) * bf16_value(wr[(size_t)e * H + h]);
    raw[e] = acc;
    logits[e] = acc + (bias ? (double)bias[e] : 0.0);
  }
  /* Repeated selection of the best remaining expert; scanning indices upward
   * with a strict '>' keeps the lower index on equal logits. */
  unsigned char* taken = (unsigned char*)calloc((size_t)E, 1);
  double ssum = 0.0;
  for (int j = 0; j < k; ++j) {
    int best = -1;
    for (int e = 0; e < E; ++e)
      if (!taken[e] && (best < 0 || logits[e] > logits[best])) best = e;
    taken[best] = 1;
    idx[j] = best;
    const double score_in = d->offset_mode == 1 ? raw[best] : logits[best];
    w[j] = 1.0 / (1.0 + exp(-score_in));
    ssum += w[j];
  }
  for (int j = 0; j < k; ++j) w[j] /= ssum;
  free(taken);
  free(raw);
}

/* Router only.  logits may be NULL. */
int ref_route(const ref_dims* d, int B, const uint16_t* x, const uint16_t* wr,
              const float* bias, double* logits, int32_t* idx, double* w) {
  const int H = d->hidden, E = d->n_experts, k = d->top_k;
  double* tmp = (double*)malloc(sizeof(double) * (size_t)E);
  if (!tmp) return 1;
  for (int t = 0; t < B; ++t) {
    route_token(d, x + (size_t)t * H, wr, bias, tmp, idx + (size_t)t * k, w + (size_t)t * k);
    if (logits) memcpy(logits + (size_t)t * E, tmp, sizeof(double) * (size_t)E);
  }
  free(tmp);
  return 0;
}

/* Expert part for given routing (idx/w per token); out = residual + shared + routed. */
static int moe_given_routing(const ref_dims* d, int B, const uint16_t* x,
                             const uint16_t* residual, const int32_t* idx, const double* w,
                             const ref_layer* L, int nthreads, double* out) {
  const int H = d->hidden, I = d->inter, k = d->top_k, S = d->n_shared;
  int err = 0;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
#endif
  for (int t = 0; t < B; ++t) {
    double* v = (double*)malloc(sizeof(double) * (size_t)H);
    double* y = (double*)malloc(sizeof(double) * (size_t)H);
    double* act = (double*)malloc(sizeof(double) * (size_t)I);
    double* o = out + (size_t)t * H;
    if (!v || !y || !act) {
      err |= 1;
    } else {
      for (int h = 0; h < H; ++h) {
        v[h] = bf16_value(x[(size_t)t * H + h]);
        o[h] = bf16_value(residual[(size_t)t * H + h]);
      }
      ref_mat m13, m2;
      for (int s = 0; s < S; ++s) {
        expert_mats(d, L, 1, s, &m13, &m2);
        expert_ffn(d, &m13, &m2, v, act, y);
        for (int h = 0; h < H; ++h) o[h] += y[h];
      }
      for (int j = 0; j < k; ++j) {
        expert_mats(d, L, 0, idx[(size_t)t * k + j], &m13, &m2);
        expert_ffn(d, &m13, &m2, v, act, y);
        for (int h = 0; h < H; ++h) o[h] += w[(size_t)t * k + j] * y[h];
      }
    }
    free(v);
    free(y);
    free(act);
  }
  return err;
}

static int moe_full(const ref_dims* d, int B, const uint16_t* x, const uint16_t* residual,
                    const uint16_t* wr, const float* bias, const ref_layer* L,
                    int nthreads, double* out, int32_t* idx, double* w) {
  if (ref_route(d, B, x, wr, bias, NULL, idx, w)) return 1;
  return moe_given_routing(d, B, x, residual, idx, w, L, nthreads, out);
}

/* ---- exported entry points ------------------------------------------------ */

int ref_moe_bf16(const ref_dims* d, int B, const uint16_t* x, const uint16_t* residual,
                 const uint16_t* wr, const float* bias,
                 const uint16_t* w13, const uint16_t* w2,
                 const uint16_t* ws13, const uint16_t* ws2,
                 int nthreads, double* out, int32_t* idx, double* w) {
  ref_layer L;
  memset(&L, 0, sizeof L);
  L.fmt = 0;
  L.w13 = w13; L.w2 = w2; L.ws13 = ws13; L.ws2 = ws2;
  return moe_full(d, B, x, residual, wr, bias, &L, nthreads, out, idx, w);
}

int ref_moe_bf16_given_routing(const ref_dims* d, int B, const uint16_t* x,
                               const uint16_t* residual, const int32_t* idx, const double* w,
                               const uint16_t* w13, const uint16_t* w2,
                               const uint16_t* ws13, const uint16_t* ws2,
                               int nthreads, double* out) {
  ref_layer L;
  memset(&L, 0, sizeof L);
  L.fmt = 0;
  L.w13 = w13; L.w2 = w2; L.ws13 = ws13; L.ws2 = ws2;
  return moe_given_routing(d, B, x, residual, idx, w, &L, nthreads, out);
}

static void nvfp4_layer(ref_layer* L,
                        const uint8_t* w13_q, const uint8_t* w13_sf, const float* w13_ts,
                        const uint8_t* w2_q, const uint8_t* w2_sf, const float* w2_ts,
                        const uint8_t* ws13_q, const uint8_t* ws13_sf, const float* ws13_ts,
                        const uint8_t* ws2_q, const uint8_t* ws2_sf, const float* ws2_ts) {
  memset(L, 0, sizeof *L);
  L->fmt = 1;
  L->w13_q = w13_q; L->w13_sf = w13_sf; L->w13_ts = w13_ts;
  L->w2_q = w2_q; L->w2_sf = w2_sf; L->w2_ts = w2_ts;
  L->ws13_q = ws13_q; L->ws13_sf = ws13_sf; L->ws13_ts = ws13_ts;
  L->ws2_q = ws2_q; L->ws2_sf = ws2_sf; L->ws2_ts = ws2_ts;
}

int ref_moe_nvfp4(const ref_dims* d, int B, const uint16_t* x, const uint16_t* residual,
                  const uint16_t* wr, const float* bias,
                  const uint8_t* w13_q, const uint8_t* w13_sf, const float* w13_ts,
                  const uint8_t* w2_q, const uint8_t* w2_sf, const float* w2_ts,
                  const uint8_t* ws13_q, const uint8_t* ws13_sf, const float* ws13_ts,
                  const uint8_t* ws2_q, const uint8_t* ws2_sf, const float* ws2_ts,
                  int nthreads, double* out, int32_t* idx, double* w) {
  ref_layer L;
  nvfp4_layer(&L, w13_q, w13_sf, w13_ts, w2_q, w2_sf, w2_ts,
              ws13_q, ws13_sf, ws13_ts, ws2_q, ws2_sf, ws2_ts);
  return moe_full(d, B, x, residual, wr, bias, &L, nthreads, out, idx, w);
}

int ref_moe_nvfp4_given_routing(const ref_dims* d, int B, const uint16_t* x,
                                const uint16_t* residual, const int32_t* idx, const double* w,
                                const uint8_t* w13_q, const uint8_t* w13_sf, const float* w13_ts,
                                const uint8_t* w2_q, const uint8_t* w2_sf, const float* w2_ts,
                                const uint8_t* ws13_q, const uint8_t* ws13_sf, const float* ws13_ts,
                                const uint8_t* ws2_q, const uint8_t* ws2_sf, const float* ws2_ts,
                                int nthreads, double* out) {
  ref_layer L;
  nvfp4_layer(&L, w13_q, w13_sf, w13_ts, w2_q, w2_sf, w2_ts,
              ws13_q, ws13_sf, ws13_ts, ws2_q, ws2_sf, ws2_ts);
  return moe_given_routing(d, B, x, residual, idx, w, &L, nthreads, out);
}

/* Token-to-expert buckets: the distinct selected experts in ascending order
 * (uniq[0..U)), where each one's (token, slot) pairs start in `pairs`
 * (offsets[0..U], offsets[U] = B*k), and the pairs themselves encoded as
 * token*8 + slot, ordered by (expert, token).  Returns U. */
int ref_bucket(int B, int k, int E, const int32_t* idx, int32_t* uniq,
               int32_t* offsets, int32_t* pairs) {
  int n = 0, U = 0;
  for (int e = 0; e < E; ++e) {
    int start = n;
    for (int t = 0; t < B; ++t)
      for (int j = 0; j < k; ++j)
        if (idx[(size_t)t * k + j] == e) pairs[n++] = t * 8 + j;
    if (n > start) {
      uniq[U] = e;
      offsets[U] = start;
      ++U;
    }
  }
  offsets[U] = n;
  return U;
}

/* Pre-norm with unit gain: out[t,h] = in[t,h] / sqrt(mean_h(in[t,:]^2) + eps). */
void ref_rmsnorm(int B, int H, const uint16_t* in, double eps, double* out) {
  for (int t = 0; t < B; ++t) {
    double ss = 0.0;
    for (int h = 0; h < H; ++h) {
      double v = bf16_value(in[(size_t)t * H + h]);
      ss += v * v;
    }
    double inv = 1.0 / sqrt(ss / H + eps);
    for (int h = 0; h < H; ++h) out[(size_t)t * H + h] = bf16_value(in[(size_t)t * H + h]) * inv;
  }
}

/* ---- attention side of a decode step: Q/K norm + RoPE + KV-cache write ----
 *
 * The pages fuse "Q/K norm, RoPE, and KV-cache write into a single kernel"
 * [vLLM Day-0 Support for Recursive's Flint, "Optimization Strategies",
 * "Fused Kernels"] for attention with "per-head Q/K RMSNorm", GQA with 32
 * query and 4 KV heads, RoPE on the sliding-window layers and no positional
 * encoding on the full-attention ones [same page, "Flint Model
 * Architecture"].  For each token t with position pos[t], its projection row
 * qkv[t] = [q_0 .. q_{nq-1} | k_0 .. k_{nkv-1} | v_0 .. v_{nkv-1}] (D values
 * per head) gives:
 *   q and k heads:  n[i] = x[i] / sqrt(mean_i x[i]^2 + eps) * g[i]
 *                   (g = q_norm for query heads, k_norm for key heads), then,
 *                   when theta > 0, for i < D/2 with a_i = pos * theta^(-2i/D):
 *                   r[i] = n[i] cos a_i - n[i + D/2] sin a_i,
 *                   r[i + D/2] = n[i + D/2] cos a_i + n[i] sin a_i;
 *   v heads:        unchanged.
 * The pairing of element i with i + D/2 (rotate-half) and theta as an input
 * are this library's readings: the pages name RoPE only.  q_out is
 * [B][nq][D], k_out and v_out [B][nkv][D]; the cache write is the caller's
 * placement of k_out and v_out at each token's slot. */
static void qk_head(int D, const uint16_t* x, const uint16_t* g, int32_t pos, double theta,
                    double eps, double* out) {
  double ss = 0.0;
  for (int i = 0; i < D; ++i) {
    double v = bf16_value(x[i]);
    ss += v * v;
  }
  double inv = 1.0 / sqrt(ss / D + eps);
  for (int i = 0; i < D; ++i) out[i] = bf16_value(x[i]) * inv * bf16_value(g[i]);
  if (theta > 0.0) {
    int half = D / 2;
    for (int i = 0; i < half; ++i) {
      double a = (double)pos * pow(theta, -2.0 * i / D);
      double c = cos(a), s = sin(a);
      double lo = out[i], hi = out[i + half];
      out[i] = lo * c - hi * s;
      out[i + half] = hi * c + lo * s;
    }
  }
}

void ref_qk_norm_rope(int B, int nq, int nkv, int D, const uint16_t* qkv, const uint16_t* q_norm,
                      const uint16_t* k_norm, const int32_t* pos, double theta, double eps,
                      double* q_out, double* k_out, double* v_out) {
  const size_t row = (size_t)(nq + 2 * nkv) * D;
  for (int t = 0; t < B; ++t) {
    const uint16_t* x = qkv + (size_t)t * row;
    for (int h = 0; h < nq; ++h)
      qk_head(D, x + (size_t)h * D, q_norm, pos[t], theta, eps, q_out + ((size_t)t * nq + h) * D);
    for (int h = 0; h < nkv; ++h)
      qk_head(D, x + (size_t)(nq + h) * D, k_norm, pos[t], theta, eps,
              k_out + ((size_t)t * nkv + h) * D);
    for (int h = 0; h < nkv; ++h)
      for (int i = 0; i < D; ++i)
        v_out[((size_t)t * nkv + h) * D + i] = bf16_value(x[(size_t)(nq + nkv + h) * D + i]);
  }
}

int ref_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
