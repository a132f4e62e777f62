/*
 * kvevict_oracle.c -- plain fp64 CPU oracle (TEST INFRASTRUCTURE; see the
 * header for who may use it, its sources and its precision rules).
 *
 * Written to be read against the pages, not to be fast: no blocking, no
 * fusion, loops in the order the method states its steps.
 *
 * Build: gcc -O2 -std=c11 -fPIC -shared -fopenmp -ffp-contract=off
 * (-ffp-contract=off matters: the fp32 RoPE re-rotation must round after
 * every multiply and every add, as plain fp32 arithmetic does.)
 */
#include "kvevict_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------------------
 * Budget schedule. PyramidKV page, "The budget schedule": a linear taper from
 * a maximum at layer 0 to a minimum at the last layer, mean = avg_budget,
 * every entry >= n_sink + 1; "Parameters": beta = 1 is flat, larger beta is
 * steeper; "Evidence": beta < 1 raises, single-layer and empty-model cases.
 *
 * Reading: the half-spread is h = min((beta-1)*avg, avg-(n_sink+1)), i.e. the
 * steepness asks for a top of beta*avg and the floor caps the spread, keeping
 * the taper centred on avg. Layer l gets avg + round(h*(1 - 2l/(L-1))), the
 * offset rounded half away from zero (symmetric, so the mean stays avg). This
 * reproduces the page's worked 12-layer example exactly.
 * ------------------------------------------------------------------------- */
static double round_half_away(double x) {
  double a = fabs(x);
  double f = floor(a);
  double r = (a - f >= 0.5) ? f + 1.0 : f;
  return x < 0 ? -r : r;
}

int orc_budgets(int32_t n_layers, int32_t avg_budget, int32_t n_sink, double beta, int32_t* out) {
  if (n_layers < 0 || n_sink < 0 || !(beta >= 1.0)) return -1;
  if (avg_budget < n_sink + 1) return -1;
  if (n_layers == 0) return 0;
  if (n_layers == 1) { out[0] = avg_budget; return 0; }
  double spread = (beta - 1.0) * (double)avg_budget;
  double room = (double)(avg_budget - (n_sink + 1));
  double h = spread < room ? spread : room;
  for (int32_t l = 0; l < n_layers; ++l) {
    double frac = 1.0 - 2.0 * (double)l / (double)(n_layers - 1);
    out[l] = avg_budget + (int32_t)round_half_away(h * frac);
  }
  return 0;
}

/* ---------------------------------------------------------------------------
 * Frozen Gumbel value. Keyformer page, "THE HONESTY CRUX" item 2 and
 * KeyformerState.gumbel: one deterministic value per inserted position, drawn
 * once and never redrawn; g = -log(-log(u)).
 *
 * Reading (the pages give no formula): SplitMix64 (Steele, Lea & Flood 2014)
 * chained over (seed, layer, head, position); the batch index is not hashed.
 * u takes the top 52 bits of the hash as k and is (2k+1)/2^53, exact in fp64
 * and strictly inside (0,1). g is computed in fp64 and stored as float32.
 * ------------------------------------------------------------------------- */
uint64_t orc_splitmix64(uint64_t x) {
  uint64_t z = x + 0x9E3779B97F4A7C15ULL;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

uint64_t orc_gumbel_hash(uint64_t seed, int64_t layer, int64_t head, int64_t pos) {
  uint64_t h = orc_splitmix64(seed);
  h = orc_splitmix64(h ^ (uint64_t)layer);
  h = orc_splitmix64(h ^ (uint64_t)head);
  h = orc_splitmix64(h ^ (uint64_t)pos);
  return h;
}

float orc_gumbel_of_hash(uint64_t h) {
  uint64_t k = h >> 12;                                            /* top 52 bits */
  double u = (double)(2 * k + 1) * 0x1p-53;                        /* (0,1) */
  double g = -log(-log(u));
  return (float)g;
}

float orc_gumbel(uint64_t seed, int64_t layer, int64_t head, int64_t pos) {
  return orc_gumbel_of_hash(orc_gumbel_hash(seed, layer, head, pos));
}

void orc_gumbel_many(uint64_t seed, int64_t layer, int64_t head, int64_t p0, int64_t count, float* out) {
  for (int64_t t = 0; t < count; ++t) out[t] = orc_gumbel(seed, layer, head, p0 + t);
}

/* ---------------------------------------------------------------------------
 * Annealed temperature. Keyformer page, GAP #1 and KeyformerState.tau_end /
 * anneal_steps; init_keyformer_state: anneal_steps = 0 means constant tau_init.
 * tau = tau_init + min(pos, T) * (tau_end - tau_init) / T.
 * ------------------------------------------------------------------------- */
double orc_tau(double tau_init, double tau_end, int64_t anneal_steps, int64_t pos) {
  if (anneal_steps <= 0 || tau_init == tau_end) return tau_init;
  int64_t t = pos < anneal_steps ? pos : anneal_steps;
  if (t < 0) t = 0;
  return tau_init + (double)t * (tau_end - tau_init) / (double)anneal_steps;
}

/* ---------------------------------------------------------------------------
 * IEEE 754 binary16, written from the format's definition: 1 sign bit, 5
 * exponent bits (bias 15), 10 fraction bits; subnormal quantum 2^-24.
 * ------------------------------------------------------------------------- */
static double round_half_even(double q) {  /* q >= 0, few significant bits */
  double f = floor(q);
  double d = q - f;
  if (d > 0.5) return f + 1.0;
  if (d < 0.5) return f;
  return (fmod(f, 2.0) == 0.0) ? f : f + 1.0;
}

uint16_t orc_f32_to_f16(float xf) {
  uint32_t u;
  memcpy(&u, &xf, sizeof u);
  uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
  uint32_t a = u & 0x7FFFFFFFu;
  if (a > 0x7F800000u) return (uint16_t)(sign | 0x7E00u);       /* NaN */
  if (a >= 0x477FF000u) return (uint16_t)(sign | 0x7C00u);      /* >= 65520 rounds past 65504 */
  if (a < 0x38800000u) {                                        /* below 2^-14: subnormal */
    double m = round_half_even(fabs((double)xf) * 0x1p24);      /* exact scaling */
    return (uint16_t)(sign | (uint16_t)m);                      /* m == 1024 is 2^-14 */
  }
  /* normal: rebias the exponent (127 -> 15), keep 10 of the 23 fraction bits
   * and round the 13 dropped bits to nearest, ties to even; a carry out of
   * the fraction correctly bumps the exponent. */
  uint32_t e = (a >> 23) - 112u;
  uint32_t frac = a & 0x7FFFFFu;
  uint32_t h = (e << 10) | (frac >> 13);
  uint32_t rest = frac & 0x1FFFu;
  if (rest > 0x1000u || (rest == 0x1000u && (h & 1u))) h += 1u;
  return (uint16_t)(sign | h);
}

/* Exact values of all 65536 binary16 patterns, from the format's definition. */
static double f16_value[65536];

static double f16_decode(uint16_t h) {
  int s = (h >> 15) & 1;
  int E = (h >> 10) & 0x1F;
  int M = h & 0x3FF;
  double v;
  if (E == 0) v = ldexp((double)M, -24);
  else if (E == 31) v = M ? NAN : INFINITY;
  else v = ldexp((double)(1024 + M), E - 25);
  return s ? -v : v;
}

__attribute__((constructor)) static void f16_table_init(void) {
  for (uint32_t h = 0; h < 65536u; ++h) f16_value[h] = f16_decode((uint16_t)h);
}

double orc_f16_to_f64(uint16_t h) { return f16_value[h]; }

void orc_f32_to_f16_array(int64_t n, const float* x, uint16_t* out) {
  for (int64_t t = 0; t < n; ++t) out[t] = orc_f32_to_f16(x[t]);
}

void orc_f16_to_f64_array(int64_t n, const uint16_t* h, double* out) {
  for (int64_t t = 0; t < n; ++t) out[t] = orc_f16_to_f64(h[t]);
}

/* ---------------------------------------------------------------------------
 * RoPE re-rotation. Keyformer page, GAP #2 (survivors that shift are
 * re-rotated so the position baked into each key stays consistent) and the
 * FUSED METAL KERNEL note (rotation in fp32, fp16 storage).
 *
 * Reading: half-split pairs (x_i, x_{i+D/2}) with w_i = theta^(-2i/D); the
 * constants cos/sin(delta*w_i) are taken in fp64 and rounded to float32; the
 * pair maps to (a*c - b*s, a*s + b*c), every product and sum rounded to
 * float32, the results rounded to fp16 (nearest, ties to even).
 * ------------------------------------------------------------------------- */
void orc_rope_consts(double theta, int32_t D, int64_t delta, float* c, float* s) {
  for (int32_t i = 0; i < D / 2; ++i) {
    double w = pow(theta, -(2.0 * (double)i) / (double)D);
    double ang = (double)delta * w;
    c[i] = (float)cos(ang);
    s[i] = (float)sin(ang);
  }
}

void orc_rotate_row(int32_t D, uint16_t* row, const float* c, const float* s) {
  int32_t half = D / 2;
  for (int32_t i = 0; i < half; ++i) {
    float a = (float)orc_f16_to_f64(row[i]);
    float b = (float)orc_f16_to_f64(row[i + half]);
    float ac = a * c[i];
    float bs = b * s[i];
    float x = ac - bs;
    float as = a * s[i];
    float bc = b * c[i];
    float y = as + bc;
    row[i] = orc_f32_to_f16(x);
    row[i + half] = orc_f32_to_f16(y);
  }
}

/* ---------------------------------------------------------------------------
 * Decode step. Keyformer page, keyformer_update steps 1-2; PyramidKV page,
 * "How it works" steps 1-2: the new key k_i is a proxy query,
 * attn = softmax(K k_i / sqrt(D)), scores += attn, new tokens start at 0.
 * The softmax runs over every stored row including the one just appended
 * (reading: the benchmark specification fixes this order).
 * mode ORC_SCORE_CURRENT is the TOVA-adapted row of the PyramidKV page's
 * method table ("current-step attention weight"): scores = attn instead.
 * ------------------------------------------------------------------------- */
int32_t orc_step_accumulate(int32_t D, int32_t n, uint16_t* K, double* score, float* g,
                            int32_t* pos, const uint16_t* k_new, int64_t p, float g_new,
                            int32_t mode) {
  memcpy(K + (size_t)n * D, k_new, sizeof(uint16_t) * (size_t)D);
  score[n] = 0.0;
  g[n] = g_new;
  pos[n] = (int32_t)p;
  int32_t n1 = n + 1;

  double* logit = (double*)malloc(sizeof(double) * (size_t)n1);
  double inv_sqrt_d = 1.0 / sqrt((double)D);
  for (int32_t j = 0; j < n1; ++j) {
    double dot = 0.0;
    for (int32_t d = 0; d < D; ++d)
      dot += orc_f16_to_f64(K[(size_t)j * D + d]) * orc_f16_to_f64(k_new[d]);
    logit[j] = dot * inv_sqrt_d;
  }
  double m = logit[0];
  for (int32_t j = 1; j < n1; ++j) if (logit[j] > m) m = logit[j];
  double l = 0.0;
  for (int32_t j = 0; j < n1; ++j) l += exp(logit[j] - m);
  for (int32_t j = 0; j < n1; ++j) {
    double attn = exp(logit[j] - m) / l;
    if (mode == ORC_SCORE_CURRENT) score[j] = attn;   /* TOVA-adapted: this step's weight */
    else score[j] += attn;                            /* H2O rule: cumulative mass */
  }
  free(logit);
  return n1;
}

/* Keyformer page, keyformer_update step 3: the eviction key is
 * score + tau * gumbel; the stored score itself stays clean. */
void orc_regularised(int32_t n, const double* score, const float* g, double tau, double* r) {
  for (int32_t j = 0; j < n; ++j) r[j] = score[j] + tau * (double)g[j];
}

/* Keyformer page, step 3, and PyramidKV page, "How it works" step 3: evict the
 * lowest non-protected row; the first n_sink rows are protected (+inf), and so
 * are the last `recent` rows (keyformer page, KeyformerState.recent: the
 * trailing protected window, 0 = off). Ties go to the lowest slot (reading
 * fixed by the benchmark specification). */
int32_t orc_argmin(int32_t n, const double* r, int32_t n_sink, int32_t recent) {
  int32_t best = -1;
  for (int32_t j = n_sink; j < n - recent; ++j)
    if (best < 0 || r[j] < r[best]) best = j;
  return best;
}

/* Keyformer page, step 3: survivors after the evicted token shift down by one
 * and are re-rotated; "Kept tokens are returned in original temporal order".
 * positions[] carries each row's original absolute position (reading). */
static int32_t evict_with_consts(int32_t D, int32_t n, uint16_t* K, double* score, float* g,
                                 int32_t* pos, int32_t e, const float* c, const float* s) {
  for (int32_t j = e + 1; j < n; ++j) {
    uint16_t* dst = K + (size_t)(j - 1) * D;
    memcpy(dst, K + (size_t)j * D, sizeof(uint16_t) * (size_t)D);
    orc_rotate_row(D, dst, c, s);
    score[j - 1] = score[j];
    g[j - 1] = g[j];
    pos[j - 1] = pos[j];
  }
  return n - 1;
}

int32_t orc_evict(int32_t D, int32_t n, uint16_t* K, double* score, float* g, int32_t* pos,
                  int32_t e, double theta) {
  float* c = (float*)malloc(sizeof(float) * (size_t)D);
  float* s = c + D / 2;
  orc_rope_consts(theta, D, -1, c, s);
  int32_t r = evict_with_consts(D, n, K, score, g, pos, e, c, s);
  free(c);
  return r;
}

/* ---------------------------------------------------------------------------
 * Value rows. Keyformer page, KeyformerState.values (one fp16 value row per
 * kept token, [n_kept, D]), keyformer_update steps 2-3 (a token is appended
 * with its key and value; survivors after the evicted token shift down by one)
 * and keyformer_get_kv (keys and values are returned together). A value row
 * carries no position, so it is only moved: the RoPE remap of step 3 applies
 * to keys alone.
 * ------------------------------------------------------------------------- */
void orc_values_append(int32_t D, int32_t n, uint16_t* V, const uint16_t* v_new) {
  memcpy(V + (size_t)n * D, v_new, sizeof(uint16_t) * (size_t)D);
}

int32_t orc_values_evict(int32_t D, int32_t n, uint16_t* V, int32_t e) {
  for (int32_t j = e + 1; j < n; ++j)
    memcpy(V + (size_t)(j - 1) * D, V + (size_t)j * D, sizeof(uint16_t) * (size_t)D);
  return n - 1;
}

/* The prompt's value rows after a bulk eviction: the survivors' rows in order. */
int32_t orc_values_prefill_apply(int32_t S, int32_t D, const uint16_t* values, const uint8_t* mask,
                                 uint16_t* V) {
  int32_t n = 0;
  for (int32_t j = 0; j < S; ++j) {
    if (mask[j]) continue;
    memcpy(V + (size_t)n * D, values + (size_t)j * D, sizeof(uint16_t) * (size_t)D);
    ++n;
  }
  return n;
}

/* ---------------------------------------------------------------------------
 * Prefill scoring: the column sums of the causal softmax(K K^T / sqrt(D)),
 * diagonal included. This is what S consecutive decode steps without eviction
 * accumulate (keyformer_update, "For each of the S incoming tokens", steps 1-2).
 * Row i: lse_i = log sum_{j<=i} exp(G_ij); colsum_j = sum_{i>=j} exp(G_ij - lse_i).
 * ------------------------------------------------------------------------- */
void orc_prefill_colsum(int32_t S, int32_t D, const uint16_t* keys, double* colsum) {
  double* kd = (double*)malloc(sizeof(double) * (size_t)S * D);
  double* row = (double*)malloc(sizeof(double) * (size_t)(S > 0 ? S : 1));
  for (size_t t = 0; t < (size_t)S * D; ++t) kd[t] = orc_f16_to_f64(keys[t]);
  double inv_sqrt_d = 1.0 / sqrt((double)D);
  for (int32_t j = 0; j < S; ++j) colsum[j] = 0.0;
  for (int32_t i = 0; i < S; ++i) {
    const double* ki = kd + (size_t)i * D;
    double m = -INFINITY;
    for (int32_t j = 0; j <= i; ++j) {
      const double* kj = kd + (size_t)j * D;
      double dot = 0.0;
      for (int32_t d = 0; d < D; ++d) dot += ki[d] * kj[d];
      row[j] = dot * inv_sqrt_d;
      if (row[j] > m) m = row[j];
    }
    double l = 0.0;
    for (int32_t j = 0; j <= i; ++j) l += exp(row[j] - m);
    double lse = m + log(l);
    for (int32_t j = 0; j <= i; ++j) colsum[j] += exp(row[j] - lse);
  }
  free(row);
  free(kd);
}

/* TOVA-adapted prompt scores: the attention the prompt's last token pays to
 * every prompt token, softmax(K k_{S-1} / sqrt(D)) over all S rows (reading:
 * "current-step attention weight" at the end of the prompt). */
void orc_prefill_lastrow(int32_t S, int32_t D, const uint16_t* keys, double* score) {
  if (S <= 0) return;
  double* logit = (double*)malloc(sizeof(double) * (size_t)S);
  const uint16_t* q = keys + (size_t)(S - 1) * D;
  double inv_sqrt_d = 1.0 / sqrt((double)D);
  double m = -INFINITY;
  for (int32_t j = 0; j < S; ++j) {
    double dot = 0.0;
    for (int32_t d = 0; d < D; ++d)
      dot += orc_f16_to_f64(keys[(size_t)j * D + d]) * orc_f16_to_f64(q[d]);
    logit[j] = dot * inv_sqrt_d;
    if (logit[j] > m) m = logit[j];
  }
  double l = 0.0;
  for (int32_t j = 0; j < S; ++j) l += exp(logit[j] - m);
  for (int32_t j = 0; j < S; ++j) score[j] = exp(logit[j] - m) / l;
  free(logit);
}

/* Bulk eviction after the prompt (reading: score the whole prompt, then evict
 * the S - budget lowest (r, slot) non-sink rows at once; lower slot first
 * among equal r). */
int32_t orc_prefill_select(int32_t S, int32_t budget, int32_t n_sink, int32_t recent,
                           const double* r, uint8_t* mask) {
  for (int32_t j = 0; j < S; ++j) mask[j] = 0;
  int32_t want = S - budget;
  if (want <= 0) return 0;
  /* order the unprotected rows (not a sink, not among the last `recent`) by
   * (r, slot) and take the first `want` */
  int32_t m = S - n_sink - recent;
  if (m < want) return -1;
  int32_t* idx = (int32_t*)malloc(sizeof(int32_t) * (size_t)(m > 0 ? m : 1));
  for (int32_t t = 0; t < m; ++t) idx[t] = n_sink + t;
  for (int32_t a = 1; a < m; ++a) {          /* stable insertion sort by r */
    int32_t v = idx[a];
    int32_t b = a - 1;
    while (b >= 0 && r[idx[b]] > r[v]) { idx[b + 1] = idx[b]; --b; }
    idx[b + 1] = v;
  }
  for (int32_t t = 0; t < want; ++t) mask[idx[t]] = 1;
  free(idx);
  return want;
}

int32_t orc_prefill_apply(int32_t S, int32_t D, const uint16_t* keys, const double* colsum,
                          const float* g, const uint8_t* mask, double theta,
                          uint16_t* K, double* score, float* g_out, int32_t* pos) {
  float* c = (float*)malloc(sizeof(float) * (size_t)D);
  float* s = c + D / 2;
  int32_t n = 0;
  for (int32_t j = 0; j < S; ++j) {
    if (mask[j]) continue;
    uint16_t* dst = K + (size_t)n * D;
    memcpy(dst, keys + (size_t)j * D, sizeof(uint16_t) * (size_t)D);
    int64_t delta = (int64_t)n - (int64_t)j;        /* new slot - old slot */
    if (delta != 0) {
      orc_rope_consts(theta, D, delta, c, s);
      orc_rotate_row(D, dst, c, s);
    }
    score[n] = colsum[j];
    g_out[n] = g[j];
    pos[n] = j;
    ++n;
  }
  free(c);
  return n;
}

/* ---------------------------------------------------------------------------
 * Whole-pass driver (own decisions): prefill, then T decode steps.
 * ------------------------------------------------------------------------- */
int32_t orc_run_head(const orc_head_cfg* cfg, int32_t S, const uint16_t* prefill_keys,
                     int32_t T, const uint16_t* decode_keys, int32_t* evicted,
                     uint16_t* K, double* score, float* g, int32_t* pos) {
  int32_t D = cfg->D, budget = cfg->budget;
  const uint16_t* decode_keys_all = decode_keys;
  int32_t n = 0;
  if (S > 0 && cfg->prefill_mode == 1) {
    /* keyformer page, keyformer_update: "For each of the S incoming tokens" --
     * every prompt token is one step, evicting inside the prompt */
    T += S;
    decode_keys = NULL;   /* handled below: the prompt comes first */
  }
  if (S > 0 && cfg->prefill_mode != 1) {
    double* colsum = (double*)malloc(sizeof(double) * (size_t)S);
    float* gp = (float*)malloc(sizeof(float) * (size_t)S);
    double* r = (double*)malloc(sizeof(double) * (size_t)S);
    uint8_t* mask = (uint8_t*)malloc((size_t)S);
    if (cfg->mode == ORC_SCORE_CURRENT) orc_prefill_lastrow(S, D, prefill_keys, colsum);
    else orc_prefill_colsum(S, D, prefill_keys, colsum);
    for (int32_t j = 0; j < S; ++j) gp[j] = orc_gumbel(cfg->seed, cfg->layer, cfg->head, j);
    double tau = orc_tau(cfg->tau_init, cfg->tau_end, cfg->anneal_steps, S - 1);
    for (int32_t j = 0; j < S; ++j) r[j] = colsum[j] + tau * (double)gp[j];
    orc_prefill_select(S, budget, cfg->n_sink, cfg->recent, r, mask);
    n = orc_prefill_apply(S, D, prefill_keys, colsum, gp, mask, cfg->theta, K, score, g, pos);
    free(mask); free(r); free(gp); free(colsum);
  }
  float* c = (float*)malloc(sizeof(float) * (size_t)D);
  float* s = c + D / 2;
  orc_rope_consts(cfg->theta, D, -1, c, s);
  double* r = (double*)malloc(sizeof(double) * (size_t)(budget + 2));
  const int32_t seq = (S > 0 && cfg->prefill_mode == 1);
  const int64_t p0 = seq ? 0 : (int64_t)S;
  for (int32_t t = 0; t < T; ++t) {
    int64_t p = p0 + t;
    const uint16_t* k = (seq && t < S) ? prefill_keys + (size_t)t * D
                                       : decode_keys_all + (size_t)(seq ? t - S : t) * D;
    float gn = orc_gumbel(cfg->seed, cfg->layer, cfg->head, p);
    int32_t n1 = orc_step_accumulate(D, n, K, score, g, pos, k, p, gn, cfg->mode);
    if (n1 > budget) {
      double tau = orc_tau(cfg->tau_init, cfg->tau_end, cfg->anneal_steps, p);
      orc_regularised(n1, score, g, tau, r);
      int32_t e = orc_argmin(n1, r, cfg->n_sink, cfg->recent);
      if (evicted && !(seq && t < S)) evicted[seq ? t - S : t] = e;
      n = evict_with_consts(D, n1, K, score, g, pos, e, c, s);
    } else {
      if (evicted && !(seq && t < S)) evicted[seq ? t - S : t] = -1;
      n = n1;
    }
  }
  free(r);
  free(c);
  return n;
}

int32_t orc_run_heads(int32_t n_heads, const orc_head_cfg* cfgs, int32_t S,
                      const uint16_t* prefill_keys, int32_t T, const uint16_t* decode_keys,
                      int32_t* evicted, int32_t cap, uint16_t* K, double* score, float* g,
                      int32_t* pos, int32_t* n_out, int32_t n_threads) {
  int32_t used = 1;
#ifdef _OPENMP
  if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel
  {
#pragma omp single
    used = omp_get_num_threads();
#pragma omp for schedule(dynamic, 1)
    for (int32_t hh = 0; hh < n_heads; ++hh) {
      n_out[hh] = orc_run_head(&cfgs[hh], S, prefill_keys + (size_t)hh * S * cfgs[hh].D, T,
                               decode_keys + (size_t)hh * T * cfgs[hh].D,
                               evicted ? evicted + (size_t)hh * T : NULL,
                               K + (size_t)hh * cap * cfgs[hh].D, score + (size_t)hh * cap,
                               g + (size_t)hh * cap, pos + (size_t)hh * cap);
    }
  }
#else
  (void)n_threads;
  for (int32_t hh = 0; hh < n_heads; ++hh)
    n_out[hh] = orc_run_head(&cfgs[hh], S, prefill_keys + (size_t)hh * S * cfgs[hh].D, T,
                             decode_keys + (size_t)hh * T * cfgs[hh].D,
                             evicted ? evicted + (size_t)hh * T : NULL,
                             K + (size_t)hh * cap * cfgs[hh].D, score + (size_t)hh * cap,
                             g + (size_t)hh * cap, pos + (size_t)hh * cap);
#endif
  return used;
}
