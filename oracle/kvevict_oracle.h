/*
 * kvevict_oracle.h -- plain fp64 CPU oracle for cumulative proxy-attention
 * KV-cache eviction (H2O-adapted, Keyformer-adapted, PyramidKV-adapted).
 *
 * TEST INFRASTRUCTURE. This oracle exists to check the CUDA library. Only the
 * test suite, the smoke check and the benchmark's CPU-baseline leg may load
 * it. It shares no code, header, table or constant generator with the CUDA
 * path, and it never reads anything the CUDA path produced.
 *
 * Sources (page title, section):
 *  - "veloxquant_mlx.quantizers.keyformer module": KeyformerState fields,
 *    init_keyformer_state (validation), keyformer_update (the three per-token
 *    steps), FUSED METAL KERNEL note (rotation in fp32, keys within 1 ULP),
 *    GAP #1 (tau annealing, Eq. 10), GAP #2 (RoPE position remap).
 *  - "PyramidKV -- Layer-Adaptive Budget Attention-Mass Eviction": "The budget
 *    schedule" (worked 12-layer example) and "How it works" (per-step rule).
 *
 * Precision: every score, softmax and regularised score is fp64. Two steps
 * decide a code and are taken in the precision the pages fix instead:
 * the RoPE re-rotation of a shifted key (fp32 arithmetic, then fp16 storage;
 * keyformer page, FUSED METAL KERNEL) and the stored Gumbel value (float32;
 * keyformer page, KeyformerState.gumbel).
 *
 * Parity pins live in tests/test_oracle_*.py. One function has no pin from
 * the pages: the way orc_gumbel_hash chains SplitMix64 over (seed, layer,
 * head, position) (the pages name no formula) is "parity unpinned". What can
 * be pinned is: SplitMix64 itself (published reference outputs), the map
 * from a hash to u and g (its end points and monotonicity, from the
 * mathematics) and the Gumbel law of the values (moments, KS test). A table
 * of hashes and values in tests/golden/ is a regression fixture, not a pin.
 */
#ifndef KVEVICT_ORACLE_H
#define KVEVICT_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Per-layer budget taper. 0 on success, -1 on invalid input. */
int orc_budgets(int32_t n_layers, int32_t avg_budget, int32_t n_sink, double beta, int32_t* out);

/* SplitMix64: the output of a generator whose state was x, after one step. */
uint64_t orc_splitmix64(uint64_t x);
/* Hash of (seed, layer, head, position) and the frozen Gumbel value. */
uint64_t orc_gumbel_hash(uint64_t seed, int64_t layer, int64_t head, int64_t pos);
/* The Gumbel value of a hash: k = top 52 bits, u = (2k+1)/2^53, -log(-log u) as f32. */
float orc_gumbel_of_hash(uint64_t h);
float orc_gumbel(uint64_t seed, int64_t layer, int64_t head, int64_t pos);
/* Gumbel values for positions p0 .. p0+count-1 of one (layer, head). */
void orc_gumbel_many(uint64_t seed, int64_t layer, int64_t head, int64_t p0, int64_t count, float* out);

/* Annealed temperature at absolute position pos (keyformer page, GAP #1). */
double orc_tau(double tau_init, double tau_end, int64_t anneal_steps, int64_t pos);

/* IEEE binary16 helpers (round to nearest, ties to even). */
uint16_t orc_f32_to_f16(float x);
double orc_f16_to_f64(uint16_t h);
void orc_f32_to_f16_array(int64_t n, const float* x, uint16_t* out);
void orc_f16_to_f64_array(int64_t n, const uint16_t* h, double* out);

/* RoPE constants for a rotation by delta positions: c[i] = f32(cos(delta*w_i)),
 * s[i] = f32(sin(delta*w_i)), w_i = theta^(-2i/D), i < D/2. */
void orc_rope_consts(double theta, int32_t D, int64_t delta, float* c, float* s);
/* Rotate one fp16 row by the given constants, fp32 arithmetic, half-split pairs. */
void orc_rotate_row(int32_t D, uint16_t* row, const float* c, const float* s);

/* Score modes: cumulative attention mass (H2O rule, Keyformer, PyramidKV) or
 * the current step's attention weight (TOVA-adapted). */
#define ORC_SCORE_CUMULATIVE 0
#define ORC_SCORE_CURRENT 1

/* One decode step, append + proxy-attention accumulation. The state holds n
 * rows; the new row goes to slot n. Returns n+1. Arrays need room for n+1 rows. */
int32_t orc_step_accumulate(int32_t D, int32_t n, uint16_t* K, double* score, float* g,
                            int32_t* pos, const uint16_t* k_new, int64_t p, float g_new,
                            int32_t mode);
/* Regularised scores r_j = score_j + tau*g_j (fp64), for all rows. */
void orc_regularised(int32_t n, const double* score, const float* g, double tau, double* r);
/* Lowest slot attaining min r over n_sink <= j < n - recent; -1 if none. */
int32_t orc_argmin(int32_t n, const double* r, int32_t n_sink, int32_t recent);
/* Evict slot e from an n-row state: rows after e move down one slot in order,
 * each moved key re-rotated by -1 position. Returns n-1. */
int32_t orc_evict(int32_t D, int32_t n, uint16_t* K, double* score, float* g, int32_t* pos,
                  int32_t e, double theta);

/* Value rows (fp16 bits [rows, D]) move with their keys and are never rotated.
 * append: V[n] = v_new. evict: rows after e move down one slot; returns n-1.
 * prefill_apply: the unmasked prompt value rows in order; returns the count. */
void orc_values_append(int32_t D, int32_t n, uint16_t* V, const uint16_t* v_new);
int32_t orc_values_evict(int32_t D, int32_t n, uint16_t* V, int32_t e);
int32_t orc_values_prefill_apply(int32_t S, int32_t D, const uint16_t* values, const uint8_t* mask,
                                 uint16_t* V);

/* Prefill scoring: column sums of the causal softmax(K K^T / sqrt(D)), the
 * diagonal included. keys [S, D] fp16 bits, out colsum [S]. */
void orc_prefill_colsum(int32_t S, int32_t D, const uint16_t* keys, double* colsum);
/* TOVA-adapted prompt scores: the last prompt token's attention over the prompt. */
void orc_prefill_lastrow(int32_t S, int32_t D, const uint16_t* keys, double* score);
/* Own bulk selection: mark the S - budget unprotected rows (not among the
 * first n_sink or the last `recent`) with the lowest (r, slot); mask[j] = 1
 * for evicted rows. Returns the evicted count, -1 if there is no room. */
int32_t orc_prefill_select(int32_t S, int32_t budget, int32_t n_sink, int32_t recent,
                           const double* r, uint8_t* mask);
/* Apply a bulk eviction mask: survivors move to consecutive slots in order,
 * each re-rotated by (new slot - old slot). Returns the kept count. */
int32_t orc_prefill_apply(int32_t S, int32_t D, const uint16_t* keys, const double* colsum,
                          const float* g, const uint8_t* mask, double theta,
                          uint16_t* K, double* score, float* g_out, int32_t* pos);

/* Whole-pass driver for one head (prefill then T decode steps), with the
 * oracle's own eviction decisions; used for the CPU baseline and self-tests.
 * evicted[T] gets the slot evicted at each step or -1. State arrays need
 * room for budget+1 rows. Returns the final kept count. */
typedef struct orc_head_cfg {
  int32_t D, budget, n_sink, layer, head;
  double tau_init, tau_end; int64_t anneal_steps;
  double theta; uint64_t seed;
  int32_t recent, mode;
  int32_t prefill_mode;   /* 0: score the whole prompt then bulk-evict; 1: one step per token */
} orc_head_cfg;
int32_t orc_run_head(const orc_head_cfg* cfg, int32_t S, const uint16_t* prefill_keys,
                     int32_t T, const uint16_t* decode_keys, int32_t* evicted,
                     uint16_t* K, double* score, float* g, int32_t* pos);
/* The same over many heads in parallel (OpenMP); arrays are per-head strided
 * by S*D, T*D, T and cap*D / cap. Returns the thread count used. */
int32_t orc_run_heads(int32_t n_heads, const orc_head_cfg* cfgs, int32_t S,
                      const uint16_t* prefill_keys, int32_t T, const uint16_t* decode_keys,
                      int32_t* evicted, int32_t cap, uint16_t* K, double* score, float* g,
                      int32_t* pos, int32_t* n_out, int32_t n_threads);

#ifdef __cplusplus
}
#endif
#endif
