/*
 * kvevict.h -- C ABI of the GB300 (sm_103a) cumulative proxy-attention
 * KV-cache eviction library: H2O-adapted, Keyformer-adapted (Gumbel
 * regulariser with an annealed temperature) and PyramidKV-adapted (per-layer
 * budget taper), all one decode step.
 *
 * What one step computes, for every (batch, layer, KV head) row of the cache
 * (page "veloxquant_mlx.quantizers.keyformer module", keyformer_update steps
 * 1-3; page "PyramidKV -- Layer-Adaptive Budget Attention-Mass Eviction",
 * "How it works"):
 *   1. append the new fp16 key k with score 0, its absolute position p and a
 *      frozen Gumbel value g(seed, layer, head, p);
 *   2. attn = softmax(K k / sqrt(D)) over every stored row, the new one
 *      included; scores += attn;
 *   3. if the layer's budget is exceeded, evict the lowest
 *      score + tau(p) * g over rows n_sink <= j < n+1-recent (lowest slot on
 *      ties); the
 *      rows after it move down one slot in order, each key re-rotated by -1
 *      RoPE position in fp32 and stored as fp16.
 *
 * Conventions shared by every entry point:
 *  - fp16 values cross the boundary as uint16_t bit patterns (IEEE binary16).
 *  - Device pointers are CUDA global-memory pointers on the device that was
 *    current at kvevict_create (mapped page-locked host memory counts as
 *    one); device key and value buffers must start on a 16-byte boundary
 *    (INVALID_ARG otherwise). Host pointers are plain host memory; the
 *    host-buffer entry point moves page-locked buffers with its own kernels
 *    (see kvevict_run_host).
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream). All work
 *    is enqueued on it; calls return before the GPU finishes unless stated.
 *  - The caller owns every buffer it passes and keeps it alive until the
 *    stream has passed the call. The library owns its state arena.
 *  - Return codes: 0 on success, else one of KVEVICT_ERR_*; the message of the
 *    last failure on the calling thread is kvevict_last_error().
 *  - One handle is not thread-safe; use one handle per thread or lock.
 */
#ifndef KVEVICT_H
#define KVEVICT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KVEVICT_OK 0
#define KVEVICT_ERR_INVALID_ARG (-1)  /* bad config, pointer or size */
#define KVEVICT_ERR_BAD_STATE (-2)    /* call out of order (e.g. prefill after a step) */
#define KVEVICT_ERR_CUDA (-3)         /* a CUDA runtime call failed */
#define KVEVICT_ERR_OOM (-4)          /* device allocation failed */
#define KVEVICT_ERR_DEVICE_CHECK (-5) /* a kernel raised its error word (bounded wait ran out) */

#define KVEVICT_MAX_LAYERS 256
#define KVEVICT_MAX_PREFILL 16384

/* Cache configuration (page "veloxquant_mlx.quantizers.keyformer module",
 * KeyformerState and init_keyformer_state; page "PyramidKV ...", Parameters). */
typedef struct kvevict_config {
  int32_t batch;          /* B >= 1 */
  int32_t n_layers;       /* L, 1 .. KVEVICT_MAX_LAYERS */
  int32_t n_kv_heads;     /* H >= 1 */
  int32_t head_dim;       /* D, 64 or 128 */
  int32_t avg_budget;     /* average kept rows per layer, sinks included */
  double pyramid_beta;    /* >= 1; 1 = the same budget in every layer (plain H2O) */
  const int32_t* layer_budgets; /* optional host array [n_layers]; overrides avg/beta */
  int32_t n_sink;         /* leading rows never evicted, >= 0; every budget >= n_sink + 1 */
  float tau_init;         /* Gumbel temperature at position 0, >= 0 */
  float tau_end;          /* temperature once position >= anneal_steps, >= 0 */
  int32_t anneal_steps;   /* >= 0; 0 = constant tau_init */
  double rope_theta;      /* RoPE base of the model's attention, > 0 */
  uint64_t seed;          /* base seed of the frozen Gumbel values */
  int32_t max_prefill;    /* longest prompt kvevict_prefill will take, 0 .. KVEVICT_MAX_PREFILL */
  int32_t recent;         /* trailing protected window, >= 0; 0 = off (keyformer page,
                             KeyformerState.recent); every budget >= n_sink + recent + 1 */
  int32_t score_mode;     /* KVEVICT_SCORE_CUMULATIVE (H2O rule) or KVEVICT_SCORE_CURRENT */
  int32_t prefill_mode;   /* KVEVICT_PREFILL_BULK or KVEVICT_PREFILL_SEQUENTIAL */
  int32_t with_values;    /* 1: the cache also holds value rows (fp16 [.., D]); they move with
                             their keys and are never rotated (keyformer page,
                             KeyformerState.values); 0: keys only */
  int32_t decode_kernel;  /* KVEVICT_DECODE_AUTO (0), KVEVICT_DECODE_STREAM or
                             KVEVICT_DECODE_RESIDENT: which kernel runs the decode steps */
} kvevict_config;

/* Decode kernels; both compute the same steps and give the same results bit
 * for bit. STREAM: every step streams each row's keys from device memory
 * through shared memory, any row length. RESIDENT: a call of several steps
 * keeps each row in one CTA's shared memory for all of them (key-only handles
 * whose rows fit: about 780 keys at head_dim 128, 1023 at 64; the rows of a
 * large cache run in waves). AUTO takes RESIDENT for calls of at least 4
 * steps on key-only handles whose rows fit in one wave of CTAs, or in two at
 * two CTAs an SM, and STREAM otherwise (kvevict_decode_kernel_for reports the
 * choice); asking for RESIDENT on a handle whose rows do not fit, or that
 * carries values, is INVALID_ARG at create. */
#define KVEVICT_DECODE_AUTO 0
#define KVEVICT_DECODE_STREAM 1
#define KVEVICT_DECODE_RESIDENT 2

/* Prompt modes. BULK: score the whole prompt, then a row over budget evicts its
 * lowest (score + tau(S-1) * g, slot) rows at once. SEQUENTIAL: every prompt
 * token is absorbed as one step (page "veloxquant_mlx.quantizers.keyformer
 * module", keyformer_update: "For each of the S incoming tokens", steps 1-3),
 * so evictions happen inside the prompt, each with tau at its own position. */
#define KVEVICT_PREFILL_BULK 0
#define KVEVICT_PREFILL_SEQUENTIAL 1

/* Score modes (page "PyramidKV ...", method table): cumulative attention mass
 * (H2O-adapted, Keyformer-adapted, PyramidKV-adapted) or the current step's
 * attention weight (TOVA-adapted; a prompt then scores each token by the
 * prompt's last token's attention). */
#define KVEVICT_SCORE_CUMULATIVE 0
#define KVEVICT_SCORE_CURRENT 1

typedef struct kvevict kvevict_t;

/* Per-layer budget taper, host only (page "PyramidKV ...", "The budget
 * schedule"): linear from its maximum at layer 0 to its minimum at the last
 * layer, mean avg_budget, each >= n_sink + 1; beta = 1 is flat. Half-spread
 * h = min((beta-1)*avg, avg-(n_sink+1)); layer l gets
 * avg + round(h*(1 - 2l/(L-1))), the offset rounded half away from zero.
 * out: host int32[n_layers]. Errors: INVALID_ARG if beta < 1, n_layers < 0,
 * n_sink < 0 or avg_budget < n_sink + 1. */
int kvevict_budgets(int32_t n_layers, int32_t avg_budget, int32_t n_sink, double beta,
                    int32_t* out);

/* Validate cfg, compute the budgets and allocate the device state on the
 * current device: per row of the cache, (budget_l + 1) x D fp16 keys plus
 * float scores, float Gumbel values and int32 positions, and prefill scratch
 * for max_prefill tokens. The state starts empty (position 0).
 * Errors: INVALID_ARG (tau < 0, beta < 1, a budget <= n_sink, D not 64/128,
 * null pointers, sizes out of range), OOM, CUDA. *out is set only on success. */
int kvevict_create(const kvevict_config* cfg, void* stream, kvevict_t** out);

/* Free the handle and its device memory (synchronises the device first).
 * The pages keep a cache's state in a KeyformerState object that lives as long
 * as its owner holds it (page "veloxquant_mlx.quantizers.keyformer module",
 * KeyformerState); this ends the life of the device arena holding it here.
 * Errors: none (a null handle is ignored). */
int kvevict_destroy(kvevict_t* h);

/* Return the handle to the empty state at position 0 (the arena is reused). */
int kvevict_reset(kvevict_t* h, void* stream);

/* Absorb a prompt of S tokens at positions 0..S-1 (the state must be empty).
 * keys: device fp16 [B, L, H, S, D], each key already RoPE-rotated at its
 * position. Scores are the column sums of the causal softmax(K K^T/sqrt(D))
 * (the diagonal included), i.e. what S decode steps without eviction would
 * accumulate. A row whose layer budget b is below S then bulk-evicts the
 * S - b non-sink rows with the lowest (score + tau(S-1) * g, slot); survivors
 * keep their order and each is re-rotated by (new slot - old slot).
 * Errors: INVALID_ARG (null keys, S < 0 or S > max_prefill), BAD_STATE (state
 * not empty), CUDA. */
int kvevict_prefill(kvevict_t* h, const uint16_t* keys, int32_t S, void* stream);

/* kvevict_prefill with an optional log of the prompt's evictions: evicted is
 * device int32 [S, B, L, H] or NULL; in SEQUENTIAL mode entry [t] is the slot
 * the token at position t evicted (index into the rows after its append) or
 * -1; in BULK mode every entry is -1 (the bulk choice shows in the kept
 * positions). SEQUENTIAL mode runs the first min(S, smallest budget) tokens
 * through the prompt scorer (no row can evict yet, so this equals as many
 * single steps) and each further token as one decode step read straight from
 * the prompt buffer. Errors: as kvevict_prefill. */
int kvevict_prefill_ex(kvevict_t* h, const uint16_t* keys, int32_t S, int32_t* evicted,
                       void* stream);

/* The value-carrying forms (handles created with with_values = 1; the
 * key-only calls above return INVALID_ARG on such a handle). values /
 * v_new have the layouts of keys / k_new: device fp16 [B, L, H, S, D],
 * [B, L, H, D] and [T, B, L, H, D]. A value row is stored, moved and evicted
 * with its key; it is never rotated. Errors: as the key-only forms. */
int kvevict_prefill_kv(kvevict_t* h, const uint16_t* keys, const uint16_t* values, int32_t S,
                       int32_t* evicted, void* stream);
int kvevict_step_kv(kvevict_t* h, const uint16_t* k_new, const uint16_t* v_new, int32_t* evicted,
                    void* stream);
int kvevict_decode_kv(kvevict_t* h, const uint16_t* keys, const uint16_t* values, int32_t T,
                      int32_t* evicted, void* stream);

/* Copy one row's value rows to host memory (synchronises the stream):
 * values [n, D] fp16 bits in slot order, n = *n_kept. Errors: INVALID_ARG
 * (indices out of range, or a key-only handle), CUDA, DEVICE_CHECK. */
int kvevict_read_values(kvevict_t* h, int32_t b, int32_t l, int32_t head, uint16_t* values,
                        int32_t* n_kept, void* stream);

/* One decode step for every row at position p = kvevict_next_pos(): the
 * three steps of keyformer_update for one incoming token (page
 * "veloxquant_mlx.quantizers.keyformer module"), applied to every (batch,
 * layer, KV head) row at once as keyformer_update_batched applies them to
 * every (batch, head) row of a layer, with each layer's own budget (page
 * "PyramidKV ...", "How it works").
 * k_new: device fp16 [B, L, H, D], RoPE-rotated at p. evicted: device int32
 * [B, L, H] or NULL; receives the evicted slot (index into the rows after the
 * append, 0..n) or -1 when the row was within budget. One fused kernel launch.
 * Errors: INVALID_ARG (null k_new), CUDA. */
int kvevict_step(kvevict_t* h, const uint16_t* k_new, int32_t* evicted, void* stream);

/* T consecutive decode steps at positions p .. p + T - 1 in one kernel launch:
 * the same result as T kvevict_step calls. Rows are independent, so a row's
 * step t + 1 starts as soon as its own step t is done, with no wait for the
 * rest of the cache between steps.
 * keys: device fp16 [T, B, L, H, D]; evicted: device int32 [T, B, L, H] or NULL.
 * Errors: as kvevict_step; T < 0 is INVALID_ARG, T = 0 does nothing,
 * BAD_STATE once more than 2^31 - 1 decode steps follow a reset. */
int kvevict_decode(kvevict_t* h, const uint16_t* keys, int32_t T, int32_t* evicted,
                   void* stream);

/* End to end from host memory: prefill S prompt keys (host fp16
 * [B, L, H, S, D]; S may be 0) then T decode steps (host fp16 [T, B, L, H, D]),
 * with the evicted slots written back to host int32 [T, B, L, H] (or NULL).
 * The state must be empty. Returns after the stream has finished.
 * Each buffer must be one allocation. A page-locked buffer (cudaHostAlloc,
 * cudaMallocHost or cudaHostRegister; both its ends are checked) is accessed
 * by the library's kernels through its device mapping: the prompt is staged
 * to the device by a copy kernel, the decode keys are read in place by the
 * decode step, and the evicted slots are written back by a copy kernel.
 * Pageable memory goes through cudaMemcpyAsync in chunks on a second stream
 * that overlap with compute. Device staging (up to 2 x 256 MiB, or one batch's
 * prompt) is allocated on first use and kept with the handle.
 * Errors: INVALID_ARG, BAD_STATE, OOM, CUDA, DEVICE_CHECK. */
int kvevict_run_host(kvevict_t* h, const uint16_t* prefill_keys, int32_t S,
                     const uint16_t* decode_keys, int32_t T, int32_t* evicted, void* stream);
/* (key-only handles; a with_values handle returns INVALID_ARG) */

/* Apply the compaction the last decode step decided: the second half of
 * keyformer_update step 3 (page "veloxquant_mlx.quantizers.keyformer module":
 * survivors after the evicted token shift down by one and are re-rotated),
 * which this library defers (the step kernel leaves
 * the evicted row in place and the next step or this call removes it while
 * re-rotating the rows that move). kvevict_read_state calls it itself; a
 * caller that reads the device arena by other means, or that wants a step's
 * work finished in full inside a timed region, calls it explicitly. One
 * kernel launch; a no-op for rows with nothing pending. Errors: CUDA. */
int kvevict_flush(kvevict_t* h, void* stream);

/* Copy one row's state to host memory (synchronises the stream): the keys
 * keyformer_get_kv returns and the KeyformerState fields scores, gumbel and
 * positions (page "veloxquant_mlx.quantizers.keyformer module"; values:
 * kvevict_read_values). Rows
 * are given in slot order: keys [n, D] fp16 bits, scores [n], gumbel [n],
 * positions [n] (the original absolute position of each kept key), n =
 * *n_kept = min(next_pos, budget of layer l). Buffers need room for
 * budget_l + 1 rows; any of the four may be NULL. Errors: INVALID_ARG
 * (indices out of range), CUDA, DEVICE_CHECK. */
int kvevict_read_state(kvevict_t* h, int32_t b, int32_t l, int32_t head, uint16_t* keys,
                       float* scores, float* gumbel, int32_t* positions, int32_t* n_kept,
                       void* stream);

/* Synchronise the stream and report a kernel error word (DEVICE_CHECK) if set.
 * After DEVICE_CHECK the state is not valid; kvevict_reset clears the error
 * word and the state, after which the handle works as a new one. */
int kvevict_check(kvevict_t* h, void* stream);

/* Test hook for the failure path, with no counterpart on the pages. With a
 * handle: in its next decode launch, the first CTA's copy of its first key
 * tile (the resident step: of its row) is never issued, so a wait on it runs
 * out (4 s) and the kernel sets the handle's error word (wait timeout) and
 * returns. With h = NULL: the next
 * launch of the tensor-core prompt scorer in this process (kvevict_prefill of
 * any handle in a cumulative score mode, or kvevict_prefill_scores_noalloc)
 * never issues the query-tile copy of its first work item, with the same
 * outcome: a
 * handle then reports DEVICE_CHECK, the allocation-free call writes NaN
 * scores. Nothing faults or hangs. One-shot. Errors: none. */
int kvevict_test_stall_next_step(kvevict_t* h);

/* Position the next decode key will occupy (= tokens absorbed so far): the
 * KeyformerState.next_pos counter, one value shared by every row (page
 * "veloxquant_mlx.quantizers.keyformer module", KeyformerState and
 * keyformer_update_batched). *p: host int64. Errors: INVALID_ARG (null). */
int kvevict_next_pos(const kvevict_t* h, int64_t* p);

/* Which decode kernel a call of T steps runs on this handle (the choice
 * kvevict_decode / kvevict_step make, see KVEVICT_DECODE_*): *kernel is
 * KVEVICT_DECODE_STREAM or KVEVICT_DECODE_RESIDENT. Host only. Errors:
 * INVALID_ARG (null pointers, T < 0). */
int kvevict_decode_kernel_for(const kvevict_t* h, int32_t T, int32_t* kernel);

/* Budget of layer l as resolved at create time. */
int kvevict_layer_budget(const kvevict_t* h, int32_t l, int32_t* budget);

/* Per-layer cache statistics, host arithmetic only (page "PyramidKV ...":
 * each layer's cache exposes layer_budget, compression_ratio and
 * tokens_kept; page "veloxquant_mlx.quantizers.keyformer module":
 * keyformer_fp16_bytes, full_keyformer_fp16_bytes). For layer l, with p the
 * tokens seen (kvevict_next_pos):
 *   tokens_kept  = min(p, budget_l), the rows each (batch, KV head) row holds;
 *   stored_bytes = B * H * tokens_kept * D * 2 bytes of fp16 keys, doubled
 *                  on a value-carrying handle (scores, Gumbel values and
 *                  positions are bookkeeping, not counted, as on the
 *                  keyformer page);
 *   full_bytes   = the same with p tokens: what keeping every token takes;
 *   compression_ratio = full_bytes / stored_bytes (1 while p = 0).
 * Any output pointer may be NULL. Errors: INVALID_ARG (null handle, layer
 * out of range). */
int kvevict_layer_stats(const kvevict_t* h, int32_t l, int32_t* tokens_kept, uint64_t* stored_bytes,
                        uint64_t* full_bytes, double* compression_ratio);

/* Device bytes held by the handle (arena + scratch + staging). */
int kvevict_device_bytes(const kvevict_t* h, size_t* bytes);

/* Checkpoint and resume. The pages keep the state in an immutable object
 * returned by each call (page "veloxquant_mlx.quantizers.keyformer module",
 * KeyformerState); here it lives in the handle's device arena, and these calls
 * copy it to and from host memory. A snapshot holds every row's keys (and
 * values), scores, Gumbel values and positions, the next position and whether
 * a decode step has run, plus the handle's shape, layer budgets and method
 * parameters (n_sink, recent, score mode, tau schedule, RoPE base, seed); the
 * frozen Gumbel values depend only on (seed, layer, head, position), so a
 * resumed handle continues exactly as the saved one would have.
 *
 * kvevict_state_bytes: size of a snapshot of this handle.
 * kvevict_save_state: applies any pending compaction (as kvevict_flush), then
 *   copies the state into buf (host memory, at least kvevict_state_bytes
 *   bytes, caller-owned); returns after the stream has finished. Errors:
 *   INVALID_ARG (null, buffer too small), CUDA, DEVICE_CHECK (the handle's
 *   error word is set; buf's contents are then unspecified).
 * kvevict_load_state: replaces this handle's state with the snapshot in buf
 *   (host memory, bytes long); returns after the stream has finished, so buf
 *   may be freed. The handle must have the snapshot's batch, layers, KV heads,
 *   head_dim, value rows, layer budgets and method parameters; max_prefill and
 *   prefill_mode may differ. Errors: INVALID_ARG (not a snapshot, a size or
 *   configuration mismatch; the handle is unchanged), CUDA. */
int kvevict_state_bytes(const kvevict_t* h, size_t* bytes);
int kvevict_save_state(kvevict_t* h, void* buf, size_t bytes, void* stream);
int kvevict_load_state(kvevict_t* h, const void* buf, size_t bytes, void* stream);

/* Prompt scoring that allocates nothing. The paper has no counterpart: this is
 * for callers that cannot call cudaMalloc -- an inference engine that reserves
 * the whole device heap for its own memory pool at start-up (a further
 * cudaMalloc then fails or fragments that pool), or a latency-bound serving
 * loop that cannot take cudaMalloc's implicit device-wide synchronisation.
 * It runs the same two tensor-core passes as kvevict_prefill's scorer and
 * writes each row's causal softmax column sums (diagonal included): the
 * scores kvevict_prefill gives a prompt before any eviction.
 *   keys:   device fp16 [heads, S, D], each key RoPE-rotated at its position.
 *   colsum: device float [heads, S], written in full by the call.
 * Working memory is a fixed 16 MiB device array inside the library, present on
 * every GPU that loads the library until the process exits. It limits a call
 * to 2 * heads * round_up(S, 128) <= 4,194,304 floats (for example 512 rows of
 * 4096 tokens); a larger call returns INVALID_ARG without launching anything.
 * Every call shares that array and leaves its contents behind; nothing in it
 * needs to start at zero, since a call reads only entries it wrote itself
 * (padding entries it reads are masked out). Calls whose work overlaps on the
 * GPU (other streams, other threads) race on the array: serialise them.
 * A failure on the GPU cannot reach the return code, which comes back before
 * the GPU runs the call: if one of the scorer's bounded waits runs out (4 s),
 * the call writes NaN to every entry of colsum instead of scores, so a caller
 * that must know checks colsum for NaN after the stream has passed the call.
 * (A device error word beside the array records it. It and the scorer's two
 * work-item counters, also beside the array, are cleared by each call first
 * with cudaMemsetAsync, which allocates nothing.)
 * The first call on each device (and head_dim) looks up the device addresses
 * of the array and the error word, the device's multiprocessor count, and sets
 * the kernels' shared-memory attribute, with that device current; make that
 * first call before any stream capture. The addresses are kept for the life of
 * the process: do not reset the device (cudaDeviceReset) after the first call.
 * With lazy module loading the driver places the array when the library's
 * kernels first load, which can be during that first call. Errors:
 * INVALID_ARG (null pointers, keys not 16-byte aligned, head_dim not 64/128,
 * negative or over-limit sizes), CUDA. */
int kvevict_prefill_scores_noalloc(const uint16_t* keys, int32_t heads, int32_t S,
                                   int32_t head_dim, float* colsum, void* stream);

/* Message of the last failure on the calling thread ("" if none). */
const char* kvevict_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* KVEVICT_H */
