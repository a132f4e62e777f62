// runtime.cu -- the C ABI declared in include/kvevict.h: validation, the
// budget taper, the device arena, launch sequencing (one decode launch per
// call, whatever its step count) and the host-buffer pipeline. Host code only; every step of the
// method runs in the kernels of decode.cu and prefill.cu.
#include "kvevict.h"
#include "kvevict_internal.cuh"

#include <nvtx3/nvToolsExt.h>

#include <atomic>
#include <climits>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <string>
#include <utility>
#include <vector>

using kvx::LayerInfo;

namespace {

thread_local std::string g_last_error;

// An NVTX range around each entry point, named after it, for profilers
// (`ncu --nvtx`, Nsight Systems); without a tool attached it costs a branch.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};
#define KV_RANGE() NvtxRange kv_range_(__func__)

int fail(int code, const std::string& msg) {
  g_last_error = msg;
  return code;
}

#define KV_CUDA(call)                                                                   \
  do {                                                                                  \
    cudaError_t e_ = (call);                                                            \
    if (e_ != cudaSuccess)                                                              \
      return fail(e_ == cudaErrorMemoryAllocation ? KVEVICT_ERR_OOM : KVEVICT_ERR_CUDA, \
                  std::string(#call) + ": " + cudaGetErrorString(e_));                  \
  } while (0)

double round_half_away(double x) {
  const double a = std::fabs(x);
  const double f = std::floor(a);
  const double r = (a - f >= 0.5) ? f + 1.0 : f;
  return x < 0 ? -r : r;
}

int compute_budgets(int32_t L, int32_t avg, int32_t n_sink, double beta, int32_t* out) {
  if (L < 0 || n_sink < 0) return fail(KVEVICT_ERR_INVALID_ARG, "n_layers and n_sink must be >= 0");
  if (!(beta >= 1.0)) return fail(KVEVICT_ERR_INVALID_ARG, "pyramid_beta must be >= 1");
  if (avg < n_sink + 1) return fail(KVEVICT_ERR_INVALID_ARG, "avg_budget must be >= n_sink + 1");
  if (L == 0) return KVEVICT_OK;
  if (L == 1) {
    out[0] = avg;
    return KVEVICT_OK;
  }
  // half-spread: steepness asks for (beta-1)*avg, the n_sink+1 floor caps it
  const double h = std::min((beta - 1.0) * (double)avg, (double)(avg - (n_sink + 1)));
  for (int32_t l = 0; l < L; ++l) {
    const double t = 1.0 - 2.0 * (double)l / (double)(L - 1);
    out[l] = avg + (int32_t)round_half_away(h * t);
  }
  return KVEVICT_OK;
}

// Annealed temperature at absolute position p (fp64, then the kernels' f32).
double tau_at(const kvevict_config& c, int64_t p) {
  if (c.anneal_steps <= 0 || c.tau_init == c.tau_end) return (double)c.tau_init;
  const int64_t t = std::max<int64_t>(0, std::min<int64_t>(p, c.anneal_steps));
  return (double)c.tau_init + (double)t * ((double)c.tau_end - (double)c.tau_init) / (double)c.anneal_steps;
}

template <typename T>
cudaError_t dalloc(T** p, size_t count) {
  *p = nullptr;
  if (count == 0) count = 1;
  return cudaMalloc(reinterpret_cast<void**>(p), count * sizeof(T));
}

}  // namespace

namespace kvx {
void set_last_error(const std::string& msg) { g_last_error = msg; }

namespace {
std::atomic<bool> g_stall_next_scorer{false};   // kvevict_test_stall_next_step(NULL)
}
bool take_scorer_stall() { return g_stall_next_scorer.exchange(false); }
}  // namespace kvx

struct kvevict {
  kvevict_config cfg{};
  int device = 0;
  int D = 0, B = 0, L = 0, H = 0, heads = 0;
  std::vector<int32_t> budgets;
  std::vector<LayerInfo> layers;
  int64_t total_rows = 0, total_meta = 0;
  int capm_max = 0;
  LayerInfo* d_layers = nullptr;
  __half* K = nullptr;
  __half* V = nullptr;      // value rows (with_values handles only)
  float* score = nullptr;
  float* gum = nullptr;
  int32_t* pos = nullptr;
  int32_t* pend = nullptr;
  int* err = nullptr;
  unsigned long long* ticket = nullptr;   // the decode step's (step, row) claim counter
  float* rope_c = nullptr;  // [max_delta + 1, D/2]; row d = f32(cos(-d * w_i))
  float* rope_s = nullptr;
  int max_delta = 1;
  float* lse2 = nullptr;    // prefill scratch [heads, Sp_max]
  int* tc_work = nullptr;   // the prompt scorer's two work-item counters
  float* colsum = nullptr;
  float* gtab = nullptr;    // [L*H, Sp_max] the prompt's Gumbel values
  int64_t Sp_max = 0;
  size_t decode_smem = 0;
  int decode_grid = 0;      // persistent decode CTAs
  size_t resident_smem = 0; // the resident decode step's shared memory
  bool resident_ok = false; // rows fit the resident decode step (key-only handle)
  bool resident_auto = false; // the automatic choice takes the resident step (long enough calls)
  int resident_warps = 8;     // its consumer warps: 8, or 16 where only one CTA fits an SM
  int sms = 0;              // SMs on the device
  int64_t next_pos = 0;
  bool stepped = false;
  size_t bytes = 0;
  unsigned long long* done = nullptr;  // [heads] steps applied << 32 | pending slot + 1
  int64_t dsteps = 0;       // decode steps launched since reset (every row takes each one)
  bool stall_next = false;  // test hook (kvevict_test_stall_next_step)
  // host pipeline staging
  cudaStream_t copy_stream = nullptr;
  cudaEvent_t ev_ready[2] = {nullptr, nullptr};
  cudaEvent_t ev_free[2] = {nullptr, nullptr};
  uint16_t* stage[2] = {nullptr, nullptr};
  int32_t* ev_stage[2] = {nullptr, nullptr};
  size_t stage_elems = 0;
  size_t ev_stage_elems = 0;
};

namespace {

// Shortest call the automatic choice gives the resident decode step (it reads
// and writes each row once per call, the streaming step once per step).
constexpr int kResidentMinSteps = 4;

// The decode kernel a call of T steps runs (kvevict_config.decode_kernel).
bool uses_resident(const kvevict* h, int64_t T) {
  const int kind = h->cfg.decode_kernel;
  return h->resident_ok && kind != KVEVICT_DECODE_STREAM &&
         (kind == KVEVICT_DECODE_RESIDENT || (h->resident_auto && T >= kResidentMinSteps));
}

int64_t BLHD(const kvevict* h) { return (int64_t)h->B * h->L * h->H * h->D; }
int64_t BLH(const kvevict* h) { return (int64_t)h->B * h->L * h->H; }

// T decode steps in one launch. Step t's key (value) of row (b, l, h) is at
// keys + t*k_step + ((b*L + l)*H + h)*k_stride; its evicted slot goes to
// evicted + t*B*L*H + (b*L + l)*H + h. The first step's position is p0.
int enqueue_steps(kvevict* h, const uint16_t* keys, const uint16_t* values, int64_t k_stride, int64_t k_step,
                  int32_t* evicted, int32_t T, int64_t p0, cudaStream_t s) {
  if (T <= 0) return KVEVICT_OK;
  if (h->dsteps + T > INT32_MAX) return fail(KVEVICT_ERR_BAD_STATE, "too many decode steps since reset");
  kvx::DecodeArgs a{};
  a.k_new = reinterpret_cast<const __half*>(keys);
  a.k_stride = k_stride;
  a.k_step = k_step;
  a.v_new = reinterpret_cast<const __half*>(values);
  a.K = h->K;
  a.V = h->V;
  a.score = h->score;
  a.gum = h->gum;
  a.pos = h->pos;
  a.pend = h->pend;
  a.done = h->done;
  a.evicted = evicted;
  a.ev_step = BLH(h);
  a.layers = h->d_layers;
  a.rope_c = h->rope_c + (size_t)(h->D / 2);  // row d = 1: shift by -1
  a.rope_s = h->rope_s + (size_t)(h->D / 2);
  a.err = h->err;
  a.ticket = h->ticket;
  a.rows = h->heads;
  a.T = T;
  a.s0 = (int)h->dsteps;
  a.capm_max = h->capm_max;
  a.B = h->B;
  a.L = h->L;
  a.H = h->H;
  a.n_sink = h->cfg.n_sink;
  a.recent = h->cfg.recent;
  a.mode = h->cfg.score_mode;
  a.p0 = p0;
  a.tau_init = h->cfg.tau_init;
  a.tau_end = h->cfg.tau_end;
  a.anneal_steps = h->cfg.anneal_steps;
  a.scale2 = (float)(1.4426950408889634 / std::sqrt((double)h->D));
  a.seed = h->cfg.seed;
  a.stall = h->stall_next ? 1 : 0;
  h->stall_next = false;
  if (uses_resident(h, T))
    KV_CUDA(kvx::launch_resident_step(a, h->D, h->resident_warps, h->resident_smem, s));
  else
    KV_CUDA(kvx::launch_decode_step(a, h->D, h->decode_grid, h->decode_smem, s));
  h->dsteps += T;
  return KVEVICT_OK;
}

// Score and bulk-evict the prompt for batches [b0, b0 + nb); keys point at
// batch b0's [nb, L, H, S, D] block; lse2/colsum hold nb*L*H rows of Sp.
int enqueue_prompt_scores(kvevict* h, const uint16_t* keys, const uint16_t* values, int32_t S,
                          int32_t S_buf, int b0, int nb, float* lse2, float* colsum, cudaStream_t s) {
  const int heads = nb * h->L * h->H;
  const int Sp = (S + kvx::kPrefillRowPad - 1) / kvx::kPrefillRowPad * kvx::kPrefillRowPad;
  kvx::PrefillScoreArgs sa{};
  sa.keys = reinterpret_cast<const __half*>(keys);
  sa.lse2 = lse2;
  sa.colsum = colsum;
  sa.S = S;
  sa.S_buf = S_buf;
  sa.Sp = Sp;
  sa.heads = heads;
  sa.scale2 = (float)(1.4426950408889634 / std::sqrt((double)h->D));
  sa.err = h->err;
  if (h->cfg.score_mode == KVEVICT_SCORE_CURRENT) {
    KV_CUDA(kvx::launch_prefill_lastrow(sa, h->D, s));
  } else {
    sa.stall = kvx::take_scorer_stall() ? 1 : 0;
    sa.work = h->tc_work;
    KV_CUDA(kvx::launch_prefill_tc(sa, h->D, h->sms, s));
  }
  kvx::PrefillSelectArgs pa{};
  pa.keys = sa.keys;
  pa.values = reinterpret_cast<const __half*>(values);
  pa.V = h->V;
  pa.colsum = colsum;
  pa.gtab = h->gtab;   // filled by enqueue_gumbel_table for this prompt length
  pa.K = h->K;
  pa.score = h->score;
  pa.gum = h->gum;
  pa.pos = h->pos;
  pa.pend = h->pend;
  pa.layers = h->d_layers;
  pa.rope_c = h->rope_c;
  pa.rope_s = h->rope_s;
  pa.err = h->err;
  pa.B = h->B;
  pa.L = h->L;
  pa.H = h->H;
  pa.n_sink = h->cfg.n_sink;
  pa.recent = h->cfg.recent;
  pa.b0 = b0;
  pa.S = S;
  pa.S_buf = S_buf;
  pa.Sp = Sp;
  pa.tau = (float)tau_at(h->cfg, (int64_t)S - 1);
  pa.seed = h->cfg.seed;
  KV_CUDA(kvx::launch_prefill_select(pa, h->D, heads, s));
  return KVEVICT_OK;
}

int enqueue_gumbel_table(kvevict* h, int32_t S, cudaStream_t s) {
  const int Sp = (S + kvx::kPrefillRowPad - 1) / kvx::kPrefillRowPad * kvx::kPrefillRowPad;
  KV_CUDA(kvx::launch_gumbel_table(h->cfg.seed, h->L, h->H, S, Sp, h->gtab, h->sms, s));
  return KVEVICT_OK;
}

// The whole prompt of every row (keys [B, L, H, S, D] on the device). BULK: one
// scoring pass + bulk eviction. SEQUENTIAL: the first S0 = min(S, smallest
// budget) tokens through the scorer (no row can evict before its budget is
// full, so this equals S0 single steps), then one decode step per further
// token with its key read from the prompt buffer (row stride S*D).
int enqueue_prefill(kvevict* h, const uint16_t* keys, const uint16_t* values, int32_t S, int32_t* evicted,
                    cudaStream_t s) {
  int32_t S0 = S;
  if (h->cfg.prefill_mode == KVEVICT_PREFILL_SEQUENTIAL)
    for (int32_t b : h->budgets) S0 = std::min(S0, b);
  int rc = enqueue_gumbel_table(h, S0, s);
  if (rc != KVEVICT_OK) return rc;
  rc = enqueue_prompt_scores(h, keys, values, S0, S, 0, h->B, h->lse2, h->colsum, s);
  if (rc != KVEVICT_OK) return rc;
  if (evicted) KV_CUDA(cudaMemsetAsync(evicted, 0xFF, (size_t)S0 * BLH(h) * 4, s));
  if (S0 < S)
    return enqueue_steps(h, keys + (size_t)S0 * h->D, values ? values + (size_t)S0 * h->D : nullptr,
                         (int64_t)S * h->D, h->D, evicted ? evicted + (size_t)S0 * BLH(h) : nullptr, S - S0, S0, s);
  return KVEVICT_OK;
}

int enqueue_flush(kvevict* h, cudaStream_t s) {
  kvx::FlushArgs f{};
  f.K = h->K;
  f.V = h->V;
  f.score = h->score;
  f.gum = h->gum;
  f.pos = h->pos;
  f.pend = h->pend;
  f.layers = h->d_layers;
  f.rope_c = h->rope_c + (size_t)(h->D / 2);
  f.rope_s = h->rope_s + (size_t)(h->D / 2);
  f.B = h->B;
  f.L = h->L;
  f.H = h->H;
  f.p = h->next_pos;
  KV_CUDA(kvx::launch_flush(f, h->D, h->heads, s));
  return KVEVICT_OK;
}

int check_error_word(kvevict* h, cudaStream_t s) {
  KV_CUDA(cudaStreamSynchronize(s));
  int e = 0;
  KV_CUDA(cudaMemcpy(&e, h->err, sizeof(int), cudaMemcpyDeviceToHost));
  if (e != 0) {
    char buf[96];
    std::snprintf(buf, sizeof buf, "kernel error word set: 0x%x (%s)", e,
                  (e & kvx::kErrWaitTimeout) ? "bounded wait ran out" : "bad index");
    return fail(KVEVICT_ERR_DEVICE_CHECK, buf);
  }
  return KVEVICT_OK;
}

void free_all(kvevict* h) {
  if (h->copy_stream) cudaStreamDestroy(h->copy_stream);
  for (int i = 0; i < 2; ++i) {
    if (h->ev_ready[i]) cudaEventDestroy(h->ev_ready[i]);
    if (h->ev_free[i]) cudaEventDestroy(h->ev_free[i]);
    cudaFree(h->stage[i]);
    cudaFree(h->ev_stage[i]);
  }
  cudaFree(h->d_layers);
  cudaFree(h->K);
  cudaFree(h->V);
  cudaFree(h->score);
  cudaFree(h->gum);
  cudaFree(h->pos);
  cudaFree(h->pend);
  cudaFree(h->done);
  cudaFree(h->err);
  cudaFree(h->ticket);
  cudaFree(h->rope_c);
  cudaFree(h->rope_s);
  cudaFree(h->lse2);
  cudaFree(h->tc_work);
  cudaFree(h->colsum);
  cudaFree(h->gtab);
}

}  // namespace

extern "C" {

const char* kvevict_last_error(void) { return g_last_error.c_str(); }

int kvevict_budgets(int32_t n_layers, int32_t avg_budget, int32_t n_sink, double beta, int32_t* out) {
  if (n_layers > 0 && !out) return fail(KVEVICT_ERR_INVALID_ARG, "out is null");
  return compute_budgets(n_layers, avg_budget, n_sink, beta, out);
}

int kvevict_create(const kvevict_config* cfg, void* stream, kvevict_t** out) {
  KV_RANGE();
  g_last_error.clear();
  if (!cfg || !out) return fail(KVEVICT_ERR_INVALID_ARG, "cfg and out must not be null");
  const kvevict_config& c = *cfg;
  if (c.batch < 1 || c.n_kv_heads < 1) return fail(KVEVICT_ERR_INVALID_ARG, "batch and n_kv_heads must be >= 1");
  if (c.n_layers < 1 || c.n_layers > KVEVICT_MAX_LAYERS)
    return fail(KVEVICT_ERR_INVALID_ARG, "n_layers must be in [1, KVEVICT_MAX_LAYERS]");
  if (c.head_dim != 64 && c.head_dim != 128) return fail(KVEVICT_ERR_INVALID_ARG, "head_dim must be 64 or 128");
  if (c.n_sink < 0) return fail(KVEVICT_ERR_INVALID_ARG, "n_sink must be >= 0");
  if (!(c.tau_init >= 0.f) || !(c.tau_end >= 0.f))
    return fail(KVEVICT_ERR_INVALID_ARG, "tau_init and tau_end must be >= 0");
  if (c.anneal_steps < 0) return fail(KVEVICT_ERR_INVALID_ARG, "anneal_steps must be >= 0");
  if (!(c.rope_theta > 0.0)) return fail(KVEVICT_ERR_INVALID_ARG, "rope_theta must be > 0");
  if (c.max_prefill < 0 || c.max_prefill > KVEVICT_MAX_PREFILL)
    return fail(KVEVICT_ERR_INVALID_ARG, "max_prefill must be in [0, KVEVICT_MAX_PREFILL]");
  if (c.recent < 0) return fail(KVEVICT_ERR_INVALID_ARG, "recent must be >= 0");
  if (c.with_values != 0 && c.with_values != 1) return fail(KVEVICT_ERR_INVALID_ARG, "with_values must be 0 or 1");
  if (c.prefill_mode != KVEVICT_PREFILL_BULK && c.prefill_mode != KVEVICT_PREFILL_SEQUENTIAL)
    return fail(KVEVICT_ERR_INVALID_ARG, "prefill_mode must be KVEVICT_PREFILL_BULK or KVEVICT_PREFILL_SEQUENTIAL");
  if (c.score_mode != KVEVICT_SCORE_CUMULATIVE && c.score_mode != KVEVICT_SCORE_CURRENT)
    return fail(KVEVICT_ERR_INVALID_ARG, "score_mode must be KVEVICT_SCORE_CUMULATIVE or KVEVICT_SCORE_CURRENT");
  if (c.decode_kernel != KVEVICT_DECODE_AUTO && c.decode_kernel != KVEVICT_DECODE_STREAM &&
      c.decode_kernel != KVEVICT_DECODE_RESIDENT)
    return fail(KVEVICT_ERR_INVALID_ARG, "decode_kernel must be KVEVICT_DECODE_AUTO, _STREAM or _RESIDENT");

  std::vector<int32_t> budgets(c.n_layers);
  if (c.layer_budgets) {
    for (int l = 0; l < c.n_layers; ++l) budgets[l] = c.layer_budgets[l];
  } else {
    const int rc = compute_budgets(c.n_layers, c.avg_budget, c.n_sink, c.pyramid_beta, budgets.data());
    if (rc != KVEVICT_OK) return rc;
  }
  for (int l = 0; l < c.n_layers; ++l)
    if (budgets[l] < c.n_sink + c.recent + 1)
      return fail(KVEVICT_ERR_INVALID_ARG,
                  "every layer budget must be >= n_sink + recent + 1 (room to evict)");

  kvevict* h = new kvevict();
  h->cfg = c;
  h->cfg.layer_budgets = nullptr;
  h->D = c.head_dim;
  h->B = c.batch;
  h->L = c.n_layers;
  h->H = c.n_kv_heads;
  h->heads = c.batch * c.n_layers * c.n_kv_heads;
  h->budgets = budgets;
  h->layers.resize(c.n_layers);
  int64_t rows = 0, meta = 0;
  for (int l = 0; l < c.n_layers; ++l) {
    LayerInfo& li = h->layers[l];
    li.budget = budgets[l];
    li.cap = budgets[l] + 1;
    li.capm = (li.cap + 3) & ~3;
    li.pad = 0;
    li.row_base = rows;
    li.meta_base = meta;
    rows += (int64_t)h->B * h->H * li.cap;
    meta += (int64_t)h->B * h->H * li.capm;
    h->capm_max = std::max(h->capm_max, li.capm);
  }
  h->total_rows = rows;
  h->total_meta = meta;
  h->decode_smem = kvx::decode_step_smem(h->D, h->capm_max);
  if (h->decode_smem > 227 * 1024) {
    delete h;
    return fail(KVEVICT_ERR_INVALID_ARG, "layer budget too large for the single-CTA decode step");
  }
  h->max_delta = std::max(1, c.max_prefill);
  h->Sp_max = (int64_t)(c.max_prefill + kvx::kPrefillRowPad - 1) / kvx::kPrefillRowPad * kvx::kPrefillRowPad;

  auto bail = [&](int code) {
    free_all(h);
    delete h;
    return code;
  };
#define KV_CUDA_CREATE(call)                                                                   \
  do {                                                                                         \
    cudaError_t e_ = (call);                                                                   \
    if (e_ != cudaSuccess)                                                                     \
      return bail(fail(e_ == cudaErrorMemoryAllocation ? KVEVICT_ERR_OOM : KVEVICT_ERR_CUDA,   \
                       std::string(#call) + ": " + cudaGetErrorString(e_)));                   \
  } while (0)

  cudaStream_t s = (cudaStream_t)stream;
  KV_CUDA_CREATE(cudaGetDevice(&h->device));
  {
    // opt-in shared memory per block on this device, less what the kernels
    // declare statically
    int optin = 0;
    KV_CUDA_CREATE(cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, h->device));
    if (h->decode_smem + 1024 > (size_t)optin ||
        kvx::prefill_select_smem(std::max(1, c.max_prefill)) + 1024 > (size_t)optin ||
        kvx::prefill_tc_smem(h->D) + 1024 > (size_t)optin)
      return bail(fail(KVEVICT_ERR_INVALID_ARG, "layer budget or max_prefill too large for shared memory"));
    h->resident_smem = kvx::resident_step_smem(h->D, h->capm_max);
    h->resident_ok = !c.with_values && h->resident_smem != (size_t)-1 && h->resident_smem + 1024 <= (size_t)optin;
    if (c.decode_kernel == KVEVICT_DECODE_RESIDENT && !h->resident_ok)
      return bail(fail(KVEVICT_ERR_INVALID_ARG,
                       "the resident decode kernel needs a key-only handle whose rows fit in shared memory"));
  }
  KV_CUDA_CREATE(kvx::decode_step_setup(h->D, h->decode_smem));
  if (h->resident_ok) {
    // The resident step runs one CTA per row, in waves when the rows outnumber
    // the CTAs that fit; each wave runs every step. Measured on GB300 it beats
    // the streaming step when the rows fit in one wave, or in two waves at two
    // or more CTAs an SM (keys up to about 400 rows of head_dim 128). Where a
    // row's shared memory leaves room for one CTA an SM, it runs 16 consumer
    // warps instead of 8.
    int per8 = 0, per16 = 0, sms = 0;
    KV_CUDA_CREATE(kvx::resident_step_setup(h->D, h->resident_smem, &per8, &per16));
    KV_CUDA_CREATE(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, h->device));
    h->resident_warps = (per8 < 2 && per16 >= 1) ? 16 : 8;
    const int per_sm = h->resident_warps == 16 ? per16 : per8;
    const int64_t slots = (int64_t)per_sm * sms;
    const int64_t waves = slots > 0 ? (h->heads + slots - 1) / slots : INT64_MAX;
    h->resident_auto = per_sm > 0 && (waves <= 1 || (waves <= 2 && per_sm >= 2));
    if (per_sm < 1) h->resident_ok = false;
    if (c.decode_kernel == KVEVICT_DECODE_RESIDENT && !h->resident_ok)
      return bail(fail(KVEVICT_ERR_INVALID_ARG, "the resident decode kernel does not fit on an SM"));
  }
  {
    int per_sm = 0, sms = 0;
    KV_CUDA_CREATE(kvx::decode_step_ctas_per_sm(h->D, h->decode_smem, &per_sm));
    KV_CUDA_CREATE(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, h->device));
    if (per_sm < 1) return bail(fail(KVEVICT_ERR_INVALID_ARG, "decode step does not fit on an SM"));
    h->decode_grid = (int)std::min<int64_t>((int64_t)per_sm * sms, h->heads);
    h->sms = sms;
  }
  KV_CUDA_CREATE(kvx::prefill_setup(h->D, c.max_prefill));
  KV_CUDA_CREATE(kvx::prefill_tc_setup(h->D));
  KV_CUDA_CREATE(dalloc(&h->d_layers, (size_t)c.n_layers));
  KV_CUDA_CREATE(dalloc(&h->K, (size_t)rows * h->D));
  if (c.with_values) KV_CUDA_CREATE(dalloc(&h->V, (size_t)rows * h->D));
  KV_CUDA_CREATE(dalloc(&h->score, (size_t)meta));
  KV_CUDA_CREATE(dalloc(&h->gum, (size_t)meta));
  KV_CUDA_CREATE(dalloc(&h->pos, (size_t)meta));
  KV_CUDA_CREATE(dalloc(&h->pend, (size_t)h->heads));
  KV_CUDA_CREATE(dalloc(&h->done, (size_t)h->heads));
  KV_CUDA_CREATE(dalloc(&h->err, 1));
  KV_CUDA_CREATE(dalloc(&h->ticket, 1));
  const size_t half = (size_t)h->D / 2;
  KV_CUDA_CREATE(dalloc(&h->rope_c, (size_t)(h->max_delta + 1) * half));
  KV_CUDA_CREATE(dalloc(&h->rope_s, (size_t)(h->max_delta + 1) * half));
  if (c.max_prefill > 0) {
    KV_CUDA_CREATE(dalloc(&h->lse2, (size_t)h->heads * h->Sp_max));
    KV_CUDA_CREATE(dalloc(&h->tc_work, 2));
    KV_CUDA_CREATE(dalloc(&h->colsum, (size_t)h->heads * h->Sp_max));
    KV_CUDA_CREATE(dalloc(&h->gtab, (size_t)h->L * h->H * h->Sp_max));
  }
  h->bytes = (size_t)rows * h->D * 2 * (c.with_values ? 2 : 1) + (size_t)meta * 12 + (size_t)h->heads * 4 +
             2 * (size_t)(h->max_delta + 1) * half * 4 + 2 * (size_t)h->heads * h->Sp_max * 4 + (size_t)h->L * h->H * h->Sp_max * 4;

  // RoPE constants for a shift back by d positions: c = f32(cos(-d w_i)),
  // s = f32(sin(-d w_i)), w_i = theta^(-2i/D), taken in fp64.
  std::vector<float> hc((size_t)(h->max_delta + 1) * half), hs(hc.size());
  for (int d = 0; d <= h->max_delta; ++d)
    for (size_t i = 0; i < half; ++i) {
      const double w = std::pow(c.rope_theta, -(2.0 * (double)i) / (double)h->D);
      const double ang = (double)(-d) * w;
      hc[(size_t)d * half + i] = (float)std::cos(ang);
      hs[(size_t)d * half + i] = (float)std::sin(ang);
    }
  KV_CUDA_CREATE(cudaMemcpy(h->rope_c, hc.data(), hc.size() * 4, cudaMemcpyHostToDevice));
  KV_CUDA_CREATE(cudaMemcpy(h->rope_s, hs.data(), hs.size() * 4, cudaMemcpyHostToDevice));
  KV_CUDA_CREATE(cudaMemcpy(h->d_layers, h->layers.data(), h->layers.size() * sizeof(LayerInfo),
                            cudaMemcpyHostToDevice));
  KV_CUDA_CREATE(cudaMemsetAsync(h->pend, 0xFF, (size_t)h->heads * 4, s));
  KV_CUDA_CREATE(cudaMemsetAsync(h->done, 0, (size_t)h->heads * 8, s));
  KV_CUDA_CREATE(cudaMemsetAsync(h->err, 0, sizeof(int), s));
  KV_CUDA_CREATE(cudaMemsetAsync(h->ticket, 0, sizeof(unsigned long long), s));
  KV_CUDA_CREATE(cudaStreamSynchronize(s));
#undef KV_CUDA_CREATE
  *out = h;
  return KVEVICT_OK;
}

int kvevict_destroy(kvevict_t* h) {
  KV_RANGE();
  if (!h) return KVEVICT_OK;
  cudaDeviceSynchronize();
  free_all(h);
  delete h;
  return KVEVICT_OK;
}

int kvevict_reset(kvevict_t* h, void* stream) {
  KV_RANGE();
  if (!h) return fail(KVEVICT_ERR_INVALID_ARG, "null handle");
  cudaStream_t s = (cudaStream_t)stream;
  KV_CUDA(cudaMemsetAsync(h->pend, 0xFF, (size_t)h->heads * 4, s));
  KV_CUDA(cudaMemsetAsync(h->done, 0, (size_t)h->heads * 8, s));
  KV_CUDA(cudaMemsetAsync(h->err, 0, sizeof(int), s));
  KV_CUDA(cudaMemsetAsync(h->ticket, 0, sizeof(unsigned long long), s));   // left set by an aborted launch
  h->next_pos = 0;
  h->dsteps = 0;
  h->stepped = false;
  return KVEVICT_OK;
}

}  // extern "C"

namespace {

// Device key and value buffers start on a 16-byte boundary (the prompt scorer
// reads them with TMA, the decode step with 4- or 8-byte words).
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

int prefill_impl(kvevict* h, const uint16_t* keys, const uint16_t* values, int32_t S, int32_t* evicted,
                 void* stream) {
  if (S < 0 || S > h->cfg.max_prefill) return fail(KVEVICT_ERR_INVALID_ARG, "S must be in [0, max_prefill]");
  if (S > 0 && (!keys || (h->V && !values))) return fail(KVEVICT_ERR_INVALID_ARG, "keys or values is null");
  if (S > 0 && (!aligned16(keys) || !aligned16(values)))
    return fail(KVEVICT_ERR_INVALID_ARG, "keys and values must be 16-byte aligned");
  if (h->next_pos != 0 || h->stepped) return fail(KVEVICT_ERR_BAD_STATE, "prefill needs an empty state");
  if (S == 0) return KVEVICT_OK;
  const int rc = enqueue_prefill(h, keys, values, S, evicted, (cudaStream_t)stream);
  if (rc != KVEVICT_OK) return rc;
  h->next_pos = S;
  return KVEVICT_OK;
}

int step_impl(kvevict* h, const uint16_t* k_new, const uint16_t* v_new, int32_t* evicted, void* stream) {
  if (!k_new || (h->V && !v_new)) return fail(KVEVICT_ERR_INVALID_ARG, "k_new or v_new is null");
  if (!aligned16(k_new) || !aligned16(v_new))
    return fail(KVEVICT_ERR_INVALID_ARG, "k_new and v_new must be 16-byte aligned");
  const int rc = enqueue_steps(h, k_new, v_new, h->D, 0, evicted, 1, h->next_pos, (cudaStream_t)stream);
  if (rc != KVEVICT_OK) return rc;
  h->next_pos += 1;
  h->stepped = true;
  return KVEVICT_OK;
}

int decode_impl(kvevict* h, const uint16_t* keys, const uint16_t* values, int32_t T, int32_t* evicted,
                void* stream) {
  if (T < 0) return fail(KVEVICT_ERR_INVALID_ARG, "T must be >= 0");
  if (T == 0) return KVEVICT_OK;
  if (!keys || (h->V && !values)) return fail(KVEVICT_ERR_INVALID_ARG, "keys or values is null");
  if (!aligned16(keys) || !aligned16(values))
    return fail(KVEVICT_ERR_INVALID_ARG, "keys and values must be 16-byte aligned");
  const int rc = enqueue_steps(h, keys, values, h->D, BLHD(h), evicted, T, h->next_pos, (cudaStream_t)stream);
  if (rc != KVEVICT_OK) return rc;
  h->next_pos += T;
  h->stepped = true;
  return KVEVICT_OK;
}

int keys_only(const kvevict* h) {
  return h->V ? fail(KVEVICT_ERR_INVALID_ARG, "this handle carries values: use the _kv entry points")
              : KVEVICT_OK;
}
int with_values(const kvevict* h) {
  return h->V ? KVEVICT_OK : fail(KVEVICT_ERR_INVALID_ARG, "this handle was created without values");
}

}  // namespace

extern "C" {

int kvevict_prefill_ex(kvevict_t* h, const uint16_t* keys, int32_t S, int32_t* evicted, void* stream) {
  KV_RANGE();
  if (!h) return fail(KVEVICT_ERR_INVALID_ARG, "null handle");
  if (int rc = keys_only(h)) return rc;
  return prefill_impl(h, keys, nullptr, S, evicted, stream);
}

int kvevict_prefill(kvevict_t* h, const uint16_t* keys, int32_t S, void* stream) {
  KV_RANGE();
  return kvevict_prefill_ex(h, keys, S, nullptr, stream);
}

int kvevict_prefill_kv(kvevict_t* h, const uint16_t* keys, const uint16_t* values, int32_t S,
                       int32_t* evicted, void* stream) {
  KV_RANGE();
  if (!h) return fail(KVEVICT_ERR_INVALID_ARG, "null handle");
  if (int rc = with_values(h)) return rc;
  return prefill_impl(h, keys, values, S, evicted, stream);
}

int kvevict_step(kvevict_t* h, const uint16_t* k_new, int32_t* evicted, void* stream) {
  KV_RANGE();
  if (!h) return fail(KVEVICT_ERR_INVALID_ARG, "null handle");
  if (int rc = keys_only(h)) return rc;
  return step_impl(h, k_new, nullptr, evicted, stream);
}

int kvevict_step_kv(kvevict_t* h, const uint16_t* k_new, const uint16_t* v_new, int32_t* evicted,
                    void* stream) {
  KV_RANGE();
  if (!h) return fail(KVEVICT_ERR_INVALID_ARG, "null handle");
  if (int rc = with_values(h)) return rc;
  return step_impl(h, k_new, v_new, evicted, stream);
}

int kvevict_decode(kvevict_t* h, const uint16_t* keys, int32_t T, int32_t* evicted, void* stream) {
  KV_RANGE();
  if (!h) return fail(KVEVICT_ERR_INVALID_ARG, "null handle");
  if (int rc = keys_only(h)) return rc;
  return decode_impl(h, keys, nullptr, T, evicted, stream);
}

int kvevict_decode_kv(kvevict_t* h, const uint16_t* keys, const uint16_t* values, int32_t T,
                      int32_t* evicted, void* stream) {
  KV_RANGE();
  if (!h) return fail(KVEVICT_ERR_INVALID_ARG, "null handle");
  if (int rc = with_values(h)) return rc;
  return decode_impl(h, keys, values, T, evicted, stream);
}

int kvevict_run_host(kvevict_t* h, const uint16_t* prefill_keys, int32_t S, const uint16_t* decode_keys,
                     int32_t T, int32_t* evicted, void* stream) {
  KV_RANGE();
  if (!h) return fail(KVEVICT_ERR_INVALID_ARG, "null handle");
  if (S < 0 || S > h->cfg.max_prefill || T < 0) return fail(KVEVICT_ERR_INVALID_ARG, "bad S or T");
  if ((S > 0 && !prefill_keys) || (T > 0 && !decode_keys)) return fail(KVEVICT_ERR_INVALID_ARG, "null keys");
  if (h->next_pos != 0 || h->stepped) return fail(KVEVICT_ERR_BAD_STATE, "run_host needs an empty state");
  if (int rc = keys_only(h)) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  const size_t per_batch = (size_t)h->L * h->H * (size_t)S * h->D;
  const size_t per_step = (size_t)BLHD(h);
  // Page-locked buffers are moved by the library's kernels through their
  // device mapping: the prompt is staged chunk by chunk by a copy kernel on the
  // copy stream (small enough to run beside the scorer), the decode keys are
  // read in place by the decode step, and the evicted slots go back by the same
  // copy kernel. Other host memory is staged with cudaMemcpyAsync on the copy
  // stream, overlapping compute.
  const void* pre_map = S > 0 ? kvx::mapped_host(prefill_keys, (size_t)h->B * per_batch * 2) : nullptr;
  const void* dec_map = T > 0 ? kvx::mapped_host(decode_keys, (size_t)T * per_step * 2) : nullptr;
  const bool dec_inplace = dec_map && aligned16(dec_map);   // else staged by the copy kernel
  void* ev_map = (evicted && T > 0) ? kvx::mapped_host(evicted, (size_t)T * BLH(h) * 4) : nullptr;
  // Staging: two buffers of up to 256 MiB (or one batch's prompt / one step,
  // whichever is larger), so copies of chunk k+1 overlap compute on chunk k.
  const size_t budget_elems = (size_t)128 << 20;  // 256 MiB of fp16
  const bool seq = h->cfg.prefill_mode == KVEVICT_PREFILL_SEQUENTIAL;
  const int bc = S <= 0 ? 0
                 : seq ? h->B   // sequential steps run over every row: stage the whole prompt
                       : (int)std::max<size_t>(1, std::min<size_t>(h->B, budget_elems / std::max<size_t>(per_batch, 1)));
  // decode chunk: bounded by the key staging, or, with the keys read in place,
  // only by the evicted-slot staging (256 MiB of int32), so one launch usually
  // runs every step
  const size_t ev_budget = (size_t)64 << 20;
  const size_t tc_cap = dec_inplace ? ev_budget / std::max<size_t>((size_t)BLH(h), 1) : budget_elems / per_step;
  const int tc = T > 0 ? (int)std::max<size_t>(1, std::min<size_t>((size_t)T, tc_cap)) : 0;
  const size_t need = std::max((size_t)bc * per_batch, dec_inplace ? (size_t)0 : (size_t)tc * per_step);
  if (!h->copy_stream) {
    KV_CUDA(cudaStreamCreateWithFlags(&h->copy_stream, cudaStreamNonBlocking));
    for (int i = 0; i < 2; ++i) {
      KV_CUDA(cudaEventCreateWithFlags(&h->ev_ready[i], cudaEventDisableTiming));
      KV_CUDA(cudaEventCreateWithFlags(&h->ev_free[i], cudaEventDisableTiming));
    }
  }
  if (need > h->stage_elems) {
    KV_CUDA(cudaStreamSynchronize(s));
    for (int i = 0; i < 2; ++i) {
      cudaFree(h->stage[i]);
      h->stage[i] = nullptr;
      KV_CUDA(dalloc(&h->stage[i], need));
    }
    h->stage_elems = need;
  }
  const size_t ev_need = (size_t)tc * BLH(h);
  if (evicted && ev_need > h->ev_stage_elems) {
    for (int i = 0; i < 2; ++i) {
      cudaFree(h->ev_stage[i]);
      h->ev_stage[i] = nullptr;
      KV_CUDA(dalloc(&h->ev_stage[i], ev_need));
    }
    h->ev_stage_elems = ev_need;
  }
  // one chunk of input into staging buffer buf on the copy stream, ordered
  // after the last work on that buffer and before the next work on s
  auto stage_in = [&](int buf, const void* host, const void* mapped, size_t off, size_t bytes) -> int {
    KV_CUDA(cudaStreamWaitEvent(h->copy_stream, h->ev_free[buf], 0));
    if (mapped)
      KV_CUDA(kvx::launch_copy(static_cast<const char*>(mapped) + off, h->stage[buf], bytes, h->sms, true,
                               h->copy_stream));
    else
      KV_CUDA(cudaMemcpyAsync(h->stage[buf], static_cast<const char*>(host) + off, bytes, cudaMemcpyHostToDevice,
                              h->copy_stream));
    KV_CUDA(cudaEventRecord(h->ev_ready[buf], h->copy_stream));
    KV_CUDA(cudaStreamWaitEvent(s, h->ev_ready[buf], 0));
    return KVEVICT_OK;
  };
  int k = 0;
  if (S > 0 && !seq) {
    const int rc = enqueue_gumbel_table(h, S, s);
    if (rc != KVEVICT_OK) return rc;
  }
  // prompt, batch chunk by batch chunk
  for (int b0 = 0; b0 < (S > 0 ? h->B : 0); b0 += bc, ++k) {
    const int nb = std::min(bc, h->B - b0);
    const int buf = k & 1;
    int rc = stage_in(buf, prefill_keys, pre_map, (size_t)b0 * per_batch * 2, (size_t)nb * per_batch * 2);
    if (rc != KVEVICT_OK) return rc;
    rc = seq ? enqueue_prefill(h, h->stage[buf], nullptr, S, nullptr, s)
             : enqueue_prompt_scores(h, h->stage[buf], nullptr, S, S, b0, nb, h->lse2, h->colsum, s);
    if (rc != KVEVICT_OK) return rc;
    KV_CUDA(cudaEventRecord(h->ev_free[buf], s));
  }
  h->next_pos = S;
  // decode, step chunk by step chunk
  for (int t0 = 0; t0 < T; t0 += tc, ++k) {
    const int nt = std::min(tc, T - t0);
    const int buf = k & 1;
    const uint16_t* keys =
        dec_inplace ? static_cast<const uint16_t*>(dec_map) + (size_t)t0 * per_step : h->stage[buf];
    if (!dec_inplace) {
      const int rc = stage_in(buf, decode_keys, dec_map, (size_t)t0 * per_step * 2, (size_t)nt * per_step * 2);
      if (rc != KVEVICT_OK) return rc;
    }
    const int rc = enqueue_steps(h, keys, nullptr, h->D, (int64_t)per_step, evicted ? h->ev_stage[buf] : nullptr,
                                 nt, h->next_pos, s);
    if (rc != KVEVICT_OK) return rc;
    h->next_pos += nt;
    h->stepped = true;
    if (evicted) {
      const size_t off = (size_t)t0 * BLH(h), bytes = (size_t)nt * BLH(h) * 4;
      if (ev_map)
        KV_CUDA(kvx::launch_copy(h->ev_stage[buf], static_cast<int32_t*>(ev_map) + off, bytes, h->sms, false, s));
      else
        KV_CUDA(cudaMemcpyAsync(evicted + off, h->ev_stage[buf], bytes, cudaMemcpyDeviceToHost, s));
    }
    KV_CUDA(cudaEventRecord(h->ev_free[buf], s));
  }
  return check_error_word(h, s);
}

int kvevict_read_state(kvevict_t* h, int32_t b, int32_t l, int32_t head, uint16_t* keys, float* scores,
                       float* gumbel, int32_t* positions, int32_t* n_kept, void* stream) {
  KV_RANGE();
  if (!h) return fail(KVEVICT_ERR_INVALID_ARG, "null handle");
  if (b < 0 || b >= h->B || l < 0 || l >= h->L || head < 0 || head >= h->H)
    return fail(KVEVICT_ERR_INVALID_ARG, "row index out of range");
  cudaStream_t s = (cudaStream_t)stream;
  int rc = enqueue_flush(h, s);
  if (rc != KVEVICT_OK) return rc;
  const LayerInfo& li = h->layers[l];
  const int n = (int)std::min<int64_t>(h->next_pos, li.budget);
  const int64_t rem = (int64_t)b * h->H + head;
  if (keys && n > 0)
    KV_CUDA(cudaMemcpyAsync(keys, h->K + (li.row_base + rem * li.cap) * h->D, (size_t)n * h->D * 2,
                            cudaMemcpyDeviceToHost, s));
  const int64_t mo = li.meta_base + rem * li.capm;
  if (scores && n > 0) KV_CUDA(cudaMemcpyAsync(scores, h->score + mo, (size_t)n * 4, cudaMemcpyDeviceToHost, s));
  if (gumbel && n > 0) KV_CUDA(cudaMemcpyAsync(gumbel, h->gum + mo, (size_t)n * 4, cudaMemcpyDeviceToHost, s));
  if (positions && n > 0)
    KV_CUDA(cudaMemcpyAsync(positions, h->pos + mo, (size_t)n * 4, cudaMemcpyDeviceToHost, s));
  rc = check_error_word(h, s);
  if (n_kept) *n_kept = n;
  return rc;
}

int kvevict_test_stall_next_step(kvevict_t* h) {
  if (!h) {
    kvx::g_stall_next_scorer.store(true);
    return KVEVICT_OK;
  }
  h->stall_next = true;
  return KVEVICT_OK;
}

int kvevict_flush(kvevict_t* h, void* stream) {
  KV_RANGE();
  if (!h) return fail(KVEVICT_ERR_INVALID_ARG, "null handle");
  return enqueue_flush(h, (cudaStream_t)stream);
}

int kvevict_read_values(kvevict_t* h, int32_t b, int32_t l, int32_t head, uint16_t* values,
                        int32_t* n_kept, void* stream) {
  KV_RANGE();
  if (!h) return fail(KVEVICT_ERR_INVALID_ARG, "null handle");
  if (int rc = with_values(h)) return rc;
  if (b < 0 || b >= h->B || l < 0 || l >= h->L || head < 0 || head >= h->H)
    return fail(KVEVICT_ERR_INVALID_ARG, "row index out of range");
  cudaStream_t s = (cudaStream_t)stream;
  int rc = enqueue_flush(h, s);
  if (rc != KVEVICT_OK) return rc;
  const LayerInfo& li = h->layers[l];
  const int n = (int)std::min<int64_t>(h->next_pos, li.budget);
  const int64_t rem = (int64_t)b * h->H + head;
  if (values && n > 0)
    KV_CUDA(cudaMemcpyAsync(values, h->V + (li.row_base + rem * li.cap) * h->D, (size_t)n * h->D * 2,
                            cudaMemcpyDeviceToHost, s));
  rc = check_error_word(h, s);
  if (n_kept) *n_kept = n;
  return rc;
}

int kvevict_check(kvevict_t* h, void* stream) {
  KV_RANGE();
  if (!h) return fail(KVEVICT_ERR_INVALID_ARG, "null handle");
  return check_error_word(h, (cudaStream_t)stream);
}

int kvevict_decode_kernel_for(const kvevict_t* h, int32_t T, int32_t* kernel) {
  if (!h || !kernel) return fail(KVEVICT_ERR_INVALID_ARG, "null argument");
  if (T < 0) return fail(KVEVICT_ERR_INVALID_ARG, "T must be >= 0");
  *kernel = uses_resident(h, T) ? KVEVICT_DECODE_RESIDENT : KVEVICT_DECODE_STREAM;
  return KVEVICT_OK;
}

int kvevict_next_pos(const kvevict_t* h, int64_t* p) {
  if (!h || !p) return fail(KVEVICT_ERR_INVALID_ARG, "null argument");
  *p = h->next_pos;
  return KVEVICT_OK;
}

int kvevict_layer_budget(const kvevict_t* h, int32_t l, int32_t* budget) {
  if (!h || !budget) return fail(KVEVICT_ERR_INVALID_ARG, "null argument");
  if (l < 0 || l >= h->L) return fail(KVEVICT_ERR_INVALID_ARG, "layer out of range");
  *budget = h->budgets[l];
  return KVEVICT_OK;
}

int kvevict_layer_stats(const kvevict_t* h, int32_t l, int32_t* tokens_kept, uint64_t* stored_bytes,
                        uint64_t* full_bytes, double* compression_ratio) {
  if (!h) return fail(KVEVICT_ERR_INVALID_ARG, "null handle");
  if (l < 0 || l >= h->L) return fail(KVEVICT_ERR_INVALID_ARG, "layer out of range");
  const int64_t p = h->next_pos;
  const int64_t kept = std::min<int64_t>(p, h->budgets[l]);
  const uint64_t per_token = (uint64_t)h->B * h->H * h->D * 2 * (h->V ? 2 : 1);
  if (tokens_kept) *tokens_kept = (int32_t)kept;
  if (stored_bytes) *stored_bytes = per_token * (uint64_t)kept;
  if (full_bytes) *full_bytes = per_token * (uint64_t)p;
  if (compression_ratio) *compression_ratio = kept > 0 ? (double)p / (double)kept : 1.0;
  return KVEVICT_OK;
}

int kvevict_device_bytes(const kvevict_t* h, size_t* bytes) {
  if (!h || !bytes) return fail(KVEVICT_ERR_INVALID_ARG, "null argument");
  *bytes = h->bytes + 2 * h->stage_elems * 2 + 2 * h->ev_stage_elems * 4;
  return KVEVICT_OK;
}

}  // extern "C"

namespace {

// ---------------------------------------------------------------- snapshots
// A snapshot is this header, the layer budgets, then the key arena, the value
// arena (value-carrying handles), scores, Gumbel values and positions, each
// array whole (kept rows and unused tail alike), in host byte order. It is
// taken after a flush, so no compaction is pending in it.
struct SnapHeader {
  char magic[8];            // "KVEVSNP1"
  uint32_t version;         // 1
  uint32_t header_bytes;    // sizeof(SnapHeader)
  int32_t batch, n_layers, n_kv_heads, head_dim, with_values, n_sink, recent, score_mode;
  int32_t anneal_steps, stepped;
  float tau_init, tau_end;
  double rope_theta;
  uint64_t seed;
  int64_t next_pos;
  int64_t total_rows, total_meta;
  uint64_t payload_bytes;   // everything after the header
};
constexpr char kSnapMagic[8] = {'K', 'V', 'E', 'V', 'S', 'N', 'P', '1'};

size_t snap_payload(const kvevict* h) {
  const size_t keys = (size_t)h->total_rows * h->D * 2;
  return (size_t)h->L * 4 + keys * (h->V ? 2 : 1) + (size_t)h->total_meta * 4 * 3;
}

SnapHeader snap_header(const kvevict* h) {
  SnapHeader sh{};
  std::memcpy(sh.magic, kSnapMagic, 8);
  sh.version = 1;
  sh.header_bytes = sizeof(SnapHeader);
  sh.batch = h->B;
  sh.n_layers = h->L;
  sh.n_kv_heads = h->H;
  sh.head_dim = h->D;
  sh.with_values = h->V ? 1 : 0;
  sh.n_sink = h->cfg.n_sink;
  sh.recent = h->cfg.recent;
  sh.score_mode = h->cfg.score_mode;
  sh.anneal_steps = h->cfg.anneal_steps;
  sh.stepped = h->stepped ? 1 : 0;
  sh.tau_init = h->cfg.tau_init;
  sh.tau_end = h->cfg.tau_end;
  sh.rope_theta = h->cfg.rope_theta;
  sh.seed = h->cfg.seed;
  sh.next_pos = h->next_pos;
  sh.total_rows = h->total_rows;
  sh.total_meta = h->total_meta;
  sh.payload_bytes = snap_payload(h);
  return sh;
}

// The device arrays of a snapshot in file order: (device pointer, bytes).
std::vector<std::pair<void*, size_t>> snap_arrays(kvevict* h) {
  std::vector<std::pair<void*, size_t>> v;
  const size_t keys = (size_t)h->total_rows * h->D * 2, meta = (size_t)h->total_meta * 4;
  v.emplace_back(h->K, keys);
  if (h->V) v.emplace_back(h->V, keys);
  v.emplace_back(h->score, meta);
  v.emplace_back(h->gum, meta);
  v.emplace_back(h->pos, meta);
  return v;
}

}  // namespace

extern "C" {

int kvevict_state_bytes(const kvevict_t* h, size_t* bytes) {
  if (!h || !bytes) return fail(KVEVICT_ERR_INVALID_ARG, "null argument");
  *bytes = sizeof(SnapHeader) + snap_payload(h);
  return KVEVICT_OK;
}

int kvevict_save_state(kvevict_t* h, void* buf, size_t bytes, void* stream) {
  KV_RANGE();
  if (!h || !buf) return fail(KVEVICT_ERR_INVALID_ARG, "null argument");
  const size_t need = sizeof(SnapHeader) + snap_payload(h);
  if (bytes < need) return fail(KVEVICT_ERR_INVALID_ARG, "buffer smaller than kvevict_state_bytes");
  cudaStream_t s = (cudaStream_t)stream;
  int rc = enqueue_flush(h, s);   // no compaction left pending in the snapshot
  if (rc != KVEVICT_OK) return rc;
  unsigned char* out = static_cast<unsigned char*>(buf);
  const SnapHeader sh = snap_header(h);
  std::memcpy(out, &sh, sizeof sh);
  size_t off = sizeof sh;
  std::memcpy(out + off, h->budgets.data(), (size_t)h->L * 4);
  off += (size_t)h->L * 4;
  for (const auto& a : snap_arrays(h)) {
    KV_CUDA(cudaMemcpyAsync(out + off, a.first, a.second, cudaMemcpyDeviceToHost, s));
    off += a.second;
  }
  return check_error_word(h, s);   // synchronises the stream
}

int kvevict_load_state(kvevict_t* h, const void* buf, size_t bytes, void* stream) {
  KV_RANGE();
  if (!h || !buf) return fail(KVEVICT_ERR_INVALID_ARG, "null argument");
  if (bytes < sizeof(SnapHeader)) return fail(KVEVICT_ERR_INVALID_ARG, "buffer too small for a snapshot header");
  SnapHeader sh;
  std::memcpy(&sh, buf, sizeof sh);
  const SnapHeader mine = snap_header(h);
  if (std::memcmp(sh.magic, kSnapMagic, 8) != 0 || sh.version != 1 || sh.header_bytes != sizeof(SnapHeader))
    return fail(KVEVICT_ERR_INVALID_ARG, "not a kvevict snapshot (magic, version or header size)");
  if (bytes < sizeof sh + sh.payload_bytes || sh.payload_bytes != mine.payload_bytes)
    return fail(KVEVICT_ERR_INVALID_ARG, "snapshot size does not match this handle");
  if (sh.batch != mine.batch || sh.n_layers != mine.n_layers || sh.n_kv_heads != mine.n_kv_heads ||
      sh.head_dim != mine.head_dim || sh.with_values != mine.with_values || sh.total_rows != mine.total_rows ||
      sh.total_meta != mine.total_meta)
    return fail(KVEVICT_ERR_INVALID_ARG, "snapshot shape (B, L, H, D, values) differs from this handle");
  if (sh.n_sink != mine.n_sink || sh.recent != mine.recent || sh.score_mode != mine.score_mode ||
      sh.anneal_steps != mine.anneal_steps || sh.tau_init != mine.tau_init || sh.tau_end != mine.tau_end ||
      sh.rope_theta != mine.rope_theta || sh.seed != mine.seed)
    return fail(KVEVICT_ERR_INVALID_ARG,
                "snapshot method parameters (sinks, recent, score mode, tau schedule, RoPE base, seed) differ");
  if (sh.next_pos < 0 || sh.stepped < 0 || sh.stepped > 1)
    return fail(KVEVICT_ERR_INVALID_ARG, "snapshot position out of range");
  const unsigned char* in = static_cast<const unsigned char*>(buf);
  size_t off = sizeof sh;
  if (std::memcmp(in + off, h->budgets.data(), (size_t)h->L * 4) != 0)
    return fail(KVEVICT_ERR_INVALID_ARG, "snapshot layer budgets differ from this handle's");
  off += (size_t)h->L * 4;
  cudaStream_t s = (cudaStream_t)stream;
  for (const auto& a : snap_arrays(h)) {
    KV_CUDA(cudaMemcpyAsync(a.first, in + off, a.second, cudaMemcpyHostToDevice, s));
    off += a.second;
  }
  KV_CUDA(cudaMemsetAsync(h->pend, 0xFF, (size_t)h->heads * 4, s));   // flushed when saved
  KV_CUDA(cudaMemsetAsync(h->done, 0, (size_t)h->heads * 8, s));
  KV_CUDA(cudaMemsetAsync(h->err, 0, sizeof(int), s));
  KV_CUDA(cudaMemsetAsync(h->ticket, 0, sizeof(unsigned long long), s));
  h->next_pos = sh.next_pos;
  h->stepped = sh.stepped != 0;
  h->dsteps = 0;
  return check_error_word(h, s);   // synchronises the stream: the caller may free buf
}

}  // extern "C"
