// kvevict_internal.cuh -- structures and device helpers shared by the runtime
// (runtime.cu) and the kernels (decode.cu, prefill.cu).
//
// Device state layout (one arena per handle, rows of the cache in
// layer-major order: head slot = (l * B + b) * H + h, so the launch visits the
// largest pyramid budgets first):
//   K      fp16 [sum_l B*H*cap_l, D]   cap_l = budget_l + 1 rows per head
//   score  f32  [sum_l B*H*capm_l]     capm_l = cap_l rounded up to 4 (16 B)
//   gum    f32  [same]                 frozen Gumbel value of each row
//   pos    i32  [same]                 original absolute position of each row
//   pend   i32  [heads]                slot evicted by the last step whose
//                                      compaction is still to be applied, or -1
// A decode step leaves the evicted row in place and records it in pend; the
// next step (or the flush kernel) applies that compaction while it streams the
// rows anyway, so each row is read once and written at most once per step.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <type_traits>

namespace kvx {

constexpr int kMaxLayers = 256;
// Bounded spin: 4 s of wall time, then the error word. Long enough that a
// stall of the host link under a step that reads its keys from host memory
// (one of about a second was seen) is not reported as a device error; short
// enough that a wait that can never end returns within seconds.
constexpr uint64_t kWaitLimitNs = 4000000000ull;
constexpr int kErrWaitTimeout = 1;
constexpr int kErrBadIndex = 2;

struct LayerInfo {
  int32_t budget;     // b_l
  int32_t cap;        // b_l + 1 key rows per head
  int32_t capm;       // cap rounded up to a multiple of 4 (metadata stride)
  int32_t pad;
  int64_t row_base;   // first K row of layer l's heads
  int64_t meta_base;  // first metadata entry of layer l's heads
};

struct DecodeArgs {
  const __half* k_new;     // step t's key of row (b, l, h) at k_new + t*k_step + ((b*L + l)*H + h)*k_stride
  int64_t k_stride;        // D for decode keys; S*D when keys come from a prompt buffer
  int64_t k_step;          // elements between consecutive steps' keys (B*L*H*D, or D in a prompt buffer)
  const __half* v_new;     // value rows, same layout and strides as k_new (null: keys only)
  __half* K;
  __half* V;               // value arena, same layout as K (null: keys only)
  float* score;
  float* gum;
  int32_t* pos;
  int32_t* pend;
  // [rows] per row: (decode steps applied since reset) << 32 | (slot the last
  // step evicted and left in place + 1, 0 for none), one release store per step
  unsigned long long* done;
  int32_t* evicted;        // [T, B, L, H] user layout (ev_step apart), or null
  int64_t ev_step;
  const LayerInfo* layers;
  const float* rope_c;     // [D/2] cos(-w_i) as f32 (shift by -1)
  const float* rope_s;     // [D/2] sin(-w_i)
  int* err;
  unsigned long long* ticket;   // (step, row) claims; 0 between launches
  int rows;                // B * L * H
  int T;                   // decode steps in this launch
  int s0;                  // steps already applied to every row before this launch
  int capm_max;            // largest metadata stride (sizes the shared-memory logits)
  int B, L, H, n_sink;
  int recent;              // trailing protected window
  int mode;                // 0 cumulative scores, 1 current-step scores
  int64_t p0;              // absolute position of step 0's key
  float tau_init, tau_end; // tau(p) = tau_init + min(p, A) * (tau_end - tau_init) / A, in fp64
  int anneal_steps;        // A (0: constant tau_init)
  float scale2;            // log2(e)/sqrt(D): logits in base-2 units
  uint64_t seed;
  int stall;               // test hook: CTA 0 never issues its first key tile's copy
};

struct FlushArgs {
  __half* K;
  __half* V;               // null: keys only
  float* score;
  float* gum;
  int32_t* pos;
  int32_t* pend;
  const LayerInfo* layers;
  const float* rope_c;
  const float* rope_s;
  int B, L, H;
  int64_t p;               // tokens absorbed so far
};

struct PrefillScoreArgs {
  const __half* keys;      // [heads, S_buf, D] for the heads of this launch; the first S rows used
  float* lse2;             // [heads, Sp] base-2 log-sum-exp of each causal row
  float* colsum;           // [heads, Sp]
  int S;
  int S_buf;               // rows per head in the key buffer (>= S)
  int Sp;                  // scratch row stride: S rounded up to 128
  int heads;
  float scale2;            // log2(e) / sqrt(D)
  int* err;                // error word for bounded waits, or null
  int stall;               // test hook: in pass 1 the copy of item 0's query tile is never issued
  int* work;               // [2] work-item counters of the two passes (zeroed by the launch)
};

// Test hook (kvevict_test_stall_next_step with a null handle): the next prompt
// scorer launch in the process takes stall = 1; returns whether one was armed.
bool take_scorer_stall();

struct PrefillSelectArgs {
  const __half* keys;      // [heads, S_buf, D] for the heads of this launch; the first S rows used
  const __half* values;    // same layout as keys (null: keys only)
  __half* V;               // value arena (null: keys only)
  const float* colsum;     // [heads, S]
  const float* gtab;       // [L*H, Sp] Gumbel value of (layer, head, prompt position)
  __half* K;
  float* score;
  float* gum;
  int32_t* pos;
  int32_t* pend;
  const LayerInfo* layers;
  const float* rope_c;     // [max_delta + 1, D/2]: row d = cos(-d * w_i)
  const float* rope_s;
  int* err;
  int B, L, H, n_sink;
  int recent;              // trailing protected window
  int b0;                  // first batch index of this launch
  int S;
  int S_buf;               // rows per head in the key buffer (>= S)
  int Sp;                  // scratch row stride
  float tau;               // tau(S - 1)
  uint64_t seed;
};

// ---------------------------------------------------------------- launchers
cudaError_t decode_step_setup(int D, size_t smem);
size_t decode_step_smem(int D, int capm_max);
// One launch runs a.T decode steps: persistent CTAs (grid = CTAs per SM x SMs,
// at most one per row) claim (step, row) pairs in order from a.ticket; a row's
// step t waits until the high half of a.done[row] shows step t - 1 applied.
cudaError_t decode_step_ctas_per_sm(int D, size_t smem, int* ctas);
cudaError_t launch_decode_step(const DecodeArgs& a, int D, int grid, size_t smem, cudaStream_t s);
cudaError_t launch_flush(const FlushArgs& a, int D, int heads, cudaStream_t s);
// The shared-memory-resident decode step (decode_resident.cu): one CTA per row
// for every step of the call. resident_step_smem returns (size_t)-1 when a
// row of capm_max slots does not fit its layout.
// It comes with 8 or 16 consumer warps: setup sets both variants' shared
// memory attribute and reports how many CTAs of each fit an SM.
size_t resident_step_smem(int D, int capm_max);
cudaError_t resident_step_setup(int D, size_t smem, int* ctas8, int* ctas16);
cudaError_t launch_resident_step(const DecodeArgs& a, int D, int warps, size_t smem, cudaStream_t s);

// Page-locked host memory (staging.cu). mapped_host: the device address of the
// host buffer [p, p + bytes) when both its ends are page-locked and mapped into
// one device range, else nullptr (pageable memory). launch_copy: bytes from src
// to dst with SM loads and stores; either side may be a mapped host address.
// background: one small block per SM, sized to run beside the prompt scorer.
void* mapped_host(const void* p, size_t bytes);
cudaError_t launch_copy(const void* src, void* dst, size_t bytes, int sms, bool background, cudaStream_t s);

cudaError_t prefill_setup(int D, int max_prefill);  // bulk-eviction kernel's shared memory
// current-step (TOVA) prompt scores: softmax of the last prompt key against every prompt key
cudaError_t launch_prefill_lastrow(const PrefillScoreArgs& a, int D, cudaStream_t s);
// tcgen05/TMEM scorer (prefill_tc.cu): a.Sp must be S rounded up to kPrefillRowPad
constexpr int kPrefillRowPad = 128;
size_t prefill_tc_smem(int D);
cudaError_t prefill_tc_setup(int D);
cudaError_t launch_prefill_tc(const PrefillScoreArgs& a, int D, int sms, cudaStream_t s);
size_t prefill_select_smem(int S);
// The prompt's Gumbel values depend on (layer, head, position) only, not on the
// batch row: out[(l*H + h)*Sp + j] = g(seed, l, h, j) for j < S.
cudaError_t launch_gumbel_table(uint64_t seed, int L, int H, int S, int Sp, float* out, int sms,
                                cudaStream_t s);
cudaError_t launch_prefill_select(const PrefillSelectArgs& a, int D, int heads, cudaStream_t s);

// ---------------------------------------------------------------- device helpers
__device__ __forceinline__ uint64_t splitmix64(uint64_t x) {
  uint64_t z = x + 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// Frozen Gumbel value of (seed, layer, head, position): SplitMix64 chained over
// the four integers, u = (2k+1)/2^53 from the top 52 bits, g = -log(-log u) in
// fp64, stored as f32.
__device__ __forceinline__ float gumbel_at(uint64_t seed, int64_t layer, int64_t head,
                                           int64_t p) {
  uint64_t h = splitmix64(seed);
  h = splitmix64(h ^ (uint64_t)layer);
  h = splitmix64(h ^ (uint64_t)head);
  h = splitmix64(h ^ (uint64_t)p);
  const uint64_t k = h >> 12;
  const double u = (double)(2 * k + 1) * 0x1p-53;
  return (float)(-log(-log(u)));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

// One-dimensional TMA bulk copy global -> this CTA's shared memory; completion
// is counted in bytes on the mbarrier. dst, src and bytes must be 16-byte
// multiples/aligned.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Wait for an mbarrier phase with a time limit; false if the limit ran out.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
}

}  // namespace kvx
