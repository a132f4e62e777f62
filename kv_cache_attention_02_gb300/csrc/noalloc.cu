// noalloc.cu -- prompt scoring for callers that cannot allocate device memory.
//
// Some callers of this library cannot call cudaMalloc: an inference engine
// that reserves the whole device heap for its own pool at start-up (an extra
// cudaMalloc then fails or fragments that pool), or a latency-bound serving
// loop that cannot afford cudaMalloc's implicit device-wide synchronisation.
// kvevict_prefill_scores_noalloc gives them the prompt scorer (causal
// column sums, the two tensor-core passes of prefill_tc.cu) with its working
// memory in a fixed file-scope device array instead of an allocation. The
// caller passes the keys and the output buffer; nothing is allocated.
//
// The array costs kNoAllocScratchFloats * 4 bytes (16 MiB) on every GPU that
// loads this library, for as long as the process lives. Every call shares it
// and the scorer's two work-item counters beside it: calls whose work overlaps
// on the GPU (different streams, or other threads) race on them and must be
// serialised by the caller.
//
// A bounded wait in the scorer that runs out (4 s) cannot be reported through
// the return code, which the call gives before the GPU runs. The scorer sets a
// file-scope error word instead, which each call clears first, and the last
// kernel of the call then writes NaN to every output instead of the scores.
#include "kvevict.h"
#include "kvevict_internal.cuh"

#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <cmath>
#include <mutex>
#include <string>

namespace kvx {
void set_last_error(const std::string& msg);  // runtime.cu: kvevict_last_error()'s message
}

namespace {

constexpr size_t kNoAllocScratchFloats = size_t(4) << 20;   // 16 MiB
constexpr int kMaxDevices = 64;

// Working memory of the allocation-free scorer: [2, heads, Sp] floats (the
// row log-sum-exps, then the padded column sums).
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchFloats];
// the scorer's two work-item counters, cleared by each call before its launches
static __device__ __align__(256) int g_noalloc_work[2];
// Error word of the allocation-free scorer's bounded waits (cleared by each call).
static __device__ __align__(256) int g_noalloc_err;

struct DeviceSetup {
  float* scratch = nullptr;   // device address of g_noalloc_scratch
  int* err = nullptr;         // device address of g_noalloc_err
  int* work = nullptr;        // device address of g_noalloc_work
  int sms = 0;                // multiprocessors, to size the gather's grid
  bool tc_ready[2] = {false, false};   // scorer's shared-memory attribute set (D = 64, 128)
};

std::mutex g_setup_mu;
DeviceSetup g_setup[kMaxDevices];

// Copy the padded column sums [heads, Sp] to the caller's [heads, S]; if a
// bounded wait of this call's scorer ran out, write NaN instead.
__global__ void gather_colsum_kernel(const float* src, int Sp, float* dst, int S, int64_t total,
                                     const int* err) {
  const bool failed = *reinterpret_cast<const volatile int*>(err) != 0;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t h = i / S;
    const int64_t j = i - h * S;
    dst[i] = failed ? __int_as_float(0x7fc00000) : src[h * Sp + j];
  }
}

// Once per device (and head_dim), with that device current: resolve the
// device addresses of the scratch array and the error word, read the SM count
// and set the scoring kernels' shared-memory attribute.
int setup_device(int D, DeviceSetup* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    kvx::set_last_error(std::string("cudaGetDevice: ") + cudaGetErrorString(e));
    return KVEVICT_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    kvx::set_last_error("device ordinal beyond the supported 64");
    return KVEVICT_ERR_INVALID_ARG;
  }
  std::lock_guard<std::mutex> lock(g_setup_mu);
  DeviceSetup& st = g_setup[dev];
  if (!st.scratch) {
    void* p = nullptr;
    void* q = nullptr;
    int sms = 0;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e == cudaSuccess) e = cudaGetSymbolAddress(&q, g_noalloc_err);
    void* w = nullptr;
    if (e == cudaSuccess) e = cudaGetSymbolAddress(&w, g_noalloc_work);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) {
      kvx::set_last_error(std::string("device set-up: ") + cudaGetErrorString(e));
      return KVEVICT_ERR_CUDA;
    }
    st.err = static_cast<int*>(q);
    st.work = static_cast<int*>(w);
    st.sms = sms > 0 ? sms : 1;
    st.scratch = static_cast<float*>(p);
  }
  const int di = D == 64 ? 0 : 1;
  if (!st.tc_ready[di]) {
    e = kvx::prefill_tc_setup(D);
    if (e != cudaSuccess) {
      kvx::set_last_error(std::string("prefill_tc_setup: ") + cudaGetErrorString(e));
      return KVEVICT_ERR_CUDA;
    }
    st.tc_ready[di] = true;
  }
  *out = st;
  return KVEVICT_OK;
}

}  // namespace

namespace {

int prefill_scores_noalloc(const uint16_t* keys, int32_t heads, int32_t S, int32_t head_dim, float* colsum,
                           void* stream) {
  if (!keys || !colsum) {
    kvx::set_last_error("keys and colsum must not be null");
    return KVEVICT_ERR_INVALID_ARG;
  }
  if ((reinterpret_cast<uintptr_t>(keys) & 15) != 0) {
    kvx::set_last_error("keys must be 16-byte aligned");
    return KVEVICT_ERR_INVALID_ARG;
  }
  if (head_dim != 64 && head_dim != 128) {
    kvx::set_last_error("head_dim must be 64 or 128");
    return KVEVICT_ERR_INVALID_ARG;
  }
  if (heads < 0 || S < 0) {
    kvx::set_last_error("heads and S must be >= 0");
    return KVEVICT_ERR_INVALID_ARG;
  }
  if (heads == 0 || S == 0) return KVEVICT_OK;
  const int64_t Sp = ((int64_t)S + kvx::kPrefillRowPad - 1) / kvx::kPrefillRowPad * kvx::kPrefillRowPad;
  if (2 * (int64_t)heads * Sp > (int64_t)kNoAllocScratchFloats) {
    kvx::set_last_error("heads * round_up(S, 128) exceeds the fixed scratch of 2,097,152 floats per pass");
    return KVEVICT_ERR_INVALID_ARG;
  }
  DeviceSetup dev;
  const int rc = setup_device(head_dim, &dev);
  if (rc != KVEVICT_OK) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  kvx::PrefillScoreArgs a{};
  a.keys = reinterpret_cast<const __half*>(keys);
  a.lse2 = dev.scratch;
  a.colsum = dev.scratch + (size_t)heads * Sp;
  a.S = S;
  a.S_buf = S;
  a.Sp = (int)Sp;
  a.heads = heads;
  a.scale2 = (float)(1.4426950408889634 / std::sqrt((double)head_dim));
  a.err = dev.err;
  a.stall = kvx::take_scorer_stall() ? 1 : 0;
  a.work = dev.work;
  cudaError_t e = cudaMemsetAsync(dev.err, 0, sizeof(int), s);   // writes, allocates nothing
  if (e == cudaSuccess) e = kvx::launch_prefill_tc(a, head_dim, dev.sms, s);
  if (e == cudaSuccess) {
    const int64_t total = (int64_t)heads * S;
    const int64_t blocks = std::min<int64_t>((total + 255) / 256, (int64_t)dev.sms * 16);
    gather_colsum_kernel<<<(unsigned)blocks, 256, 0, s>>>(a.colsum, (int)Sp, colsum, S, total, dev.err);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) {
    kvx::set_last_error(std::string("launch: ") + cudaGetErrorString(e));
    return KVEVICT_ERR_CUDA;
  }
  return KVEVICT_OK;
}

}  // namespace

// The exported call, inside an NVTX range named after it (for profilers; a
// branch when no tool is attached).
extern "C" int kvevict_prefill_scores_noalloc(const uint16_t* keys, int32_t heads, int32_t S,
                                              int32_t head_dim, float* colsum, void* stream) {
  nvtxRangePushA("kvevict_prefill_scores_noalloc");
  const int rc = prefill_scores_noalloc(keys, heads, S, head_dim, colsum, stream);
  nvtxRangePop();
  return rc;
}
