// decode_common.cuh -- device helpers shared by the decode kernels (the
// streaming step in decode.cu and the shared-memory-resident step in
// decode_resident.cu): row geometry, the fp16 dot product, the fp32 RoPE
// re-rotation, the consumer warps' block reductions and bounded waits.
#pragma once

#include "kvevict_internal.cuh"

#include <cfloat>
#include <climits>
#include <type_traits>

namespace kvx {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;   // 256 threads work on key rows
constexpr int kTPR = 8;                           // threads per key row
constexpr int kRowsPerPass = kConsumers / kTPR;   // 32
constexpr int kTile = 64;                         // rows per TMA tile

template <int D>
struct Geo {
  static constexpr int CH = D / 16;            // halves per chunk
  static constexpr int HALF = D / 2;
  static constexpr int ROWB = D * 2;
  static constexpr int TILEB = kTile * ROWB;
  static constexpr int SLOTB = 64 + 2 * ROWB;   // header (padded) + new key + new value
  using Chunk = typename std::conditional<CH == 8, uint4, uint2>::type;
  using Word = typename std::conditional<D == 128, uint2, uint32_t>::type;   // a row over 32 lanes
};
static_assert(Geo<128>::SLOTB % 16 == 0 && Geo<64>::SLOTB % 16 == 0, "16-byte aligned rows in a slot");

// fp16 chunk <-> float2 pairs
template <int CH>
__device__ __forceinline__ void unpack2(const typename std::conditional<CH == 8, uint4, uint2>::type& c,
                                        float2* f) {
  const __half2* h = reinterpret_cast<const __half2*>(&c);
#pragma unroll
  for (int k = 0; k < CH / 2; ++k) f[k] = __half22float2(h[k]);
}

template <int CH>
__device__ __forceinline__ typename std::conditional<CH == 8, uint4, uint2>::type pack2(const float2* f) {
  typename std::conditional<CH == 8, uint4, uint2>::type c;
  __half2* h = reinterpret_cast<__half2*>(&c);
#pragma unroll
  for (int k = 0; k < CH / 2; ++k) h[k] = __float22half2_rn(f[k]);
  return c;
}

// Rotate pair halves (a, b) by the shift-by-one constants: x = a*c - b*s,
// y = a*s + b*c, each product and each sum rounded to f32 on its own. Scalar
// __fmul_rn/__fsub_rn/__fadd_rn on purpose: on sm_103a with CUDA 13.0 a packed
// mul.rn.f32x2 + add.rn.f32x2 pair was measured to return the fused result
// (an fp16 midpoint case came out one ULP off), which would break the op-by-op
// fp32 rotation the stored keys must follow.
template <int CH>
__device__ __forceinline__ void rotate2(float2* a, float2* b, const float2* c, const float2* s) {
#pragma unroll
  for (int k = 0; k < CH / 2; ++k) {
    const float x0 = __fsub_rn(__fmul_rn(a[k].x, c[k].x), __fmul_rn(b[k].x, s[k].x));
    const float y0 = __fadd_rn(__fmul_rn(a[k].x, s[k].x), __fmul_rn(b[k].x, c[k].x));
    const float x1 = __fsub_rn(__fmul_rn(a[k].y, c[k].y), __fmul_rn(b[k].y, s[k].y));
    const float y1 = __fadd_rn(__fmul_rn(a[k].y, s[k].y), __fmul_rn(b[k].y, c[k].y));
    a[k] = make_float2(x0, x1);
    b[k] = make_float2(y0, y1);
  }
}

// fp32 accumulation of fp16 x fp16 products with the mixed-precision FMA
// (the product of two fp16 values is exact in f32, so this equals converting
// both operands and using an f32 FMA). Two independent chains, one per chunk.
__device__ __forceinline__ float fma_f16(__half a, __half b, float c) {
  float d;
  asm("fma.rn.f32.f16 %0, %1, %2, %3;" : "=f"(d) : "h"(__half_as_ushort(a)), "h"(__half_as_ushort(b)), "f"(c));
  return d;
}
template <int CH>
__device__ __forceinline__ float dot_chunks(const typename std::conditional<CH == 8, uint4, uint2>::type& klo,
                                            const typename std::conditional<CH == 8, uint4, uint2>::type& khi,
                                            const typename std::conditional<CH == 8, uint4, uint2>::type& qlo,
                                            const typename std::conditional<CH == 8, uint4, uint2>::type& qhi) {
  const __half2* a = reinterpret_cast<const __half2*>(&klo);
  const __half2* b = reinterpret_cast<const __half2*>(&khi);
  const __half2* qa = reinterpret_cast<const __half2*>(&qlo);
  const __half2* qb = reinterpret_cast<const __half2*>(&qhi);
  float s0 = 0.f, s1 = 0.f;
#pragma unroll
  for (int k = 0; k < CH / 2; ++k) {
    s0 = fma_f16(__low2half(a[k]), __low2half(qa[k]), s0);
    s1 = fma_f16(__low2half(b[k]), __low2half(qb[k]), s1);
    s0 = fma_f16(__high2half(a[k]), __high2half(qa[k]), s0);
    s1 = fma_f16(__high2half(b[k]), __high2half(qb[k]), s1);
  }
  return s0 + s1;
}

// 2^x on the MUFU (ex2.approx: relative error below 2^-22; a result below the
// smallest normal flushes to zero, which only drops terms smaller than 2^-126
// of the row's largest from a softmax sum).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// The softmax statistics of a step, in two block-wide passes over the logits
// in shared memory (base-2 units). First the block max of every thread's
// running max (one redux per warp, one barrier; a max is exact, so which
// thread saw which logit does not matter). Then each thread sums
// 2^(logit - max) over the rows R = tid, tid + 256, ... in ascending order,
// storing each term back in place (the score update reuses it), and the block
// adds the threads' sums with a butterfly per warp and the eight warp sums in
// warp order (one barrier). Both decode kernels use exactly these two
// functions and this row-to-thread assignment, so their sums agree bit for bit
// whichever threads computed the dot products.
//
// NT is the number of consumer threads taking part (256 in the streaming
// kernel; 256 or 512 in the resident one). The sum's assignment is the 256-
// thread one whatever NT is: threads beyond 256 add nothing. Scratch: red[w]
// holds warp maxima (w < 16), red[16 + w] warp sums (w < 8).
template <int NT = kConsumers>
__device__ float block_max(float m, float* red) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float wm;
  asm("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(wm) : "f"(m));
  if (lane == 0) red[w] = wm;
  asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory");
  float M = red[0];
#pragma unroll
  for (int k = 1; k < NT / 32; ++k) M = fmaxf(M, red[k]);
  return M;
}

// Sum of 2^(lg[R] - M) over R < NR, R != skip; the terms replace the logits.
template <int NT = kConsumers>
__device__ float block_expsum(float* lg, int NR, int skip, float M, float* red) {
  static_assert(NT >= kConsumers, "the sum's row assignment needs 256 threads");
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x < kConsumers) {   // whole warps
    float ls = 0.f;
    for (int R = threadIdx.x; R < NR; R += kConsumers) {
      if (R == skip) continue;
      const float e = ex2(lg[R] - M);
      lg[R] = e;
      ls += e;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, o);
    if (lane == 0) red[16 + w] = ls;
  }
  asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory");
  float L = red[16];
#pragma unroll
  for (int k = 1; k < kConsumerWarps; ++k) L += red[16 + k];
  return L;
}

// Order-preserving map of a float onto an unsigned key (-0 taken as +0).
__device__ __forceinline__ uint32_t float_key(float f) {
  const uint32_t u = __float_as_uint(f + 0.f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Block-wide (r, slot) argmin, lowest slot on ties: per warp two redux
// minima (the key of r, then the slot among the lanes holding it), then every
// thread merges the eight warp candidates itself.
template <int NT = kConsumers>
__device__ int block_argmin(float r, int i, float* redf, int* redi) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t key = float_key(r);
  uint32_t kmin, imin;
  asm("redux.sync.min.u32 %0, %1, 0xffffffff;" : "=r"(kmin) : "r"(key));
  const uint32_t cand = key == kmin ? (uint32_t)i : 0xffffffffu;
  asm("redux.sync.min.u32 %0, %1, 0xffffffff;" : "=r"(imin) : "r"(cand));
  if (lane == 0) { redf[40 + w] = __uint_as_float(kmin); redi[40 + w] = (int)imin; }
  asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory");
  uint32_t kb = __float_as_uint(redf[40]);
  int ib = redi[40];
#pragma unroll
  for (int k = 1; k < NT / 32; ++k) {
    const uint32_t k2 = __float_as_uint(redf[40 + k]);
    const int i2 = redi[40 + k];
    if (k2 < kb || (k2 == kb && i2 < ib)) { kb = k2; ib = i2; }
  }
  return ib;
}

__device__ __forceinline__ void mbar_arrive_cta(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Order this thread's later async-proxy (TMA) reads of global memory after the
// generic-proxy writes it has synchronised with.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// tau(p) = tau_init + min(p, A) (tau_end - tau_init) / A, each operation in
// fp64 and the result rounded to f32.
__device__ __forceinline__ float tau_at(const DecodeArgs& a, int64_t p) {
  if (a.anneal_steps <= 0 || a.tau_init == a.tau_end) return a.tau_init;
  const int64_t t = p < 0 ? 0 : (p < a.anneal_steps ? p : (int64_t)a.anneal_steps);
  const double span = __dsub_rn((double)a.tau_end, (double)a.tau_init);
  return (float)__dadd_rn((double)a.tau_init, __ddiv_rn(__dmul_rn((double)t, span), (double)a.anneal_steps));
}

// Named barrier 1 over the consumer warps only (the producer and scheduler
// warps run ahead on their own): a plain sync, and one that ORs a predicate.
template <int NT = kConsumers>
__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory");
}
template <int NT = kConsumers>
__device__ __forceinline__ bool consumers_any(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "n"(NT)
      : "memory");
  return r != 0;
}

// Bounded wait that also gives up as soon as another thread raised the abort flag.
__device__ __forceinline__ bool wait_watch(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                           int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      *abort_flag = 1;
      atomicOr(err, kErrWaitTimeout);
      return false;
    }
  }
}

}  // namespace
}  // namespace kvx
