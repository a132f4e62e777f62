// prefill.cu -- prompt bulk eviction (the prompt's scores come from the
// tensor-core scorer in prefill_tc.cu).
//
// Bulk eviction (reading: the whole prompt is scored first, then the S - b
// non-sink rows with the lowest (score + tau(S-1) * gumbel, slot) go at once):
// one CTA per cache row sorts (r, slot) keys in shared memory (the Gumbel
// values come from a per-prompt (layer, head, position) table), scans the
// survivors' new slots and writes them, each key re-rotated by
// (new slot - old slot) RoPE positions in fp32 and stored as fp16.
#include "kvevict_internal.cuh"

#include <algorithm>
#include <cfloat>

namespace kvx {
namespace {

// ---------------------------------------------------------------- bulk eviction
// 256 threads a CTA, four CTAs an SM: while one CTA sorts (barrier-bound,
// no HBM traffic) the others move rows.
constexpr int kSThreads = 256;
constexpr int kSWarps = kSThreads / 32;

__device__ __forceinline__ uint32_t ordered_bits(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

template <int D>
__global__ void __launch_bounds__(kSThreads, 4) prefill_select_kernel(const PrefillSelectArgs a) {
  constexpr int CH = D / 16, HALF = D / 2;
  using Chunk = typename std::conditional<CH == 8, uint4, uint2>::type;
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x;
  const int S = a.S;
  const int hi = blockIdx.x;                     // cache row within this launch (user order)
  const int LH = a.L * a.H;
  const int b = a.b0 + hi / LH;
  const int rem2 = hi - (hi / LH) * LH;
  const int l = rem2 / a.H;
  const int hh = rem2 - l * a.H;
  const LayerInfo li = a.layers[l];
  const int slot_rem = b * a.H + hh;
  const int slot = l * (a.B * a.H) + slot_rem;
  __half* Kg = a.K + (li.row_base + (int64_t)slot_rem * li.cap) * D;
  float* scg = a.score + li.meta_base + (int64_t)slot_rem * li.capm;
  float* gg = a.gum + li.meta_base + (int64_t)slot_rem * li.capm;
  int32_t* pg = a.pos + li.meta_base + (int64_t)slot_rem * li.capm;
  const __half* src = a.keys + (size_t)hi * a.S_buf * D;
  const __half* vsrc = a.V ? a.values + (size_t)hi * a.S_buf * D : nullptr;
  __half* Vg = a.V ? a.V + (li.row_base + (int64_t)slot_rem * li.cap) * D : nullptr;
  const float* col = a.colsum + (size_t)hi * a.Sp;
  const float* gs = a.gtab + ((size_t)l * a.H + hh) * a.Sp;
  const int budget = li.budget;
  const int c = tid & 7;

  // Rows move 8 threads to a row, kRowsInFlight rows per thread per round:
  // every load of a round is issued before the first store, so a thread keeps
  // several HBM reads in flight instead of one (as many as fit in the 64
  // registers a thread has at four 256-thread CTAs an SM).
  constexpr int RPP = kSThreads / 8;   // rows per pass
  constexpr int kRowsInFlight = D == 128 ? 3 : 4;

  if (S <= budget) {  // the whole prompt fits: keep every row where it is
    for (int j0 = 0; j0 < S; j0 += RPP * kRowsInFlight) {
      Chunk lo[kRowsInFlight], hi2[kRowsInFlight];
      float sv[kRowsInFlight], gv[kRowsInFlight];
#pragma unroll
      for (int u = 0; u < kRowsInFlight; ++u) {
        const int j = j0 + u * RPP + (tid >> 3);
        if (j < S) {
          lo[u] = *reinterpret_cast<const Chunk*>(src + (size_t)j * D + c * CH);
          hi2[u] = *reinterpret_cast<const Chunk*>(src + (size_t)j * D + HALF + c * CH);
          if (c == 0) { sv[u] = col[j]; gv[u] = gs[j]; }
        }
      }
#pragma unroll
      for (int u = 0; u < kRowsInFlight; ++u) {
        const int j = j0 + u * RPP + (tid >> 3);
        if (j < S) {
          *reinterpret_cast<Chunk*>(Kg + (size_t)j * D + c * CH) = lo[u];
          *reinterpret_cast<Chunk*>(Kg + (size_t)j * D + HALF + c * CH) = hi2[u];
          if (c == 0) { scg[j] = sv[u]; gg[j] = gv[u]; pg[j] = j; }
          if (Vg) {
            *reinterpret_cast<Chunk*>(Vg + (size_t)j * D + c * CH) =
                *reinterpret_cast<const Chunk*>(vsrc + (size_t)j * D + c * CH);
            *reinterpret_cast<Chunk*>(Vg + (size_t)j * D + HALF + c * CH) =
                *reinterpret_cast<const Chunk*>(vsrc + (size_t)j * D + HALF + c * CH);
          }
        }
      }
    }
    if (tid == 0) a.pend[slot] = -1;
    return;
  }

  const int m = S - a.n_sink - a.recent;   // evictable rows: not a sink, not in the recent window
  // m <= S keys; an even count keeps the next region 16-byte aligned
  uint64_t* keys = reinterpret_cast<uint64_t*>(smem);
  unsigned char* flag = smem + (size_t)((S + 1) & ~1) * 8;
  int16_t* newslot = reinterpret_cast<int16_t*>(flag + ((S + 15) & ~15));
  int* wsum = reinterpret_cast<int*>(newslot + ((S + 7) & ~7));

  for (int t = tid; t < m; t += kSThreads) {
    const int j = a.n_sink + t;
    const float r = fmaf(a.tau, gs[j], col[j]);
    keys[t] = ((uint64_t)ordered_bits(r) << 32) | (uint32_t)j;
  }
  for (int j = tid; j < S; j += kSThreads) flag[j] = 0;
  const int n_ev = S - budget;   // 1 <= n_ev < m
  {
    // Radix select of the n_ev smallest (r, slot) keys. The keys are distinct
    // (the slot is in the low bits), so the n_ev-th smallest key K* is found
    // one byte at a time from the top, and exactly the keys <= K* are evicted:
    // the set an ascending sort's first n_ev entries would give. A slot takes
    // at most 14 bits (S <= 16384), so bits 16..31 are zero in every key and
    // are not visited: six passes (bytes 7..4 of r, then bytes 1, 0).
    static_assert(kSThreads == 256, "one histogram bin per thread");
    int* hist = wsum + 32;   // 256 bins
    int* sel = hist + 256;   // [0] the digit, [1] keys below it
    const int lane = tid & 31, wid = tid >> 5;
    uint64_t prefix = 0, pmask = 0;
    int rank = n_ev;         // 1-based rank of K* among the keys matching the prefix
    for (int pass = 0; pass < 6; ++pass) {
      const int shift = pass < 4 ? 56 - 8 * pass : (pass == 4 ? 8 : 0);
      hist[tid] = 0;
      __syncthreads();
      for (int base = 0; base < m; base += kSThreads) {
        const int t = base + tid;
        const uint64_t key = t < m ? keys[t] : 0ull;
        const bool in = t < m && (key & pmask) == prefix;
        const int bin = in ? (int)((key >> shift) & 255) : 256 + lane;   // no dummy shares a bin
        const unsigned peers = __match_any_sync(0xffffffffu, bin);
        if (in && lane == __ffs(peers) - 1) atomicAdd(&hist[bin], __popc(peers));
      }
      __syncthreads();
      const int v = hist[tid];
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
      }
      if (lane == 31) wsum[wid] = incl;
      __syncthreads();
      int excl = incl - v;
      for (int w = 0; w < wid; ++w) excl += wsum[w];
      if (v > 0 && excl < rank && rank <= excl + v) {   // exactly one bin holds rank
        sel[0] = tid;
        sel[1] = excl;
      }
      __syncthreads();
      rank -= sel[1];
      prefix |= (uint64_t)sel[0] << shift;
      pmask |= (uint64_t)0xFF << shift;
      if (pass == 3) pmask |= 0xFFFF0000ull;
      __syncthreads();   // hist, wsum and sel are rewritten by the next pass
    }
    for (int t = tid; t < m; t += kSThreads)
      if (keys[t] <= prefix) flag[(uint32_t)keys[t]] = 1;
  }
  __syncthreads();

  // exclusive scan of survivors -> new slot (each thread owns a contiguous segment)
  const int seg = (S + kSThreads - 1) / kSThreads;
  const int s0 = min(S, tid * seg), s1 = min(S, s0 + seg);
  int cnt = 0;
  for (int j = s0; j < s1; ++j) cnt += flag[j] ? 0 : 1;
  const int lane = tid & 31, wid = tid >> 5;
  int incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) wsum[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    int v = lane < kSWarps ? wsum[lane] : 0;
    int iv = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, iv, o);
      if (lane >= o) iv += u;
    }
    wsum[lane] = iv - v;  // exclusive prefix over warps
  }
  __syncthreads();
  int run = wsum[wid] + incl - cnt;
  for (int j = s0; j < s1; ++j) {
    newslot[j] = (int16_t)run;
    run += flag[j] ? 0 : 1;
  }
  __syncthreads();

  // write survivors, each re-rotated by (new slot - old slot)
  for (int j0 = 0; j0 < S; j0 += RPP * kRowsInFlight) {
    Chunk lo[kRowsInFlight], hi2[kRowsInFlight];
    float sv[kRowsInFlight], gv[kRowsInFlight];
    bool live[kRowsInFlight];
#pragma unroll
    for (int u = 0; u < kRowsInFlight; ++u) {
      const int j = j0 + u * RPP + (tid >> 3);
      live[u] = j < S && !flag[j];
      if (live[u]) {
        lo[u] = *reinterpret_cast<const Chunk*>(src + (size_t)j * D + c * CH);
        hi2[u] = *reinterpret_cast<const Chunk*>(src + (size_t)j * D + HALF + c * CH);
        if (c == 0) { sv[u] = col[j]; gv[u] = gs[j]; }
      }
    }
#pragma unroll
    for (int u = 0; u < kRowsInFlight; ++u) {
      if (!live[u]) continue;
      const int j = j0 + u * RPP + (tid >> 3);
      const int ns = newslot[j];
      const int d = j - ns;   // shift back by d positions
      if (d > 0) {
        const float* tc = a.rope_c + (size_t)d * HALF + c * CH;
        const float* ts = a.rope_s + (size_t)d * HALF + c * CH;
        __half2* h_lo = reinterpret_cast<__half2*>(&lo[u]);
        __half2* h_hi = reinterpret_cast<__half2*>(&hi2[u]);
#pragma unroll
        for (int k = 0; k < CH / 2; ++k) {
          const float2 fa = __half22float2(h_lo[k]);
          const float2 fb = __half22float2(h_hi[k]);
          const float c0 = tc[2 * k], c1 = tc[2 * k + 1], s0v = ts[2 * k], s1v = ts[2 * k + 1];
          const float x0 = __fsub_rn(__fmul_rn(fa.x, c0), __fmul_rn(fb.x, s0v));
          const float y0 = __fadd_rn(__fmul_rn(fa.x, s0v), __fmul_rn(fb.x, c0));
          const float x1 = __fsub_rn(__fmul_rn(fa.y, c1), __fmul_rn(fb.y, s1v));
          const float y1 = __fadd_rn(__fmul_rn(fa.y, s1v), __fmul_rn(fb.y, c1));
          h_lo[k] = __halves2half2(__float2half_rn(x0), __float2half_rn(x1));
          h_hi[k] = __halves2half2(__float2half_rn(y0), __float2half_rn(y1));
        }
      }
      *reinterpret_cast<Chunk*>(Kg + (size_t)ns * D + c * CH) = lo[u];
      *reinterpret_cast<Chunk*>(Kg + (size_t)ns * D + HALF + c * CH) = hi2[u];
      if (c == 0) { scg[ns] = sv[u]; gg[ns] = gv[u]; pg[ns] = j; }
      if (Vg) {   // value rows move with their keys, never rotated
        *reinterpret_cast<Chunk*>(Vg + (size_t)ns * D + c * CH) =
            *reinterpret_cast<const Chunk*>(vsrc + (size_t)j * D + c * CH);
        *reinterpret_cast<Chunk*>(Vg + (size_t)ns * D + HALF + c * CH) =
            *reinterpret_cast<const Chunk*>(vsrc + (size_t)j * D + HALF + c * CH);
      }
    }
  }
  if (tid == 0) a.pend[slot] = -1;
}

__global__ void gumbel_table_kernel(uint64_t seed, int H, int S, int Sp, int64_t n, float* out) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t lh = i / S;
    const int j = (int)(i - lh * S);
    out[lh * Sp + j] = gumbel_at(seed, lh / H, lh % H, j);
  }
}

// Current-step (TOVA-adapted) prompt scores: the prompt's last key attends
// over every prompt key; score_j = softmax_j(K_j . k_{S-1} / sqrt(D)). One CTA
// per cache row, 8 threads per key row, fp16 products accumulated in f32.
template <int D>
__global__ void __launch_bounds__(256) prefill_lastrow_kernel(const PrefillScoreArgs a) {
  constexpr int CH = D / 16, HALF = D / 2;
  using Chunk = typename std::conditional<CH == 8, uint4, uint2>::type;
  extern __shared__ __align__(128) unsigned char smem[];
  float* lg = reinterpret_cast<float*>(smem);          // [S] base-2 logits
  __shared__ float red[64];
  const int tid = threadIdx.x, c = tid & 7, rg = tid >> 3, lane = tid & 31, w = tid >> 5;
  const int S = a.S;
  const __half* Kh = a.keys + (size_t)blockIdx.x * a.S_buf * D;
  const __half* q = Kh + (size_t)(S - 1) * D;
  const Chunk qlo = *reinterpret_cast<const Chunk*>(q + c * CH);
  const Chunk qhi = *reinterpret_cast<const Chunk*>(q + HALF + c * CH);
  const __half2* qa = reinterpret_cast<const __half2*>(&qlo);
  const __half2* qb = reinterpret_cast<const __half2*>(&qhi);
  float mx = -INFINITY;
  for (int j0 = 0; j0 < S; j0 += 32) {
    const int j = j0 + rg;
    float dot = 0.f;
    if (j < S) {
      const Chunk klo = *reinterpret_cast<const Chunk*>(Kh + (size_t)j * D + c * CH);
      const Chunk khi = *reinterpret_cast<const Chunk*>(Kh + (size_t)j * D + HALF + c * CH);
      const __half2* ka = reinterpret_cast<const __half2*>(&klo);
      const __half2* kb = reinterpret_cast<const __half2*>(&khi);
#pragma unroll
      for (int k = 0; k < CH / 2; ++k) {
        const float2 x = __half22float2(ka[k]), y = __half22float2(kb[k]);
        const float2 u = __half22float2(qa[k]), v = __half22float2(qb[k]);
        dot = fmaf(x.x, u.x, fmaf(x.y, u.y, fmaf(y.x, v.x, fmaf(y.y, v.y, dot))));
      }
    }
    dot += __shfl_xor_sync(0xffffffffu, dot, 1);
    dot += __shfl_xor_sync(0xffffffffu, dot, 2);
    dot += __shfl_xor_sync(0xffffffffu, dot, 4);
    if (j < S && c == 0) {
      lg[j] = dot * a.scale2;
      mx = fmaxf(mx, lg[j]);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (lane == 0) red[w] = mx;
  __syncthreads();
  mx = -INFINITY;
  for (int i = 0; i < 8; ++i) mx = fmaxf(mx, red[i]);
  float sum = 0.f;
  for (int j = tid; j < S; j += 256) sum += exp2f(lg[j] - mx);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  __syncthreads();
  if (lane == 0) red[w] = sum;
  __syncthreads();
  sum = 0.f;
  for (int i = 0; i < 8; ++i) sum += red[i];
  float* out = a.colsum + (size_t)blockIdx.x * a.Sp;
  for (int j = tid; j < S; j += 256) out[j] = exp2f(lg[j] - mx) / sum;
}

}  // namespace

size_t prefill_select_smem(int S) {
  // keys, flags, new slots, the scan's warp sums, the select's histogram and result
  return (size_t)((S + 1) & ~1) * 8 + ((S + 15) & ~15) + ((S + 7) & ~7) * 2 + (32 + 256 + 4) * sizeof(int) + 64;
}

cudaError_t prefill_setup(int D, int max_prefill) {
  const int select = (int)prefill_select_smem(max_prefill > 0 ? max_prefill : 1);
  const int last = (max_prefill > 0 ? max_prefill : 1) * (int)sizeof(float);
  const auto attr = cudaFuncAttributeMaxDynamicSharedMemorySize;
  cudaError_t e;
  if (D == 64) {
    e = cudaFuncSetAttribute(prefill_select_kernel<64>, attr, select);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(prefill_lastrow_kernel<64>, attr, last);
  } else {
    e = cudaFuncSetAttribute(prefill_select_kernel<128>, attr, select);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(prefill_lastrow_kernel<128>, attr, last);
  }
  return e;
}

cudaError_t launch_prefill_lastrow(const PrefillScoreArgs& a, int D, cudaStream_t s) {
  if (a.S <= 0 || a.heads <= 0) return cudaSuccess;
  const size_t smem = (size_t)a.S * sizeof(float);
  if (D == 64)
    prefill_lastrow_kernel<64><<<a.heads, 256, smem, s>>>(a);
  else
    prefill_lastrow_kernel<128><<<a.heads, 256, smem, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_gumbel_table(uint64_t seed, int L, int H, int S, int Sp, float* out, int sms,
                                cudaStream_t s) {
  const int64_t n = (int64_t)L * H * S;
  if (n <= 0) return cudaSuccess;
  const int blocks = (int)std::min<int64_t>((n + 255) / 256, (int64_t)std::max(sms, 1) * 16);
  gumbel_table_kernel<<<blocks, 256, 0, s>>>(seed, H, S, Sp, n, out);
  return cudaGetLastError();
}

cudaError_t launch_prefill_select(const PrefillSelectArgs& a, int D, int heads, cudaStream_t s) {
  if (a.S <= 0 || heads <= 0) return cudaSuccess;
  const size_t smem = prefill_select_smem(a.S);
  if (D == 64)
    prefill_select_kernel<64><<<heads, kSThreads, smem, s>>>(a);
  else
    prefill_select_kernel<128><<<heads, kSThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace kvx
