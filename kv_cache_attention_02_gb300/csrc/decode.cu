// decode.cu -- the fused decode step (one launch per step over every row of
// the cache) and the flush kernel that applies a pending compaction.
//
// What a step computes per (batch, layer, KV head) row follows page
// "veloxquant_mlx.quantizers.keyformer module", keyformer_update steps 1-3 and
// page "PyramidKV -- Layer-Adaptive Budget Attention-Mass Eviction", "How it
// works": append the new key, softmax(K k / sqrt(D)) over every row including
// the new one, scores += attn, and when over the layer's budget evict the
// lowest score + tau * gumbel among non-sink rows (lowest slot on ties); rows
// after the evicted one move down one slot, keys re-rotated by -1 RoPE
// position in fp32 (FUSED METAL KERNEL note) and stored as fp16.
//
// Design (GB300): one CTA per cache row. The row's keys stream through a
// 4-stage shared-memory ring filled by 1-D TMA bulk copies (16 KB tiles),
// completion tracked by mbarriers. 8 threads share a key row (two 16-byte
// chunks each: the pair halves (i, i + D/2) a RoPE rotation needs), so bank
// access is conflict-free without a swizzle and the dot product reduces with
// three shuffles. The compaction decided by the previous step is applied to
// each row as it passes through (rotate, write to slot R-1), so a key row is
// read from HBM once per step and written only if it moves. Softmax max/sum,
// score update and the (r, slot) argmin then run over shared memory.
#include "kvevict_internal.cuh"

#include <cfloat>
#include <climits>
#include <type_traits>

namespace kvx {
namespace {

constexpr int kThreads = 256;
constexpr int kTPR = 8;                       // threads per key row
constexpr int kRowsPerPass = kThreads / kTPR;  // 32
constexpr int kTile = 64;                      // rows per TMA tile
constexpr int kStages = 4;

template <int D>
struct Geo {
  static constexpr int CH = D / 16;            // halves per chunk
  static constexpr int HALF = D / 2;
  static constexpr int ROWB = D * 2;
  static constexpr int TILEB = kTile * ROWB;
  using Chunk = typename std::conditional<CH == 8, uint4, uint2>::type;
};

struct SmemLayout {
  size_t ring, bars, slog, ssc, sg, redf, redi, total;
};

template <int D>
__host__ __device__ inline SmemLayout decode_layout(int capm) {
  SmemLayout L{};
  size_t o = 0;
  L.ring = o;  o += (size_t)kStages * Geo<D>::TILEB;
  L.bars = o;  o += 64;
  const size_t arr = ((size_t)(capm + 4) * 4 + 127) / 128 * 128;
  L.slog = o;  o += arr;
  L.ssc = o;   o += arr;
  L.sg = o;    o += arr;
  L.redf = o;  o += 64 * 4;
  L.redi = o;  o += 64 * 4;
  L.total = o;
  return L;
}

template <int CH>
__device__ __forceinline__ void unpack(const typename std::conditional<CH == 8, uint4, uint2>::type& c,
                                       float* f) {
  const __half2* h = reinterpret_cast<const __half2*>(&c);
#pragma unroll
  for (int k = 0; k < CH / 2; ++k) {
    const float2 v = __half22float2(h[k]);
    f[2 * k] = v.x;
    f[2 * k + 1] = v.y;
  }
}

template <int CH>
__device__ __forceinline__ typename std::conditional<CH == 8, uint4, uint2>::type pack(const float* f) {
  typename std::conditional<CH == 8, uint4, uint2>::type c;
  __half2* h = reinterpret_cast<__half2*>(&c);
#pragma unroll
  for (int k = 0; k < CH / 2; ++k) h[k] = __halves2half2(__float2half_rn(f[2 * k]), __float2half_rn(f[2 * k + 1]));
  return c;
}

// Rotate the pair halves (a_i, b_i) by the shift-by-one constants: every product
// and sum rounded to f32 (no contraction), then fp16 round-to-nearest-even.
template <int CH>
__device__ __forceinline__ void rotate_pairs(float* a, float* b, const float* c, const float* s) {
#pragma unroll
  for (int k = 0; k < CH; ++k) {
    const float x = __fsub_rn(__fmul_rn(a[k], c[k]), __fmul_rn(b[k], s[k]));
    const float y = __fadd_rn(__fmul_rn(a[k], s[k]), __fmul_rn(b[k], c[k]));
    a[k] = x;
    b[k] = y;
  }
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ void warp_argmin(float& r, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float r2 = __shfl_xor_sync(0xffffffffu, r, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, i, o);
    if (r2 < r || (r2 == r && i2 < i)) { r = r2; i = i2; }
  }
}

__device__ float block_max(float v, float* red) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  v = warp_max(v);
  if (lane == 0) red[w] = v;
  __syncthreads();
  if (w == 0) {
    v = lane < kThreads / 32 ? red[lane] : -INFINITY;
    v = warp_max(v);
    if (lane == 0) red[32] = v;
  }
  __syncthreads();
  return red[32];
}

__device__ float block_sum(float v, float* red) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  v = warp_sum(v);
  if (lane == 0) red[w] = v;
  __syncthreads();
  if (w == 0) {
    v = lane < kThreads / 32 ? red[lane] : 0.f;
    v = warp_sum(v);
    if (lane == 0) red[33] = v;
  }
  __syncthreads();
  return red[33];
}

__device__ int block_argmin(float r, int i, float* redf, int* redi) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  warp_argmin(r, i);
  if (lane == 0) { redf[40 + w] = r; redi[40 + w] = i; }
  __syncthreads();
  if (w == 0) {
    r = lane < kThreads / 32 ? redf[40 + lane] : INFINITY;
    i = lane < kThreads / 32 ? redi[40 + lane] : INT_MAX;
    warp_argmin(r, i);
    if (lane == 0) redi[63] = i;
  }
  __syncthreads();
  return redi[63];
}

template <int D>
__global__ void __launch_bounds__(kThreads) decode_step_kernel(const DecodeArgs a) {
  using G = Geo<D>;
  using Chunk = typename G::Chunk;
  constexpr int CH = G::CH, HALF = G::HALF;

  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x;
  const int c = tid & (kTPR - 1);   // chunk index within a row
  const int rg = tid >> 3;          // row within a pass

  const int head = blockIdx.x;
  const int BH = a.B * a.H;
  const int l = head / BH;
  const int rem = head - l * BH;
  const int b = rem / a.H;
  const int hh = rem - b * a.H;
  const LayerInfo li = a.layers[l];
  const SmemLayout SL = decode_layout<D>(li.capm);
  unsigned char* ring = smem + SL.ring;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SL.bars);
  float* s_log = reinterpret_cast<float*>(smem + SL.slog);
  float* s_sc = reinterpret_cast<float*>(smem + SL.ssc);
  float* s_g = reinterpret_cast<float*>(smem + SL.sg);
  float* redf = reinterpret_cast<float*>(smem + SL.redf);
  int* redi = reinterpret_cast<int*>(smem + SL.redi);
  __shared__ float s_gnew;
  __shared__ int s_abort;

  const int n = (int)(a.p < (int64_t)li.budget ? a.p : (int64_t)li.budget);  // rows before append
  const int e_prev = a.pend[head];                                          // dead row or -1
  const int shift = e_prev >= 0 ? 1 : 0;
  const int nphys = n + shift;                                              // stored rows
  const int NR = nphys + 1;                                                 // + the new row
  const bool evict = (n + 1) > li.budget;
  const int ntiles = (nphys + kTile - 1) / kTile;

  __half* Kg = a.K + (li.row_base + (int64_t)rem * li.cap) * D;
  float* scg = a.score + li.meta_base + (int64_t)rem * li.capm;
  float* gg = a.gum + li.meta_base + (int64_t)rem * li.capm;
  int32_t* pg = a.pos + li.meta_base + (int64_t)rem * li.capm;
  const __half* qg = a.k_new + (((int64_t)b * a.L + l) * a.H + hh) * D;

  if (tid == 0) {
    for (int s = 0; s <= kStages; ++s) mbar_init(smem_addr(&bars[s]), 1);
    fence_mbar_init();
    s_abort = 0;
  }
  __syncthreads();

  int issued = 0;  // tiles issued so far (thread 0 only)
  if (tid == 0) {
    if (nphys > 0) {
      const uint32_t mbytes = (uint32_t)(((nphys + 3) & ~3) * 4);
      mbar_expect_tx(smem_addr(&bars[kStages]), 2 * mbytes);
      bulk_g2s(smem_addr(s_sc), scg, mbytes, smem_addr(&bars[kStages]));
      bulk_g2s(smem_addr(s_g), gg, mbytes, smem_addr(&bars[kStages]));
    }
    for (; issued < ntiles && issued < kStages; ++issued) {
      const int rows = min(kTile, nphys - issued * kTile);
      const uint32_t bytes = (uint32_t)rows * G::ROWB;
      const uint32_t bar = smem_addr(&bars[issued % kStages]);
      mbar_expect_tx(bar, bytes);
      bulk_g2s(smem_addr(ring + (size_t)(issued % kStages) * G::TILEB),
               Kg + (size_t)issued * kTile * D, bytes, bar);
    }
  }

  // The proxy query (the new key) and the shift-by-one RoPE constants this
  // thread's pair indices need, kept in registers for the whole pass.
  const Chunk q_lo = *reinterpret_cast<const Chunk*>(qg + c * CH);
  const Chunk q_hi = *reinterpret_cast<const Chunk*>(qg + HALF + c * CH);
  float qa[CH], qb[CH], rc[CH], rs[CH];
  unpack<CH>(q_lo, qa);
  unpack<CH>(q_hi, qb);
#pragma unroll
  for (int k = 0; k < CH; ++k) {
    rc[k] = a.rope_c[c * CH + k];
    rs[k] = a.rope_s[c * CH + k];
  }
  if (tid == 32) s_gnew = gumbel_at(a.seed, l, hh, a.p);
  if (tid < 32) {  // logit of the new row against itself
    float d = 0.f;
#pragma unroll
    for (int k = 0; k < CH; ++k) d = fmaf(qa[k], qa[k], fmaf(qb[k], qb[k], d));
    d += __shfl_xor_sync(0xffffffffu, d, 1);
    d += __shfl_xor_sync(0xffffffffu, d, 2);
    d += __shfl_xor_sync(0xffffffffu, d, 4);
    if (tid == 0) s_log[nphys] = d * a.scale;
  }

  // ---------------------------------------------------------------- stream K
  bool abort = false;
  int t = 0;
  for (; t < ntiles; ++t) {
    const int st = t % kStages;
    const bool ok = mbar_wait_bounded(smem_addr(&bars[st]), (uint32_t)((t / kStages) & 1));
    if (__syncthreads_or(!ok)) { abort = true; break; }
    const unsigned char* tile = ring + (size_t)st * G::TILEB;
    const int r0 = t * kTile;
#pragma unroll
    for (int pass = 0; pass < kTile / kRowsPerPass; ++pass) {
      const int rr = pass * kRowsPerPass + rg;
      const int R = r0 + rr;
      const bool live = (R < nphys) && (R != e_prev);
      float dot = 0.f;
      if (live) {
        const unsigned char* row = tile + (size_t)rr * G::ROWB;
        Chunk lo = *reinterpret_cast<const Chunk*>(row + c * CH * 2);
        Chunk hi = *reinterpret_cast<const Chunk*>(row + (HALF + c * CH) * 2);
        float fa[CH], fb[CH];
        unpack<CH>(lo, fa);
        unpack<CH>(hi, fb);
        if (shift && R > e_prev) {   // apply last step's compaction to this row
          rotate_pairs<CH>(fa, fb, rc, rs);
          lo = pack<CH>(fa);
          hi = pack<CH>(fb);
          unpack<CH>(lo, fa);         // the stored fp16 values are what gets scored
          unpack<CH>(hi, fb);
          __half* dst = Kg + (size_t)(R - 1) * D;
          *reinterpret_cast<Chunk*>(dst + c * CH) = lo;
          *reinterpret_cast<Chunk*>(dst + HALF + c * CH) = hi;
        }
        float d0 = 0.f, d1 = 0.f;
#pragma unroll
        for (int k = 0; k < CH; ++k) {
          d0 = fmaf(fa[k], qa[k], d0);
          d1 = fmaf(fb[k], qb[k], d1);
        }
        dot = d0 + d1;
      }
      dot += __shfl_xor_sync(0xffffffffu, dot, 1);
      dot += __shfl_xor_sync(0xffffffffu, dot, 2);
      dot += __shfl_xor_sync(0xffffffffu, dot, 4);
      if (live && c == 0) s_log[R] = dot * a.scale;
    }
    __syncthreads();  // every thread is done with stage st
    if (tid == 0 && issued < ntiles) {
      const int rows = min(kTile, nphys - issued * kTile);
      const uint32_t bytes = (uint32_t)rows * G::ROWB;
      const uint32_t bar = smem_addr(&bars[issued % kStages]);
      mbar_expect_tx(bar, bytes);
      bulk_g2s(smem_addr(ring + (size_t)(issued % kStages) * G::TILEB),
               Kg + (size_t)issued * kTile * D, bytes, bar);
      ++issued;
    }
  }
  if (!abort && nphys > 0) {
    const bool ok = mbar_wait_bounded(smem_addr(&bars[kStages]), 0);
    if (__syncthreads_or(!ok)) abort = true;
  }
  if (abort) {
    // Record the failure, then wait (briefly, bounded) for copies still in flight.
    if (tid == 0) {
      atomicOr(a.err, kErrWaitTimeout);
      for (int u = t; u < issued; ++u)
        (void)mbar_wait_bounded(smem_addr(&bars[u % kStages]), (uint32_t)((u / kStages) & 1),
                                10000000ull);
      if (nphys > 0) (void)mbar_wait_bounded(smem_addr(&bars[kStages]), 0, 10000000ull);
    }
    __syncthreads();
    return;
  }
  __syncthreads();

  // ---------------------------------------------------------------- softmax
  float m = -INFINITY;
  for (int R = tid; R < NR; R += kThreads)
    if (R != e_prev) m = fmaxf(m, s_log[R]);
  m = block_max(m, redf);
  float lsum = 0.f;
  for (int R = tid; R < NR; R += kThreads)
    if (R != e_prev) {
      const float ex = expf(s_log[R] - m);
      s_log[R] = ex;
      lsum += ex;
    }
  lsum = block_sum(lsum, redf);

  // ------------------------------------------------- accumulate + select
  const float gnew = s_gnew;
  float best_r = INFINITY;
  int best_R = INT_MAX;
  for (int R = tid; R < NR; R += kThreads) {
    if (R == e_prev) continue;
    const float old = R < nphys ? s_sc[R] : 0.f;
    const float ns = old + s_log[R] / lsum;
    s_log[R] = ns;
    if (evict && R >= a.n_sink) {
      const float gv = R < nphys ? s_g[R] : gnew;
      const float r = fmaf(a.tau, gv, ns);
      if (r < best_r) { best_r = r; best_R = R; }
    }
  }
  int R_e = -1;
  if (evict) R_e = block_argmin(best_r, best_R, redf, redi);

  // ---------------------------------------------------------------- write back
  for (int R = tid; R < NR; R += kThreads)
    if (R != e_prev) scg[R - ((shift && R > e_prev) ? 1 : 0)] = s_log[R];
  if (shift) {
    for (int R = e_prev + 1 + tid; R < nphys; R += kThreads) gg[R - 1] = s_g[R];
    for (int base = e_prev + 1; base < nphys; base += kThreads) {
      const int R = base + tid;
      const int v = R < nphys ? pg[R] : 0;
      __syncthreads();
      if (R < nphys) pg[R - 1] = v;
    }
  }
  if (R_e != nphys && tid < kTPR) {   // the new key, unless it was evicted itself
    __half* dst = Kg + (size_t)n * D;
    *reinterpret_cast<Chunk*>(dst + c * CH) = q_lo;
    *reinterpret_cast<Chunk*>(dst + HALF + c * CH) = q_hi;
  }
  if (tid == 0) {
    gg[n] = gnew;
    pg[n] = (int32_t)a.p;
    const int e_log = evict ? R_e - ((shift && R_e > e_prev) ? 1 : 0) : -1;
    a.pend[head] = e_log;
    if (a.evicted) a.evicted[((int64_t)b * a.L + l) * a.H + hh] = e_log;
    if (evict && (R_e < a.n_sink || R_e > nphys)) atomicOr(a.err, kErrBadIndex);
  }
}

// Apply a pending compaction: rows after the recorded slot move down one,
// keys re-rotated by -1 position. Read a chunk of rows into registers, barrier,
// write them one slot lower; chunks ascend so no row is overwritten unread.
template <int D>
__global__ void __launch_bounds__(kThreads) flush_kernel(const FlushArgs a) {
  using G = Geo<D>;
  using Chunk = typename G::Chunk;
  constexpr int CH = G::CH, HALF = G::HALF;
  const int head = blockIdx.x;
  const int e = a.pend[head];
  if (e < 0) return;
  const int tid = threadIdx.x, c = tid & (kTPR - 1), rg = tid >> 3;
  const int BH = a.B * a.H;
  const int l = head / BH;
  const int rem = head - l * BH;
  const LayerInfo li = a.layers[l];
  const int n = (int)(a.p < (int64_t)li.budget ? a.p : (int64_t)li.budget);
  const int nphys = n + 1;
  __half* Kg = a.K + (li.row_base + (int64_t)rem * li.cap) * D;
  float* scg = a.score + li.meta_base + (int64_t)rem * li.capm;
  float* gg = a.gum + li.meta_base + (int64_t)rem * li.capm;
  int32_t* pg = a.pos + li.meta_base + (int64_t)rem * li.capm;
  float rc[CH], rs[CH];
#pragma unroll
  for (int k = 0; k < CH; ++k) {
    rc[k] = a.rope_c[c * CH + k];
    rs[k] = a.rope_s[c * CH + k];
  }
  for (int base = e + 1; base < nphys; base += kRowsPerPass) {
    const int R = base + rg;
    const bool live = R < nphys;
    Chunk lo{}, hi{};
    float sv = 0.f, gv = 0.f;
    int pv = 0;
    if (live) {
      lo = *reinterpret_cast<const Chunk*>(Kg + (size_t)R * D + c * CH);
      hi = *reinterpret_cast<const Chunk*>(Kg + (size_t)R * D + HALF + c * CH);
      if (c == 0) { sv = scg[R]; gv = gg[R]; pv = pg[R]; }
    }
    __syncthreads();
    if (live) {
      float fa[CH], fb[CH];
      unpack<CH>(lo, fa);
      unpack<CH>(hi, fb);
      rotate_pairs<CH>(fa, fb, rc, rs);
      __half* dst = Kg + (size_t)(R - 1) * D;
      *reinterpret_cast<Chunk*>(dst + c * CH) = pack<CH>(fa);
      *reinterpret_cast<Chunk*>(dst + HALF + c * CH) = pack<CH>(fb);
      if (c == 0) { scg[R - 1] = sv; gg[R - 1] = gv; pg[R - 1] = pv; }
    }
    __syncthreads();
  }
  if (tid == 0) a.pend[head] = -1;
}

}  // namespace

size_t decode_step_smem(int D, int capm_max) {
  return D == 64 ? decode_layout<64>(capm_max).total : decode_layout<128>(capm_max).total;
}

cudaError_t decode_step_setup(int D, size_t smem) {
  if (D == 64)
    return cudaFuncSetAttribute(decode_step_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  return cudaFuncSetAttribute(decode_step_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

cudaError_t launch_decode_step(const DecodeArgs& a, int D, int heads, size_t smem, cudaStream_t s) {
  if (heads <= 0) return cudaSuccess;
  if (D == 64)
    decode_step_kernel<64><<<heads, kThreads, smem, s>>>(a);
  else
    decode_step_kernel<128><<<heads, kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_flush(const FlushArgs& a, int D, int heads, cudaStream_t s) {
  if (heads <= 0) return cudaSuccess;
  if (D == 64)
    flush_kernel<64><<<heads, kThreads, 0, s>>>(a);
  else
    flush_kernel<128><<<heads, kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace kvx
