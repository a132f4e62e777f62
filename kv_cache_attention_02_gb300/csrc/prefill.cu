// prefill.cu -- prompt scoring and bulk eviction.
//
// Scoring: the column sums of the causal softmax(K K^T / sqrt(D)), the
// diagonal included -- exactly what the prompt's S tokens would accumulate as
// S decode steps without eviction (page "veloxquant_mlx.quantizers.keyformer
// module", keyformer_update: "For each of the S incoming tokens", steps 1-2).
// Two passes over 64x64 tiles of S = K K^T on the tensor cores:
//   pass 1: per row i, the base-2 log-sum-exp over columns j <= i;
//   pass 2: per column j, sum over rows i >= j of exp2(S_ij*log2e/sqrt(D) - lse2_i).
// Pass 2 computes the transposed tile (rows = j, columns = i), so each thread
// accumulates its own columns' sums in registers with no cross-thread traffic.
//
// Bulk eviction (reading: the whole prompt is scored first, then the S - b
// non-sink rows with the lowest (score + tau(S-1) * gumbel, slot) go at once):
// one CTA per cache row sorts (r, slot) keys in shared memory, scans the
// survivors' new slots and writes them, each key re-rotated by
// (new slot - old slot) RoPE positions in fp32 and stored as fp16.
#include "kvevict_internal.cuh"

#include <cfloat>

namespace kvx {
namespace {

// ---------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void ldmatrix_x4(uint32_t* r, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void mma_16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

constexpr int kBM = 64;        // tile rows
constexpr int kPThreads = 128; // 4 warps x 16 rows

template <int D>
struct PGeo {
  static constexpr int ROWB = D * 2;
  static constexpr int CHR = D / 8;         // 16-byte chunks per row
  static constexpr int TILEB = kBM * ROWB;
  static constexpr int KS = D / 16;         // k-steps of 16
};

// Swizzled shared-memory offset of (row, 16-byte chunk): chunk ^ (row & 7), so
// eight consecutive rows at one chunk index hit eight different bank groups.
__device__ __forceinline__ uint32_t swz(int row, int ch, int rowb) {
  return (uint32_t)(row * rowb + ((ch ^ (row & 7)) << 4));
}

template <int D>
__device__ __forceinline__ void load_tile(uint32_t base, const __half* src, int r0, int S) {
  using G = PGeo<D>;
  for (int idx = threadIdx.x; idx < kBM * G::CHR; idx += kPThreads) {
    const int row = idx / G::CHR, ch = idx - row * G::CHR;
    const int gr = r0 + row;
    const bool ok = gr < S;
    const __half* p = src + (size_t)(ok ? gr : 0) * D + ch * 8;
    cp_async16(base + swz(row, ch, G::ROWB), p, ok ? 16 : 0);
  }
}

// COLSUM = false: pass 1 (row lse2). COLSUM = true: pass 2 (column sums).
template <int D, bool COLSUM>
__global__ void __launch_bounds__(kPThreads) prefill_score_kernel(const PrefillScoreArgs a) {
  using G = PGeo<D>;
  extern __shared__ __align__(128) unsigned char smem[];
  const uint32_t sA = smem_addr(smem);
  const uint32_t sB0 = sA + G::TILEB;
  float* s_lse = reinterpret_cast<float*>(smem + 3 * G::TILEB);  // [2][64]

  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int g = lane >> 2, c4 = lane & 3;
  const int S = a.S;
  const int nb = (S + kBM - 1) / kBM;
  // one flat grid, head-major: a head's causal blocks run together and share
  // its keys through L2; within a head the heaviest block goes first
  const int head = (int)(blockIdx.x / (unsigned)nb);
  const int bidx = (int)(blockIdx.x - (unsigned)head * (unsigned)nb);
  const __half* Kh = a.keys + (size_t)head * S * D;
  const float* lse_h = a.lse2 + (size_t)head * a.Sp;

  // pass 1: this CTA owns rows ia (query block), visits column blocks 0..ia
  // pass 2: this CTA owns rows ja (key block, transposed), visits row blocks ja..nb-1
  const int ablk = COLSUM ? bidx : nb - 1 - bidx;
  const int first = COLSUM ? ablk : 0;
  const int last = COLSUM ? nb - 1 : ablk;
  const int nblk = last - first + 1;

  load_tile<D>(sA, Kh, ablk * kBM, S);
  cp_async_commit();
  load_tile<D>(sB0, Kh, first * kBM, S);
  if (COLSUM && tid < 16) cp_async16(smem_addr(s_lse) + tid * 16, lse_h + first * kBM + tid * 4, 16);
  cp_async_commit();

  uint32_t af[G::KS][4];
  float run_m[2] = {-INFINITY, -INFINITY}, run_l[2] = {0.f, 0.f};  // pass 1
  float csum[2] = {0.f, 0.f};                                        // pass 2
  const int rowA0 = ablk * kBM + w * 16 + g;                          // rows g and g+8

  for (int k = 0; k < nblk; ++k) {
    const int bblk = first + k;
    if (k + 1 < nblk) {
      const uint32_t dst = sB0 + ((k + 1) & 1) * G::TILEB;
      load_tile<D>(dst, Kh, (bblk + 1) * kBM, S);
      if (COLSUM && tid < 16)
        cp_async16(smem_addr(s_lse + ((k + 1) & 1) * kBM) + tid * 16,
                   lse_h + (bblk + 1) * kBM + tid * 4, 16);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    if (k == 0) {
#pragma unroll
      for (int ks = 0; ks < G::KS; ++ks) {
        const int row = w * 16 + (lane & 15), ch = ks * 2 + (lane >> 4);
        ldmatrix_x4(af[ks], sA + swz(row, ch, G::ROWB));
      }
    }
    const uint32_t sB = sB0 + (k & 1) * G::TILEB;
    float acc[8][4];
#pragma unroll
    for (int nf = 0; nf < 8; ++nf) acc[nf][0] = acc[nf][1] = acc[nf][2] = acc[nf][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < G::KS; ++ks) {
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        uint32_t bf[4];
        const int row = np * 16 + (lane & 7) + ((lane >> 4) << 3);
        const int ch = ks * 2 + ((lane >> 3) & 1);
        ldmatrix_x4(bf, sB + swz(row, ch, G::ROWB));
        mma_16816(acc[2 * np], af[ks], bf[0], bf[1]);
        mma_16816(acc[2 * np + 1], af[ks], bf[2], bf[3]);
      }
    }
    const int colB0 = bblk * kBM;
    if (!COLSUM) {
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int i = rowA0 + hr * 8;
        float bm = -INFINITY;
        float v[16];
#pragma unroll
        for (int nf = 0; nf < 8; ++nf)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int j = colB0 + nf * 8 + 2 * c4 + e;
            const float s = acc[nf][hr * 2 + e] * a.scale2;
            v[nf * 2 + e] = (j <= i && j < S) ? s : -INFINITY;
            bm = fmaxf(bm, v[nf * 2 + e]);
          }
        const float mn = fmaxf(run_m[hr], bm);
        if (mn != -INFINITY) {
          float sum = 0.f;
#pragma unroll
          for (int t = 0; t < 16; ++t) sum += exp2f(v[t] - mn);
          run_l[hr] = run_l[hr] * exp2f(run_m[hr] - mn) + sum;
          run_m[hr] = mn;
        }
      }
    } else {
      const float* lse_t = s_lse + (k & 1) * kBM;
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int j = rowA0 + hr * 8;
        float sum = 0.f;
#pragma unroll
        for (int nf = 0; nf < 8; ++nf)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int cl = nf * 8 + 2 * c4 + e;
            const int i = colB0 + cl;
            const float p = exp2f(acc[nf][hr * 2 + e] * a.scale2 - lse_t[cl]);
            sum += (i >= j && i < S) ? p : 0.f;
          }
        csum[hr] += sum;
      }
    }
    __syncthreads();
  }

  // combine the four threads that share a row
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    const int row = rowA0 + hr * 8;
    if (!COLSUM) {
      float m = run_m[hr], l = run_l[hr];
#pragma unroll
      for (int o = 1; o <= 2; o <<= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
        const float l2 = __shfl_xor_sync(0xffffffffu, l, o);
        const float mn = fmaxf(m, m2);
        l = (m == -INFINITY ? 0.f : l * exp2f(m - mn)) + (m2 == -INFINITY ? 0.f : l2 * exp2f(m2 - mn));
        m = mn;
      }
      if (c4 == 0 && row < S) a.lse2[(size_t)head * a.Sp + row] = m + log2f(l);
    } else {
      float s = csum[hr];
      s += __shfl_xor_sync(0xffffffffu, s, 1);
      s += __shfl_xor_sync(0xffffffffu, s, 2);
      if (c4 == 0 && row < S) a.colsum[(size_t)head * a.Sp + row] = s;
    }
  }
}

// ---------------------------------------------------------------- bulk eviction
constexpr int kSThreads = 1024;

__device__ __forceinline__ uint32_t ordered_bits(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

template <int D>
__global__ void __launch_bounds__(kSThreads) prefill_select_kernel(const PrefillSelectArgs a) {
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
  const __half* src = a.keys + (size_t)hi * S * D;
  const float* col = a.colsum + (size_t)hi * a.Sp;
  float* gs = a.gscr + (size_t)hi * a.Sp;
  const int budget = li.budget;
  const int c = tid & 7;

  for (int j = tid; j < S; j += kSThreads) gs[j] = gumbel_at(a.seed, l, hh, j);
  __syncthreads();

  if (S <= budget) {  // the whole prompt fits: keep every row where it is
    for (int j0 = 0; j0 < S; j0 += kSThreads / 8) {
      const int j = j0 + (tid >> 3);
      if (j < S) {
        const Chunk lo = *reinterpret_cast<const Chunk*>(src + (size_t)j * D + c * CH);
        const Chunk hi2 = *reinterpret_cast<const Chunk*>(src + (size_t)j * D + HALF + c * CH);
        *reinterpret_cast<Chunk*>(Kg + (size_t)j * D + c * CH) = lo;
        *reinterpret_cast<Chunk*>(Kg + (size_t)j * D + HALF + c * CH) = hi2;
        if (c == 0) { scg[j] = col[j]; gg[j] = gs[j]; pg[j] = j; }
      }
    }
    if (tid == 0) a.pend[slot] = -1;
    return;
  }

  const int m = S - a.n_sink;       // evictable rows
  int P2 = 1;
  while (P2 < m) P2 <<= 1;
  uint64_t* keys = reinterpret_cast<uint64_t*>(smem);
  unsigned char* flag = smem + (size_t)P2 * 8;
  int16_t* newslot = reinterpret_cast<int16_t*>(flag + ((S + 15) & ~15));
  int* wsum = reinterpret_cast<int*>(newslot + ((S + 7) & ~7));

  for (int t = tid; t < P2; t += kSThreads) {
    uint64_t key = ~0ull;
    if (t < m) {
      const int j = a.n_sink + t;
      const float r = fmaf(a.tau, gs[j], col[j]);
      key = ((uint64_t)ordered_bits(r) << 32) | (uint32_t)j;
    }
    keys[t] = key;
  }
  for (int j = tid; j < S; j += kSThreads) flag[j] = 0;
  __syncthreads();
  // bitonic sort, ascending by (r, slot)
  for (int k = 2; k <= P2; k <<= 1) {
    for (int jj = k >> 1; jj > 0; jj >>= 1) {
      for (int t = tid; t < P2; t += kSThreads) {
        const int ixj = t ^ jj;
        if (ixj > t) {
          const uint64_t x = keys[t], y = keys[ixj];
          const bool up = (t & k) == 0;
          if ((x > y) == up) { keys[t] = y; keys[ixj] = x; }
        }
      }
      __syncthreads();
    }
  }
  const int n_ev = S - budget;
  for (int t = tid; t < n_ev; t += kSThreads) flag[(uint32_t)keys[t]] = 1;
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
    int v = wsum[lane];
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
  for (int j0 = 0; j0 < S; j0 += kSThreads / 8) {
    const int j = j0 + (tid >> 3);
    if (j < S && !flag[j]) {
      const int ns = newslot[j];
      const int d = j - ns;   // shift back by d positions
      Chunk lo = *reinterpret_cast<const Chunk*>(src + (size_t)j * D + c * CH);
      Chunk hi2 = *reinterpret_cast<const Chunk*>(src + (size_t)j * D + HALF + c * CH);
      if (d > 0) {
        const float* tc = a.rope_c + (size_t)d * HALF + c * CH;
        const float* ts = a.rope_s + (size_t)d * HALF + c * CH;
        __half2* h_lo = reinterpret_cast<__half2*>(&lo);
        __half2* h_hi = reinterpret_cast<__half2*>(&hi2);
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
      *reinterpret_cast<Chunk*>(Kg + (size_t)ns * D + c * CH) = lo;
      *reinterpret_cast<Chunk*>(Kg + (size_t)ns * D + HALF + c * CH) = hi2;
      if (c == 0) { scg[ns] = col[j]; gg[ns] = gs[j]; pg[ns] = j; }
    }
  }
  if (tid == 0) a.pend[slot] = -1;
}

}  // namespace

size_t prefill_select_smem(int S) {
  int P2 = 1;
  while (P2 < S) P2 <<= 1;
  return (size_t)P2 * 8 + ((S + 15) & ~15) + ((S + 7) & ~7) * 2 + 32 * sizeof(int) + 64;
}

size_t prefill_score_smem(int D) { return 3 * (size_t)kBM * D * 2 + 2 * kBM * sizeof(float); }

cudaError_t prefill_setup(int D, int max_prefill) {
  const int score = (int)prefill_score_smem(D);
  const int select = (int)prefill_select_smem(max_prefill > 0 ? max_prefill : 1);
  const auto attr = cudaFuncAttributeMaxDynamicSharedMemorySize;
  cudaError_t e;
  if (D == 64) {
    e = cudaFuncSetAttribute(prefill_score_kernel<64, false>, attr, score);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(prefill_score_kernel<64, true>, attr, score);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(prefill_select_kernel<64>, attr, select);
  } else {
    e = cudaFuncSetAttribute(prefill_score_kernel<128, false>, attr, score);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(prefill_score_kernel<128, true>, attr, score);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(prefill_select_kernel<128>, attr, select);
  }
  return e;
}

cudaError_t prefill_score_setup(int D) {
  const int score = (int)prefill_score_smem(D);
  const auto attr = cudaFuncAttributeMaxDynamicSharedMemorySize;
  cudaError_t e;
  if (D == 64) {
    e = cudaFuncSetAttribute(prefill_score_kernel<64, false>, attr, score);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(prefill_score_kernel<64, true>, attr, score);
  } else {
    e = cudaFuncSetAttribute(prefill_score_kernel<128, false>, attr, score);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(prefill_score_kernel<128, true>, attr, score);
  }
  return e;
}

cudaError_t launch_prefill_scores(const PrefillScoreArgs& a, int D, cudaStream_t s) {
  if (a.S <= 0 || a.heads <= 0) return cudaSuccess;
  const int nb = (a.S + kBM - 1) / kBM;
  const dim3 grid((unsigned)(a.heads * nb));
  const size_t smem = prefill_score_smem(D);
  if (D == 64) {
    prefill_score_kernel<64, false><<<grid, kPThreads, smem, s>>>(a);
    prefill_score_kernel<64, true><<<grid, kPThreads, smem, s>>>(a);
  } else {
    prefill_score_kernel<128, false><<<grid, kPThreads, smem, s>>>(a);
    prefill_score_kernel<128, true><<<grid, kPThreads, smem, s>>>(a);
  }
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
