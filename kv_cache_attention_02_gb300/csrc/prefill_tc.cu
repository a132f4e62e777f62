// prefill_tc.cu -- the prompt scorer on the 5th-generation tensor cores.
//
// Computes, per cache row, the column sums of the causal softmax(K K^T/sqrt(D))
// (diagonal included): what the prompt's S tokens would accumulate as S decode
// steps without eviction (page "veloxquant_mlx.quantizers.keyformer module",
// keyformer_update, "For each of the S incoming tokens", steps 1-2).
//
//   pass 1 (COLSUM = false): work item = (row, 128-query block I); tiles J = 0..I;
//            per query row i: lse2_i = log2 sum_{j<=i} 2^(s_ij), s = K_i.K_j*log2e/sqrt(D)
//   pass 2 (COLSUM = true):  work item = (row, 128-key block J); tiles I = J..nb-1 of
//            the transposed product (TMEM lanes = key j, columns = query i);
//            colsum_j = sum_{i>=j} 2^(s_ij - lse2_i), summed per lane in registers.
//
// Persistent CTAs, two per SM, take work items in row-major order (a row's
// blocks together, so its keys are reused from L2; each row's blocks heaviest
// first) from a launch-wide counter; TMEM, the barriers and the tile ring stay
// live from one item to the next. Roles in a 320-thread CTA:
//   warp 0      one thread claims the items and issues TMA loads (3-D tensor map
//               [heads, S, D], 128-byte swizzle, two 64-element halves per 128-row
//               tile): an item's stationary tile once the previous item's MMAs are
//               done with it, then its streamed tiles into a 2-stage ring;
//   warp 1      allocates 256 TMEM columns (two 128x128 fp32 accumulators, used in
//               turn by the CTA's running tile count) and one thread issues
//               tcgen05.mma (M=128, N=128, K=16, f16 in, f32 out); tcgen05.commit
//               releases the ring stage and publishes the accumulator;
//   warps 2..9  two epilogue warpgroups; warpgroup w takes tiles k = w, w + 2, ...
//               of every item (so a row's result does not depend on which CTA
//               ran it): tcgen05.ld, causal mask on diagonal tiles only, exp2 on
//               the MUFU, online row max/sum (pass 1) or column sums (pass 2); the
//               two combine their per-row results at the end of the item. An
//               accumulator goes back to the MMA issuer as soon as its last 64
//               columns are in registers, before their exponentials run.
// Every mbarrier wait is bounded; on expiry the CTA sets the error word, drains
// and frees its TMEM.
#include "kvevict_internal.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

namespace kvx {
namespace {

constexpr int kTB = 128;           // tile rows (M) and columns (N)
constexpr int kTCThreads = 320;   // TMA warp, MMA warp, two epilogue warpgroups
constexpr int kStagesTC = 2;
constexpr int kTmemCols = 256;     // two 128-column fp32 accumulators

template <int D>
struct TCGeo {
  static constexpr int KH = D / 64;              // 128-byte K-halves per row
  static constexpr int HALFB = kTB * 128;        // one half tile, 16 KB
  static constexpr int TILEB = KH * HALFB;
  static constexpr int KSTEPS = D / 16;
};

struct TCSmem {
  size_t a, b, lse, comb, bars, tmem, total;
};

template <int D>
__host__ __device__ constexpr TCSmem tc_layout() {
  TCSmem L{};
  size_t o = 0;
  L.a = o;    o += TCGeo<D>::TILEB;
  L.b = o;    o += (size_t)kStagesTC * TCGeo<D>::TILEB;
  L.lse = o;  o += 2 * kTB * sizeof(float);
  L.comb = o; o += 2 * 2 * kTB * sizeof(float);   // per item parity: WG 1's (m, l) or sum
  L.bars = o; o += 16 * 8;
  L.tmem = o; o += 16;                            // TMEM base, then the two queued items
  L.total = o + 1024;  // slack to align the tile region to 1024 bytes
  return L;
}

// ---------------------------------------------------------------- tcgen05 / TMA PTX
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of
// 128 bytes, 8-row groups 1024 bytes apart (stride byte offset), descriptor
// version 1. The leading byte offset is unused for swizzled K-major layouts.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)(1024u >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor, kind::f16: f32 accumulator, A and B f16, both
// K-major, N = 128 (N>>3 at bit 17), M = 128 (M>>4 at bit 24).
constexpr uint32_t kIdesc = (1u << 4) | ((uint32_t)(kTB >> 3) << 17) | ((uint32_t)(kTB >> 4) << 24);

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

// 32 consecutive fp32 accumulator columns of this warp's 32 TMEM lanes.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(r[e]);
}

// 64 consecutive fp32 accumulator columns of this warp's 32 TMEM lanes (one
// per thread), waited for before returning.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float* v) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int e = 0; e < 64; ++e) v[e] = __uint_as_float(r[e]);
}

// 2^x on the MUFU (ex2.approx: relative error below 2^-22; subnormal results
// flush to zero, which only drops terms below 2^-126 from a sum of terms <= 1).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Named barriers: 1 + w for the 128 threads of epilogue warpgroup w, 3 for
// both warpgroups (256 threads).
__device__ __forceinline__ void wg_bar(int w) {
  if (w == 0)
    asm volatile("bar.sync 1, 128;" ::: "memory");
  else
    asm volatile("bar.sync 2, 128;" ::: "memory");
}
// Barrier of both epilogue warpgroups (256 threads) that also ORs a predicate.
__device__ __forceinline__ bool epi_any(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 3, 256, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred)
      : "memory");
  return r != 0;
}

// Barrier of warpgroup w that also ORs a predicate across it, so the whole
// warpgroup leaves its loop together.
__device__ __forceinline__ bool wg_any(int w, bool pred) {
  uint32_t r;
  if (w == 0)
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred)
        : "memory");
  else
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 2, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred)
        : "memory");
  return r != 0;
}

// Bounded wait that also watches the CTA's abort flag.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                              int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      *abort_flag = 1;
      if (err) atomicOr(err, kErrWaitTimeout);
      return false;
    }
  }
}


// Two f32 lanes per instruction (sm_100+ packed FP32): the same per-lane
// rounding as fmaf / a + b.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mov.b64 rc, {%6, %7};\n\tfma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

template <int D, bool COLSUM>
__global__ void __launch_bounds__(kTCThreads, 2)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap kmap, const PrefillScoreArgs a) {
  using G = TCGeo<D>;
  constexpr TCSmem SL = tc_layout<D>();
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* smem = smem_raw + (base - raw);
  const uint32_t sA = base + (uint32_t)SL.a;
  const uint32_t sB = base + (uint32_t)SL.b;
  float* lse_s = reinterpret_cast<float*>(smem + SL.lse);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SL.bars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SL.tmem);
  volatile int* item_s = reinterpret_cast<volatile int*>(smem + SL.tmem + 4);   // [2]
  __shared__ int s_abort;
  auto full = [&](int s) { return smem_addr(&bars[s]); };
  auto empty = [&](int s) { return smem_addr(&bars[2 + s]); };
  auto acc_full = [&](int b) { return smem_addr(&bars[4 + b]); };
  auto acc_empty = [&](int b) { return smem_addr(&bars[6 + b]); };
  const uint32_t a_full = smem_addr(&bars[8]);
  const uint32_t drain = smem_addr(&bars[9]);
  const uint32_t a_empty = smem_addr(&bars[10]);
  auto item_full = [&](int q) { return smem_addr(&bars[11 + q]); };
  auto item_empty = [&](int q) { return smem_addr(&bars[13 + q]); };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = a.S;
  const int nb = (S + kTB - 1) / kTB;
  const int total = a.heads * nb;   // work items (row, 128-row block), row-major
  int* work = a.work + (COLSUM ? 1 : 0);
  // Item x: row x / nb, block x % nb taken heaviest first; the CTA keeps one
  // query (pass 1) or key (pass 2) tile and streams the other operand's tiles.
  auto item_geom = [&](int x, int& head, int& ablk, int& first, int& nblk) {
    head = x / nb;
    const int bidx = x - head * nb;
    ablk = COLSUM ? bidx : nb - 1 - bidx;
    first = COLSUM ? ablk : 0;
    nblk = (COLSUM ? nb - 1 : ablk) - first + 1;
  };

  if (tid == 0) {
    for (int s = 0; s < kStagesTC; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(acc_full(b), 1);
      mbar_init(acc_empty(b), 4);
      mbar_init(item_full(b), 1);
      mbar_init(item_empty(b), 2);   // the MMA issuer and the epilogue
    }
    mbar_init(a_full, 1);
    mbar_init(drain, 1);             // abort path only
    mbar_init(a_empty, 1);
    fence_mbar_init();
    s_abort = 0;
  }
  if (warp == 1) tmem_alloc(smem_addr(tmem_slot), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  volatile int* abort_flag = &s_abort;

  if (warp == 0) {
    // ------------------------------------------------------------ scheduler + TMA producer
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&kmap)) : "memory");
      int gb = 0;            // B tiles issued over all items
      int a_issued = 0;      // query/key tiles issued
      for (int it = 0;; ++it) {
        const int q = it & 1;
        if (it >= 2 && !wait_or_abort(item_empty(q), (uint32_t)(((it >> 1) - 1) & 1), abort_flag, a.err))
          break;
        const int x = atomicAdd(work, 1);
        item_s[q] = x < total ? x : -1;
        mbar_arrive(item_full(q));
        if (x >= total) break;
        int head, ablk, first, nblk;
        item_geom(x, head, ablk, first, nblk);
        // the stationary tile, once the previous item's MMAs are done with it;
        // test hook: in pass 1 the CTA that claims item 0 leaves that tile's
        // barrier incomplete
        if (it >= 1 && !wait_or_abort(a_empty, (uint32_t)((it - 1) & 1), abort_flag, a.err)) break;
        if (!(!COLSUM && a.stall && x == 0)) {
          mbar_expect_tx(a_full, G::TILEB);
          for (int kh = 0; kh < G::KH; ++kh)
            tma_load_3d(sA + kh * G::HALFB, &kmap, kh * 64, ablk * kTB, head, a_full);
        }
        a_issued = it + 1;
        bool ok = true;
        for (int k = 0; k < nblk; ++k, ++gb) {
          const int s = gb % kStagesTC;
          if (gb >= kStagesTC &&
              !wait_or_abort(empty(s), (uint32_t)((gb / kStagesTC - 1) & 1), abort_flag, a.err)) {
            ok = false;
            break;
          }
          mbar_expect_tx(full(s), G::TILEB);
          for (int kh = 0; kh < G::KH; ++kh)
            tma_load_3d(sB + s * G::TILEB + kh * G::HALFB, &kmap, kh * 64, (first + k) * kTB, head,
                        full(s));
        }
        if (!ok) break;
      }
      if (*abort_flag) {  // give copies still in flight a moment to land before exit
        if (a_issued > 0) (void)mbar_wait_bounded(a_full, (uint32_t)((a_issued - 1) & 1), 10000000ull);
        for (int k = gb > kStagesTC ? gb - kStagesTC : 0; k < gb; ++k)
          (void)mbar_wait_bounded(full(k % kStagesTC), (uint32_t)((k / kStagesTC) & 1), 10000000ull);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int gb = 0, g = 0;     // B tiles consumed, accumulator tiles issued
      for (int it = 0;; ++it) {
        const int q = it & 1;
        if (!wait_or_abort(item_full(q), (uint32_t)((it >> 1) & 1), abort_flag, a.err)) break;
        const int x = item_s[q];
        mbar_arrive(item_empty(q));
        if (x < 0) break;
        int head, ablk, first, nblk;
        item_geom(x, head, ablk, first, nblk);
        if (!wait_or_abort(a_full, (uint32_t)(it & 1), abort_flag, a.err)) break;
        bool ok = true;
        for (int k = 0; k < nblk; ++k, ++gb, ++g) {
          const int s = gb % kStagesTC, b = g & 1;
          if (!wait_or_abort(full(s), (uint32_t)((gb / kStagesTC) & 1), abort_flag, a.err) ||
              (g >= 2 && !wait_or_abort(acc_empty(b), (uint32_t)((g / 2 - 1) & 1), abort_flag, a.err))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem + (uint32_t)(b * kTB);
#pragma unroll
          for (int kk = 0; kk < G::KSTEPS; ++kk) {
            const uint32_t off = (uint32_t)((kk >> 2) * G::HALFB + (kk & 3) * 32);
            tc_mma(d, sw128_desc(sA + off), sw128_desc(sB + s * G::TILEB + off), kk > 0 ? 1u : 0u);
          }
          tc_commit(empty(s));
          tc_commit(acc_full(b));
        }
        if (!ok) break;
        tc_commit(a_empty);   // the stationary tile is free once these MMAs finish
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue warpgroups
    // Warpgroup wg (warps 2..5: 0, warps 6..9: 1) takes tiles k = wg, wg + 2, ...
    // of every item, whichever accumulator the CTA's running tile count puts
    // them in, so each row's result does not depend on the schedule; the two
    // combine their per-row results at the end of the item. A warp reaches
    // TMEM lanes 32 * (warp % 4) .. + 31.
    // The parity waits on acc_full stay unambiguous because a warpgroup's
    // consecutive tiles of an item use the same accumulator (it has seen that
    // accumulator's previous phase itself) and both warpgroups meet at the end
    // of every item (all earlier phases seen): no wait can be issued while its
    // accumulator is two phases behind. More warpgroups than accumulators would
    // break this and need the waits ordered explicitly.
    const int wg = (warp - 2) >> 2;
    const int q = warp & 3;
    const int r = q * 32 + lane;                  // tile row = TMEM lane
    const int et = tid - 64 - wg * kTB;           // 0..127 within the warpgroup
    float* comb = reinterpret_cast<float*>(smem + SL.comb);
    constexpr int CW = 64;                        // accumulator columns per TMEM read
    int g = 0;                                    // the CTA's tiles before this item
    for (int it = 0;; ++it) {
      const int qi = it & 1;
      const bool got = wait_or_abort(item_full(qi), (uint32_t)((it >> 1) & 1), abort_flag, a.err);
      const int x = got ? item_s[qi] : -1;
      if (epi_any(x < 0)) break;
      int head, ablk, first, nblk;
      item_geom(x, head, ablk, first, nblk);
      const int rowA = ablk * kTB + r;            // query row i (pass 1) / key row j (pass 2)
      float run_m = -INFINITY, run_l = 0.f, csum = 0.f;
      bool aborted = false;
      float* lsb = lse_s + wg * kTB;
      const int tend = first + nblk;
      for (int tb = first + wg, gt = g + wg; tb < tend; tb += 2, gt += 2) {
        const int b = gt & 1;
        const int colB0 = tb * kTB;
        // the tile's 128 query -lse values (0 past S, where the scratch holds no
        // value and the masked -inf products must still give exp2 = +0)
        if (COLSUM) lsb[et] = colB0 + et < S ? -a.lse2[(size_t)head * a.Sp + colB0 + et] : 0.f;
        const bool ok = wait_or_abort(acc_full(b), (uint32_t)((gt >> 1) & 1), abort_flag, a.err);
        if (wg_any(wg, !ok)) {                    // also publishes lsb to the warpgroup
          aborted = true;
          break;
        }
        tc_fence_after();
        const bool full_tile = COLSUM ? (colB0 > ablk * kTB + kTB - 1 && colB0 + kTB <= S)
                                      : (colB0 + kTB - 1 < ablk * kTB && ablk * kTB + kTB <= S);
        // Interior tiles take no mask; the scale rides in one FMA per element
        // (max over the raw dot products: scale2 > 0 keeps the order).
#pragma unroll 1
        for (int c = 0; c < kTB / CW; ++c) {
          float v[CW];
          const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * kTB + c * CW);
          if (CW == 64)
            tmem_ld64(taddr, v);
          else
            tmem_ld32(taddr, v);
          if (c == kTB / CW - 1) {
            // the whole accumulator has reached registers: hand it back to the
            // MMA issuer before the last chunk's exponentials run
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty(b));
          }
          const int c0 = colB0 + c * CW;
          if (!COLSUM) {
            if (!full_tile) {
#pragma unroll
              for (int e = 0; e < CW; ++e) {
                const int j = c0 + e;
                v[e] = (j <= rowA && j < S) ? v[e] : -INFINITY;
              }
            }
            float m8[8];   // independent max chains
#pragma unroll
            for (int e = 0; e < 8; ++e) m8[e] = v[e];
#pragma unroll
            for (int e = 8; e < CW; ++e) m8[e & 7] = fmaxf(m8[e & 7], v[e]);
#pragma unroll
            for (int e = 0; e < 4; ++e) m8[e] = fmaxf(m8[e], m8[e + 4]);
            const float cm = fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3]));
            if (cm != -INFINITY) {
              const float mn = fmaxf(run_m, cm * a.scale2);
              const float nm = -mn;
              const float2 sc2 = make_float2(a.scale2, a.scale2), nm2 = make_float2(nm, nm);
              float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);   // sums of e % 4 = 0, 1 | 2, 3
#pragma unroll
              for (int e = 0; e < CW; e += 4) {
                const float2 t0 = ffma2(make_float2(v[e], v[e + 1]), sc2, nm2);
                const float2 t1 = ffma2(make_float2(v[e + 2], v[e + 3]), sc2, nm2);
                acc0 = fadd2(acc0, make_float2(ex2(t0.x), ex2(t0.y)));
                acc1 = fadd2(acc1, make_float2(ex2(t1.x), ex2(t1.y)));
              }
              run_l = run_l * ex2(run_m - mn) + ((acc0.x + acc0.y) + (acc1.x + acc1.y));
              run_m = mn;
            }
          } else {
            // -lse2 of the chunk's queries, read as 16-byte broadcasts where used
            const float* nlp = lsb + c * CW;
            if (!full_tile) {
              // queries outside i >= j, i < S: -inf, whose exp2 adds +0
#pragma unroll
              for (int e = 0; e < CW; ++e) {
                const int i = c0 + e;
                v[e] = (i >= rowA && i < S) ? v[e] : -INFINITY;
              }
            }
            float s4[4];
            {
              const float2 sc2 = make_float2(a.scale2, a.scale2);
              float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
              for (int e = 0; e < CW; e += 4) {
                const float4 nl = *reinterpret_cast<const float4*>(nlp + e);
                const float2 t0 = ffma2(make_float2(v[e], v[e + 1]), sc2, make_float2(nl.x, nl.y));
                const float2 t1 = ffma2(make_float2(v[e + 2], v[e + 3]), sc2, make_float2(nl.z, nl.w));
                acc0 = fadd2(acc0, make_float2(ex2(t0.x), ex2(t0.y)));
                acc1 = fadd2(acc1, make_float2(ex2(t1.x), ex2(t1.y)));
              }
              s4[0] = acc0.x;
              s4[1] = acc0.y;
              s4[2] = acc1.x;
              s4[3] = acc1.y;
            }
            csum += (s4[0] + s4[1]) + (s4[2] + s4[3]);
          }
        }
        if (COLSUM) wg_bar(wg);                   // lsb free for this warpgroup's next tile
      }
      g += nblk;
      // warpgroup 1 hands its per-row results to warpgroup 0 (buffers alternate
      // by item, so warpgroup 1 may run one item ahead)
      float* cb = comb + qi * 2 * kTB;
      if (wg == 1) {
        cb[r] = COLSUM ? csum : run_m;
        cb[kTB + r] = run_l;
      }
      if (epi_any(aborted || *abort_flag)) break;
      if (tid == 64) mbar_arrive(item_empty(qi));   // every epilogue thread has read the item
      if (wg == 0 && rowA < S) {
        if (COLSUM) {
          a.colsum[(size_t)head * a.Sp + rowA] = csum + cb[r];
        } else {
          const float m2 = cb[r], l2 = cb[kTB + r];
          const float m = fmaxf(run_m, m2);
          const float l = (run_m == -INFINITY ? 0.f : run_l * exp2f(run_m - m)) +
                          (m2 == -INFINITY ? 0.f : l2 * exp2f(m2 - m));
          a.lse2[(size_t)head * a.Sp + rowA] = m + log2f(l);
        }
      }
    }
  }

  // ------------------------------------------------------------------ teardown
  __syncthreads();
  if (*abort_flag && tid == 32) {
    // let any MMA still in flight finish before the accumulators are freed
    tc_commit(drain);
    (void)mbar_wait_bounded(drain, 0, 10000000ull);
  }
  __syncwarp();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

}  // namespace

size_t prefill_tc_smem(int D) { return D == 64 ? tc_layout<64>().total : tc_layout<128>().total; }

cudaError_t prefill_tc_setup(int D) {
  const int smem = (int)prefill_tc_smem(D);
  const auto attr = cudaFuncAttributeMaxDynamicSharedMemorySize;
  cudaError_t e;
  if (D == 64) {
    e = cudaFuncSetAttribute(prefill_tc_kernel<64, false>, attr, smem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(prefill_tc_kernel<64, true>, attr, smem);
  } else {
    e = cudaFuncSetAttribute(prefill_tc_kernel<128, false>, attr, smem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(prefill_tc_kernel<128, true>, attr, smem);
  }
  return e;
}

// Both passes over a.heads rows of S keys; a.Sp must be S rounded up to 128.
cudaError_t launch_prefill_tc(const PrefillScoreArgs& a, int D, int sms, cudaStream_t s) {
  if (a.S <= 0 || a.heads <= 0) return cudaSuccess;
  if (!a.work) return cudaErrorInvalidValue;
  auto enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  // keys as a 3-D tensor [heads, S, D] (rows S_buf apart): box = 64 elements (128 bytes)
  // x 128 rows x 1 row; rows past S read as zeros
  CUtensorMap map;
  const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)a.S, (cuuint64_t)a.heads};
  const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)a.S_buf * D * 2};
  const cuuint32_t box[3] = {64, (cuuint32_t)kTB, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = enc(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<__half*>(a.keys), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  const int64_t items = (int64_t)a.heads * ((a.S + kTB - 1) / kTB);
  const dim3 grid((unsigned)std::min<int64_t>(items, (int64_t)2 * std::max(sms, 1)));   // two CTAs an SM
  const size_t smem = prefill_tc_smem(D);
  const cudaError_t z = cudaMemsetAsync(a.work, 0, 2 * sizeof(int), s);
  if (z != cudaSuccess) return z;
  if (D == 64) {
    prefill_tc_kernel<64, false><<<grid, kTCThreads, smem, s>>>(map, a);
    prefill_tc_kernel<64, true><<<grid, kTCThreads, smem, s>>>(map, a);
  } else {
    prefill_tc_kernel<128, false><<<grid, kTCThreads, smem, s>>>(map, a);
    prefill_tc_kernel<128, true><<<grid, kTCThreads, smem, s>>>(map, a);
  }
  return cudaGetLastError();
}

}  // namespace kvx
