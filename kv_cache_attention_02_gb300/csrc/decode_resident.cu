// decode_resident.cu -- the decode step with each cache row held in shared
// memory for a whole multi-step call.
//
// It computes exactly what decode_step_kernel computes (page
// "veloxquant_mlx.quantizers.keyformer module", keyformer_update steps 1-3;
// page "PyramidKV -- Layer-Adaptive Budget Attention-Mass Eviction", "How it
// works"): per step, append the new key, softmax(K k / sqrt(D)) over every
// row including the new one, scores += attn (or = attn, current-step mode),
// and over budget evict the lowest score + tau * gumbel among the rows that
// are neither sinks nor in the recent window (lowest slot on ties); the rows
// after it move down one slot, keys re-rotated by -1 position in fp32.
//
// Design (GB300): when a row's keys and metadata fit in one CTA's shared
// memory and a call runs several steps, one CTA takes one row for every step
// of the call. It loads the row once (a 1-D TMA bulk copy of its keys), runs
// the T steps out of shared memory, and writes the row back once, so a step
// costs no HBM or L2 round trip: the few-row shapes, whose steps are a chain
// of such round trips in the streaming kernel, run at the speed of one SM's
// shared memory instead. A helper warp runs ahead of the step: it reads the
// next steps' keys (several in flight), computes their frozen Gumbel values
// (fp64 logs, eight steps at once on eight lanes) and temperatures, and hands
// them over through a ring of shared-memory slots. The eight consumer warps
// keep the physical key rows in place and a logical-slot -> physical-row map:
// an eviction shifts the map and the per-slot scores, Gumbel values and
// positions (a few words per row), the evicted row's storage takes the next
// step's new key, and every row that moved is re-rotated in place by the
// threads that read it in the next step's dot products (the deferred
// compaction of the streaming kernel, without the move). The call ends by
// writing the row back in the arena's layout, with the last step's
// compaction left pending exactly as the streaming kernel leaves it.
//
// Rows are independent, so a grid with more rows than fit on the GPU at once
// runs in waves; nothing waits across CTAs.
#include "decode_common.cuh"

namespace kvx {
namespace {

// NW consumer warps (8, or 16 when a row's shared memory leaves room for one
// CTA an SM only) and one helper warp that stages each step's inputs.
template <int NW>
struct Res {
  static constexpr int NT = NW * 32;           // consumer threads
  static constexpr int HELPER = NW;            // the helper's warp index
  static constexpr int THREADS = NT + 32;
  static constexpr int RPP = NT / kTPR;        // rows per pass (8 threads a row)
};
constexpr int kQ = 16;                        // input slots (steps the helper may run ahead)
constexpr int kGroup = 8;                     // steps the helper prepares at once
constexpr int kResidentMaxCap = 1024;         // rows a CTA holds

// One step's inputs as the helper leaves them in a slot; the new key follows.
struct StepIn {
  int64_t p;    // absolute position of the incoming key
  float gnew;   // its frozen Gumbel value
  float tau;    // tau(p)
};
static_assert(sizeof(StepIn) == 16, "step input header");

struct ResLayout {
  size_t keys, meta, logit, rope, queue, bars, redf, redi, total;
  size_t arr_stride;   // words between consecutive slot arrays
};

template <int D>
__host__ __device__ inline size_t res_slot_bytes() { return sizeof(StepIn) + (size_t)D * 2; }

// cap: physical key rows (the largest budget + 1, rounded up to 4)
template <int D>
__host__ __device__ inline ResLayout resident_layout(int cap) {
  ResLayout L{};
  const size_t c4 = ((size_t)cap + 3) / 4 * 4;
  size_t o = 0;
  L.arr_stride = c4;
  L.keys = o;  o += c4 * D * 2;
  // two copies of the four slot arrays (score, Gumbel value, position,
  // physical row), each copy the four arrays back to back
  L.meta = o;  o += 2 * 4 * c4 * 4;
  L.logit = o; o += (c4 + 4) * 4;
  o = (o + 15) / 16 * 16;
  L.rope = o;  o += (size_t)D * 4;   // cos then sin of the shift by -1, D/2 each
  L.queue = o; o += (size_t)kQ * res_slot_bytes<D>();
  o = (o + 7) / 8 * 8;
  L.bars = o;  o += (size_t)8 * (2 * kQ + 1);
  L.redf = o;  o += 64 * 4;
  L.redi = o;  o += 64 * 4;
  L.total = o;
  return L;
}

// With 8 consumer warps two CTAs (18 warps) fit on an SM at up to 96 registers
// a thread; at 104 the register file of the SM sub-partition holding a CTA's
// ninth warp runs out. With 16 (17 warps, one CTA an SM) 96 registers keep the
// busiest sub-partition's five warps within its share.
template <int D, int NW>
__global__ void __launch_bounds__(Res<NW>::THREADS, NW == 8 ? 2 : 1) resident_step_kernel(const DecodeArgs a) {
  using RC = Res<NW>;
  constexpr int NT = RC::NT, RPP = RC::RPP;
  using G = Geo<D>;
  using Chunk = typename G::Chunk;
  using Word = typename G::Word;
  constexpr int CH = G::CH, HALF = G::HALF, ROWB = G::ROWB;

  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const ResLayout SL = resident_layout<D>(a.capm_max);
  __half* Ks = reinterpret_cast<__half*>(smem + SL.keys);
  float* lg = reinterpret_cast<float*>(smem + SL.logit);
  unsigned char* queue = smem + SL.queue;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SL.bars);
  float* redf = reinterpret_cast<float*>(smem + SL.redf);
  int* redi = reinterpret_cast<int*>(smem + SL.redi);
  __shared__ int s_abort;
  auto kfull = [&](int q) { return smem_addr(&bars[q]); };
  auto kempty = [&](int q) { return smem_addr(&bars[kQ + q]); };
  const uint32_t loaded = smem_addr(&bars[2 * kQ]);

  if (tid == 0) {
    for (int q = 0; q < kQ; ++q) {
      mbar_init(kfull(q), 32);               // every helper lane
      mbar_init(kempty(q), NW);  // each consumer warp
    }
    mbar_init(loaded, 1);
    fence_mbar_init();
    s_abort = 0;
  }
  __syncthreads();
  volatile int* abort_flag = &s_abort;

  const int row = blockIdx.x;   // layer-major cache row
  const int BH = a.B * a.H;
  const int l = row / BH;
  const int rem = row - l * BH;
  const int b = rem / a.H;
  const int hh = rem - b * a.H;
  const LayerInfo li = a.layers[l];
  const int budget = li.budget;
  const int64_t in_off = (((int64_t)b * a.L + l) * a.H + hh);

  if (warp == RC::HELPER) {
    // ------------------------------------------------------------ helper
    // Eight steps at a time: their keys are read together (eight loads in
    // flight per lane) and lanes 0..7 take one step's Gumbel value each.
    for (int t0 = 0; t0 < a.T; t0 += kGroup) {
      const int cnt = min(kGroup, a.T - t0);
      Word w[kGroup];
#pragma unroll
      for (int u = 0; u < kGroup; ++u)
        if (u < cnt)
          w[u] = reinterpret_cast<const Word*>(a.k_new + (int64_t)(t0 + u) * a.k_step + in_off * a.k_stride)[lane];
      float gv = 0.f, tv = 0.f;
      if (lane < cnt) {
        gv = gumbel_at(a.seed, l, hh, a.p0 + t0 + lane);
        tv = tau_at(a, a.p0 + t0 + lane);
      }
      bool ok = true;
#pragma unroll
      for (int u = 0; u < kGroup; ++u) {
        const float g_u = __shfl_sync(0xffffffffu, gv, u);
        const float t_u = __shfl_sync(0xffffffffu, tv, u);
        if (u >= cnt || !ok) continue;
        const int t = t0 + u;
        const int q = t % kQ;
        if (t >= kQ) ok = wait_watch(kempty(q), (uint32_t)((t / kQ - 1) & 1), abort_flag, a.err);
        ok = __all_sync(0xffffffffu, ok);   // the lanes leave together
        if (!ok) continue;
        unsigned char* slot = queue + (size_t)q * res_slot_bytes<D>();
        reinterpret_cast<Word*>(slot + sizeof(StepIn))[lane] = w[u];
        if (lane == 0) {
          StepIn* si = reinterpret_cast<StepIn*>(slot);
          si->p = a.p0 + t;
          si->gnew = g_u;
          si->tau = t_u;
        }
        __syncwarp();
        mbar_arrive_cta(kfull(q));
      }
      if (!ok) break;
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int c = tid & (kTPR - 1);   // chunk index within a row
  const int rg = tid >> 3;          // row within a pass
  // the row in the arena (recomputed where used, to keep registers free)
  auto arena_keys = [&]() { return a.K + (li.row_base + (int64_t)rem * li.cap) * D; };
  auto arena_meta = [&]() { return li.meta_base + (int64_t)rem * li.capm; };

  // The per-slot arrays are double-buffered: a step reads one copy and writes
  // the other, so the compaction needs no barrier between its reads and writes.
  // Copy `cur` holds, at word offsets 0, c4, 2 c4, 3 c4: scores, Gumbel values,
  // positions and the physical row of each logical slot.
  const int c4 = (int)SL.arr_stride;
  uint32_t* meta0 = reinterpret_cast<uint32_t*>(smem + SL.meta);
  int cur = 0;
  auto sc_at = [&](int j) -> float& { return reinterpret_cast<float*>(meta0)[cur + j]; };
  auto gm_at = [&](int j) -> float& { return reinterpret_cast<float*>(meta0)[cur + c4 + j]; };
  auto ps_at = [&](int j) -> int& { return reinterpret_cast<int*>(meta0)[cur + 2 * c4 + j]; };
  auto pm_at = [&](int j) -> int& { return reinterpret_cast<int*>(meta0)[cur + 3 * c4 + j]; };

  // the row as the arena holds it: n kept rows, plus the slot e0 the last
  // step evicted and left in place (rows after it not yet moved or rotated)
  int n = (int)(a.p0 < (int64_t)budget ? a.p0 : (int64_t)budget);
  const int e0 = __ldcg(a.pend + row);
  const int nphys0 = n + (e0 >= 0 ? 1 : 0);
  if (tid == 0) {
    const bool stall = a.stall && blockIdx.x == 0;   // test hook: a barrier nothing completes
    const uint32_t lo_rows = (uint32_t)(e0 >= 0 ? e0 : nphys0);
    const uint32_t hi_rows = (uint32_t)(e0 >= 0 ? nphys0 - e0 - 1 : 0);
    const uint32_t bytes = (lo_rows + hi_rows) * ROWB;
    if (!stall) {   // one arrival, completing once the copies' bytes have landed
      mbar_expect_tx(loaded, bytes);
      const __half* Kg = arena_keys();
      if (lo_rows) bulk_g2s(smem_addr(Ks), Kg, lo_rows * ROWB, loaded);
      if (hi_rows) bulk_g2s(smem_addr(Ks + (size_t)e0 * D), Kg + (size_t)(e0 + 1) * D, hi_rows * ROWB, loaded);
    }
  }
  {
    const int64_t mb = arena_meta();
    for (int j = tid; j < n; j += NT) {
      const int src = (e0 >= 0 && j >= e0) ? j + 1 : j;
      sc_at(j) = a.score[mb + src];
      gm_at(j) = a.gum[mb + src];
      ps_at(j) = a.pos[mb + src];
      pm_at(j) = j;
    }
  }
  // shift-by-one RoPE constants, read from shared memory where a row moved
  // (registers are the resident step's scarcest resource)
  float* rope_s_c = reinterpret_cast<float*>(smem + SL.rope);
  for (int i = tid; i < D; i += NT) rope_s_c[i] = i < HALF ? a.rope_c[i] : a.rope_s[i - HALF];
  bool got = wait_watch(loaded, 0, abort_flag, a.err);
  if (got && a.T > 0) got = wait_watch(kfull(0), 0, abort_flag, a.err);
  bool aborted = consumers_any<NT>(!got || *abort_flag);   // also publishes the slot arrays

  int e_prev = e0;     // physical slot the last step evicted (left in place), or -1
  int fr = n;          // the physical row the next new key goes to
  int t = 0;
  for (; t < a.T && !aborted; ++t) {
    const int q = t % kQ;
    const unsigned char* slot = queue + (size_t)q * res_slot_bytes<D>();
    const StepIn si = *reinterpret_cast<const StepIn*>(slot);
    const unsigned char* qs = slot + sizeof(StepIn);
    const Chunk q_lo = *reinterpret_cast<const Chunk*>(qs + c * CH * 2);
    const Chunk q_hi = *reinterpret_cast<const Chunk*>(qs + (HALF + c * CH) * 2);
    __syncwarp();
    if (lane == 0) mbar_arrive_cta(kempty(q));   // the slot's contents are in registers
    if (tid < kTPR) {                            // the new key's storage for the coming steps
      __half* dst = Ks + (size_t)fr * D;
      *reinterpret_cast<Chunk*>(dst + c * CH) = q_lo;
      *reinterpret_cast<Chunk*>(dst + HALF + c * CH) = q_hi;
    }
    // Rows are visited in the streaming kernel's numbering: "physical" index R
    // runs over the kept rows with the slot the last step evicted still in
    // place (dead, skipped) and the new row last, and every row's logit is
    // summed, and accumulated into the softmax statistics, by the same thread
    // in the same order as there, so the two kernels agree bit for bit.
    const bool shift = e_prev >= 0;
    const int nphys = n + (shift ? 1 : 0);
    const int NR = nphys + 1;
    const bool evict = n + 1 > budget;

    // ------------------------------------------------ logits (and pending rotations)
    float run_m = -INFINITY;   // the largest logit this thread wrote
    if (tid < 32) {   // the new row against itself
      float d = dot_chunks<CH>(q_lo, q_hi, q_lo, q_hi);
      d += __shfl_xor_sync(0xffffffffu, d, 1);
      d += __shfl_xor_sync(0xffffffffu, d, 2);
      d += __shfl_xor_sync(0xffffffffu, d, 4);
      if (tid == 0) {
        lg[nphys] = d * a.scale2;
        run_m = d * a.scale2;
      }
    }
    // Four rows per thread per round: R = r0 + 32u + rg, u = 0..3. Which thread
    // writes a logit does not matter: the softmax statistics are a block max and
    // a sum in a fixed row order (block_max, block_expsum).
    for (int r0 = 0; r0 < nphys; r0 += 4 * RPP) {
      Chunk lo[4], hi[4];
      bool live[4];
      int Rr[4], ph[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        Rr[u] = r0 + u * RPP + rg;
        live[u] = Rr[u] < nphys && Rr[u] != e_prev;
        ph[u] = live[u] ? pm_at((shift && Rr[u] > e_prev) ? Rr[u] - 1 : Rr[u]) : 0;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {   // every row's loads before any arithmetic
        const __half* src = Ks + (size_t)ph[u] * D;
        lo[u] = *reinterpret_cast<const Chunk*>(src + c * CH);
        hi[u] = *reinterpret_cast<const Chunk*>(src + HALF + c * CH);
      }
      float dot[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (live[u] && shift && Rr[u] > e_prev) {   // moved last step: re-rotate in place
          // one half2 pair at a time (the same operations, in the same order, as
          // unpack2 + rotate2 + pack2), so few values are live at once
          __half2* la = reinterpret_cast<__half2*>(&lo[u]);
          __half2* hb = reinterpret_cast<__half2*>(&hi[u]);
#pragma unroll
          for (int k = 0; k < CH / 2; ++k) {
            float2 fa = __half22float2(la[k]), fb = __half22float2(hb[k]);
            const float2 rc = *reinterpret_cast<const float2*>(rope_s_c + c * CH + 2 * k);
            const float2 rs = *reinterpret_cast<const float2*>(rope_s_c + HALF + c * CH + 2 * k);
            rotate2<2>(&fa, &fb, &rc, &rs);
            la[k] = __float22half2_rn(fa);
            hb[k] = __float22half2_rn(fb);
          }
          __half* dst = Ks + (size_t)ph[u] * D;
          *reinterpret_cast<Chunk*>(dst + c * CH) = lo[u];
          *reinterpret_cast<Chunk*>(dst + HALF + c * CH) = hi[u];
        }
        dot[u] = live[u] ? dot_chunks<CH>(lo[u], hi[u], q_lo, q_hi) : 0.f;
      }
      {
        // Reduce-scatter of the four rows' partial sums over the 8 threads of a
        // row group, with the streaming kernel's association ((c, c^1), then
        // (c, c^2), then (c, c^4)), so each logit is bit for bit the one the
        // streaming kernel computes: after the first exchange even threads hold
        // rows 0 and 2, odd threads rows 1 and 3; after the second, thread c
        // holds row (c & 1) + 2 ((c >> 1) & 1), and threads 0..3 write one each.
        const bool odd = (c & 1) != 0;
        const bool b1 = (c & 2) != 0;
        const float p0 = (odd ? dot[1] : dot[0]) + __shfl_xor_sync(0xffffffffu, odd ? dot[0] : dot[1], 1);
        const float p1 = (odd ? dot[3] : dot[2]) + __shfl_xor_sync(0xffffffffu, odd ? dot[2] : dot[3], 1);
        float mine = (b1 ? p1 : p0) + __shfl_xor_sync(0xffffffffu, b1 ? p0 : p1, 2);
        mine += __shfl_xor_sync(0xffffffffu, mine, 4);
        if (c < 4) {   // thread c holds row u = (c & 1) + 2 ((c >> 1) & 1)
          const int u = (c & 1) + 2 * ((c >> 1) & 1);
          const bool lv = u == 0 ? live[0] : u == 1 ? live[1] : u == 2 ? live[2] : live[3];
          if (lv) {
            const float sv = mine * a.scale2;   // base-2 logit
            lg[r0 + u * RPP + rg] = sv;
            run_m = fmaxf(run_m, sv);
          }
        }
      }
    }

    // ------------------------------------------------ softmax, scores, selection
    const float m = block_max<NT>(run_m, redf);
    const float inv_l = 1.f / block_expsum<NT>(lg, NR, e_prev, m, redf);   // lg now holds the terms
    float best_r = INFINITY;
    int best_R = INT_MAX;
    for (int R0 = tid; R0 < NR; R0 += 2 * NT) {   // two rows per thread per round
      float ns[2], rr[2];
      bool ok[2], cand[2];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int R = R0 + k * NT;
        ok[k] = R < NR && R != e_prev;
        const int j = (shift && R > e_prev) ? R - 1 : R;   // logical slot (the new row: n)
        const float lgv = ok[k] ? lg[R] : 0.f;
        const float old = (ok[k] && j < n) ? sc_at(j) : 0.f;
        const float gv = (ok[k] && j < n) ? gm_at(j) : si.gnew;
        const float attn = lgv * inv_l;
        ns[k] = a.mode ? attn : old + attn;   // current-step or cumulative
        cand[k] = ok[k] && evict && R >= a.n_sink && j < n + 1 - a.recent;
        rr[k] = fmaf(si.tau, gv, ns[k]);
      }
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int R = R0 + k * NT;
        if (ok[k]) lg[R] = ns[k];
        if (cand[k] && rr[k] < best_r) { best_r = rr[k]; best_R = R; }
      }
    }
    int e = -1;   // the evicted slot, numbered over the n + 1 rows after the append
    if (evict) {
      const int R_e = block_argmin<NT>(best_r, best_R, redf, redi);   // its barrier also publishes lg
      e = (shift && R_e > e_prev) ? R_e - 1 : R_e;
    } else {
      consumers_sync<NT>();
    }
    if (tid == 0) {
      if (a.evicted) a.evicted[(int64_t)t * a.ev_step + in_off] = e;
      if (evict && (e < a.n_sink || e >= n + 1 - a.recent)) atomicOr(a.err, kErrBadIndex);
    }

    // ------------------------------------------------ compaction of the slot arrays
    // Slot j of the kept rows takes logical slot src = j (+1 from the evicted
    // slot on) of the rows after the append; written to the other copy.
    const int NK = evict ? n : n + 1;
    const int fr_next = !evict ? n + 1 : (e < n ? pm_at(e) : fr);
    const int nxt = cur ^ (4 * c4);   // the other copy
    for (int j = tid; j < NK; j += NT) {
      const int src = (evict && j >= e) ? j + 1 : j;
      const bool old = src < n;
      reinterpret_cast<float*>(meta0)[nxt + j] = lg[(shift && src >= e_prev) ? src + 1 : src];
      reinterpret_cast<float*>(meta0)[nxt + c4 + j] = old ? gm_at(src) : si.gnew;
      reinterpret_cast<int*>(meta0)[nxt + 2 * c4 + j] = old ? ps_at(src) : (int)si.p;
      reinterpret_cast<int*>(meta0)[nxt + 3 * c4 + j] = old ? pm_at(src) : fr;
    }
    cur = nxt;
    fr = fr_next;
    n = NK;
    e_prev = evict ? e : -1;
    // the next step's inputs, and the barrier that publishes this step's
    // slot arrays (and frees lg and the reduction scratch) before it
    got = true;
    if (t + 1 < a.T) got = wait_watch(kfull((t + 1) % kQ), (uint32_t)(((t + 1) / kQ) & 1), abort_flag, a.err);
    aborted = consumers_any<NT>(!got || *abort_flag);
  }

  if (aborted) {
    if (tid == 0) (void)mbar_wait_bounded(loaded, 0, 10000000ull);   // no copy may still be landing
    return;
  }

  // ------------------------------------------------------------ write-back
  // The arena's layout after a step: the slot the last step evicted stays in
  // place, dead, and the rows after it keep their slots and their
  // un-re-rotated keys; the next step (or a flush) applies that compaction.
  const int gshift = e_prev;   // -1: nothing pending
  __half* Kg = arena_keys();
  for (int j0 = 0; j0 < n; j0 += RPP) {
    const int j = j0 + rg;
    if (j < n) {
      const int gs = (gshift >= 0 && j >= gshift) ? j + 1 : j;
      const __half* src = Ks + (size_t)pm_at(j) * D;
      __half* dst = Kg + (size_t)gs * D;
      *reinterpret_cast<Chunk*>(dst + c * CH) = *reinterpret_cast<const Chunk*>(src + c * CH);
      *reinterpret_cast<Chunk*>(dst + HALF + c * CH) = *reinterpret_cast<const Chunk*>(src + HALF + c * CH);
    }
  }
  const int64_t mb = arena_meta();
  for (int j = tid; j < n; j += NT) {
    const int gs = (gshift >= 0 && j >= gshift) ? j + 1 : j;
    a.score[mb + gs] = sc_at(j);
    a.gum[mb + gs] = gm_at(j);
    a.pos[mb + gs] = ps_at(j);
  }
  if (tid == 0) {
    a.pend[row] = gshift;
    a.done[row] = ((unsigned long long)(unsigned)(a.s0 + a.T) << 32) | (unsigned)(gshift + 1);
  }
}

}  // namespace

size_t resident_step_smem(int D, int capm_max) {
  if (capm_max > kResidentMaxCap) return (size_t)-1;
  return D == 64 ? resident_layout<64>(capm_max).total : resident_layout<128>(capm_max).total;
}

namespace {
template <int D, int NW>
cudaError_t resident_setup_one(size_t smem, int* ctas) {
  cudaError_t e = cudaFuncSetAttribute(resident_step_kernel<D, NW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas, resident_step_kernel<D, NW>, Res<NW>::THREADS, smem);
  return e;
}
}  // namespace

cudaError_t resident_step_setup(int D, size_t smem, int* ctas8, int* ctas16) {
  cudaError_t e = D == 64 ? resident_setup_one<64, 8>(smem, ctas8) : resident_setup_one<128, 8>(smem, ctas8);
  if (e == cudaSuccess)
    e = D == 64 ? resident_setup_one<64, 16>(smem, ctas16) : resident_setup_one<128, 16>(smem, ctas16);
  return e;
}

cudaError_t launch_resident_step(const DecodeArgs& a, int D, int warps, size_t smem, cudaStream_t s) {
  if (a.rows <= 0 || a.T <= 0) return cudaSuccess;
  if (warps == 16) {
    if (D == 64)
      resident_step_kernel<64, 16><<<a.rows, Res<16>::THREADS, smem, s>>>(a);
    else
      resident_step_kernel<128, 16><<<a.rows, Res<16>::THREADS, smem, s>>>(a);
  } else {
    if (D == 64)
      resident_step_kernel<64, 8><<<a.rows, Res<8>::THREADS, smem, s>>>(a);
    else
      resident_step_kernel<128, 8><<<a.rows, Res<8>::THREADS, smem, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace kvx
