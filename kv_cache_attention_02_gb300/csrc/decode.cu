// decode.cu -- the fused decode step (one launch runs a call's steps over
// every row of the cache) and the flush kernel that applies a pending
// compaction.
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
// Design (GB300): one launch runs T decode steps. Persistent CTAs (as many as
// fit, at most one per row) claim (step, row) pairs from a launch-wide
// counter, heaviest layers first within a step; rows are independent, so a
// row's next step starts as soon as its own previous step has been published
// (a per-row release/acquire counter), never waiting for the whole cache to
// finish a step; when there are no more rows than CTAs, each CTA keeps one
// row for all the steps and hands them over internally. In each CTA a
// scheduler warp claims the next row and stages its header, new key and
// Gumbel value in shared memory; a producer warp streams the row's keys
// through a 6-stage shared-memory ring with 1-D TMA bulk copies (16 KB tiles,
// mbarrier completion) and runs on into the next row while eight consumer
// warps finish the current one. 8 threads share a key row (two 16-byte
// chunks each: the pair halves (i, i + D/2) a RoPE rotation needs), so bank
// access is conflict-free without a swizzle and the dot product reduces with
// three shuffles. The compaction decided by the previous step is applied to
// each row as it passes through (rotate, write to slot R-1), so a key row is
// read from HBM once per step and written only if it moves. Softmax max/sum,
// score update and the (r, slot) argmin then run over shared memory.
#include "decode_common.cuh"

#include <cfloat>
#include <climits>
#include <type_traits>

namespace kvx {
namespace {

constexpr int kProducerWarp = kConsumerWarps;     // issues the TMA copies
constexpr int kSchedulerWarp = kConsumerWarps + 1;  // claims rows and stages their inputs
constexpr int kThreads = kConsumers + 64;
constexpr int kStages = 6;
constexpr int kRowQ = 2;                          // the row in work + the one claimed next

// A claimed (step, row) pair as the scheduler warp leaves it in shared memory;
// the new key row (and value row) follow the header.
struct RowHdr {
  int64_t kbase;   // first key row of this head in the arena
  int64_t mbase;   // first metadata entry of this head
  int64_t p;       // absolute position of the incoming key
  int head;        // row index (layer-major), or -1: nothing left to claim
  int t;           // step within the launch
  int n;           // rows kept before the append
  int e_prev;      // row the previous step evicted but left in place, or -1
  int budget;
  int capm;
  float gnew;      // Gumbel value of the incoming key
  float tau;       // tau(p)
};
static_assert(sizeof(RowHdr) == 56, "row header layout");


struct SmemLayout {
  size_t ring, bars, rowq, redf, redi, slog, total;
};

__host__ __device__ inline size_t meta_stride(int capm) { return ((size_t)(capm + 4) * 4 + 127) / 128 * 128; }

template <int D>
__host__ __device__ inline SmemLayout decode_layout(int capm_max) {
  SmemLayout L{};
  size_t o = 0;
  L.ring = o;  o += (size_t)kStages * Geo<D>::TILEB;
  L.bars = o;  o += (size_t)8 * (2 * kStages + 2 * kRowQ);
  o = (o + 127) / 128 * 128;
  L.rowq = o;  o += (size_t)kRowQ * Geo<D>::SLOTB;
  o = (o + 127) / 128 * 128;
  L.redf = o;  o += 64 * 4;
  L.redi = o;  o += 64 * 4;
  L.slog = o;  o += meta_stride(capm_max);
  L.total = o;
  return L;
}

// Tile accounting of one row, computed alike by the producer and the consumers.
struct RowPlan {
  int nphys;     // stored rows (kept rows + the dead one still in place)
  int ntiles;    // key tiles
  int vstart;    // first value row that moves
  int ntot;      // key + value tiles
  int nm;        // metadata tiles (the whole ring when the row is too long to stage)
  int pos0;      // 16-byte aligned start of the moving positions
  bool move_pos;
  bool staged;   // metadata as one ring tile per array
  bool packed;   // all three metadata arrays in one ring tile (at stride meta_stride)
};

template <int D>
__device__ __forceinline__ RowPlan row_plan(const RowHdr& h, bool values) {
  RowPlan P;
  const bool shift = h.e_prev >= 0;
  P.nphys = h.n + (shift ? 1 : 0);
  P.ntiles = (P.nphys + kTile - 1) / kTile;
  P.vstart = h.e_prev + 1;
  const int nvt = (values && shift && P.vstart < P.nphys) ? (P.nphys - P.vstart + kTile - 1) / kTile : 0;
  P.ntot = P.ntiles + nvt;
  P.pos0 = (h.e_prev + 1) & ~3;
  P.move_pos = shift && h.e_prev + 1 < P.nphys;
  P.staged = (size_t)(h.capm + 4) * 4 <= (size_t)Geo<D>::TILEB;
  P.packed = 3 * meta_stride(h.capm) <= (size_t)Geo<D>::TILEB;
  P.nm = P.nphys == 0 ? 0 : P.packed ? 1 : P.staged ? (P.move_pos ? 3 : 2) : kStages;
  return P;
}

// Largest metadata stride the ring can host after the stream (scores, Gumbel
// values and positions: three arrays of capm floats).
template <int D>
__host__ __device__ constexpr int decode_max_capm() {
  return (int)(((size_t)kStages * Geo<D>::TILEB / 3) / 128 * 128 / 4) - 4;
}


__device__ __forceinline__ unsigned long long ld_acquire(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
// A row's published state: steps applied, and the slot its last step evicted
// (left in place for the next step to compact), -1 for none.
__device__ __forceinline__ unsigned long long pack_done(int steps, int e_log) {
  return ((unsigned long long)(unsigned)steps << 32) | (unsigned)(e_log + 1);
}
__device__ __forceinline__ int done_steps(unsigned long long w) { return (int)(w >> 32); }
__device__ __forceinline__ int done_pending(unsigned long long w) { return (int)(unsigned)(w & 0xffffffffull) - 1; }

template <int D>
__global__ void __launch_bounds__(kThreads, 2) decode_step_kernel(const DecodeArgs a) {
  using G = Geo<D>;
  using Chunk = typename G::Chunk;
  constexpr int CH = G::CH, HALF = G::HALF;

  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const SmemLayout SL = decode_layout<D>(a.capm_max);
  unsigned char* ring = smem + SL.ring;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SL.bars);
  unsigned char* rowq = smem + SL.rowq;
  float* s_log = reinterpret_cast<float*>(smem + SL.slog);
  float* redf = reinterpret_cast<float*>(smem + SL.redf);
  int* redi = reinterpret_cast<int*>(smem + SL.redi);
  __shared__ int s_abort;
  auto full = [&](int s) { return smem_addr(&bars[s]); };
  auto empty = [&](int s) { return smem_addr(&bars[kStages + s]); };
  auto rfull = [&](int q) { return smem_addr(&bars[2 * kStages + q]); };
  auto rempty = [&](int q) { return smem_addr(&bars[2 * kStages + kRowQ + q]); };

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), kConsumerWarps);
    }
    for (int q = 0; q < kRowQ; ++q) {
      mbar_init(rfull(q), 32);                    // every scheduler lane
      mbar_init(rempty(q), 1 + kConsumerWarps);   // the producer + each consumer warp
    }
    fence_mbar_init();
    s_abort = 0;
  }
  __syncthreads();
  volatile int* abort_flag = &s_abort;
  const bool values = a.V != nullptr;
  const int BH = a.B * a.H;
  // When every row has its own CTA, CTA r runs all of row r's steps in order
  // and hands each step to the next inside the CTA: the consumers leave the
  // evicted slot in the row slot's spare header word and the scheduler waits
  // on the slot's barrier, instead of the release/acquire step word and the
  // claim counter (a global round trip off each step's chain).
  const bool static_rows = a.rows <= (int)gridDim.x;

  if (warp == kSchedulerWarp) {
    // ------------------------------------------------------- row scheduler
    // Claims (step, row) pairs from the launch-wide counter in order (step by
    // step, heaviest layers first within a step) and stages each one's header,
    // new key and new value one row ahead. A row's step t first waits until
    // the row's step t - 1 has been published (in practice long done: the row
    // was claimed a whole step of the cache earlier).
    const unsigned long long total = (unsigned long long)a.T * (unsigned long long)a.rows;
    for (int seq = 0;; ++seq) {
      const int q = seq % kRowQ;
      if (seq >= kRowQ && !wait_watch(rempty(q), (uint32_t)((seq / kRowQ - 1) & 1), abort_flag, a.err)) break;
      unsigned long long k = 0;
      if (static_rows) {
        k = seq < a.T ? (unsigned long long)seq * a.rows + blockIdx.x : total;
      } else {
        if (lane == 0) {
          k = atomicAdd(a.ticket, 1ull);
          if (k == total + gridDim.x - 1) atomicExch(a.ticket, 0ull);   // the launch's last claim
        }
        k = __shfl_sync(0xffffffffu, k, 0);
      }
      unsigned char* slot = rowq + (size_t)q * G::SLOTB;
      RowHdr* hd = reinterpret_cast<RowHdr*>(slot);
      const bool claimed = k < total;
      bool ready = true;
      if (claimed) {
        const int t = (int)(k / (unsigned long long)a.rows);
        const int row = (int)(k - (unsigned long long)t * a.rows);
        const int l = row / BH;
        const int rem = row - l * BH;
        const int b = rem / a.H;
        const int hh = rem - b * a.H;
        const int64_t src = (int64_t)t * a.k_step + (((int64_t)b * a.L + l) * a.H + hh) * a.k_stride;
        using Word = typename G::Word;   // this lane's share of a new row
        reinterpret_cast<Word*>(slot + 64)[lane] = reinterpret_cast<const Word*>(a.k_new + src)[lane];
        if (values)
          reinterpret_cast<Word*>(slot + 64 + G::ROWB)[lane] = reinterpret_cast<const Word*>(a.v_new + src)[lane];
        if (lane == 0) {
          // What does not depend on the row's previous step is staged before
          // waiting for it (the Gumbel value's fp64 logs are slow on this GPU
          // and would otherwise lengthen each row's step-to-step chain).
          const LayerInfo li = a.layers[l];
          const int64_t p = a.p0 + t;
          hd->kbase = li.row_base + (int64_t)rem * li.cap;
          hd->mbase = li.meta_base + (int64_t)rem * li.capm;
          hd->p = p;
          hd->head = row;
          hd->t = t;
          hd->n = (int)(p < (int64_t)li.budget ? p : (int64_t)li.budget);
          hd->budget = li.budget;
          hd->capm = li.capm;
          hd->gnew = gumbel_at(a.seed, l, hh, p);
          hd->tau = tau_at(a, p);
          // step t of this row needs step t - 1 applied (by whichever CTA ran
          // it); that step's published word also carries the slot it left to
          // compact. A launch's first step takes it from the pending array
          // (written by the previous launch, the prompt, or a flush).
          if (t > 0 && static_rows) {
            // this CTA ran step t - 1 (its sequence number seq - 1): wait for its
            // consumers, who leave the evicted slot in the slot header's spare word
            const int qp = (seq - 1) % kRowQ;
            ready = wait_watch(rempty(qp), (uint32_t)(((seq - 1) / kRowQ) & 1), abort_flag, a.err);
            hd->e_prev = ready ? *reinterpret_cast<volatile int*>(rowq + (size_t)qp * G::SLOTB + 56) : -1;
          } else if (t > 0) {
            unsigned long long w = ld_acquire(a.done + row);
            if (done_steps(w) < a.s0 + t) {
              const uint64_t t0 = global_timer_ns();
              while (done_steps(w = ld_acquire(a.done + row)) < a.s0 + t) {
                if (*abort_flag) { ready = false; break; }
                if (global_timer_ns() - t0 > kWaitLimitNs) {
                  *abort_flag = 1;
                  atomicOr(a.err, kErrWaitTimeout);
                  ready = false;
                  break;
                }
              }
            }
            hd->e_prev = done_pending(w);
          } else {
            hd->e_prev = __ldcg(a.pend + row);
          }
        }
        ready = __shfl_sync(0xffffffffu, ready, 0);
      } else if (lane == 0) {
        hd->head = -1;
      }
      if (!ready) break;   // aborted while waiting: the other roles see the flag
      __syncwarp();
      mbar_arrive_cta(rfull(q));
      if (!claimed) break;
    }
  } else if (warp == kProducerWarp) {
    // ---------------------------------------------------------- TMA producer
    // Tile sequence tg runs across rows: a row's key tiles, its value tiles,
    // then its metadata (scores, Gumbel values, moving positions): one more tile
    // holding all three arrays when they fit, else up to three tiles, or, for
    // rows too long for that, the whole ring.
    if (lane == 0) {
      int tg = 0;
      for (int seq = 0;; ++seq) {
        const int q = seq % kRowQ;
        if (!wait_watch(rfull(q), (uint32_t)((seq / kRowQ) & 1), abort_flag, a.err)) break;
        const RowHdr hd = *reinterpret_cast<const RowHdr*>(rowq + (size_t)q * G::SLOTB);
        mbar_arrive_cta(rempty(q));
        if (hd.head < 0) break;
        const RowPlan P = row_plan<D>(hd, values);
        const __half* Kg = a.K + hd.kbase * D;
        const __half* Vg = values ? a.V + hd.kbase * D : nullptr;
        if (hd.t > 0) fence_proxy_async_global();   // the row's previous step was written in this launch
        bool ok = true;
        for (int t = 0; t < P.ntot; ++t) {
          const int s = tg % kStages;
          if (tg >= kStages && !(ok = wait_watch(empty(s), (uint32_t)((tg / kStages - 1) & 1), abort_flag, a.err)))
            break;
          if (a.stall && blockIdx.x == 0 && seq == 0 && t == 0) {   // test hook: a barrier nothing completes
            ++tg;
            continue;
          }
          const int r0 = t < P.ntiles ? t * kTile : P.vstart + (t - P.ntiles) * kTile;
          const int rows = min(kTile, P.nphys - r0);
          const uint32_t bytes = (uint32_t)rows * G::ROWB;
          mbar_expect_tx(full(s), bytes);
          bulk_g2s(smem_addr(ring + (size_t)s * G::TILEB), (t < P.ntiles ? Kg : Vg) + (size_t)r0 * D, bytes,
                   full(s));
          ++tg;
        }
        if (!ok) break;
        if (P.nm == 0) continue;
        const float* scg = a.score + hd.mbase;
        const float* gg = a.gum + hd.mbase;
        const int32_t* pg = a.pos + hd.mbase;
        const uint32_t mbytes = (uint32_t)(((P.nphys + 3) & ~3) * 4);
        const uint32_t pbytes = P.move_pos ? (uint32_t)(((P.nphys - P.pos0 + 3) & ~3) * 4) : 0u;
        if (P.packed) {   // short rows: all three arrays in one stage, so the row needs fewer ring slots
          const int s = tg % kStages;
          if (tg >= kStages && !(ok = wait_watch(empty(s), (uint32_t)((tg / kStages - 1) & 1), abort_flag, a.err)))
            break;
          const size_t arr = meta_stride(hd.capm);
          unsigned char* st = ring + (size_t)s * G::TILEB;
          mbar_expect_tx(full(s), 2 * mbytes + pbytes);
          bulk_g2s(smem_addr(st), scg, mbytes, full(s));
          bulk_g2s(smem_addr(st + arr), gg, mbytes, full(s));
          if (pbytes) bulk_g2s(smem_addr(st + 2 * arr), pg + P.pos0, pbytes, full(s));
          ++tg;
        } else if (P.staged) {
          for (int k = 0; k < P.nm; ++k) {
            const int s = tg % kStages;
            if (tg >= kStages && !(ok = wait_watch(empty(s), (uint32_t)((tg / kStages - 1) & 1), abort_flag, a.err)))
              break;
            const void* src = k == 0 ? (const void*)scg : k == 1 ? (const void*)gg : (const void*)(pg + P.pos0);
            const uint32_t bytes = k < 2 ? mbytes : pbytes;
            mbar_expect_tx(full(s), bytes);
            bulk_g2s(smem_addr(ring + (size_t)s * G::TILEB), src, bytes, full(s));
            ++tg;
          }
        } else {
          for (int k = 0; k < kStages && ok; ++k) {   // wait until every stage is free
            const int u = tg + k;
            if (u >= kStages)
              ok = wait_watch(empty(u % kStages), (uint32_t)((u / kStages - 1) & 1), abort_flag, a.err);
          }
          if (ok) {
            const size_t arr = meta_stride(hd.capm);
            const int s0 = tg % kStages;
            mbar_expect_tx(full(s0), 2 * mbytes + pbytes);
            bulk_g2s(smem_addr(ring), scg, mbytes, full(s0));
            bulk_g2s(smem_addr(ring + arr), gg, mbytes, full(s0));
            if (pbytes) bulk_g2s(smem_addr(ring + 2 * arr), pg + P.pos0, pbytes, full(s0));
            for (int k = 1; k < kStages; ++k) mbar_arrive_cta(full((tg + k) % kStages));
            tg += kStages;
          }
        }
        if (!ok) break;
      }
      // no copy may still be landing in shared memory when the CTA leaves
      for (int u = tg > kStages ? tg - kStages : 0; u < tg; ++u)
        (void)mbar_wait_bounded(full(u % kStages), (uint32_t)((u / kStages) & 1), 10000000ull);
    }
  } else {
    // ---------------------------------------------------------- consumers
    const int c = tid & (kTPR - 1);   // chunk index within a row
    const int rg = tid >> 3;          // row within a pass
    // shift-by-one RoPE constants of this thread's pair indices, for every row
    float2 rc[CH / 2], rs[CH / 2];
#pragma unroll
    for (int k = 0; k < CH / 2; ++k) {
      rc[k] = make_float2(a.rope_c[c * CH + 2 * k], a.rope_c[c * CH + 2 * k + 1]);
      rs[k] = make_float2(a.rope_s[c * CH + 2 * k], a.rope_s[c * CH + 2 * k + 1]);
    }
    int tg = 0;
    for (int seq = 0;; ++seq) {
      const int q = seq % kRowQ;
      const bool got = wait_watch(rfull(q), (uint32_t)((seq / kRowQ) & 1), abort_flag, a.err);
      if (consumers_any(!got || *abort_flag)) break;
      const unsigned char* slot = rowq + (size_t)q * G::SLOTB;
      const RowHdr hd = *reinterpret_cast<const RowHdr*>(slot);
      if (hd.head < 0) break;
      const RowPlan P = row_plan<D>(hd, values);
      // the proxy query (the new key) stays in registers for the whole row
      const unsigned char* qs = slot + 64;
      const Chunk q_lo = *reinterpret_cast<const Chunk*>(qs + c * CH * 2);
      const Chunk q_hi = *reinterpret_cast<const Chunk*>(qs + (HALF + c * CH) * 2);
      Chunk v_lo{}, v_hi{};
      if (values && tid < kTPR) {
        v_lo = *reinterpret_cast<const Chunk*>(qs + G::ROWB + c * CH * 2);
        v_hi = *reinterpret_cast<const Chunk*>(qs + G::ROWB + (HALF + c * CH) * 2);
      }
      const int n = hd.n, e_prev = hd.e_prev, nphys = P.nphys, NR = nphys + 1;
      const bool shift = e_prev >= 0;
      const bool evict = (n + 1) > hd.budget;
      __half* Kg = a.K + hd.kbase * D;
      __half* Vg = values ? a.V + hd.kbase * D : nullptr;
      float* scg = a.score + hd.mbase;
      float* gg = a.gum + hd.mbase;
      int32_t* pg = a.pos + hd.mbase;
      const size_t arr = meta_stride(hd.capm);
      const int um = tg + P.ntot;   // first metadata tile
      const unsigned char* mtile = ring + (size_t)(um % kStages) * G::TILEB;   // the packed form's tile
      const float* s_sc = reinterpret_cast<const float*>(P.packed ? mtile : P.staged ? ring + (size_t)(um % kStages) * G::TILEB : ring);
      const float* s_g =
          reinterpret_cast<const float*>(P.packed ? mtile + arr : P.staged ? ring + (size_t)((um + 1) % kStages) * G::TILEB : ring + arr);
      const int32_t* s_pos =
          reinterpret_cast<const int32_t*>(P.packed ? mtile + 2 * arr : P.staged ? ring + (size_t)((um + 2) % kStages) * G::TILEB : ring + 2 * arr);

      float run_m = -INFINITY;   // the largest logit this thread wrote
      if (tid < 32) {   // logit of the new row against itself
        float d = dot_chunks<CH>(q_lo, q_hi, q_lo, q_hi);
        d += __shfl_xor_sync(0xffffffffu, d, 1);
        d += __shfl_xor_sync(0xffffffffu, d, 2);
        d += __shfl_xor_sync(0xffffffffu, d, 4);
        if (tid == 0) {
          s_log[nphys] = d * a.scale2;
          run_m = d * a.scale2;
        }
      }
      for (int t = 0; t < P.ntiles; ++t) {
        const int u = tg + t;
        const int st = u % kStages;
        if (!wait_watch(full(st), (uint32_t)((u / kStages) & 1), abort_flag, a.err)) break;
        const unsigned char* tile = ring + (size_t)st * G::TILEB;
        const int r0 = t * kTile;
        constexpr int PR = kTile / kRowsPerPass;   // rows per thread in this tile
        Chunk lo[PR], hi[PR];
        bool live[PR];
        int Rr[PR];
#pragma unroll
        for (int pass = 0; pass < PR; ++pass) {     // both rows' loads first
          const int rr = pass * kRowsPerPass + rg;
          Rr[pass] = r0 + rr;
          live[pass] = (Rr[pass] < nphys) && (Rr[pass] != e_prev);
          const unsigned char* row = tile + (size_t)rr * G::ROWB;
          lo[pass] = *reinterpret_cast<const Chunk*>(row + c * CH * 2);
          hi[pass] = *reinterpret_cast<const Chunk*>(row + (HALF + c * CH) * 2);
        }
        float dot[PR];
#pragma unroll
        for (int pass = 0; pass < PR; ++pass) {
          if (live[pass] && shift && Rr[pass] > e_prev) {   // apply last step's compaction
            float2 fa[CH / 2], fb[CH / 2];
            unpack2<CH>(lo[pass], fa);
            unpack2<CH>(hi[pass], fb);
            rotate2<CH>(fa, fb, rc, rs);
            lo[pass] = pack2<CH>(fa);                      // the stored fp16 values are scored
            hi[pass] = pack2<CH>(fb);
            __half* dst = Kg + (size_t)(Rr[pass] - 1) * D;
            *reinterpret_cast<Chunk*>(dst + c * CH) = lo[pass];
            *reinterpret_cast<Chunk*>(dst + HALF + c * CH) = hi[pass];
          }
          dot[pass] = live[pass] ? dot_chunks<CH>(lo[pass], hi[pass], q_lo, q_hi) : 0.f;
        }
        static_assert(PR == 2, "the reduce-scatter below pairs two rows per thread");
        {
          // reduce-scatter over the 8 threads of a row group: after the first
          // exchange even threads carry row 0's partial sums and odd ones row
          // 1's; two more rounds finish both (the association is the plain
          // butterfly's, so the sums are the same)
          const bool odd = (c & 1) != 0;
          float mine = odd ? dot[1] : dot[0];
          mine += __shfl_xor_sync(0xffffffffu, odd ? dot[0] : dot[1], 1);
          mine += __shfl_xor_sync(0xffffffffu, mine, 2);
          mine += __shfl_xor_sync(0xffffffffu, mine, 4);
          const bool lv = odd ? live[1] : live[0];
          const int Rw = odd ? Rr[1] : Rr[0];
          if (lv && c < 2) {
            const float sv = mine * a.scale2;   // base-2 logit
            s_log[Rw] = sv;
            run_m = fmaxf(run_m, sv);
          }
        }
        // Hand the stage back only after the arithmetic has consumed every
        // value loaded from it: the TMA refill this permits is an async-proxy
        // write ordered only through the barrier, so loads still in flight
        // could read the next tile's bytes.
        __syncwarp();
        if (lane == 0) mbar_arrive_cta(empty(st));
      }
      for (int t = P.ntiles; t < P.ntot && !*abort_flag; ++t) {   // value rows: move down one slot
        const int u = tg + t;
        const int st = u % kStages;
        if (!wait_watch(full(st), (uint32_t)((u / kStages) & 1), abort_flag, a.err)) break;
        const unsigned char* tile = ring + (size_t)st * G::TILEB;
        const int r0 = P.vstart + (t - P.ntiles) * kTile;
#pragma unroll
        for (int pass = 0; pass < kTile / kRowsPerPass; ++pass) {
          const int rr = pass * kRowsPerPass + rg;
          const int R = r0 + rr;
          if (R < nphys) {
            const unsigned char* row = tile + (size_t)rr * G::ROWB;
            __half* dst = Vg + (size_t)(R - 1) * D;
            *reinterpret_cast<Chunk*>(dst + c * CH) = *reinterpret_cast<const Chunk*>(row + c * CH * 2);
            *reinterpret_cast<Chunk*>(dst + HALF + c * CH) =
                *reinterpret_cast<const Chunk*>(row + (HALF + c * CH) * 2);
          }
        }
        __syncwarp();   // the stores above have consumed the loaded values
        if (lane == 0) mbar_arrive_cta(empty(st));
      }
      for (int k = 0; k < P.nm && !*abort_flag; ++k)   // the metadata
        if (!wait_watch(full((um + k) % kStages), (uint32_t)(((um + k) / kStages) & 1), abort_flag, a.err)) break;
      if (consumers_any(*abort_flag)) break;

      // -------------------------------------------------------------- softmax
      const float m = block_max(run_m, redf);
      const float inv_l = 1.f / block_expsum(s_log, NR, e_prev, m, redf);   // s_log now holds the terms

      // --------------------------- accumulate, write back, select (one pass)
      // Every source is in shared memory, so each row's new score, its moved
      // Gumbel value and position go straight to their (compacted) global slots.
      const float gnew = hd.gnew;
      float best_r = INFINITY;
      int best_R = INT_MAX;
      for (int R = tid; R < NR; R += kConsumers) {
        if (R == e_prev) continue;
        const float attn = s_log[R] * inv_l;
        const float ns = a.mode ? attn : (R < nphys ? s_sc[R] : 0.f) + attn;   // current-step or cumulative
        const bool moved = shift && R > e_prev;
        const int j = R - (moved ? 1 : 0);                                     // slot after compaction
        scg[j] = ns;
        if (moved && R < nphys) {
          gg[j] = s_g[R];
          pg[j] = s_pos[R - P.pos0];
        }
        if (evict && R >= a.n_sink && j < n + 1 - a.recent) {
          const float gv = R < nphys ? s_g[R] : gnew;
          const float r = fmaf(hd.tau, gv, ns);
          if (r < best_r) { best_r = r; best_R = R; }
        }
      }
      int R_e = -1;
      if (evict) R_e = block_argmin(best_r, best_R, redf, redi);

      if (R_e != nphys && tid < kTPR) {   // the new key (and value), unless it was evicted itself
        __half* dst = Kg + (size_t)n * D;
        *reinterpret_cast<Chunk*>(dst + c * CH) = q_lo;
        *reinterpret_cast<Chunk*>(dst + HALF + c * CH) = q_hi;
        if (Vg) {
          __half* vd = Vg + (size_t)n * D;
          *reinterpret_cast<Chunk*>(vd + c * CH) = v_lo;
          *reinterpret_cast<Chunk*>(vd + HALF + c * CH) = v_hi;
        }
      }
      // the slot this step evicts, numbered after the previous compaction; -1 within budget
      const int e_log = evict ? R_e - ((shift && R_e > e_prev) ? 1 : 0) : -1;
      if (tid == 0) {
        const int head = hd.head;
        gg[n] = gnew;
        pg[n] = (int32_t)hd.p;
        a.pend[head] = e_log;
        if (a.evicted) {
          const int l = head / BH;
          const int rem = head - l * BH;
          const int b = rem / a.H;
          a.evicted[hd.t * a.ev_step + ((int64_t)b * a.L + l) * a.H + (rem - b * a.H)] = e_log;
        }
        if (evict && (R_e < a.n_sink || R_e > nphys || e_log >= n + 1 - a.recent)) atomicOr(a.err, kErrBadIndex);
      }
      // every consumer is done with s_log, the metadata and the reduction
      // scratch, and every write of this row's step has been issued: publish
      // the step (its count and the slot it leaves to compact, one word), free
      // the metadata stages and the row's slot. The named
      // barrier orders every consumer's writes before thread 0's release (the
      // barrier synchronises at CTA scope, and a release is cumulative over
      // what precedes it in causality order), so no separate fence is needed
      // for a CTA that acquires the counter to see them.
      if (static_rows) {
        // this CTA's producer reads these rows with TMA at the row's next step:
        // each writer orders its generic-proxy writes before those async-proxy
        // reads (the producer fences again before issuing them)
        fence_proxy_async_global();
        if (tid == 0) *reinterpret_cast<volatile int*>(const_cast<unsigned char*>(slot) + 56) = e_log;
      }
      consumers_sync();
      if (tid == 0 && !static_rows) st_release(a.done + hd.head, pack_done(a.s0 + hd.t + 1, e_log));
      if (lane == 0) {
        for (int k = 0; k < P.nm; ++k) mbar_arrive_cta(empty((um + k) % kStages));
        mbar_arrive_cta(rempty(q));
      }
      tg = um + P.nm;
    }
  }
}

// Apply a pending compaction: rows after the recorded slot move down one,
// keys re-rotated by -1 position. Read a chunk of rows into registers, barrier,
// write them one slot lower; chunks ascend so no row is overwritten unread.
template <int D>
__global__ void __launch_bounds__(kConsumers) flush_kernel(const FlushArgs a) {
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
  __half* Vg = a.V ? a.V + (li.row_base + (int64_t)rem * li.cap) * D : nullptr;
  float* scg = a.score + li.meta_base + (int64_t)rem * li.capm;
  float* gg = a.gum + li.meta_base + (int64_t)rem * li.capm;
  int32_t* pg = a.pos + li.meta_base + (int64_t)rem * li.capm;
  float2 rc[CH / 2], rs[CH / 2];
#pragma unroll
  for (int k = 0; k < CH / 2; ++k) {
    rc[k] = make_float2(a.rope_c[c * CH + 2 * k], a.rope_c[c * CH + 2 * k + 1]);
    rs[k] = make_float2(a.rope_s[c * CH + 2 * k], a.rope_s[c * CH + 2 * k + 1]);
  }
  for (int base = e + 1; base < nphys; base += kRowsPerPass) {
    const int R = base + rg;
    const bool live = R < nphys;
    Chunk lo{}, hi{}, vlo{}, vhi{};
    float sv = 0.f, gv = 0.f;
    int pv = 0;
    if (live) {
      lo = *reinterpret_cast<const Chunk*>(Kg + (size_t)R * D + c * CH);
      hi = *reinterpret_cast<const Chunk*>(Kg + (size_t)R * D + HALF + c * CH);
      if (Vg) {
        vlo = *reinterpret_cast<const Chunk*>(Vg + (size_t)R * D + c * CH);
        vhi = *reinterpret_cast<const Chunk*>(Vg + (size_t)R * D + HALF + c * CH);
      }
      if (c == 0) { sv = scg[R]; gv = gg[R]; pv = pg[R]; }
    }
    __syncthreads();
    if (live) {
      float2 fa[CH / 2], fb[CH / 2];
      unpack2<CH>(lo, fa);
      unpack2<CH>(hi, fb);
      rotate2<CH>(fa, fb, rc, rs);
      __half* dst = Kg + (size_t)(R - 1) * D;
      *reinterpret_cast<Chunk*>(dst + c * CH) = pack2<CH>(fa);
      *reinterpret_cast<Chunk*>(dst + HALF + c * CH) = pack2<CH>(fb);
      if (c == 0) { scg[R - 1] = sv; gg[R - 1] = gv; pg[R - 1] = pv; }
      if (Vg) {
        __half* vd = Vg + (size_t)(R - 1) * D;
        *reinterpret_cast<Chunk*>(vd + c * CH) = vlo;
        *reinterpret_cast<Chunk*>(vd + HALF + c * CH) = vhi;
      }
    }
    __syncthreads();
  }
  if (tid == 0) a.pend[head] = -1;
}

}  // namespace

size_t decode_step_smem(int D, int capm_max) {
  const int lim = D == 64 ? decode_max_capm<64>() : decode_max_capm<128>();
  if (capm_max > lim) return (size_t)-1;   // the ring cannot host this row's metadata
  return D == 64 ? decode_layout<64>(capm_max).total : decode_layout<128>(capm_max).total;
}

cudaError_t decode_step_setup(int D, size_t smem) {
  if (D == 64)
    return cudaFuncSetAttribute(decode_step_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  return cudaFuncSetAttribute(decode_step_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

cudaError_t decode_step_ctas_per_sm(int D, size_t smem, int* ctas) {
  if (D == 64)
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas, decode_step_kernel<64>, kThreads, smem);
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas, decode_step_kernel<128>, kThreads, smem);
}

cudaError_t launch_decode_step(const DecodeArgs& a, int D, int grid, size_t smem, cudaStream_t s) {
  if (a.rows <= 0 || grid <= 0) return cudaSuccess;
  if (D == 64)
    decode_step_kernel<64><<<grid, kThreads, smem, s>>>(a);
  else
    decode_step_kernel<128><<<grid, kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_flush(const FlushArgs& a, int D, int heads, cudaStream_t s) {
  if (heads <= 0) return cudaSuccess;
  if (D == 64)
    flush_kernel<64><<<heads, kConsumers, 0, s>>>(a);
  else
    flush_kernel<128><<<heads, kConsumers, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace kvx
