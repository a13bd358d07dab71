// Persistent step kernel: one SPD cycle (or one plain AR step) in one cooperative launch.
//
// One CTA per SM runs a program of phases (SPD summary 方法步骤详情 steps 1-5 for a cycle):
//   GEMV   the grouped GEMV engine over this CTA's share of the phase's weight bytes
//   ATTN   decode attention items (tile, kv head, 64-key chunk), CTA-strided; the producer streams
//          their K/V chunks through the same ring (chunks of earlier cycles before the QKV phase's
//          barrier, the chunks holding this cycle's keys after it)
//   CTRL   verify / accept / rollback / reseed on CTA 0 (the last phase)
// Consecutive phases are separated by a grid barrier of the consumer warps.  The producer warp
// does not take part in the barriers: the weights of every GEMV phase are known when the cycle
// starts (they depend on the control block only, which changes in the last phase), so it streams
// the tensor copies of phase after phase into the shared-memory ring while the consumers wait at a
// barrier; HBM stays busy across phase boundaries and no launch gaps remain inside a cycle.
//
// Grid barrier: count + generation words in global memory; every CTA adds 1 to the count, the last
// one resets it and advances the generation, the others wait (bounded: 2 s of %globaltimer, then
// the error flag is set and the CTA leaves; the producer's bounded waits then run out too).  The
// cooperative launch guarantees that all CTAs are resident.
#include <mutex>

#include "spd_attn.cuh"
#include "spd_ctrl.cuh"
#include "spd_engine.cuh"

namespace spd {

namespace {

using namespace eng;

constexpr int kStepGroups = 36;   // groups of one phase: n target + n+1 draft rows (n <= 16)
constexpr int kStepTiles = 28;    // attention tiles of one phase: n target tiles + ceil((n+1)/2) draft-row tiles
constexpr int kProdWarp = kNCW;       // warp 8: producer (weights and K/V chunks into the ring)
constexpr int kPlanWarp = kNCW + 1;   // warp 9: planner (resolves the next phase)
constexpr int kStepThreads = (kNCW + 2) * 32;
constexpr int kNCT = kNCW * 32;       // consumer threads
constexpr int kStepQT = 2;            // query rows per attention tile of the draft module's rows

struct StepParams {
  EngineCfg cfg;
  const Phase* prog;
  int nphases;
  unsigned* bar;                  // [0] count, [1] generation
  unsigned long long* phase_ns;   // accumulated per-phase time (CTA 0), or null
  int union_bytes;                // tensor-core partials / attention query vectors / control scratch
};

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void red_add_release(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Grid barrier of the 256 consumer threads of every CTA.  One monotonic arrival counter: every
// CTA adds 1 (a release reduction, no round trip) when it arrives; barrier k of a launch is passed
// once the counter reaches (g0 + k + 1) * gridDim.x, where g0 = barriers completed before the
// launch (the counter is zeroed with the control block at prefill and rollback).  Arrival and wait
// are separate so that the next phase can be prepared in between.  Writes before grid_arrive are
// visible to every CTA after grid_wait.
__device__ __forceinline__ void grid_arrive(unsigned* bar) { red_add_release(bar, 1u); }  // thread 0

// Thread 0: bounded wait for the counter to reach `target`.  False if it gave up.
__device__ __forceinline__ bool grid_wait(const unsigned* bar, unsigned target, DevState* st,
                                          uint64_t limit_ns = kWaitLimitNs) {
  if ((int)(ld_acquire(bar) - target) >= 0) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0; (int)(ld_acquire(bar) - target) < 0; ++it) {
    if ((it & 63u) == 63u && globaltimer_ns() - t0 > limit_ns) {
      set_err(st, ERR_TIMEOUT, 70);
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ int qt_of(const Launch& lc) {
  return (lc.kind == LK_PDMROWS || lc.kind == LK_ROWS) ? kStepQT : 1;
}

__device__ __forceinline__ void st_release_cta(int* p, int v) {
  asm volatile("st.release.cta.shared.s32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_acquire_cta(const int* p) {
  int v;
  asm volatile("ld.acquire.cta.shared.s32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)) : "memory");
  return v;
}
// Bounded wait (lane 0 of a warp) for a shared progress counter to reach `v`.
__device__ __forceinline__ bool wait_progress(const int* p, int v, uint64_t limit_ns = kWaitLimitNs) {
  if (ld_acquire_cta(p) >= v) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0; ld_acquire_cta(p) < v; ++it)
    if ((it & 63u) == 63u && globaltimer_ns() - t0 > limit_ns) return false;
  return true;
}

// Self-check of the bounded waits: one thread runs the chosen wait on a condition that nothing
// satisfies (a grid-barrier count that no CTA adds to, an mbarrier nobody arrives on, a progress
// counter nobody advances) with a short limit; each must give up and flag ERR_TIMEOUT.
__global__ void wait_selftest_kernel(DevState* st, unsigned* counter, int which, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int progress;
  if (threadIdx.x != 0) return;
  bool ok = true;
  if (which == 0) {
    ok = grid_wait(counter, ld_acquire(counter) + 1u, st, limit_ns);  // sets the flag itself
  } else if (which == 1) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    ok = mbar_wait_bounded(&bar, 0, limit_ns);
    if (!ok) set_err(st, ERR_TIMEOUT, 71);
  } else {
    progress = 0;
    ok = wait_progress(&progress, 1, limit_ns);
    if (!ok) set_err(st, ERR_TIMEOUT, 72);
  }
}

__device__ __forceinline__ void mbar_arrive_cnt(uint64_t* bar, uint32_t n) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(n) : "memory");
}

// Cooperative 16-byte copy global -> shared by threads [t0, t0 + nthr) of the caller's set.
__device__ __forceinline__ void copy16(void* dst, const void* src, int bytes, int t, int nthr) {
  const uint4* s4 = reinterpret_cast<const uint4*>(src);
  uint4* d4 = reinterpret_cast<uint4*>(dst);
  for (int i = t; i < bytes / 16; i += nthr) d4[i] = s4[i];
}

// Items of one attention phase for this CTA: pass 0 = chunks written in earlier cycles, pass 1 =
// chunks holding this cycle's keys; each list is dealt to the CTAs round robin, each pass padded to
// whole ring stages of `ips` items.
struct AttnPlan {
  int n0, n1;      // this CTA's items of pass 0 and 1
  int q0, q1;      // the same, padded to multiples of ips
  __device__ __forceinline__ int stages(int ips) const { return (q0 + q1) / ips; }
};
__device__ __forceinline__ AttnPlan attn_plan(int n_old, int n_new, int ips) {
  AttnPlan a;
  const int b = blockIdx.x, G = gridDim.x;
  a.n0 = n_old > b ? (n_old - b + G - 1) / G : 0;
  a.n1 = n_new > b ? (n_new - b + G - 1) / G : 0;
  a.q0 = (a.n0 + ips - 1) / ips * ips;
  a.q1 = (a.n1 + ips - 1) / ips * ips;
  return a;
}
// Item at padded position q of this CTA's sequence: pass and index in that pass's list (-1: padding).
__device__ __forceinline__ int attn_item_at(const AttnPlan& a, int q, int& pass) {
  pass = q < a.q0 ? 0 : 1;
  const int k = pass ? q - a.q0 : q;
  if (k >= (pass ? a.n1 : a.n0)) return -1;
  return blockIdx.x + k * gridDim.x;
}

constexpr int kMergeList = 64;  // (tile, kv head) pairs one CTA can hold for its end-of-phase merge

// Consumer warps of an attention phase.  Warp w takes padded positions q = w / wpi + j * (8 / wpi)
// of this CTA's item sequence (ring stage q / ips, slot q % ips); wpi warps share an item (each takes
// every wpi-th query head) and the two warps of a stage release it with 4 arrivals each.  The next
// item's first query is loaded while the current one is computed; tickets are batched per warp
// (one lane per (tile, kv head) touched) and flushed at the end.  A pair whose last ticket a warp
// takes goes on the CTA's merge list (mlist, *mcount); the caller merges the list with all warps
// once every warp is done (attn_merge_list).
template <typename WT, int DPL>
__device__ void attn_consume(const Dims& D, const att::Tile* tb, int nt, const AttnPlan& A, int nst, int ips,
                             int item_bytes, Ring& R, float* qb, int* s_fail, DevState* st, int* mlist,
                             int* mcount) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wpi = 2 / ips;
  const int qh0 = warp % wpi;
  const int qend = nst * ips, qstride = kNCW / wpi;
  int pT = 0, pkh = 0, pc = 0, npend = 0;  // pending tickets: lane i holds entry i
  auto flush = [&]() {
    __threadfence();  // this warp's partials before its tickets
    __syncwarp();
    int last = 0;
    if (lane < npend) {
      const att::Tile& T = tb[pT];
      const int old = atomicAdd(&T.tick[T.tick_off + pkh], pc);
      last = old + pc == T.nch * wpi;
    }
    unsigned mask = __ballot_sync(0xffffffffu, last);
    if (mask) __threadfence();  // the other warps' partials of the (tile, kv head) are visible
    while (mask) {
      const int b = __ffs(mask) - 1;
      mask &= mask - 1;
      const int T_ = __shfl_sync(0xffffffffu, pT, b), kh_ = __shfl_sync(0xffffffffu, pkh, b);
      int slot = 0;
      if (lane == 0) slot = atomicAdd(mcount, 1);
      slot = __shfl_sync(0xffffffffu, slot, 0);
      if (slot < kMergeList) {
        if (lane == 0) mlist[slot] = (T_ << 16) | kh_;
      } else {  // list full: merge here, one query head after the other
        const att::Tile& T = tb[T_];
        for (int qh = 0; qh < T.nq * D.gq; ++qh) att::merge_qh<DPL>(D, T, kh_, qh);
        __syncwarp();
        if (lane == 0) T.tick[T.tick_off + kh_] = 0;
      }
    }
    npend = 0;
  };
  att::Item it{0, 0, 0, 0};
  int g = -1;
  constexpr int HP = att::kHeadsPerPass;
  float qv[HP][DPL];
  auto fetch = [&](int qpos) {  // identity of the item at qpos and its first pass of query heads
    int pass = 0;
    g = qpos < qend ? attn_item_at(A, qpos, pass) : -1;
    if (g >= 0) {
      it = att::item_of_pass(tb, nt, pass, g, att::kWarpCK);
      const int QH = tb[it.T].nq * D.gq;
#pragma unroll
      for (int h = 0; h < HP; ++h)
        if (qh0 + h * wpi < QH) att::load_q<DPL>(D, tb[it.T], it.kh, qh0 + h * wpi, qv[h]);
    }
  };
  fetch(warp / wpi);
  for (int q = warp / wpi; q < qend; q += qstride) {
    const att::Item cur = it;
    const int gcur = g;
    float qc[HP][DPL];
#pragma unroll
    for (int h = 0; h < HP; ++h)
#pragma unroll
      for (int e = 0; e < DPL; ++e) qc[h][e] = qv[h][e];
    fetch(q + qstride);
    const uint32_t ctr = R.ctr + (uint32_t)(q / ips);
    const int s = ctr % kStages;
    bool ok = !(R.failed || *(volatile int*)s_fail);
    if (ok && !mbar_wait_bounded(&R.full[s], (ctr / kStages) & 1)) {
      if (lane == 0) set_err(st, ERR_TIMEOUT, 31);
      *(volatile int*)s_fail = 1;
      ok = false;
    }
    if (ok && gcur >= 0) {
      const unsigned char* slot = R.base + (size_t)s * kStageBytes + (size_t)(q % ips) * item_bytes;
      att::warp_item<WT, DPL>(D, tb[cur.T], cur, reinterpret_cast<const WT*>(slot),
                              reinterpret_cast<const WT*>(slot + item_bytes / 2), qb, qh0, wpi, qc);
      const unsigned hit = __ballot_sync(0xffffffffu, lane < npend && pT == cur.T && pkh == cur.kh);
      if (hit) {
        if (lane == __ffs(hit) - 1) ++pc;
      } else {
        if (lane == npend) { pT = cur.T; pkh = cur.kh; pc = 1; }
        ++npend;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive_cnt(&R.empty[s], kNCW / 2);
    if (npend == 32) flush();
  }
  if (npend > 0 && !*(volatile int*)s_fail) flush();
}

// All consumer warps, after every warp's attn_consume of the phase (named barrier 1 in between):
// merge the CTA's listed pairs, one (pair, query head) per warp at a time, and reset their tickets.
template <int DPL>
__device__ void attn_merge_list(const Dims& D, const att::Tile* tb, const int* mlist, int n) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  n = min(n, kMergeList);
  int u = warp;  // units (pair, query head) in list order; warp w takes units w, w + 8, ...
  for (int i = 0; i < n; ++i) {
    const att::Tile& T = tb[mlist[i] >> 16];
    const int kh = mlist[i] & 0xFFFF;
    const int QH = T.nq * D.gq;
    for (; u < QH; u += kNCW) att::merge_qh<DPL>(D, T, kh, u);
    u -= QH;  // the next pair's query heads continue the warp's turn
    if (lane == 0 && warp == 0) T.tick[T.tick_off + kh] = 0;
  }
}

template <typename WT>
__global__ void __launch_bounds__(kStepThreads, 1) step_kernel(const __grid_constant__ StepParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* ring =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  unsigned char* uni = ring + kStages * kStageBytes;
  GG* gg = reinterpret_cast<GG*>(uni + p.union_bytes);                // 2 tables (phase parity)
  att::Tile* tiles = reinterpret_cast<att::Tile*>(gg + 2 * kStepGroups);  // 2 tables (phase parity)
  LayerW* lw = reinterpret_cast<LayerW*>(  // target layers, then draft layers (16-byte aligned)
      (reinterpret_cast<uintptr_t>(tiles + 2 * kStepTiles) + 15) & ~(uintptr_t)15);

  __shared__ __align__(8) uint64_t full_bar[kStages];
  __shared__ __align__(8) uint64_t empty_bar[kStages];
  __shared__ int s_planned, s_produced;         // last phase resolved (planner) / streamed (producer)
  __shared__ __align__(16) DevState s_sv;        // control block as the cycle starts
  __shared__ __align__(16) Phase s_ph[2];        // descriptors of the phases by parity
  __shared__ int s_ng[2], s_gb[2], s_rb[2], s_ge[2], s_re[2];  // GEMV: groups, this CTA's share
  __shared__ int s_nt[2], s_nold[2], s_nnew[2];                // attention: tiles, item counts
  __shared__ int s_fail, s_abort, s_tok, s_slot;
  __shared__ int s_mlist[kMergeList], s_mcount;  // attention pairs this CTA merges at the phase end
  __shared__ float rstd_s[16 * kMaxMT];
  __shared__ float wpart[kNCW];
  __shared__ Top2 hred[kNCW * 8][2];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const EngineCfg& cfg = p.cfg;
  const Dims& D = cfg.D;
  DevState* st = cfg.B.st;
  constexpr int ESZ = sizeof(WT);
  // one attention item = K and V chunks of kWarpCK keys; ips items per ring stage (at most 2)
  const int item_bytes = 2 * att::kWarpCK * D.hd * ESZ;
  const int ips = kStageBytes / item_bytes >= 2 ? 2 : 1;
  // snapshots: control block, per-layer tables
  copy16(&s_sv, st, sizeof(DevState), tid, kStepThreads);
  copy16(lw, cfg.B.tl, D.L * (int)sizeof(LayerW), tid, kStepThreads);
  if (D.Ls > 0) copy16(lw + D.L, cfg.B.pl, D.Ls * (int)sizeof(LayerW), tid, kStepThreads);
  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], kNCW);
    }
    fence_mbar_init();
    s_planned = -1;
    s_produced = -1;
    s_fail = 0;
    s_abort = 0;
    s_mcount = 0;
  }
  __syncthreads();
  if (s_sv.done || s_sv.err) return;  // every CTA reads the same control block: a uniform decision
  const View vw{&s_sv, lw, lw + D.L};
  Ring R{ring, full_bar, empty_bar, 0u, false};

  if (warp == kPlanWarp) {
    // ------------------------------ planner warp ------------------------------
    // Resolves phase ph+1 (descriptor, groups and this CTA's share, or attention tiles) while the
    // consumers run phase ph; named barrier 4 with the consumers at every phase boundary.  Tables
    // alternate by phase parity: those of phase ph are rewritten for ph+2 once the consumers have
    // finished ph (barrier 4) and the producer has streamed it (s_produced).
    auto plan = [&](int ph) {
      const int b = ph & 1;
      int ok = 1;
      if (lane == 0 && ph >= 2 && !wait_progress(&s_produced, ph - 2)) {
        set_err(st, ERR_TIMEOUT, 44);
        ok = 0;
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) {  // the producer is gone: the consumers stop waiting
        if (lane == 0) { s_abort = 1; st_release_cta(&s_planned, ph); }
        __syncwarp();
        return;
      }
      copy16(&s_ph[b], p.prog + ph, sizeof(Phase), lane, 32);
      __syncwarp();
      if (lane == 0) {
        const Phase& P = s_ph[b];
        if (P.type == PH_GEMV) {
          s_ng[b] = resolve_parts(cfg, P.part, P.nparts, gg + b * kStepGroups, kStepGroups, vw);
          span_of(gg + b * kStepGroups, s_ng[b], blockIdx.x, gridDim.x, s_gb[b], s_rb[b], s_ge[b], s_re[b]);
        } else if (P.type == PH_ATTN) {
          att::Tile* tb = tiles + b * kStepTiles;
          int nt = 0, items = 0;
          for (int i = 0; i < P.nparts && nt >= 0; ++i)
            nt = att::add_tiles(D, cfg.B, P.part[i].lc, qt_of(P.part[i].lc), att::kWarpCK, tb, nt, &items,
                                kStepTiles, &s_sv);
          if (nt < 0) nt = 0;
          s_nt[b] = nt;
          att::split_items(D, tb, nt, att::kWarpCK, &s_nold[b], &s_nnew[b]);
        }
        st_release_cta(&s_planned, ph);  // releases the tables to the producer
      }
      __syncwarp();
    };
    plan(0);
    named_bar(4, kNCT + 32);
    for (int ph = 0; ph + 1 < p.nphases; ++ph) {
      plan(ph + 1);
      named_bar(4, kNCT + 32);
    }
    return;
  }

  if (warp == kProdWarp) {
    // ------------------------------ producer warp ------------------------------
    const uint64_t pol = l2_evict_first_policy();
    // arrivals before this launch; phase ph starts once the counter reaches base + ph * gridDim.x
    const unsigned base = __shfl_sync(0xffffffffu, lane == 0 ? ld_acquire(p.bar) / gridDim.x : 0u, 0) * gridDim.x;
    for (int ph = 0; ph < p.nphases && !R.failed; ++ph) {
      const int b = ph & 1;
      int ok = 1;
      if (lane == 0 && !wait_progress(&s_planned, ph)) {
        set_err(st, ERR_TIMEOUT, 43);
        ok = 0;
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) { R.failed = true; break; }
      const Phase& P = s_ph[b];
      if (P.type == PH_GEMV) {
        produce_span<WT>(gg + b * kStepGroups, s_gb[b], s_rb[b], s_ge[b], s_re[b], D.hd, D.box3 != 0, R, st, pol, lane);
      } else if (P.type == PH_ATTN) {
        const att::Tile* tb = tiles + b * kStepTiles;
        const int nt = s_nt[b];
        const AttnPlan A = attn_plan(s_nold[b], s_nnew[b], ips);
        const int nst = nt > 0 ? A.stages(ips) : 0;
        for (int k = 0; k < nst && !R.failed; ++k) {
          if (k * ips == A.q0 && A.q1 > 0) {
            // chunks holding this cycle's keys: wait for the QKV phase's grid barrier
            int ok = 1;
            if (lane == 0) {
              const uint64_t t0 = globaltimer_ns();
              const unsigned target = base + (unsigned)ph * gridDim.x;
              for (uint32_t it = 0; (int)(ld_acquire(p.bar) - target) < 0; ++it)
                if ((it & 63u) == 63u && globaltimer_ns() - t0 > kWaitLimitNs) {
                  set_err(st, ERR_TIMEOUT, 41);
                  ok = 0;
                  break;
                }
            }
            if (!__shfl_sync(0xffffffffu, ok, 0)) { R.failed = true; break; }
          }
          const int s = R.ctr % kStages;
          if (R.ctr >= (uint32_t)kStages && !mbar_wait_bounded(&R.empty[s], ((R.ctr / kStages) - 1) & 1)) {
            if (lane == 0) set_err(st, ERR_TIMEOUT, 42);
            R.failed = true;
            break;
          }
          if (lane == 0) {
            att::Item its[2];
            int idx[2];
            uint32_t tot = 0;
            for (int h = 0; h < ips; ++h) {
              int pass;
              idx[h] = attn_item_at(A, k * ips + h, pass);
              if (idx[h] >= 0) {
                its[h] = att::item_of_pass(tb, nt, pass, idx[h], att::kWarpCK);
                tot += 2u * (uint32_t)its[h].nk * D.hd * ESZ;
              }
            }
            mbar_arrive_expect_tx(&R.full[s], tot);
            for (int h = 0; h < ips; ++h) {
              if (idx[h] < 0) continue;
              const att::Tile& Ti = tb[its[h].T];
              const uint32_t bytes = (uint32_t)its[h].nk * D.hd * ESZ;
              const size_t off = ((size_t)its[h].kh * D.max_seq + (size_t)its[h].c * att::kWarpCK) * D.hd * ESZ;
              unsigned char* dst = R.base + (size_t)s * kStageBytes + (size_t)h * item_bytes;
              bulk_g2s(dst, Ti.kc + off, bytes, &R.full[s], pol);
              bulk_g2s(dst + item_bytes / 2, Ti.vc + off, bytes, &R.full[s], pol);
            }
          }
          __syncwarp();
          ++R.ctr;
        }
      }
      __syncwarp();
      if (lane == 0) st_release_cta(&s_produced, ph);  // the tables of phase ph are no longer read
    }
    if (lane == 0) st_release_cta(&s_produced, 1 << 30);  // leaving (done or failed)
    drain_ring(R, lane);
    return;
  }

  // ------------------------------ consumer warps ------------------------------
  uint64_t t_prev = (blockIdx.x == 0 && tid == 0) ? globaltimer_ns() : 0;
  // arrivals before this launch (fewer than gridDim.x of this launch can have been added yet)
  const unsigned bar_base = tid == 0 ? (ld_acquire(p.bar) / gridDim.x) * gridDim.x : 0u;
  named_bar(4, kNCT + 32);  // phase 0 resolved
  // tcgen05 tiles: consumer warp 0 holds the TMEM accumulator columns for the whole launch
  __shared__ uint32_t s_tmem;
  __shared__ __align__(8) uint64_t s_tc_done;
  __shared__ __align__(8) uint64_t s_tc_bfull[kStages];
  TcCtx tcx{uni, 0u, &s_tc_done, 0u, s_tc_bfull, 0u};
  if (cfg.has_tc) {
    if (warp == 0) tc::alloc_cols(&s_tmem, tc::kColsStep);
    if (tid == 0) {
      mbar_init(&s_tc_done, 1);
      for (int i = 0; i < kStages; ++i) mbar_init(&s_tc_bfull[i], kNCW - 1);  // the builder warps
      fence_mbar_init();
    }
    tc::fence_before();
    named_bar(1, kNCT);
    tc::fence_after();
    tcx.tmem = s_tmem;
  }
  for (int ph = 0; ph < p.nphases; ++ph) {
    const int b = ph & 1;
    const Phase& P = s_ph[b];
    if (s_abort) R.failed = true;
    if (P.type == PH_GEMV) {
      Top2 loc[2];
      top2_init(loc[0]);
      top2_init(loc[1]);
      consume_span<WT, 16>(cfg, gg + b * kStepGroups, s_gb[b], s_rb[b], s_ge[b], s_re[b], R, uni, rstd_s, wpart,
                       loc, &tcx);
      if (P.nparts > 0 && P.part[0].op == OP_HEAD)
        write_head_partial(loc, hred, cfg.B.head_part + (size_t)blockIdx.x * 8);
    } else if (P.type == PH_ATTN) {
      const att::Tile* tb = tiles + b * kStepTiles;
      const int nt = s_nt[b];
      const AttnPlan A = attn_plan(s_nold[b], s_nnew[b], ips);
      const int nst = nt > 0 ? A.stages(ips) : 0;
      float* qb = reinterpret_cast<float*>(uni) + (size_t)warp * att::kHeadsPerPass * D.hd;
      if (D.hd == 64) attn_consume<WT, 2>(D, tb, nt, A, nst, ips, item_bytes, R, qb, &s_fail, st, s_mlist, &s_mcount);
      else attn_consume<WT, 4>(D, tb, nt, A, nst, ips, item_bytes, R, qb, &s_fail, st, s_mlist, &s_mcount);
      R.ctr += (uint32_t)nst;
      named_bar(1, kNCT);
      if (s_fail) R.failed = true;
      if (!R.failed && s_mcount > 0) {
        if (D.hd == 64) attn_merge_list<2>(D, tb, s_mlist, s_mcount);
        else attn_merge_list<4>(D, tb, s_mlist, s_mcount);
      }
      named_bar(1, kNCT);  // every warp has read the count
      if (tid == 0) s_mcount = 0;
    } else if (blockIdx.x == 0 && !R.failed) {  // control: the last phase
      Top2 (*red)[2] = reinterpret_cast<Top2(*)[2]>(uni);
      // the ring is idle in the control phase (every stage of the head phase was consumed): the
      // sampled control step borrows its first bytes as scratch
      static_assert(sizeof(ctl::SampleSmem) <= kStageBytes, "sampling scratch exceeds a ring stage");
      ctl::SampleSmem& S = *reinterpret_cast<ctl::SampleSmem*>(ring);
      if (P.type == PH_CTRL_CYCLE) ctl::control_cycle<WT>(D, cfg.B, red, s_tok, s_slot, kNCT, 1, S);
      else ctl::control_ar<WT>(D, cfg.B, red, s_tok, s_slot, kNCT, 1, S);
    }
    if (ph + 1 < p.nphases) {
      named_bar(1, kNCT);  // this phase's writes are done
      if (tid == 0 && !s_abort) {
        grid_arrive(p.bar);
        if (!grid_wait(p.bar, bar_base + (unsigned)(ph + 1) * gridDim.x, st)) s_abort = 1;
      }
      named_bar(4, kNCT + 32);  // with the planner: phase ph+1 resolved; s_abort visible
    }
    if (p.phase_ns && blockIdx.x == 0 && tid == 0) {
      const uint64_t t = globaltimer_ns();
      atomicAdd(p.phase_ns + ph, (unsigned long long)(t - t_prev));
      t_prev = t;
    }
  }
  if (cfg.has_tc) {  // every MMA this CTA issued has completed and every tcgen05.ld is done
    if (tid == 0) tc::commit(&s_tc_done);
    mbar_wait_bounded(&s_tc_done, tcx.phase);
    tc::fence_before();
    named_bar(1, kNCT);
    if (warp == 0) tc::free_cols(tcx.tmem, tc::kColsStep);
  }
}

static_assert(sizeof(Phase) % 16 == 0, "phase descriptors are copied in 16-byte pieces");
static_assert(sizeof(DevState) % 16 == 0 && sizeof(LayerW) % 16 == 0, "16-byte snapshots");

}  // namespace

// Union scratch: tensor-core partial tiles (GEMV), per-warp query vectors (attention), top-2 merge
// (control).
static size_t step_union_bytes(const Dims& D) {
  size_t uni = (size_t)kMmaScratch;
  const size_t q = (size_t)kNCW * att::kHeadsPerPass * D.hd * sizeof(float);
  if (uni < q) uni = q;
  if (uni < (size_t)kNCW * 32 * 2 * sizeof(Top2)) uni = (size_t)kNCW * 32 * 2 * sizeof(Top2);
  return (uni + 127) & ~(size_t)127;
}

size_t step_smem_bytes(const Dims& D) {
  const int esz = D.dtype == SPD_DTYPE_BF16 ? 2 : 4;
  // an attention item (K and V chunks of kWarpCK keys) must fit one ring stage; hd 64 or 128 (other
  // head sizes run on the per-operator launches)
  if ((size_t)2 * att::kWarpCK * D.hd * esz > (size_t)kStageBytes) return 0;
  if (D.hd != 64 && D.hd != 128) return 0;
  const size_t total = 1024 + (size_t)kStages * kStageBytes + step_union_bytes(D) + 2 * kStepGroups * sizeof(GG) +
                       (size_t)2 * kStepTiles * sizeof(att::Tile) + 16 + (size_t)(D.L + D.Ls) * sizeof(LayerW);
  const size_t static_bytes = 8 * 1024;  // barriers, snapshots, per-vector 1/rms, head merge scratch
  return total + static_bytes <= 227 * 1024 ? total : 0;
}

cudaError_t launch_wait_selftest(DevState* st, unsigned* counter, int which, uint64_t limit_ns, cudaStream_t s) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(st, counter, which, limit_ns);
  return cudaGetLastError();
}

// The dynamic shared-memory limit is an attribute of the kernel on the current device, shared by every
// handle of the process: it is only ever raised (a handle of a smaller model must not lower the limit
// another live handle launches with), per device ordinal, under a mutex.
cudaError_t step_setup_attributes(size_t smem) {
  static std::mutex mu;
  static size_t current[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (dev >= 0 && dev < 64 && smem <= current[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(step_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(step_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess && dev >= 0 && dev < 64) current[dev] = smem;
  return e;
}

cudaError_t launch_step(const Dims& D, const Bufs& B, const LaunchCfg& lcfg, const Phase* prog, int nphases,
                        unsigned* bar, unsigned long long* phase_ns, size_t smem, cudaStream_t s) {
  StepParams p;
  memset(&p, 0, sizeof(p));
  p.cfg.debug_logits = lcfg.debug_logits;
  p.cfg.has_mma = D.dtype == SPD_DTYPE_BF16;
  p.cfg.has_tc = D.tc;
  p.cfg.tc_nv_max = 16;  // the union scratch holds the B ring of 16-vector tiles
  p.cfg.eps = D.eps;
  p.cfg.D = D;
  p.cfg.B = B;
  p.prog = prog;
  p.nphases = nphases;
  p.bar = bar;
  p.phase_ns = phase_ns;
  p.union_bytes = (int)step_union_bytes(D);
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(num_sms());
  cfg.blockDim = dim3(kStepThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (D.dtype == SPD_DTYPE_BF16) return cudaLaunchKernelEx(&cfg, step_kernel<__nv_bfloat16>, p);
  return cudaLaunchKernelEx(&cfg, step_kernel<float>, p);
}

}  // namespace spd
