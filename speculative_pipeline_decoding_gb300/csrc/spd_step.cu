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
#include "spd_attn.cuh"
#include "spd_ctrl.cuh"
#include "spd_engine.cuh"

namespace spd {

namespace {

using namespace eng;

constexpr int kStepGroups = 36;   // groups of one phase: n target + n+1 draft rows (n <= 16)
constexpr int kStepTiles = 24;    // attention tiles of one phase: n target tiles + draft-row tiles
constexpr int kKVHalf = kStageBytes / 2;  // an attention item's ring stage: K chunk | V chunk

struct StepParams {
  EngineCfg cfg;
  const Phase* prog;
  int nphases;
  unsigned* bar;                  // [0] count, [1] generation
  unsigned long long* phase_ns;   // accumulated per-phase time (CTA 0), or null
  int union_bytes;                // attention items / tensor-core partials / control scratch
  int attn_qh_max;
};

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ void red_add_release(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Grid barrier of the 256 consumer threads of every CTA, in two halves so that thread 0 can
// prepare the next phase between its arrival and its wait.  Writes before grid_arrive are visible
// to every CTA after grid_wait.
__device__ __forceinline__ unsigned grid_arrive(unsigned* bar) {  // thread 0 only
  unsigned* count = bar;
  unsigned* gen = bar + 1;
  const unsigned g0 = ld_acquire(gen);
  const unsigned old = atom_add_acq_rel(count, 1u);
  if (old == gridDim.x - 1) {
    atomicExch(count, 0u);
    red_add_release(gen, 1u);
  }
  return g0;
}

// Thread 0: bounded wait for the generation to move past g0.  False if it gave up.
__device__ __forceinline__ bool grid_wait(unsigned* bar, unsigned g0, DevState* st) {
  const unsigned* gen = bar + 1;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0; ld_acquire(gen) == g0; ++it) {
    if ((it & 63u) == 63u && globaltimer_ns() - t0 > 2000000000ull) {
      set_err(st, ERR_TIMEOUT, 70);
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ int qt_of(const Launch& lc) {
  return (lc.kind == LK_PDMROWS || lc.kind == LK_ROWS) ? kAttnQT : 1;
}

template <typename WT>
__global__ void __launch_bounds__(kThreads, 1) step_kernel(const __grid_constant__ StepParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* ring =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  unsigned char* uni = ring + kStages * kStageBytes;
  GG* gg_c = reinterpret_cast<GG*>(uni + p.union_bytes);  // consumers: 2 tables (this / next phase)
  GG* gg_p = gg_c + 2 * kStepGroups;                       // producer
  att::Tile* tiles = reinterpret_cast<att::Tile*>(gg_p + kStepGroups);  // consumers
  att::Tile* tiles_p = tiles + kStepTiles;                                 // producer

  __shared__ __align__(8) uint64_t full_bar[kStages];
  __shared__ __align__(8) uint64_t empty_bar[kStages];
  __shared__ int s_ng[2], s_gb[2], s_rb[2], s_ge[2], s_re[2];
  __shared__ int s_skip, s_nt, s_items, s_fail, s_last, s_tok, s_slot, s_ok;
  __shared__ float rstd_s[16 * kMaxMT];
  __shared__ float wpart[kNCW];
  __shared__ Top2 hred[kNCW * 8][2];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const EngineCfg& cfg = p.cfg;
  const Dims& D = cfg.D;
  DevState* st = cfg.B.st;
  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], kNCW);
    }
    fence_mbar_init();
    s_skip = (st->done || st->err) ? 1 : 0;
  }
  __syncthreads();
  if (s_skip) return;  // every CTA reads the same control block: a uniform decision
  Ring R{ring, full_bar, empty_bar, 0u, false};

  if (warp == kNCW) {
    // ------------------------------ producer warp ------------------------------
    const uint64_t pol = l2_evict_first_policy();
    // grid barriers completed before phase ph = ph; the generation word counts them
    const unsigned g_start = __shfl_sync(0xffffffffu, lane == 0 ? ld_acquire(p.bar + 1) : 0u, 0);
    constexpr int ESZ = sizeof(WT);
    for (int ph = 0; ph < p.nphases && !R.failed; ++ph) {
      const Phase& P = p.prog[ph];
      if (P.type == PH_GEMV) {
        int gb = 0, rb = 0, ge = 0, re = 0;
        if (lane == 0) {
          const int ng = resolve_parts(cfg, P.part, P.nparts, gg_p, kStepGroups);
          span_of(gg_p, ng, blockIdx.x, gridDim.x, gb, rb, ge, re);
        }
        __syncwarp();
        gb = __shfl_sync(0xffffffffu, gb, 0); rb = __shfl_sync(0xffffffffu, rb, 0);
        ge = __shfl_sync(0xffffffffu, ge, 0); re = __shfl_sync(0xffffffffu, re, 0);
        produce_span<WT>(gg_p, gb, rb, ge, re, D.hd, R, st, pol, lane);
        __syncwarp();  // gg_p is rewritten by the next phase
      } else if (P.type == PH_ATTN) {
        // this CTA's items: chunks written in earlier cycles first, then -- once the QKV phase's
        // grid barrier has passed -- the chunks holding this cycle's keys
        int nt = 0, items = 0;
        if (lane == 0) {
          for (int i = 0; i < P.nparts && nt >= 0; ++i)
            nt = att::add_tiles(D, cfg.B, P.part[i].lc, qt_of(P.part[i].lc), kStepChunk, tiles_p, nt, &items,
                                kStepTiles);
        }
        __syncwarp();
        nt = __shfl_sync(0xffffffffu, nt, 0);
        items = __shfl_sync(0xffffffffu, items, 0);
        if (nt <= 0) continue;
        for (int pass = 0; pass < 2 && !R.failed; ++pass) {
          if (pass == 1) {
            int ok = 1;
            if (lane == 0) {
              const uint64_t t0 = globaltimer_ns();
              for (uint32_t it = 0; (ld_acquire(p.bar + 1) - g_start) < (unsigned)ph; ++it)
                if ((it & 63u) == 63u && globaltimer_ns() - t0 > 2000000000ull) {
                  set_err(st, ERR_TIMEOUT, 41);
                  ok = 0;
                  break;
                }
            }
            if (!__shfl_sync(0xffffffffu, ok, 0)) { R.failed = true; break; }
          }
          for (int item = blockIdx.x; item < items && !R.failed; item += gridDim.x) {
            const att::Item it = att::item_of(tiles_p, nt, item, kStepChunk);
            const att::Tile& Ti = tiles_p[it.T];
            if (att::chunk_is_new(Ti, it.c, kStepChunk) != (pass == 1)) continue;
            const int s = R.ctr % kStages;
            if (R.ctr >= (uint32_t)kStages && !mbar_wait_bounded(&R.empty[s], ((R.ctr / kStages) - 1) & 1)) {
              if (lane == 0) set_err(st, ERR_TIMEOUT, 42);
              R.failed = true;
              break;
            }
            if (lane == 0) {
              const uint32_t bytes = (uint32_t)it.nk * D.hd * ESZ;
              const size_t off = ((size_t)it.kh * D.max_seq + (size_t)it.c * kStepChunk) * D.hd * ESZ;
              unsigned char* dst = R.base + (size_t)s * kStageBytes;
              mbar_arrive_expect_tx(&R.full[s], 2 * bytes);
              bulk_g2s(dst, Ti.kc + off, bytes, &R.full[s], pol);
              bulk_g2s(dst + kKVHalf, Ti.vc + off, bytes, &R.full[s], pol);
            }
            __syncwarp();
            ++R.ctr;
          }
        }
      }
    }
    drain_ring(R, lane);
    return;
  }

  // ------------------------------ consumer warps ------------------------------
  constexpr int NCT = kNCW * 32;
  uint64_t t_prev = (blockIdx.x == 0 && tid == 0) ? globaltimer_ns() : 0;
  // groups (table ph & 1) or attention tiles of phase ph; they depend on the control block only,
  // so phase ph+1 is prepared before the grid barrier that ends phase ph
  auto prepare = [&](int ph) {
    const Phase& P = p.prog[ph];
    const int b = ph & 1;
    if (P.type == PH_GEMV) {
      s_ng[b] = resolve_parts(cfg, P.part, P.nparts, gg_c + b * kStepGroups, kStepGroups);
      span_of(gg_c + b * kStepGroups, s_ng[b], blockIdx.x, gridDim.x, s_gb[b], s_rb[b], s_ge[b], s_re[b]);
    } else if (P.type == PH_ATTN) {
      int nt = 0, items = 0;
      for (int i = 0; i < P.nparts && nt >= 0; ++i)
        nt = att::add_tiles(D, cfg.B, P.part[i].lc, qt_of(P.part[i].lc), kStepChunk, tiles, nt, &items,
                            kStepTiles);
      s_nt = nt > 0 ? nt : 0;
      s_items = nt > 0 ? items : 0;
      s_fail = 0;
    }
  };
  if (tid == 0) prepare(0);
  named_bar(1, NCT);
  for (int ph = 0; ph < p.nphases; ++ph) {
    const Phase& P = p.prog[ph];
    const int b = ph & 1;
    if (P.type == PH_GEMV) {
      Top2 loc[2];
      top2_init(loc[0]);
      top2_init(loc[1]);
      consume_span<WT>(cfg, gg_c + b * kStepGroups, s_gb[b], s_rb[b], s_ge[b], s_re[b], R, uni, rstd_s, wpart,
                       loc);
      if (P.nparts > 0 && P.part[0].op == OP_HEAD)
        write_head_partial(loc, hred, cfg.B.head_part + (size_t)blockIdx.x * 8);
    } else if (P.type == PH_ATTN) {
      // items from the ring, in the producer's order (older chunks, then this cycle's)
      float* qs = reinterpret_cast<float*>(uni);
      float* sc = qs + (size_t)p.attn_qh_max * D.hd;
      float* m_s = sc + (size_t)p.attn_qh_max * kStepChunk;
      float* l_s = m_s + p.attn_qh_max;
      for (int pass = 0; pass < 2 && s_items > 0; ++pass) {
        for (int item = blockIdx.x; item < s_items; item += gridDim.x) {
          const att::Item it = att::item_of(tiles, s_nt, item, kStepChunk);
          if (att::chunk_is_new(tiles[it.T], it.c, kStepChunk) != (pass == 1)) continue;
          const int s = R.ctr % kStages;
          if (!R.failed && !mbar_wait_bounded(&R.full[s], (R.ctr / kStages) & 1)) {
            set_err(st, ERR_TIMEOUT, 31);
            s_fail = 1;
          }
          named_bar(1, NCT);  // uniform decision
          if (s_fail) R.failed = true;
          if (!R.failed) {
            const WT* kst = reinterpret_cast<const WT*>(R.base + (size_t)s * kStageBytes);
            const WT* vst = reinterpret_cast<const WT*>(R.base + (size_t)s * kStageBytes + kKVHalf);
            att::item_compute<WT, kStepChunk>(D, tiles[it.T], it, kst, vst, qs, sc, m_s, l_s, &s_last);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&R.empty[s]);
          ++R.ctr;
        }
      }
    } else if (blockIdx.x == 0) {  // control: the last phase
      Top2 (*red)[2] = reinterpret_cast<Top2(*)[2]>(uni);
      if (P.type == PH_CTRL_CYCLE) ctl::control_cycle<WT>(D, cfg.B, red, s_tok, s_slot, NCT, 1);
      else ctl::control_ar<WT>(D, cfg.B, red, s_tok, s_slot, NCT, 1);
    }
    if (ph + 1 < p.nphases) {
      named_bar(1, NCT);  // this phase's writes are done; its tables / tiles are no longer read
      if (tid == 0) {
        const unsigned g0 = grid_arrive(p.bar);
        prepare(ph + 1);
        s_ok = grid_wait(p.bar, g0, st) ? 1 : 0;
      }
      named_bar(1, NCT);
      if (!s_ok) break;
    }
    if (p.phase_ns && blockIdx.x == 0 && tid == 0) {
      const uint64_t t = globaltimer_ns();
      atomicAdd(p.phase_ns + ph, (unsigned long long)(t - t_prev));
      t_prev = t;
    }
  }
}

}  // namespace

size_t step_smem_bytes(const Dims& D) {
  const int esz = D.dtype == SPD_DTYPE_BF16 ? 2 : 4;
  if ((size_t)kStepChunk * D.hd * esz > (size_t)kKVHalf) return 0;  // a K or V chunk fills half a stage
  size_t uni = att::smem_bytes(D.hd, D.gq, esz, kAttnQT, kStepChunk) - (size_t)2 * kStepChunk * D.hd * esz;
  if (uni < (size_t)kMmaScratch) uni = (size_t)kMmaScratch;
  if (uni < (size_t)kNCW * 32 * 2 * sizeof(Top2)) uni = (size_t)kNCW * 32 * 2 * sizeof(Top2);
  uni = (uni + 127) & ~(size_t)127;
  const size_t total = 1024 + (size_t)kStages * kStageBytes + uni + 3 * kStepGroups * sizeof(GG) +
                       (size_t)2 * kStepTiles * sizeof(att::Tile);
  const size_t static_bytes = 8 * 1024;  // barriers, per-vector 1/rms, head merge scratch
  return total + static_bytes <= 227 * 1024 ? total : 0;
}

cudaError_t step_setup_attributes(size_t smem) {
  cudaError_t e = cudaFuncSetAttribute(step_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(step_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

cudaError_t launch_step(const Dims& D, const Bufs& B, const LaunchCfg& lcfg, const Phase* prog, int nphases,
                        unsigned* bar, unsigned long long* phase_ns, size_t smem, cudaStream_t s) {
  StepParams p;
  memset(&p, 0, sizeof(p));
  p.cfg.debug_logits = lcfg.debug_logits;
  p.cfg.has_mma = D.dtype == SPD_DTYPE_BF16;
  p.cfg.eps = D.eps;
  p.cfg.D = D;
  p.cfg.B = B;
  p.prog = prog;
  p.nphases = nphases;
  p.bar = bar;
  p.phase_ns = phase_ns;
  const int esz = D.dtype == SPD_DTYPE_BF16 ? 2 : 4;
  size_t uni = att::smem_bytes(D.hd, D.gq, esz, kAttnQT, kStepChunk) - (size_t)2 * kStepChunk * D.hd * esz;
  if (uni < (size_t)kMmaScratch) uni = (size_t)kMmaScratch;
  if (uni < (size_t)kNCW * 32 * 2 * sizeof(Top2)) uni = (size_t)kNCW * 32 * 2 * sizeof(Top2);
  p.union_bytes = (int)((uni + 127) & ~(size_t)127);
  p.attn_qh_max = kAttnQT * D.gq;
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(num_sms());
  cfg.blockDim = dim3(kThreads);
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
