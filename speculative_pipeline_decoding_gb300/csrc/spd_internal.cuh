// Internal types and device helpers shared by the SPD kernels and the C-ABI layer.
//
// Memory layout in HBM (all device-resident for the lifetime of a handle):
//   target KV   [L ][Hkv][max_seq][hd]  (K and V separate), storage dtype
//   draft KV    [Ls][Hkv][max_seq][hd]
//   resid ring  [n+1][d]    fp32: residual stream of the n+1 trailing positions, row = pos % (n+1)
//   anchor ring [n+1][m][d] fp32: h^(b_i) of those positions; row i = anchor b_i (b_0 = embedding)
//   decode scratch (target): qkv [n][(Hq+2Hkv)hd], attn [n][Hq hd], u [n][ffn]
//   draft rows (<= n+1 per cycle): z [n+2][d], qkv, attn, u
//   prefill block scratch (PB rows): h, anchors [PB][m][d], z, qkv, attn, u
//   rope tables cos/sin [max_seq][hd/2] fp32 (angles formed in fp64)
//   control block (DevState), token sequence, verification trace, draft override arrays.
#pragma once
#include <cuda.h>  // CUtensorMap (the type only; maps are encoded through the runtime's entry point)
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/spd.h"

namespace spd {

constexpr int kMaxGroups = 72;      // one launch: n_stages target groups + n_stages+1 draft rows (+ splits)
constexpr int kMaxAttnRows = 32;    // query rows of the stand-alone attention operators
constexpr int kMaxExplicit = 34;    // groups of the stand-alone grouped GEMV
constexpr int kMaxTiles = 64;       // attention query tiles per launch
constexpr int kPrefillBlock = 32;   // prompt rows per prefill pass
constexpr int kAttnChunk = 128;     // keys per attention split (fixed: split count depends on length only)
constexpr int kAttnQT = 8;          // query rows per attention tile for multi-row launches
constexpr int kAttnThreads = 256;

// ------------------------------------------------------------------------------------------
// control block
// ------------------------------------------------------------------------------------------
struct DevState {
  int t, a, v, pdm_len;        // newest position, fill, verified length, draft cache length
  int P, cycles, exits, rejects;
  int err, done, max_commit, flags;
  int last_exited, last_exit_pos, last_accept, target_top1;
  int pdm_top1, pdm_top2, draft, pushed;
  int err_where, pad0, pad1, pad2;
};

enum ErrCode { ERR_TIMEOUT = 1, ERR_PDM_ROWS = 2, ERR_BOUNDS = 4 };
enum StateFlags { SF_TARGET_ONLY = 1, SF_POST_STEP = 2 };  // SF_POST_STEP: draft module after the step

struct LayerW {
  const void *attn_norm, *wq, *wk, *wv, *wo, *ffn_norm, *wg, *wu, *wd;
  const CUtensorMap *tq, *tk, *tv, *to, *tg, *tu, *td;  // tensor maps of the seven matrices
};

constexpr int kMaxTopK = 64;  // largest top-k of sampled decoding

struct Dims {
  int L, d, hq, hkv, hd, ffn, V, n, S, Ls, m;
  int max_seq, dtype, qkv_rows, gq;
  int box3;         // weight tensor maps are 3-D (see box3_cols): two copies per GEMV stage
  int tc;           // tcgen05 draft tiles: every stream map is followed by its 128-row map
  int top_k;        // sampled decoding: top-k (0: greedy decoding)
  float temp;       // sampled decoding: temperature T > 0
  int anchors[SPD_MAX_ANCHORS];
  int ftab[SPD_MAX_STAGES + 1];
  float eps;
};

struct Bufs {
  DevState* st;
  int* seq;          // [max_seq + 2]
  int* trace;        // [2][max_seq]
  int* kvlen;        // [L]
  int* ovr_ref;      // [max_seq + 2]
  unsigned char* ovr_mode;
  float* resid;      // [(n+1)][d]
  float* anch;       // [(n+1)][m][d]
  void *kc, *vc, *pkc, *pvc;
  const float *rope_cos, *rope_sin;
  float* head_part;  // [grid][2][4]
  float* logits;     // [2][V] (debug, and the heads' logits of sampled decoding)
  const float* u_smp;  // sampled decoding: [4][max_seq + 2] uniforms by position (draft, accept,
                       // resample, ar)
  float* q_prob;     // sampled decoding: draft distribution of position q in slot q % (n+1):
  int* q_id;         //   [(n+1)][kMaxTopK] probabilities and token ids, canonical order
  int head_grid;
  const LayerW* tl;
  const LayerW* pl;
  const void* embed;
  const void* lm_head;
  const void* pdm_head;
  const float* final_norm;
  const float* pdm_norm;
  const void* fc[SPD_MAX_ANCHORS];
  const CUtensorMap* tm_fc[SPD_MAX_ANCHORS];
  const CUtensorMap* tm_lm;
  const CUtensorMap* tm_pdm;
  float* tc_part;    // split-K partial tiles of the tcgen05 groups of one launch or phase (or null)
  int* tc_tick;      // their tickets (left at zero)
  int tc_part_cap, tc_tick_cap;  // floats / tickets available
};

// How the rows of one launch are formed from the control block.
enum LaunchKind {
  LK_DIAG = 0,     // target stage-diagonal sub-step `sub`: token at depth j runs layer j*S+sub
  LK_PDMROWS = 1,  // draft rows pdm_len+1..t through draft layer `sub`
  LK_ROWS = 2,     // explicit consecutive rows pos0..pos0+cnt-1 through layer `sub` of `stack`
  LK_AR = 3,       // one token at position t through target layer `sub`
  LK_EXPLICIT = 4  // stand-alone operator: caller-given rows
};

// Activation buffers a launch reads and writes.
struct Act {
  float* resid; int resid_ring;   // residual rows; ring size (huge = linear)
  float* qkv;                     // [rows][qkv_rows]
  float* attn;                    // [rows][hq*hd]
  float* u;                       // [rows][ffn]
  float* anch; int anch_ring;     // anchor rows [row][m][d] (target stacks only; may be null)
  float* part; int* tick;         // attention split partials and tickets
  const int* pos_arr;             // LK_EXPLICIT: positions
  const void* kc; const void* vc; // LK_EXPLICIT: cache bases
};

struct Launch {
  int kind, stack, sub, pos0, cnt;
  Act act;
};

// ------------------------------------------------------------------------------------------
// small device helpers
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

template <typename WT> struct WTraits;
template <> struct WTraits<float> {
  static constexpr int kVec = 4;  // elements per 16 bytes
  __device__ static __forceinline__ void unpack(const uint4& q, float* f) {
    f[0] = __uint_as_float(q.x); f[1] = __uint_as_float(q.y);
    f[2] = __uint_as_float(q.z); f[3] = __uint_as_float(q.w);
  }
  __device__ static __forceinline__ float to_f(float x) { return x; }
  __device__ static __forceinline__ float from_f(float x) { return x; }
};
template <> struct WTraits<__nv_bfloat16> {
  static constexpr int kVec = 8;
  __device__ static __forceinline__ void unpack(const uint4& q, float* f) {
    f[0] = bf16_lo(q.x); f[1] = bf16_hi(q.x); f[2] = bf16_lo(q.y); f[3] = bf16_hi(q.y);
    f[4] = bf16_lo(q.z); f[5] = bf16_hi(q.z); f[6] = bf16_lo(q.w); f[7] = bf16_hi(q.w);
  }
  __device__ static __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
  __device__ static __forceinline__ __nv_bfloat16 from_f(float x) { return __float2bfloat16_rn(x); }
};

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---- mbarrier / bulk-copy PTX (sm_90+ forms, valid on sm_103a) ----
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
  return ok != 0;
}
// Limit of every bounded device wait: after this much wall time (%globaltimer) the wait gives up,
// the kernel sets the control block's error word and leaves; the host reports SPD_ETIMEOUT.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// Bounded wait: gives up after `limit_ns` of wall time and reports false.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 255u && globaltimer_ns() - t0 > limit_ns) return false;
  }
}
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
// 1-D bulk copy global -> shared, completion counted on `bar` (bytes % 16 == 0, both 16B aligned).
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
// Programmatic dependent launch: wait for the previous kernel of the stream (no-op when the kernel
// was launched without the attribute), and allow the next kernel to be scheduled.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void named_bar(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ void set_err(DevState* st, int code, int where) {
  if (st == nullptr) return;
  atomicOr(&st->err, code);
  atomicCAS(&st->err_where, 0, where);
}

// top-2 with a total order: larger value first, lower index on ties
struct Top2 {
  float v1, v2;
  int i1, i2;
};
__device__ __forceinline__ bool better(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}
__device__ __forceinline__ void top2_init(Top2& t) {
  t.v1 = -INFINITY; t.v2 = -INFINITY; t.i1 = 0x7fffffff; t.i2 = 0x7fffffff;
}
__device__ __forceinline__ void top2_push(Top2& t, float v, int i) {
  if (better(v, i, t.v1, t.i1)) {
    t.v2 = t.v1; t.i2 = t.i1; t.v1 = v; t.i1 = i;
  } else if (better(v, i, t.v2, t.i2)) {
    t.v2 = v; t.i2 = i;
  }
}
__device__ __forceinline__ void top2_merge(Top2& a, const Top2& b) {
  top2_push(a, b.v1, b.i1);
  top2_push(a, b.v2, b.i2);
}

// Row-set of one launch: groups of consecutive rows that share a layer.
struct RowGroup {
  int layer, nv, pos0, vid0, rrow0;
};

// Where row and group resolution reads the control block and the per-layer tables: global memory
// in the stand-alone kernels; shared-memory snapshots taken at the start of the step kernel (the
// control block changes only in its last phase), so that resolving a phase costs no global loads.
struct View {
  const DevState* sv;
  const LayerW* tl;
  const LayerW* pl;
};

// Fill `g` from the launch kind and the control block `sv`; returns the group count (0 if none).
// Executed by one thread.  Sets an error flag in `st` for an out-of-step draft cache.
__device__ __forceinline__ int build_rows(const Launch& lc, const Dims& D, const DevState* sv, DevState* st,
                                          RowGroup* g) {
  switch (lc.kind) {
    case LK_DIAG: {
      const int a = sv->a, t = sv->t;
      for (int j = 0; j < a; ++j) {
        g[j].layer = j * D.S + lc.sub; g[j].nv = 1; g[j].pos0 = t - j; g[j].vid0 = j;
        g[j].rrow0 = (t - j) % (D.n + 1);
      }
      return a;
    }
    case LK_PDMROWS: {
      const int R = sv->t - sv->pdm_len;
      if (R < 1 || R > D.n + 1) {
        set_err(st, ERR_PDM_ROWS, 100 + lc.sub);
        return 0;
      }
      g[0].layer = lc.sub; g[0].nv = R; g[0].pos0 = sv->pdm_len + 1; g[0].vid0 = 0; g[0].rrow0 = 0;
      return 1;
    }
    case LK_ROWS:
      g[0].layer = lc.sub; g[0].nv = lc.cnt; g[0].pos0 = lc.pos0; g[0].vid0 = 0; g[0].rrow0 = 0;
      return 1;
    case LK_AR:
      g[0].layer = lc.sub; g[0].nv = 1; g[0].pos0 = sv->t; g[0].vid0 = 0;
      g[0].rrow0 = sv->t % (D.n + 1);
      return 1;
    default:
      return 0;
  }
}

// ------------------------------------------------------------------------------------------
// host-side launchers (implemented in the kernel translation units)
// ------------------------------------------------------------------------------------------
enum GemvOp { OP_QKV = 0, OP_O = 1, OP_GATEUP = 2, OP_DOWN = 3, OP_FC = 4, OP_HEAD = 5 };
enum KernelKind { KK_QKV = 0, KK_ROPE = 1, KK_ATTN = 2, KK_O = 3, KK_GATEUP = 4, KK_DOWN = 5,
                  KK_FC = 6, KK_HEAD = 7, KK_CTRL = 8 };

struct GemvExplicit {  // stand-alone grouped GEMV
  const CUtensorMap* tm[kMaxExplicit];  // device copies of the weights' tensor maps
  const void* W[kMaxExplicit];
  const float* x[kMaxExplicit];
  float* y[kMaxExplicit];
  int G, rows, cols;
  const float* nw;
};

struct LaunchCfg {
  int sms;
  int gemv_grid;
  int attn_grid_decode, attn_grid_multi;
  int debug_logits;
};

// One operator over the rows a launch descriptor selects; a GEMV launch carries one or two parts
// (the target's stage-diagonal groups and the draft module's rows of the same operator).
struct GemvPart {
  int op;
  Launch lc;
};

// ---- persistent step kernel: one cooperative launch runs a program of phases ----
enum PhaseType { PH_GEMV = 0, PH_ATTN = 1, PH_CTRL_CYCLE = 2, PH_CTRL_AR = 3 };
struct Phase {
  int type;        // PhaseType
  int kind;        // kernel kind charged with the phase's time (KK_*, +9 for draft-only phases)
  int nparts;      // GEMV / attention parts (target rows, draft rows)
  GemvPart part[2];
};
constexpr int kStepChunk = 32;   // attention keys per split inside the step kernel (one warp item)

// Dynamic shared memory the step kernel needs for this model (0: it does not fit on one SM).
size_t step_smem_bytes(const Dims& D);
cudaError_t step_setup_attributes(size_t smem);
// One cooperative launch (one CTA per SM) running `prog[0..nphases)`.  `bar` = 2 words of grid
// barrier state (zero-initialised), `phase_ns` = per-phase accumulated nanoseconds (or null).
cudaError_t launch_step(const Dims& D, const Bufs& B, const LaunchCfg& cfg, const Phase* prog,
                        int nphases, unsigned* bar, unsigned long long* phase_ns, size_t smem,
                        cudaStream_t s);

// pdl: launch with programmatic stream serialisation (the kernel may start before its predecessor
// ends; it waits with griddepcontrol.wait before touching activations).  resolve_after_wait: the
// predecessor may have written the control block, so the rows are resolved after that wait.
cudaError_t launch_gemv(const GemvPart* parts, int nparts, const Dims& D, const Bufs& B,
                        const LaunchCfg& cfg, bool pdl, bool resolve_after_wait, cudaStream_t s);
cudaError_t launch_gemv_explicit(const GemvExplicit& ge, int dtype, float eps, cudaStream_t s);
cudaError_t launch_attn(const Dims& D, const Bufs& B, const Launch& lc, const LaunchCfg& cfg,
                        bool pdl, cudaStream_t s);
size_t attn_smem_bytes(const Dims& D, bool multi);
size_t attn_part_floats(int rows, int hq, int hd, int max_seq, int ck = kAttnChunk);
cudaError_t gemv_setup_attributes();
// A row-major [rows, cols] weight matrix is streamed through 3-D tensor maps when its rows are whole
// 128-byte chunks: (128-byte chunk, row, chunk index), box = 4 chunks x 32 rows (16 KB), so one copy
// brings a 32-row band of a 512-byte column slice; other widths use 2-D maps with boxes of
// 128 bytes x 32 rows (four copies per band).  Both land in shared memory as [chunk][row][128 B]
// with the 128-byte swizzle.
inline bool box3_cols(int cols, int dtype) { return cols % (dtype == SPD_DTYPE_BF16 ? 64 : 32) == 0; }
// Encodes that tensor map (3-D when box3, else 2-D).  Host call; returns a CUDA error code.
cudaError_t gemv_encode_map(CUtensorMap* out, const void* W, int rows, int cols, int dtype, bool box3);
// The 128-row map of a bf16 matrix for tcgen05 tiles: 3-D (chunk, row, chunk index), box 128 rows x
// 2 chunks (32 KB, one ring stage), 128-byte swizzle.
cudaError_t gemv_encode_tc_map(CUtensorMap* out, const void* W, int rows, int cols);
int gemv_head_grid(int dtype);
int num_sms();
cudaError_t attn_setup_attributes(size_t max_smem);
int attn_grid(const Dims& D, bool multi);

// control kernels
cudaError_t launch_control_cycle(const Dims& D, const Bufs& B, cudaStream_t s);
cudaError_t launch_control_ar(const Dims& D, const Bufs& B, cudaStream_t s);
cudaError_t launch_prefill_embed(const Dims& D, const Bufs& B, float* h, float* anch, int pos0,
                                 int cnt, cudaStream_t s);
cudaError_t launch_prefill_finish(const Dims& D, const Bufs& B, int P, cudaStream_t s);
cudaError_t launch_rollback(const Dims& D, const Bufs& B, int keep_len, int reseed,
                            cudaStream_t s);
cudaError_t launch_begin_generate(const Dims& D, const Bufs& B, int max_new, cudaStream_t s);
cudaError_t launch_rope_tables(float* cosv, float* sinv, int max_seq, int hd, float theta,
                               cudaStream_t s);

// Runs one of the step kernel's bounded waits on a condition nothing satisfies (which: 0 grid barrier
// counter, 1 mbarrier phase, 2 shared progress counter), with limit `limit_ns`; the wait sets the
// ERR_TIMEOUT bit of st->err when it gives up.
cudaError_t launch_wait_selftest(DevState* st, unsigned* counter, int which, uint64_t limit_ns, cudaStream_t s);

// Causal attention of one prefill block on the tensor cores (spd_pfattn.cu): nq <= 32 query rows at
// positions pos0..pos0+nq-1, keys and values of the layer already in its bf16 cache.
struct PfAttnArgs {
  const CUtensorMap* kmap;  // host copies of the 2-D maps over the K / V caches (pfattn_encode_map)
  const CUtensorMap* vmap;
  const float* q; int q_stride;  // query rows (rotated q of head h at h*hd)
  float* out;                    // attention rows [row][hq*hd]
  float* part; int* tick;        // split partials (pfattn_part_floats) and tickets (>= hq ints, zeroed)
  DevState* st;                  // error word, or null
  int kv_row0;                   // map row of position 1 of kv head 0 of the layer
  int max_seq, hq, hkv, hd, pos0, nq, sms;
};
bool pfattn_supported(int dtype, int hd, int nq, int gq);
size_t pfattn_smem_bytes(int hd);
size_t pfattn_part_floats(int hkv, int gq, int max_seq, int sms);
cudaError_t pfattn_encode_map(CUtensorMap* out, const void* cache, long long rows, int hd);
cudaError_t pfattn_setup_attributes();
cudaError_t launch_pfattn(const PfAttnArgs& a, cudaStream_t s);

// records `msg` as the text spd_last_error(NULL) returns; gives back `code`
int spd_internal_fail(int code, const char* msg);

}  // namespace spd
