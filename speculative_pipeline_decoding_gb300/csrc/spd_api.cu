// C ABI of the SPD engine (declared in include/spd.h): handle, memory, and the enqueueing of
// prefill, SPD cycles, plain AR steps and the host-side rollback.
//
// A cycle is enqueued as (SPD summary, 方法步骤详情 steps 1-5), all on one stream:
//   anchor FC over the staircase rows of the draft module                       (steps 2-3)
//   for s in 0..S-1: QKV(+RoPE, KV append), attention, o-proj, gate/up, down of the stage
//     diagonal (step 1); draft layer s (s < Ls) rides in the same GEMV launches (step 4)
//   vocab head (exiting token + draft row), control (verify / rollback / reseed, step 5)
// With SPD_OPT_PDL every launch may start while its predecessor drains (weights stream early; the
// activations are read after griddepcontrol.wait).  With graphs enabled the whole cycle is captured
// once and replayed; all per-cycle state lives in the device control block, so replays run back to
// back without host synchronisation.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "spd_internal.cuh"

using namespace spd;

namespace {

constexpr int kBigRing = 1 << 30;
thread_local std::string g_create_error;

struct EvRec {
  int kind;
  cudaEvent_t a, b;
};

}  // namespace

struct spd_handle {
  spd_config cfg;
  Dims D;
  Bufs B;
  LaunchCfg LC;
  int esz = 2;
  cudaStream_t s_main = nullptr;
  bool own_main = false;
  cudaEvent_t ev_t0 = nullptr, ev_t1 = nullptr;
  std::vector<void*> allocs;
  Act act_t{}, act_p{}, act_head{}, act_pf{}, act_pfp{};
  float* p_z = nullptr;
  int opts = SPD_OPT_GRAPHS | SPD_OPT_PDL | SPD_OPT_COSCHED | SPD_OPT_STEP;
  // persistent step kernel: programs of phases for one cycle and one AR step
  size_t step_smem = 0;               // 0: the step kernel does not fit this model
  Phase* d_prog_cycle = nullptr;
  Phase* d_prog_ar = nullptr;
  int n_prog_cycle = 0, n_prog_ar = 0, cap_prog_cycle = 0, cap_prog_ar = 0;
  std::vector<int> kinds_cycle, kinds_ar;
  unsigned* d_bar = nullptr;          // grid barrier words
  unsigned long long* d_ns_cycle = nullptr;  // per-phase accumulated time while timing
  unsigned long long* d_ns_ar = nullptr;
  int64_t timed_cycles = 0, timed_ar = 0;
  bool st_dirty = true;         // the last kernel enqueued may have written the control block
  bool prefilled = false;
  int P = 0;
  cudaGraphExec_t g_cycle = nullptr;
  cudaGraphExec_t g_ar = nullptr;
  std::string err;
  bool timing = false;
  std::vector<EvRec> recs;
  std::vector<cudaEvent_t> pool;
  size_t pool_used = 0;
  int64_t n_launch = 0;         // kernels enqueued (eager) or captured
  int64_t graph_nodes_cycle = 0, graph_nodes_ar = 0;
  int64_t launches[SPD_NUM_KINDS] = {0};
  double ms[SPD_NUM_KINDS] = {0};
  DevState* host_state = nullptr;  // pinned mirror
  // prefill blocks' causal attention on the tensor cores (bf16, head size 64 or 128)
  bool pf_on = false;
  CUtensorMap pf_map[4];          // K, V of the target cache; K, V of the draft-module cache
  float* pf_part = nullptr;       // split partials
  int* pf_tick = nullptr;         // merge tickets (left at zero)
};

namespace {

int fail(spd_handle* h, int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  if (h) h->err = buf; else g_create_error = buf;
  return code;
}

#define SPD_CUDA(h, call)                                                                   \
  do {                                                                                      \
    cudaError_t e_ = (call);                                                                \
    if (e_ != cudaSuccess) return fail((h), SPD_ECUDA, "%s: %s", #call, cudaGetErrorString(e_)); \
  } while (0)

template <typename T>
T* dalloc(spd_handle* h, size_t count, cudaError_t* e) {
  void* p = nullptr;
  const size_t bytes = count * sizeof(T) + 16;
  *e = cudaMalloc(&p, bytes);
  if (*e != cudaSuccess) return nullptr;
  *e = cudaMemset(p, 0, bytes);
  h->allocs.push_back(p);
  return reinterpret_cast<T*>(p);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---- launch wrappers with optional per-kind event timing (eager mode only) ----
cudaEvent_t pool_event(spd_handle* h) {
  if (h->pool_used == h->pool.size()) {
    cudaEvent_t e;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    h->pool.push_back(e);
  }
  return h->pool[h->pool_used++];
}

struct Timed {
  spd_handle* h;
  int kind;
  cudaStream_t s;
  cudaEvent_t a = nullptr, b = nullptr;
  Timed(spd_handle* h_, int k, cudaStream_t s_) : h(h_), kind(k), s(s_) {
    h->n_launch += 1;
    if (h->timing && h->pool_used + 2 <= 65536) {
      a = pool_event(h);
      b = pool_event(h);
      if (a && b) cudaEventRecord(a, s);
    }
  }
  ~Timed() {
    if (a && b) {
      cudaEventRecord(b, s);
      h->recs.push_back({kind, a, b});
    }
  }
};

constexpr int kDraftKinds = 9;  // kinds 9..17: the same operators on the draft-module stack

bool use_pdl(const spd_handle* h) { return (h->opts & SPD_OPT_PDL) != 0; }

// One GEMV launch of operator `op` over the rows of `a` and, when given, the rows of `b` (the
// draft module's rows riding in a target launch).
int run_gemv(spd_handle* h, int op, const Launch& a, const Launch* b, cudaStream_t s) {
  static const int kind_of[] = {KK_QKV, KK_O, KK_GATEUP, KK_DOWN, KK_FC, KK_HEAD};
  GemvPart parts[2];
  parts[0].op = op;
  parts[0].lc = a;
  int np = 1;
  if (b) {
    parts[1].op = op;
    parts[1].lc = *b;
    np = 2;
  }
  Timed tm(h, kind_of[op] + (a.stack == 1 ? kDraftKinds : 0), s);
  SPD_CUDA(h, launch_gemv(parts, np, h->D, h->B, h->LC, use_pdl(h), h->st_dirty, s));
  h->st_dirty = false;
  return SPD_OK;
}

int run_attn(spd_handle* h, const Launch& lc, cudaStream_t s) {
  Timed tm(h, KK_ATTN + (lc.stack == 1 ? kDraftKinds : 0), s);
  SPD_CUDA(h, launch_attn(h->D, h->B, lc, h->LC, use_pdl(h) && !h->st_dirty, s));
  h->st_dirty = false;
  return SPD_OK;
}

// Causal attention of a prefill block (rows pos0..pos0+cnt-1 of layer `sub` of `stack`) on the
// tensor-core kernel.
int run_pfattn(spd_handle* h, const Launch& lc, cudaStream_t s) {
  Timed tm(h, KK_ATTN + (lc.stack == 1 ? kDraftKinds : 0), s);
  const Dims& D = h->D;
  PfAttnArgs a;
  memset(&a, 0, sizeof(a));
  a.kmap = &h->pf_map[lc.stack == 1 ? 2 : 0];
  a.vmap = &h->pf_map[lc.stack == 1 ? 3 : 1];
  a.q = lc.act.qkv; a.q_stride = D.qkv_rows;
  a.out = lc.act.attn;
  a.part = h->pf_part; a.tick = h->pf_tick; a.st = h->B.st;
  a.kv_row0 = lc.sub * D.hkv * D.max_seq;
  a.max_seq = D.max_seq; a.hq = D.hq; a.hkv = D.hkv; a.hd = D.hd;
  a.pos0 = lc.pos0; a.nq = lc.cnt; a.sms = h->LC.sms;
  SPD_CUDA(h, launch_pfattn(a, s));
  h->st_dirty = false;
  return SPD_OK;
}

// One decoder layer (or the layer-s slice of a co-scheduled step) for the rows of `lc` and, when
// given, `extra` (5 launches; the draft rows need their own attention launch).
int enqueue_layer(spd_handle* h, const Launch& lc, const Launch* extra, cudaStream_t s) {
  int rc;
  if ((rc = run_gemv(h, OP_QKV, lc, extra, s))) return rc;
  if ((rc = (lc.kind == LK_ROWS && h->pf_on) ? run_pfattn(h, lc, s) : run_attn(h, lc, s))) return rc;
  if (extra && (rc = run_attn(h, *extra, s))) return rc;
  if ((rc = run_gemv(h, OP_O, lc, extra, s))) return rc;
  if ((rc = run_gemv(h, OP_GATEUP, lc, extra, s))) return rc;
  return run_gemv(h, OP_DOWN, lc, extra, s);
}

Launch mk(int kind, int stack, int sub, const Act& act, int pos0, int cnt) {
  Launch lc;
  memset(&lc, 0, sizeof(lc));
  lc.kind = kind; lc.stack = stack; lc.sub = sub; lc.pos0 = pos0; lc.cnt = cnt; lc.act = act;
  return lc;
}

bool use_step(const spd_handle* h) { return (h->opts & SPD_OPT_STEP) && h->step_smem > 0; }

// Control-block flags of an option set: the device side reads which schedule runs.
int state_flags(int opts) {
  if (opts & SPD_OPT_TARGET_ONLY) return SF_TARGET_ONLY;
  return (opts & SPD_OPT_POST_STEP) ? SF_POST_STEP : 0;
}

Phase ph_gemv(int op, int kind, const Launch& a, const Launch* b) {
  Phase P;
  memset(&P, 0, sizeof(P));
  P.type = PH_GEMV; P.kind = kind; P.nparts = b ? 2 : 1;
  P.part[0].op = op; P.part[0].lc = a;
  if (b) { P.part[1].op = op; P.part[1].lc = *b; }
  return P;
}

Phase ph_attn(int kind, const Launch& a, const Launch* b) {
  Phase P = ph_gemv(0, kind, a, b);
  P.type = PH_ATTN;
  return P;
}

// The five phases of one decoder layer (or of one co-scheduled stage-diagonal sub-step).
void layer_phases(std::vector<Phase>& v, const Launch& lc, const Launch* extra) {
  const int off = lc.stack == 1 ? 9 : 0;
  v.push_back(ph_gemv(OP_QKV, KK_QKV + off, lc, extra));
  v.push_back(ph_attn(KK_ATTN + off, lc, extra));
  v.push_back(ph_gemv(OP_O, KK_O + off, lc, extra));
  v.push_back(ph_gemv(OP_GATEUP, KK_GATEUP + off, lc, extra));
  v.push_back(ph_gemv(OP_DOWN, KK_DOWN + off, lc, extra));
}

Launch mk(int kind, int stack, int sub, const Act& act, int pos0, int cnt);

// Builds the cycle and AR programs for the current options and copies them to the device.
int build_programs(spd_handle* h) {
  if (h->step_smem == 0) return SPD_OK;
  const Dims& D = h->D;
  std::vector<Phase> cyc, ar;
  const bool pdm = !(h->opts & SPD_OPT_TARGET_ONLY);
  const bool post = pdm && (h->opts & SPD_OPT_POST_STEP);
  const bool cos = pdm && !post && (h->opts & SPD_OPT_COSCHED);
  auto draft_serial = [&]() {  // anchor FC, then the Ls draft layers on their own phases
    cyc.push_back(ph_gemv(OP_FC, KK_FC + 9, mk(LK_PDMROWS, 1, 0, h->act_p, 0, 0), nullptr));
    for (int lp = 0; lp < D.Ls; ++lp) layer_phases(cyc, mk(LK_PDMROWS, 1, lp, h->act_p, 0, 0), nullptr);
  };
  if (pdm && !post) {
    if (cos) cyc.push_back(ph_gemv(OP_FC, KK_FC + 9, mk(LK_PDMROWS, 1, 0, h->act_p, 0, 0), nullptr));
    else draft_serial();
  }
  for (int s = 0; s < D.S; ++s) {
    const Launch lt = mk(LK_DIAG, 0, s, h->act_t, 0, 0);
    const Launch lp = mk(LK_PDMROWS, 1, s, h->act_p, 0, 0);
    layer_phases(cyc, lt, (cos && s < D.Ls) ? &lp : nullptr);
  }
  if (post) draft_serial();  // on the step's output state
  cyc.push_back(ph_gemv(OP_HEAD, KK_HEAD, mk(LK_DIAG, 0, 0, h->act_head, 0, 0), nullptr));
  {
    Phase c;
    memset(&c, 0, sizeof(c));
    c.type = PH_CTRL_CYCLE; c.kind = KK_CTRL;
    cyc.push_back(c);
  }
  for (int l = 0; l < D.L; ++l) layer_phases(ar, mk(LK_AR, 0, l, h->act_t, 0, 0), nullptr);
  ar.push_back(ph_gemv(OP_HEAD, KK_HEAD, mk(LK_AR, 0, 0, h->act_head, 0, 0), nullptr));
  {
    Phase c;
    memset(&c, 0, sizeof(c));
    c.type = PH_CTRL_AR; c.kind = KK_CTRL;
    ar.push_back(c);
  }
  if ((int)cyc.size() > h->cap_prog_cycle || (int)ar.size() > h->cap_prog_ar)
    return fail(h, SPD_ESTATE, "step program larger than its buffer");
  SPD_CUDA(h, cudaMemcpy(h->d_prog_cycle, cyc.data(), sizeof(Phase) * cyc.size(), cudaMemcpyHostToDevice));
  SPD_CUDA(h, cudaMemcpy(h->d_prog_ar, ar.data(), sizeof(Phase) * ar.size(), cudaMemcpyHostToDevice));
  h->n_prog_cycle = (int)cyc.size();
  h->n_prog_ar = (int)ar.size();
  h->kinds_cycle.clear();
  h->kinds_ar.clear();
  for (const Phase& P : cyc) h->kinds_cycle.push_back(P.kind);
  for (const Phase& P : ar) h->kinds_ar.push_back(P.kind);
  return SPD_OK;
}

int enqueue_step(spd_handle* h, bool cycle) {
  h->n_launch += 1;
  unsigned long long* ns = nullptr;
  if (h->timing) {
    ns = cycle ? h->d_ns_cycle : h->d_ns_ar;
    (cycle ? h->timed_cycles : h->timed_ar) += 1;
  }
  SPD_CUDA(h, launch_step(h->D, h->B, h->LC, cycle ? h->d_prog_cycle : h->d_prog_ar,
                          cycle ? h->n_prog_cycle : h->n_prog_ar, h->d_bar, ns, h->step_smem, h->s_main));
  h->st_dirty = true;
  return SPD_OK;
}

int enqueue_cycle(spd_handle* h) {
  if (use_step(h)) return enqueue_step(h, true);
  int rc;
  const bool pdm = !(h->opts & SPD_OPT_TARGET_ONLY);
  const bool post = pdm && (h->opts & SPD_OPT_POST_STEP);
  const bool cos = pdm && !post && (h->opts & SPD_OPT_COSCHED);
  cudaStream_t sm = h->s_main;
  h->st_dirty = true;  // the previous cycle's control kernel (or the host) wrote the control block
  auto draft_fc = [&]() { return run_gemv(h, OP_FC, mk(LK_PDMROWS, 1, 0, h->act_p, 0, 0), nullptr, sm); };
  auto draft_layers = [&]() {  // serialised draft module: its Ls layers on their own launches
    for (int lp = 0; lp < h->D.Ls; ++lp)
      if (int r = enqueue_layer(h, mk(LK_PDMROWS, 1, lp, h->act_p, 0, 0), nullptr, sm)) return r;
    return (int)SPD_OK;
  };
  if (pdm && !post) {  // before the target step, on its input state
    if ((rc = draft_fc())) return rc;
    if (!cos && (rc = draft_layers())) return rc;
  }
  for (int s = 0; s < h->D.S; ++s) {
    const Launch lt = mk(LK_DIAG, 0, s, h->act_t, 0, 0);
    const Launch lp = mk(LK_PDMROWS, 1, s, h->act_p, 0, 0);
    if ((rc = enqueue_layer(h, lt, (cos && s < h->D.Ls) ? &lp : nullptr, sm))) return rc;
  }
  if (post) {  // post-step schedule: after the target step, on its output state
    if ((rc = draft_fc())) return rc;
    if ((rc = draft_layers())) return rc;
  }
  if ((rc = run_gemv(h, OP_HEAD, mk(LK_DIAG, 0, 0, h->act_head, 0, 0), nullptr, sm))) return rc;
  Timed tm(h, KK_CTRL, sm);
  SPD_CUDA(h, launch_control_cycle(h->D, h->B, sm));
  h->st_dirty = true;
  return SPD_OK;
}

int enqueue_ar_step(spd_handle* h) {
  if (use_step(h)) return enqueue_step(h, false);
  int rc;
  cudaStream_t sm = h->s_main;
  h->st_dirty = true;
  for (int l = 0; l < h->D.L; ++l)
    if ((rc = enqueue_layer(h, mk(LK_AR, 0, l, h->act_t, 0, 0), nullptr, sm))) return rc;
  if ((rc = run_gemv(h, OP_HEAD, mk(LK_AR, 0, 0, h->act_head, 0, 0), nullptr, sm))) return rc;
  Timed tm(h, KK_CTRL, sm);
  SPD_CUDA(h, launch_control_ar(h->D, h->B, sm));
  h->st_dirty = true;
  return SPD_OK;
}

void drop_graphs(spd_handle* h) {
  if (h->g_cycle) cudaGraphExecDestroy(h->g_cycle);
  if (h->g_ar) cudaGraphExecDestroy(h->g_ar);
  h->g_cycle = h->g_ar = nullptr;
}

int capture(spd_handle* h, int (*fn)(spd_handle*), cudaGraphExec_t* out, int64_t* nodes) {
  SPD_CUDA(h, cudaStreamBeginCapture(h->s_main, cudaStreamCaptureModeThreadLocal));
  const bool saved = h->timing;
  h->timing = false;
  const int64_t n0 = h->n_launch;
  const int rc = fn(h);
  *nodes = h->n_launch - n0;
  h->n_launch = n0;
  h->timing = saved;
  cudaGraph_t g = nullptr;
  const cudaError_t e = cudaStreamEndCapture(h->s_main, &g);
  if (rc) { if (g) cudaGraphDestroy(g); return rc; }
  if (e != cudaSuccess) return fail(h, SPD_ECUDA, "graph capture: %s", cudaGetErrorString(e));
  const cudaError_t e2 = cudaGraphInstantiate(out, g, 0);
  cudaGraphDestroy(g);
  if (e2 != cudaSuccess) return fail(h, SPD_ECUDA, "graph instantiate: %s", cudaGetErrorString(e2));
  return SPD_OK;
}

int run_cycle(spd_handle* h) {
  if ((h->opts & SPD_OPT_GRAPHS) && !h->timing) {
    if (!h->g_cycle) {
      const int rc = capture(h, enqueue_cycle, &h->g_cycle, &h->graph_nodes_cycle);
      if (rc) return rc;
    }
    SPD_CUDA(h, cudaGraphLaunch(h->g_cycle, h->s_main));
    h->n_launch += h->graph_nodes_cycle;
    return SPD_OK;
  }
  return enqueue_cycle(h);
}

int run_ar(spd_handle* h) {
  if ((h->opts & SPD_OPT_GRAPHS) && !h->timing) {
    if (!h->g_ar) {
      const int rc = capture(h, enqueue_ar_step, &h->g_ar, &h->graph_nodes_ar);
      if (rc) return rc;
    }
    SPD_CUDA(h, cudaGraphLaunch(h->g_ar, h->s_main));
    h->n_launch += h->graph_nodes_ar;
    return SPD_OK;
  }
  return enqueue_ar_step(h);
}

int read_state(spd_handle* h) {
  SPD_CUDA(h, cudaMemcpyAsync(h->host_state, h->B.st, sizeof(DevState), cudaMemcpyDeviceToHost,
                              h->s_main));
  SPD_CUDA(h, cudaStreamSynchronize(h->s_main));
  return SPD_OK;
}

int state_error(spd_handle* h) {
  const DevState& s = *h->host_state;
  if (s.err & ERR_TIMEOUT)
    return fail(h, SPD_ETIMEOUT, "a bounded device wait gave up (site %d)", s.err_where);
  if (s.err & ERR_PDM_ROWS)
    return fail(h, SPD_ESTATE, "draft-module cache out of step (t=%d, cached=%d); call spd_rollback",
                s.t, s.pdm_len);
  if (s.err)
    return fail(h, SPD_ESTATE, "device error flag %d (site %d)", s.err, s.err_where);
  return SPD_OK;
}

int copy_out(spd_handle* h, int32_t* out, int count) {
  if (!out || count <= 0) return SPD_OK;
  SPD_CUDA(h, cudaMemcpyAsync(out, h->B.seq + h->P + 1, sizeof(int32_t) * count, cudaMemcpyDefault,
                              h->s_main));
  SPD_CUDA(h, cudaStreamSynchronize(h->s_main));
  return SPD_OK;
}

int generate(spd_handle* h, int32_t max_new, int32_t* out, int32_t* n_out, spd_stats* stats,
             bool ar) {
  if (!h) return SPD_EINVAL;
  if (!h->prefilled) return fail(h, SPD_ESTATE, "generate before prefill");
  if (max_new < 1) return fail(h, SPD_EINVAL, "max_new must be >= 1");
  if (h->P + max_new + h->D.n + 1 > h->D.max_seq)
    return fail(h, SPD_EINVAL, "P + max_new + n + 1 = %d exceeds max_seq %d",
                h->P + max_new + h->D.n + 1, h->D.max_seq);
  int rc;
  const int64_t launches0 = h->n_launch;
  SPD_CUDA(h, launch_begin_generate(h->D, h->B, max_new, h->s_main));
  h->n_launch += 1;
  if ((rc = read_state(h))) return rc;
  if ((rc = state_error(h))) return rc;
  const DevState s0 = *h->host_state;
  SPD_CUDA(h, cudaEventRecord(h->ev_t0, h->s_main));
  int committed = s0.v + 1 - s0.P;
  while (committed < max_new) {
    const int batch = max_new - committed;  // each cycle commits at most one token
    for (int i = 0; i < batch; ++i)
      if ((rc = ar ? run_ar(h) : run_cycle(h))) return rc;
    if ((rc = read_state(h))) return rc;
    if ((rc = state_error(h))) return rc;
    committed = h->host_state->v + 1 - h->host_state->P;
  }
  SPD_CUDA(h, cudaEventRecord(h->ev_t1, h->s_main));
  SPD_CUDA(h, cudaEventSynchronize(h->ev_t1));
  if ((rc = copy_out(h, out, max_new))) return rc;
  if (n_out) *n_out = out ? max_new : 0;
  if (stats) {
    float ms = 0.f;
    cudaEventElapsedTime(&ms, h->ev_t0, h->ev_t1);
    stats->cycles = h->host_state->cycles - s0.cycles;
    stats->exits = h->host_state->exits - s0.exits;
    stats->rejects = h->host_state->rejects - s0.rejects;
    stats->committed = committed;
    stats->device_ms = ms;
    stats->kernel_launches = h->n_launch - launches0;
  }
  return SPD_OK;
}

}  // namespace

namespace spd {
int spd_internal_fail(int code, const char* msg) { return fail(nullptr, code, "%s", msg); }
}  // namespace spd

extern "C" {

const char* spd_last_error(const spd_handle* h) {
  return h ? h->err.c_str() : g_create_error.c_str();
}

void spd_destroy(spd_handle* h) {
  if (!h) return;
  if (h->s_main) cudaStreamSynchronize(h->s_main);
  drop_graphs(h);
  for (void* p : h->allocs) cudaFree(p);
  for (cudaEvent_t e : h->pool) cudaEventDestroy(e);
  if (h->ev_t0) cudaEventDestroy(h->ev_t0);
  if (h->ev_t1) cudaEventDestroy(h->ev_t1);
  if (h->own_main && h->s_main) cudaStreamDestroy(h->s_main);
  if (h->host_state) cudaFreeHost(h->host_state);
  delete h;
}

int spd_create(const spd_config* cfg, const spd_weights* w, void* cuda_stream, spd_handle** out) {
  if (out) *out = nullptr;
  if (!cfg || !w || !out) return fail(nullptr, SPD_EINVAL, "NULL argument");
  const spd_config& c = *cfg;
  if (c.n_layers < 1 || c.d_model < 8 || c.n_heads < 1 || c.n_kv_heads < 1 || c.head_dim < 16 ||
      c.d_ffn < 8 || c.vocab < 2 || c.n_stages < 1 || c.n_stages > SPD_MAX_STAGES ||
      c.n_anchors < 1 || c.n_anchors > SPD_MAX_ANCHORS || c.max_seq < 4)
    return fail(nullptr, SPD_EINVAL, "config value out of range");
  if (c.n_layers % c.n_stages != 0)
    return fail(nullptr, SPD_EINVAL, "n_stages=%d must divide n_layers=%d", c.n_stages, c.n_layers);
  const int S = c.n_layers / c.n_stages;
  if (c.pdm_layers < 1 || c.pdm_layers > S)
    return fail(nullptr, SPD_EINVAL, "pdm_layers=%d must satisfy 1 <= Ls <= L/n = %d", c.pdm_layers, S);
  if (c.anchors[0] != 0) return fail(nullptr, SPD_EINVAL, "anchors[0] must be 0 (the embedding)");
  for (int i = 1; i < c.n_anchors; ++i)
    if (c.anchors[i] <= c.anchors[i - 1])
      return fail(nullptr, SPD_EINVAL, "anchors must increase strictly");
  if (c.anchors[c.n_anchors - 1] > c.n_layers)
    return fail(nullptr, SPD_EINVAL, "anchors must be <= n_layers");
  if (c.n_heads % c.n_kv_heads != 0) return fail(nullptr, SPD_EINVAL, "n_heads %% n_kv_heads != 0");
  if (c.head_dim % 64 != 0 || c.head_dim > 256)
    return fail(nullptr, SPD_EINVAL, "head_dim must be a multiple of 64, <= 256");
  if (c.d_model % 8 || c.d_ffn % 8) return fail(nullptr, SPD_EINVAL, "d_model and d_ffn must be multiples of 8");
  if (c.dtype != SPD_DTYPE_F32 && c.dtype != SPD_DTYPE_BF16) return fail(nullptr, SPD_EINVAL, "bad dtype");
  const int gq = c.n_heads / c.n_kv_heads;
  if (kAttnQT * gq > 64) return fail(nullptr, SPD_EINVAL, "query heads per kv head too large");

  spd_handle* h = new spd_handle();
  h->cfg = c;
  h->esz = c.dtype == SPD_DTYPE_BF16 ? 2 : 4;
  Dims& D = h->D;
  memset(&D, 0, sizeof(D));
  D.L = c.n_layers; D.d = c.d_model; D.hq = c.n_heads; D.hkv = c.n_kv_heads; D.hd = c.head_dim;
  D.ffn = c.d_ffn; D.V = c.vocab; D.n = c.n_stages; D.S = S; D.Ls = c.pdm_layers; D.m = c.n_anchors;
  D.max_seq = c.max_seq; D.dtype = c.dtype; D.qkv_rows = (c.n_heads + 2 * c.n_kv_heads) * c.head_dim;
  D.gq = gq; D.eps = c.norm_eps;
  D.box3 = box3_cols(c.d_model, c.dtype) && box3_cols(c.d_ffn, c.dtype);  // every streamed matrix's cols
  D.tc = D.box3 && c.dtype == SPD_DTYPE_BF16 && c.head_dim <= 128;       // tcgen05 draft tiles
  for (int i = 0; i < c.n_anchors; ++i) D.anchors[i] = c.anchors[i];
  // f(k) = max{i : b_i <= lmax(k)}, lmax(k) = min(L, k*L/n)   (SPD summary, 核心方法)
  for (int k = 0; k <= c.n_stages; ++k) {
    const int lm = k * S < c.n_layers ? k * S : c.n_layers;
    int f = 0;
    for (int i = 0; i < c.n_anchors; ++i)
      if (c.anchors[i] <= lm) f = i;
    D.ftab[k] = f;
  }
  // weights
  auto bad = [&](const void* p) { return p == nullptr || !aligned16(p); };
  if (bad(w->embed) || bad(w->final_norm) || bad(w->lm_head) || bad(w->pdm_norm) || bad(w->pdm_lm_head) ||
      !w->layers || !w->pdm_layers || !w->pdm_fc) {
    delete h;
    return fail(nullptr, SPD_EINVAL, "a weight pointer is NULL or not 16-byte aligned");
  }
  std::vector<LayerW> tl(c.n_layers), pl(c.pdm_layers);
  auto conv = [&](const spd_layer_weights& s, LayerW& o) {
    o.attn_norm = s.attn_norm; o.wq = s.wq; o.wk = s.wk; o.wv = s.wv; o.wo = s.wo;
    o.ffn_norm = s.ffn_norm; o.wg = s.w_gate; o.wu = s.w_up; o.wd = s.w_down;
    return !(bad(o.attn_norm) || bad(o.wq) || bad(o.wk) || bad(o.wv) || bad(o.wo) || bad(o.ffn_norm) ||
             bad(o.wg) || bad(o.wu) || bad(o.wd));
  };
  for (int l = 0; l < c.n_layers; ++l)
    if (!conv(w->layers[l], tl[l])) { delete h; return fail(nullptr, SPD_EINVAL, "target layer %d: bad pointer", l); }
  for (int l = 0; l < c.pdm_layers; ++l)
    if (!conv(w->pdm_layers[l], pl[l])) { delete h; return fail(nullptr, SPD_EINVAL, "draft layer %d: bad pointer", l); }
  Bufs& B = h->B;
  memset(&B, 0, sizeof(B));
  for (int j = 0; j < c.n_anchors; ++j) {
    B.fc[j] = w->pdm_fc[j];
    if (B.fc[j] && !aligned16(B.fc[j])) { delete h; return fail(nullptr, SPD_EINVAL, "pdm_fc[%d] not aligned", j); }
  }
  for (int k = 0; k <= c.n_stages; ++k)
    if (!B.fc[D.ftab[k]]) {
      delete h;
      return fail(nullptr, SPD_EINVAL, "pdm_fc[%d] is needed (depth %d) but NULL", D.ftab[k], k);
    }
  B.embed = w->embed; B.lm_head = w->lm_head; B.pdm_head = w->pdm_lm_head;
  B.final_norm = (const float*)w->final_norm; B.pdm_norm = (const float*)w->pdm_norm;

  cudaError_t e = cudaSuccess;
  const int n = c.n_stages, d = c.d_model, m = c.n_anchors;
  const size_t ms = c.max_seq, hd = c.head_dim;
  const int PB = kPrefillBlock;
#define ALLOC(ptr, T, count)                                                       \
  do {                                                                             \
    ptr = dalloc<T>(h, (count), &e);                                               \
    if (e != cudaSuccess) {                                                        \
      std::string msg = std::string("cudaMalloc: ") + cudaGetErrorString(e);       \
      spd_destroy(h);                                                              \
      return fail(nullptr, e == cudaErrorMemoryAllocation ? SPD_ENOMEM : SPD_ECUDA, "%s", msg.c_str()); \
    }                                                                              \
  } while (0)
  // tensor maps of every weight matrix the GEMV engine streams (7 per layer, FCs, two heads)
  {
    const int per = D.tc ? 2 : 1;  // with tcgen05 tiles every stream map is followed by its 128-row map
    const int nmaps = per * (7 * (c.n_layers + c.pdm_layers) + c.n_anchors + 2);
    CUtensorMap* dmaps;
    ALLOC(dmaps, CUtensorMap, nmaps);
    std::vector<CUtensorMap> hm(nmaps);
    int k = 0;
    const int qr = c.n_heads * c.head_dim, kr = c.n_kv_heads * c.head_dim;
    auto enc = [&](const void* W, int rows, int cols) -> const CUtensorMap* {
      if (e == cudaSuccess) e = gemv_encode_map(&hm[k], W, rows, cols, c.dtype, D.box3 != 0);
      if (per == 2 && e == cudaSuccess) e = gemv_encode_tc_map(&hm[k + 1], W, rows, cols);
      const CUtensorMap* m = dmaps + k;
      k += per;
      return m;
    };
    auto layer_maps = [&](LayerW& o) {
      o.tq = enc(o.wq, qr, c.d_model); o.tk = enc(o.wk, kr, c.d_model); o.tv = enc(o.wv, kr, c.d_model);
      o.to = enc(o.wo, c.d_model, qr);
      o.tg = enc(o.wg, c.d_ffn, c.d_model); o.tu = enc(o.wu, c.d_ffn, c.d_model);
      o.td = enc(o.wd, c.d_model, c.d_ffn);
    };
    for (auto& o : tl) layer_maps(o);
    for (auto& o : pl) layer_maps(o);
    for (int j = 0; j < c.n_anchors; ++j)
      B.tm_fc[j] = B.fc[j] ? enc(B.fc[j], c.d_model, (j + 1) * c.d_model) : nullptr;
    B.tm_lm = enc(B.lm_head, c.vocab, c.d_model);
    B.tm_pdm = enc(B.pdm_head, c.vocab, c.d_model);
    if (e == cudaSuccess) e = cudaMemcpy(dmaps, hm.data(), sizeof(CUtensorMap) * nmaps, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) {
      std::string msg = cudaGetErrorString(e);
      spd_destroy(h);
      return fail(nullptr, SPD_ECUDA, "tensor maps: %s", msg.c_str());
    }
  }
  LayerW *dtl, *dpl;
  ALLOC(dtl, LayerW, c.n_layers);
  ALLOC(dpl, LayerW, c.pdm_layers);
  e = cudaMemcpy(dtl, tl.data(), sizeof(LayerW) * c.n_layers, cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(dpl, pl.data(), sizeof(LayerW) * c.pdm_layers, cudaMemcpyHostToDevice);
  if (e != cudaSuccess) { spd_destroy(h); return fail(nullptr, SPD_ECUDA, "cudaMemcpy: %s", cudaGetErrorString(e)); }
  B.tl = dtl; B.pl = dpl;
  unsigned char *kc, *vc, *pkc, *pvc;
  const size_t kv_t = (size_t)c.n_layers * c.n_kv_heads * ms * hd * h->esz;
  const size_t kv_p = (size_t)c.pdm_layers * c.n_kv_heads * ms * hd * h->esz;
  ALLOC(kc, unsigned char, kv_t); ALLOC(vc, unsigned char, kv_t);
  ALLOC(pkc, unsigned char, kv_p); ALLOC(pvc, unsigned char, kv_p);
  B.kc = kc; B.vc = vc; B.pkc = pkc; B.pvc = pvc;
  ALLOC(B.st, DevState, 1);
  ALLOC(B.seq, int, ms + 2);
  ALLOC(B.trace, int, 2 * ms);
  ALLOC(B.kvlen, int, c.n_layers);
  ALLOC(B.ovr_ref, int, ms + 2);
  ALLOC(B.ovr_mode, unsigned char, ms + 2);
  ALLOC(B.resid, float, (size_t)(n + 1) * d);
  ALLOC(B.anch, float, (size_t)(n + 1) * m * d);
  float *rc_, *rs_;
  ALLOC(rc_, float, ms * hd / 2);
  ALLOC(rs_, float, ms * hd / 2);
  B.rope_cos = rc_; B.rope_sin = rs_;
  B.head_grid = gemv_head_grid(c.dtype);
  ALLOC(B.head_part, float, (size_t)B.head_grid * 8);
  ALLOC(B.logits, float, (size_t)2 * c.vocab);
  {  // sampled decoding: uniforms by position, draft distributions by position % (n+1)
    float* u;
    ALLOC(u, float, (size_t)4 * (c.max_seq + 2));
    B.u_smp = u;
    ALLOC(B.q_prob, float, (size_t)(n + 1) * kMaxTopK);
    ALLOC(B.q_id, int, (size_t)(n + 1) * kMaxTopK);
  }
  const int qkvr = D.qkv_rows, hqd = c.n_heads * c.head_dim, f = c.d_ffn;
  // target decode scratch
  Act& T = h->act_t;
  T.resid = B.resid; T.resid_ring = n + 1; T.anch = B.anch; T.anch_ring = n + 1;
  ALLOC(T.qkv, float, (size_t)n * qkvr);
  ALLOC(T.attn, float, (size_t)n * hqd);
  ALLOC(T.u, float, (size_t)n * f);
  const int part_rows_t = n > PB ? n : PB;
  {  // prefill blocks use 128-key chunks, the step kernel 64-key chunks
    const size_t a1 = attn_part_floats(part_rows_t, c.n_heads, c.head_dim, c.max_seq, kAttnChunk);
    const size_t a2 = attn_part_floats(n, c.n_heads, c.head_dim, c.max_seq, kStepChunk);
    ALLOC(T.part, float, a1 > a2 ? a1 : a2);
  }
  ALLOC(T.tick, int, (size_t)kMaxTiles * c.n_kv_heads);
  // draft rows
  Act& Pm = h->act_p;
  ALLOC(h->p_z, float, (size_t)(n + 2) * d);
  Pm.resid = h->p_z; Pm.resid_ring = kBigRing; Pm.anch = nullptr;
  ALLOC(Pm.qkv, float, (size_t)(n + 2) * qkvr);
  ALLOC(Pm.attn, float, (size_t)(n + 2) * hqd);
  ALLOC(Pm.u, float, (size_t)(n + 2) * f);
  ALLOC(Pm.part, float, attn_part_floats(n + 2, c.n_heads, c.head_dim, c.max_seq, kStepChunk));
  ALLOC(Pm.tick, int, (size_t)kMaxTiles * c.n_kv_heads);
  // head: target rows in the ring, draft row z in act.qkv
  h->act_head = T;
  h->act_head.qkv = h->p_z;
  // prefill blocks
  Act& F = h->act_pf;
  ALLOC(F.resid, float, (size_t)PB * d);
  F.resid_ring = kBigRing;
  ALLOC(F.anch, float, (size_t)PB * m * d);
  F.anch_ring = kBigRing;
  ALLOC(F.qkv, float, (size_t)PB * qkvr);
  ALLOC(F.attn, float, (size_t)PB * hqd);
  ALLOC(F.u, float, (size_t)PB * f);
  F.part = T.part; F.tick = T.tick;
  Act& FP = h->act_pfp;
  FP = F;
  ALLOC(FP.resid, float, (size_t)PB * d);
  FP.anch = F.anch;  // anchor source of the prefix rows for the draft FC
  // split-K partials and tickets of the tcgen05 groups (one launch or one step-kernel phase at a time)
  if (D.tc) {
    B.tc_part_cap = 8 << 20;
    B.tc_tick_cap = 4096;
    ALLOC(B.tc_part, float, (size_t)B.tc_part_cap);
    ALLOC(B.tc_tick, int, (size_t)B.tc_tick_cap);
  }
  // prefill attention on the tensor cores: maps over the whole caches (row = layer, kv head, position)
  if (pfattn_supported(c.dtype, hd, PB, gq)) {
    const int sms = num_sms();
    ALLOC(h->pf_part, float, pfattn_part_floats(c.n_kv_heads, gq, ms, sms));
    ALLOC(h->pf_tick, int, (size_t)c.n_heads);
    const long long rt = (long long)c.n_layers * c.n_kv_heads * ms, rp = (long long)c.pdm_layers * c.n_kv_heads * ms;
    e = pfattn_encode_map(&h->pf_map[0], kc, rt, hd);
    if (e == cudaSuccess) e = pfattn_encode_map(&h->pf_map[1], vc, rt, hd);
    if (e == cudaSuccess) e = pfattn_encode_map(&h->pf_map[2], pkc, rp, hd);
    if (e == cudaSuccess) e = pfattn_encode_map(&h->pf_map[3], pvc, rp, hd);
    if (e == cudaSuccess) e = pfattn_setup_attributes();
    if (e != cudaSuccess) { spd_destroy(h); return fail(nullptr, SPD_ECUDA, "prefill attention set-up: %s", cudaGetErrorString(e)); }
    h->pf_on = true;
  }
  e = cudaMallocHost(reinterpret_cast<void**>(&h->host_state), sizeof(DevState));
  if (e != cudaSuccess) { spd_destroy(h); return fail(nullptr, SPD_ENOMEM, "cudaMallocHost failed"); }
  memset(h->host_state, 0, sizeof(DevState));

  if (cuda_stream) {
    h->s_main = reinterpret_cast<cudaStream_t>(cuda_stream);
  } else {
    e = cudaStreamCreate(&h->s_main);  // blocking: orders with the legacy default stream
    h->own_main = true;
  }
  if (e == cudaSuccess) e = cudaEventCreate(&h->ev_t0);
  if (e == cudaSuccess) e = cudaEventCreate(&h->ev_t1);
  if (e == cudaSuccess) e = gemv_setup_attributes();
  const size_t asm_ = attn_smem_bytes(D, true) > attn_smem_bytes(D, false) ? attn_smem_bytes(D, true)
                                                                           : attn_smem_bytes(D, false);
  if (e == cudaSuccess) e = attn_setup_attributes(asm_);
  // persistent step kernel: programs, grid barrier, per-phase timers
  h->step_smem = step_smem_bytes(D);
  if (e == cudaSuccess && h->step_smem) {
    e = step_setup_attributes(h->step_smem);
    if (e != cudaSuccess) {  // the per-operator path remains
      cudaGetLastError();
      e = cudaSuccess;
      h->step_smem = 0;
    }
  }
  if (e == cudaSuccess && h->step_smem) {
    h->cap_prog_cycle = 1 + 5 * (D.S + D.Ls) + 2;
    h->cap_prog_ar = 5 * D.L + 2;
    ALLOC(h->d_prog_cycle, Phase, h->cap_prog_cycle);
    ALLOC(h->d_prog_ar, Phase, h->cap_prog_ar);
    ALLOC(h->d_bar, unsigned, 2);
    ALLOC(h->d_ns_cycle, unsigned long long, h->cap_prog_cycle);
    ALLOC(h->d_ns_ar, unsigned long long, h->cap_prog_ar);
  }
#undef ALLOC
  if (e == cudaSuccess) {
    h->LC.sms = num_sms();
    h->LC.gemv_grid = 0;
    h->LC.attn_grid_decode = attn_grid(D, false);
    h->LC.attn_grid_multi = attn_grid(D, true);
    h->LC.debug_logits = 0;
    e = launch_rope_tables(rc_, rs_, c.max_seq, c.head_dim, c.rope_theta, h->s_main);
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(h->s_main);
  if (e != cudaSuccess) {
    std::string msg = cudaGetErrorString(e);
    spd_destroy(h);
    return fail(nullptr, SPD_ECUDA, "setup: %s", msg.c_str());
  }
  int rcp;
  if ((rcp = build_programs(h))) {
    const std::string msg = h->err;
    spd_destroy(h);
    return fail(nullptr, rcp, "%s", msg.c_str());
  }
  *out = h;
  return SPD_OK;
}

int spd_prefill(spd_handle* h, const int32_t* tokens, int32_t P, int32_t* first_token) {
  if (!h) return SPD_EINVAL;
  if (!tokens || P < 1) return fail(h, SPD_EINVAL, "need a prompt of >= 1 token");
  if (P + h->D.n + 2 > h->D.max_seq) return fail(h, SPD_EINVAL, "prompt too long for max_seq");
  for (int i = 0; i < P; ++i)
    if (tokens[i] < 0 || tokens[i] >= h->D.V) return fail(h, SPD_EINVAL, "token %d out of range", i);
  cudaStream_t s = h->s_main;
  const Dims& D = h->D;
  h->prefilled = false;
  SPD_CUDA(h, cudaMemcpyAsync(h->B.seq + 1, tokens, sizeof(int32_t) * P, cudaMemcpyHostToDevice, s));
  SPD_CUDA(h, cudaMemsetAsync(h->B.ovr_mode, 0, D.max_seq + 2, s));
  SPD_CUDA(h, cudaMemsetAsync(h->B.st, 0, sizeof(DevState), s));
  if (h->d_bar) SPD_CUDA(h, cudaMemsetAsync(h->d_bar, 0, 2 * sizeof(unsigned), s));
  const int flags = state_flags(h->opts);
  h->host_state->flags = flags;
  SPD_CUDA(h, cudaMemcpyAsync(&h->B.st->flags, &h->host_state->flags, sizeof(int),
                              cudaMemcpyHostToDevice, s));
  SPD_CUDA(h, cudaStreamSynchronize(s));  // host_state is reused below
  int rc, cnt = 0;
  for (int p0 = 1; p0 <= P; p0 += kPrefillBlock) {
    cnt = P - p0 + 1 < kPrefillBlock ? P - p0 + 1 : kPrefillBlock;
    SPD_CUDA(h, launch_prefill_embed(D, h->B, h->act_pf.resid, h->act_pf.anch, p0, cnt, s));
    h->st_dirty = true;
    for (int l = 0; l < D.L; ++l)
      if ((rc = enqueue_layer(h, mk(LK_ROWS, 0, l, h->act_pf, p0, cnt), nullptr, s))) return rc;
    // draft-module prefix rows at depth n (cached verified features, SPD v3 App. A.1)
    if ((rc = run_gemv(h, OP_FC, mk(LK_ROWS, 1, 0, h->act_pfp, p0, cnt), nullptr, s))) return rc;
    for (int lp = 0; lp < D.Ls; ++lp)
      if ((rc = enqueue_layer(h, mk(LK_ROWS, 1, lp, h->act_pfp, p0, cnt), nullptr, s))) return rc;
  }
  if ((rc = run_gemv(h, OP_HEAD, mk(LK_ROWS, 0, 0, h->act_pf, P - cnt + 1, cnt), nullptr, s))) return rc;
  SPD_CUDA(h, launch_prefill_finish(D, h->B, P, s));
  h->P = P;
  h->prefilled = true;
  if (first_token) {
    if ((rc = read_state(h))) return rc;
    if ((rc = state_error(h))) return rc;
    *first_token = h->host_state->pushed;
  }
  return SPD_OK;
}

int spd_cycle(spd_handle* h, spd_cycle_info* info) {
  if (!h) return SPD_EINVAL;
  if (!h->prefilled) return fail(h, SPD_ESTATE, "cycle before prefill");
  int rc;
  SPD_CUDA(h, launch_begin_generate(h->D, h->B, 0x7fffffff, h->s_main));
  if ((rc = run_cycle(h))) return rc;
  if (info) {
    if ((rc = read_state(h))) return rc;
    if ((rc = state_error(h))) return rc;
    const DevState& s = *h->host_state;
    info->t = s.t; info->a = s.a; info->v = s.v;
    info->exited = s.last_exited; info->exit_pos = s.last_exit_pos; info->accepted = s.last_accept;
    info->target_top1 = s.target_top1; info->pdm_top1 = s.pdm_top1; info->pdm_top2 = s.pdm_top2;
    info->draft_token = s.draft; info->pushed_token = s.pushed;
  }
  return SPD_OK;
}

int spd_generate(spd_handle* h, int32_t max_new, int32_t* out, int32_t* n_out, spd_stats* stats) {
  return generate(h, max_new, out, n_out, stats, false);
}

int spd_generate_ar(spd_handle* h, int32_t max_new, int32_t* out, int32_t* n_out, spd_stats* stats) {
  return generate(h, max_new, out, n_out, stats, true);
}

int spd_rollback(spd_handle* h, int32_t keep_len, int32_t reseed_token) {
  if (!h) return SPD_EINVAL;
  if (!h->prefilled) return fail(h, SPD_ESTATE, "rollback before prefill");
  int rc;
  if ((rc = read_state(h))) return rc;
  const int v = h->host_state->v;
  if (keep_len < 1 || keep_len > v)
    return fail(h, SPD_EINVAL, "keep_len %d outside 1..verified length %d", keep_len, v);
  if (reseed_token < 0 || reseed_token >= h->D.V) return fail(h, SPD_EINVAL, "reseed token out of range");
  if (keep_len + h->D.n + 2 > h->D.max_seq) return fail(h, SPD_EINVAL, "keep_len too large");
  SPD_CUDA(h, cudaMemsetAsync(&h->B.st->err, 0, sizeof(int), h->s_main));
  if (h->d_bar) SPD_CUDA(h, cudaMemsetAsync(h->d_bar, 0, 2 * sizeof(unsigned), h->s_main));
  SPD_CUDA(h, launch_rollback(h->D, h->B, keep_len, reseed_token, h->s_main));
  return SPD_OK;
}

int spd_set_draft_override(spd_handle* h, int32_t first_pos, int32_t count, const int32_t* ref,
                           const uint8_t* modes) {
  if (!h) return SPD_EINVAL;
  if (count < 0 || first_pos < 1 || first_pos + count > h->D.max_seq + 2 || (count && (!ref || !modes)))
    return fail(h, SPD_EINVAL, "override range outside 1..max_seq");
  for (int i = 0; i < count; ++i) {
    if (modes[i] > 2) return fail(h, SPD_EINVAL, "mode %d at %d", modes[i], i);
    if (ref[i] < 0 || ref[i] >= h->D.V) return fail(h, SPD_EINVAL, "ref token out of range at %d", i);
  }
  if (!count) return SPD_OK;
  SPD_CUDA(h, cudaMemcpyAsync(h->B.ovr_ref + first_pos, ref, sizeof(int32_t) * count,
                              cudaMemcpyHostToDevice, h->s_main));
  SPD_CUDA(h, cudaMemcpyAsync(h->B.ovr_mode + first_pos, modes, count, cudaMemcpyHostToDevice,
                              h->s_main));
  SPD_CUDA(h, cudaStreamSynchronize(h->s_main));
  return SPD_OK;
}

int spd_acceptance_modes(double alpha, uint64_t seed, int32_t first_pos, int32_t count, uint8_t* modes) {
  if (count < 0 || (count && !modes) || first_pos < 0)
    return fail(nullptr, SPD_EINVAL, "acceptance modes: bad range or NULL output");
  // SplitMix64 (Steele, Lea, Flood, OOPSLA 2014): one step from state x = seed ^ q * golden, i.e.
  // mix(x + golden); the coin is its top 53 bits over 2^53, compared with alpha in double precision
  const uint64_t golden = 0x9E3779B97F4A7C15ull;
  for (int32_t i = 0; i < count; ++i) {
    const uint64_t q = (uint64_t)(first_pos + i);
    uint64_t z = (seed ^ (q * golden)) + golden;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    z ^= z >> 31;
    const double coin = (double)(z >> 11) / 9007199254740992.0;  // 2^53
    modes[i] = coin < alpha ? 1 : 2;
  }
  return SPD_OK;
}

int spd_set_acceptance(spd_handle* h, double alpha, uint64_t seed, const int32_t* ref_tokens, int32_t n_ref) {
  if (!h) return SPD_EINVAL;
  if (!h->prefilled) return fail(h, SPD_ESTATE, "set_acceptance before prefill");
  const int P = h->P;
  if (alpha < 0.0) {  // knob off: raw draft-module drafts
    SPD_CUDA(h, cudaMemsetAsync(h->B.ovr_mode, 0, h->D.max_seq + 2, h->s_main));
    SPD_CUDA(h, cudaStreamSynchronize(h->s_main));
    return SPD_OK;
  }
  if (!(alpha <= 1.0)) return fail(h, SPD_EINVAL, "alpha must be <= 1 (or < 0 to switch the knob off)");
  if (n_ref < 1 || !ref_tokens) return fail(h, SPD_EINVAL, "need >= 1 reference token");
  if (P + n_ref > h->D.max_seq) return fail(h, SPD_EINVAL, "P + n_ref exceeds max_seq");
  // positions P+2..P+n_ref are drafted (P+1 comes from the prefill); ref_tokens[i] is position P+1+i
  const int count = n_ref - 1;
  if (!count) return SPD_OK;
  std::vector<uint8_t> modes(count);
  int rc;
  if ((rc = spd_acceptance_modes(alpha, seed, P + 2, count, modes.data()))) return fail(h, rc, "%s", g_create_error.c_str());
  return spd_set_draft_override(h, P + 2, count, ref_tokens + 1, modes.data());
}

int spd_debug_wait_timeout(spd_handle* h, int32_t which, int64_t limit_ns) {
  if (!h) return SPD_EINVAL;
  if (which < 0 || which > 2 || limit_ns < 1000 || limit_ns > (int64_t)kWaitLimitNs)
    return fail(h, SPD_EINVAL, "which must be 0..2 and limit_ns in [1e3, %llu]", (unsigned long long)kWaitLimitNs);
  cudaStream_t s = h->s_main;
  SPD_CUDA(h, cudaMemsetAsync(&h->B.st->err, 0, sizeof(int), s));
  SPD_CUDA(h, cudaMemsetAsync(&h->B.st->err_where, 0, sizeof(int), s));
  // a word of the control block that no kernel writes stands for a grid-barrier count nobody adds to
  SPD_CUDA(h, launch_wait_selftest(h->B.st, reinterpret_cast<unsigned*>(&h->B.st->pad0), which,
                                   (uint64_t)limit_ns, s));
  int rc;
  if ((rc = read_state(h))) return rc;
  const int verdict = state_error(h);  // SPD_ETIMEOUT when the wait gave up, as it must
  SPD_CUDA(h, cudaMemsetAsync(&h->B.st->err, 0, sizeof(int), s));
  SPD_CUDA(h, cudaMemsetAsync(&h->B.st->err_where, 0, sizeof(int), s));
  SPD_CUDA(h, cudaStreamSynchronize(s));
  return verdict;
}

int spd_set_sampling(spd_handle* h, float temperature, int32_t top_k, int32_t first_pos, int32_t count,
                     const float* uniforms) {
  if (!h) return SPD_EINVAL;
  const bool on = temperature > 0.f;
  if (on && (top_k < 1 || top_k > kMaxTopK || !(temperature < 1e30f)))
    return fail(h, SPD_EINVAL, "top_k must be 1..%d and the temperature finite", kMaxTopK);
  if (count < 0 || first_pos < 1 || (size_t)first_pos + count > (size_t)h->D.max_seq + 2 || (count && !uniforms))
    return fail(h, SPD_EINVAL, "uniform range outside 1..max_seq+1");
  for (int i = 0; i < 4 * count; ++i)
    if (!(uniforms[i] >= 0.f && uniforms[i] < 1.f)) return fail(h, SPD_EINVAL, "uniform %d outside [0, 1)", i);
  SPD_CUDA(h, cudaStreamSynchronize(h->s_main));
  const int k = on ? top_k : 0;
  const float T = on ? temperature : 0.f;
  if (k != h->D.top_k || T != h->D.temp) drop_graphs(h);  // graphs hold the kernels' parameters
  h->D.top_k = k;
  h->D.temp = T;
  h->LC.debug_logits = ((h->opts & SPD_OPT_DEBUG_LOGITS) || k > 0) ? 1 : 0;
  const size_t L = (size_t)h->D.max_seq + 2;
  float* u = const_cast<float*>(h->B.u_smp);
  for (int s = 0; s < 4 && count; ++s)
    SPD_CUDA(h, cudaMemcpyAsync(u + s * L + first_pos, uniforms + (size_t)s * count, sizeof(float) * count,
                                cudaMemcpyHostToDevice, h->s_main));
  SPD_CUDA(h, cudaStreamSynchronize(h->s_main));
  return SPD_OK;
}

int spd_set_options(spd_handle* h, int32_t flags) {
  if (!h) return SPD_EINVAL;
  if (flags & ~(SPD_OPT_GRAPHS | SPD_OPT_COSCHED | SPD_OPT_TARGET_ONLY | SPD_OPT_DEBUG_LOGITS | SPD_OPT_PDL |
                SPD_OPT_STEP | SPD_OPT_POST_STEP))
    return fail(h, SPD_EINVAL, "unknown option bits");
  SPD_CUDA(h, cudaStreamSynchronize(h->s_main));
  if ((flags ^ h->opts) & (SPD_OPT_COSCHED | SPD_OPT_TARGET_ONLY | SPD_OPT_DEBUG_LOGITS | SPD_OPT_PDL |
                           SPD_OPT_STEP | SPD_OPT_POST_STEP))
    drop_graphs(h);
  h->opts = flags;
  int rcp;
  if ((rcp = build_programs(h))) return rcp;
  h->LC.debug_logits = ((flags & SPD_OPT_DEBUG_LOGITS) || h->D.top_k > 0) ? 1 : 0;
  h->host_state->flags = state_flags(flags);
  SPD_CUDA(h, cudaMemcpyAsync(&h->B.st->flags, &h->host_state->flags, sizeof(int),
                              cudaMemcpyHostToDevice, h->s_main));
  SPD_CUDA(h, cudaStreamSynchronize(h->s_main));
  return SPD_OK;
}

size_t spd_dump_size(const spd_handle* h, int32_t what) {
  if (!h) return 0;
  const Dims& D = h->D;
  switch (what) {
    case SPD_DUMP_STATE: return sizeof(DevState);
    case SPD_DUMP_RESID: return sizeof(float) * (D.n + 1) * D.d;
    case SPD_DUMP_ANCHORS: return sizeof(float) * (D.n + 1) * D.m * D.d;
    case SPD_DUMP_PDM_Z: return sizeof(float) * (D.n + 2) * D.d;
    case SPD_DUMP_LOGITS: return sizeof(float) * 2 * D.V;
    case SPD_DUMP_SEQ: return sizeof(int32_t) * (D.max_seq + 2);
    case SPD_DUMP_TRACE: return sizeof(int32_t) * 2 * D.max_seq;
    case SPD_DUMP_KVLEN: return sizeof(int32_t) * D.L;
    case SPD_DUMP_PREFILL_H: return sizeof(float) * kPrefillBlock * D.d;
    default: return 0;
  }
}

int spd_debug_dump(spd_handle* h, int32_t what, void* dst, size_t bytes) {
  if (!h) return SPD_EINVAL;
  const size_t want = spd_dump_size(h, what);
  if (!want || bytes != want || !dst) return fail(h, SPD_EINVAL, "dump %d wants %zu bytes", what, want);
  const void* src = nullptr;
  switch (what) {
    case SPD_DUMP_STATE: src = h->B.st; break;
    case SPD_DUMP_RESID: src = h->B.resid; break;
    case SPD_DUMP_ANCHORS: src = h->B.anch; break;
    case SPD_DUMP_PDM_Z: src = h->p_z; break;
    case SPD_DUMP_LOGITS: src = h->B.logits; break;
    case SPD_DUMP_SEQ: src = h->B.seq; break;
    case SPD_DUMP_TRACE: src = h->B.trace; break;
    case SPD_DUMP_PREFILL_H: src = h->act_pf.resid; break;
    default: src = h->B.kvlen; break;
  }
  SPD_CUDA(h, cudaStreamSynchronize(h->s_main));
  SPD_CUDA(h, cudaMemcpy(dst, src, bytes, cudaMemcpyDeviceToHost));
  return SPD_OK;
}

int spd_time_kernels(spd_handle* h, int32_t enable) {
  if (!h) return SPD_EINVAL;
  SPD_CUDA(h, cudaStreamSynchronize(h->s_main));
  h->timing = enable != 0;
  return SPD_OK;
}

int spd_kernel_times(spd_handle* h, int64_t* launches, double* ms, int32_t n_kinds) {
  if (!h || n_kinds < 0) return SPD_EINVAL;
  SPD_CUDA(h, cudaDeviceSynchronize());
  for (const EvRec& r : h->recs) {
    float t = 0.f;
    if (cudaEventElapsedTime(&t, r.a, r.b) == cudaSuccess) {
      h->launches[r.kind] += 1;
      h->ms[r.kind] += t;
    }
  }
  h->recs.clear();
  h->pool_used = 0;
  // step kernel: per-phase times (barrier to barrier on CTA 0) charged to the phases' kinds
  auto take = [&](unsigned long long* dns, const std::vector<int>& kinds, int64_t runs) -> int {
    if (!dns || kinds.empty()) return SPD_OK;
    std::vector<unsigned long long> ns(kinds.size());
    SPD_CUDA(h, cudaMemcpy(ns.data(), dns, sizeof(unsigned long long) * ns.size(), cudaMemcpyDeviceToHost));
    SPD_CUDA(h, cudaMemset(dns, 0, sizeof(unsigned long long) * ns.size()));
    if (!runs) return SPD_OK;
    for (size_t i = 0; i < kinds.size(); ++i) {
      h->launches[kinds[i]] += runs;
      h->ms[kinds[i]] += ns[i] * 1e-6;
    }
    return SPD_OK;
  };
  int rc;
  if ((rc = take(h->d_ns_cycle, h->kinds_cycle, h->timed_cycles))) return rc;
  if ((rc = take(h->d_ns_ar, h->kinds_ar, h->timed_ar))) return rc;
  h->timed_cycles = h->timed_ar = 0;
  for (int k = 0; k < n_kinds && k < SPD_NUM_KINDS; ++k) {
    if (launches) launches[k] = h->launches[k];
    if (ms) ms[k] = h->ms[k];
    h->launches[k] = 0;
    h->ms[k] = 0;
  }
  return SPD_OK;
}

int spd_cycle_bytes(const spd_handle* h, int32_t t, int32_t fill, int32_t exited, int32_t with_pdm,
                    double* out, int32_t n_kinds) {
  if (!h || !out || n_kinds < SPD_NUM_KINDS) return SPD_EINVAL;
  const Dims& D = h->D;
  const double e = h->esz;
  for (int k = 0; k < SPD_NUM_KINDS; ++k) out[k] = 0.0;
  const double qkv = (double)D.qkv_rows * D.d * e, wo = (double)D.d * D.hq * D.hd * e;
  const double gu = 2.0 * D.ffn * D.d * e, dn = (double)D.d * D.ffn * e;
  const double kvrow = 2.0 * D.hkv * D.hd * e;  // K and V of one position at one layer
  const int a = fill < 0 ? 0 : (fill > D.n ? D.n : fill);
  double kv = 0.0;
  for (int j = 0; j < a; ++j) kv += (double)(t - j) * D.S * kvrow;
  out[KK_QKV] = a * D.S * (qkv + kvrow);  // the QKV launch also appends K and V to the cache
  out[KK_ROPE] = 0.0;
  out[KK_ATTN] = kv;
  out[KK_O] = a * D.S * wo;
  out[KK_GATEUP] = a * D.S * gu;
  out[KK_DOWN] = a * D.S * dn;
  out[KK_HEAD] = exited ? (double)D.V * D.d * e : 0.0;
  if (with_pdm) {  // draft-module kinds 9..17
    const int o = 9;
    // draft rows of a cycle: about fill + 1 (the in-flight rows and the row verified last cycle)
    out[o + KK_QKV] = D.Ls * (qkv + (double)(a + 1) * kvrow);
    out[o + KK_O] = D.Ls * wo;
    out[o + KK_GATEUP] = D.Ls * gu;
    out[o + KK_DOWN] = D.Ls * dn;
    out[o + KK_ATTN] = (double)t * D.Ls * kvrow;
    bool used[SPD_MAX_ANCHORS] = {false};
    for (int k = 0; k <= D.n; ++k) used[D.ftab[k]] = true;
    for (int j = 0; j < D.m; ++j)
      if (used[j]) out[o + KK_FC] += (double)D.d * (j + 1) * D.d * e;
    out[KK_HEAD] += (double)D.V * D.d * e;  // the draft head rides in the same head launch
  }
  return SPD_OK;
}

size_t spd_attention_workspace_bytes(int32_t R, int32_t n_heads, int32_t n_kv_heads, int32_t head_dim,
                                     int32_t max_pos) {
  if (R < 1 || n_heads < 1 || n_kv_heads < 1 || head_dim < 16 || max_pos < 1) return 0;
  return 256 + (size_t)kMaxTiles * n_kv_heads * sizeof(int) +
         attn_part_floats(R, n_heads, head_dim, max_pos) * sizeof(float);
}

int spd_attention(const float* q, const void* k_cache, const void* v_cache, int32_t dtype,
                  const int32_t* pos, int32_t R, int32_t n_heads, int32_t n_kv_heads, int32_t head_dim,
                  int32_t max_seq, float* out, void* workspace, size_t ws_bytes, void* stream) {
  if (!q || !k_cache || !v_cache || !pos || !out || !workspace || R < 1 || R > kMaxAttnRows ||
      n_kv_heads < 1 || n_heads % n_kv_heads || head_dim % 16 || head_dim > 256 || max_seq < 1 ||
      (dtype != SPD_DTYPE_F32 && dtype != SPD_DTYPE_BF16))
    return fail(nullptr, SPD_EINVAL, "spd_attention: bad arguments");
  if (ws_bytes < spd_attention_workspace_bytes(R, n_heads, n_kv_heads, head_dim, max_seq))
    return fail(nullptr, SPD_EINVAL, "spd_attention: workspace too small");
  Dims D;
  memset(&D, 0, sizeof(D));
  D.hq = n_heads; D.hkv = n_kv_heads; D.hd = head_dim; D.gq = n_heads / n_kv_heads;
  D.max_seq = max_seq; D.dtype = dtype; D.qkv_rows = n_heads * head_dim;
  Bufs B;
  memset(&B, 0, sizeof(B));
  Launch lc;
  memset(&lc, 0, sizeof(lc));
  lc.kind = LK_EXPLICIT; lc.cnt = R;
  lc.act.qkv = const_cast<float*>(q);
  lc.act.attn = out;
  lc.act.tick = reinterpret_cast<int*>(workspace);
  lc.act.part = reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(workspace) + 256 +
                                         (size_t)kMaxTiles * n_kv_heads * sizeof(int));
  lc.act.pos_arr = pos;
  lc.act.kc = k_cache; lc.act.vc = v_cache;
  cudaGetLastError();  // start from a clean error state
  cudaError_t e = attn_setup_attributes(attn_smem_bytes(D, false));
  if (e != cudaSuccess)
    return fail(nullptr, SPD_ECUDA, "attention smem attribute (%zu B): %s", attn_smem_bytes(D, false),
                cudaGetErrorString(e));
  LaunchCfg LC;
  memset(&LC, 0, sizeof(LC));
  LC.attn_grid_decode = attn_grid(D, false);
  e = launch_attn(D, B, lc, LC, false, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess)
    return fail(nullptr, SPD_ECUDA, "attention launch (grid %d): %s", LC.attn_grid_decode,
                cudaGetErrorString(e));
  return SPD_OK;
}

size_t spd_prefill_attention_workspace_bytes(int32_t n_heads, int32_t n_kv_heads, int32_t head_dim,
                                             int32_t max_seq) {
  if (n_heads < 1 || n_kv_heads < 1 || n_heads % n_kv_heads || max_seq < 1 || (head_dim != 64 && head_dim != 128))
    return 0;
  return 256 + (size_t)n_heads * sizeof(int) +
         pfattn_part_floats(n_kv_heads, n_heads / n_kv_heads, max_seq, num_sms()) * sizeof(float);
}

int spd_prefill_attention(const float* q, const void* k_cache, const void* v_cache, int32_t pos0, int32_t R,
                          int32_t n_heads, int32_t n_kv_heads, int32_t head_dim, int32_t max_seq, float* out,
                          void* workspace, size_t ws_bytes, void* stream) {
  if (!q || !k_cache || !v_cache || !out || !workspace || n_kv_heads < 1 || n_heads < 1 || n_heads % n_kv_heads ||
      !pfattn_supported(SPD_DTYPE_BF16, head_dim, R, n_heads / n_kv_heads) || pos0 < 1 ||
      (long long)pos0 + R - 1 > max_seq)
    return fail(nullptr, SPD_EINVAL, "spd_prefill_attention: bad arguments");
  if (!aligned16(q) || !aligned16(out) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(workspace))
    return fail(nullptr, SPD_EINVAL, "spd_prefill_attention: pointers must be 16-byte aligned");
  if (ws_bytes < spd_prefill_attention_workspace_bytes(n_heads, n_kv_heads, head_dim, max_seq))
    return fail(nullptr, SPD_EINVAL, "spd_prefill_attention: workspace too small");
  cudaGetLastError();
  CUtensorMap km, vm;
  const long long rows = (long long)n_kv_heads * max_seq;
  cudaError_t e = pfattn_encode_map(&km, k_cache, rows, head_dim);
  if (e == cudaSuccess) e = pfattn_encode_map(&vm, v_cache, rows, head_dim);
  if (e == cudaSuccess) e = pfattn_setup_attributes();
  if (e != cudaSuccess) return fail(nullptr, SPD_ECUDA, "spd_prefill_attention: set-up: %s", cudaGetErrorString(e));
  PfAttnArgs a;
  memset(&a, 0, sizeof(a));
  a.kmap = &km; a.vmap = &vm;
  a.q = q; a.q_stride = n_heads * head_dim; a.out = out;
  a.tick = reinterpret_cast<int*>(workspace);
  a.part = reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(workspace) + 256 + (size_t)n_heads * sizeof(int));
  a.part = reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(a.part) + 15) & ~(uintptr_t)15);
  a.st = nullptr; a.kv_row0 = 0; a.max_seq = max_seq;
  a.hq = n_heads; a.hkv = n_kv_heads; a.hd = head_dim; a.pos0 = pos0; a.nq = R; a.sms = num_sms();
  e = launch_pfattn(a, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(nullptr, SPD_ECUDA, "spd_prefill_attention: launch: %s", cudaGetErrorString(e));
  return SPD_OK;
}

int spd_grouped_gemv(const void* const* W, const float* const* x, float* const* y, int32_t G,
                     int32_t rows, int32_t cols, int32_t dtype, const float* nw, float eps,
                     void* stream) {
  if (!W || !x || !y || G < 1 || G > kMaxExplicit || rows < 1 || cols < 8 || cols % 8 ||
      (dtype != SPD_DTYPE_F32 && dtype != SPD_DTYPE_BF16))
    return fail(nullptr, SPD_EINVAL, "spd_grouped_gemv: bad arguments");
  GemvExplicit ge;
  memset(&ge, 0, sizeof(ge));
  for (int g = 0; g < G; ++g) {
    if (!aligned16(W[g]) || !aligned16(x[g]) || !W[g] || !x[g] || !y[g])
      return fail(nullptr, SPD_EINVAL, "spd_grouped_gemv: pointer %d NULL or unaligned", g);
    ge.W[g] = W[g]; ge.x[g] = x[g]; ge.y[g] = y[g];
  }
  if (nw && !aligned16(nw)) return fail(nullptr, SPD_EINVAL, "spd_grouped_gemv: norm weight unaligned");
  ge.G = G; ge.rows = rows; ge.cols = cols; ge.nw = nw;
  // tensor maps of the G weights: encoded here, held in stream-ordered scratch for this launch
  std::vector<CUtensorMap> maps(G);
  for (int g = 0; g < G; ++g) {
    const cudaError_t em = gemv_encode_map(&maps[g], W[g], rows, cols, dtype, box3_cols(cols, dtype));
    if (em != cudaSuccess)
      return fail(nullptr, SPD_ECUDA, "spd_grouped_gemv: tensor map %d: %s", g, cudaGetErrorString(em));
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  CUtensorMap* dmaps = nullptr;
  cudaError_t e = cudaMallocAsync(reinterpret_cast<void**>(&dmaps), sizeof(CUtensorMap) * G, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(dmaps, maps.data(), sizeof(CUtensorMap) * G, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) {
    for (int g = 0; g < G; ++g) ge.tm[g] = dmaps + g;
    e = gemv_setup_attributes();
  }
  if (e == cudaSuccess) e = launch_gemv_explicit(ge, dtype, eps, st);
  if (dmaps) {
    const cudaError_t ef = cudaFreeAsync(dmaps, st);
    if (e == cudaSuccess) e = ef;
  }
  if (e != cudaSuccess) return fail(nullptr, SPD_ECUDA, "%s", cudaGetErrorString(e));
  return SPD_OK;
}

}  // extern "C"
