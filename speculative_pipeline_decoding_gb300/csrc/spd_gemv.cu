// Grouped GEMV engine for the SPD cycle.
//
// One launch computes y_g = W_g x_g for up to kMaxGroups groups.  Each group has its own weights,
// operator and epilogue, so one launch can carry the stage-diagonal step of the target (the token
// at depth j runs layer j*S+s, SPD summary 方法步骤详情 step 1) together with the draft module's rows
// (steps 3-4).  Weight rows are streamed once from HBM with 1-D bulk copies (cp.async.bulk,
// L2 evict-first) into a 4-deep ring of shared-memory stages guarded by mbarriers; one producer
// warp issues the copies, eight consumer warps compute.
//
// Work split: every CTA of the persistent grid (one per SM) takes a contiguous share of the
// launch's weight bytes, cut at row boundaries; tiles never straddle a group or a share.
//
// Two compute paths:
//  * single input vector (target step, plain AR, heads): the group's activation, RMS-normalised
//    when the operator has a norm, is staged once in shared memory as fp32.  A stage holds 16
//    weight rows x 2 KB; consumer warp w owns rows w and w+8 of the stage (for gate/up: the gate
//    and up rows of one output), lane l the 16-byte column vectors l, l+32, l+64, l+96 of each
//    2 KB chunk.  Partial sums stay in registers across chunks; a row ends with one xor-tree warp
//    reduction.  A row's arithmetic depends only on its column count, never on the other groups
//    of the launch, so a token's results are bit-identical in plain AR and in the SPD step.
//  * several input vectors sharing the weights (draft-module rows, prefill blocks; bf16 weights):
//    m16n8k16 bf16 tensor-core MMAs with fp32 accumulation.  A stage holds 32 rows x 1 KB; the fp32
//    activations are split into bf16 high and low halves (x = hi + lo keeps ~16 significant bits)
//    and both are multiplied into the accumulator; warps take interleaved 16-column k-steps and
//    their partial tiles are added in warp order.
//
// Epilogues (per group):
//   STORE   y = W x                                  (anchor FC, stand-alone operator)
//   RESID   h += W x, anchor capture when the layer index + 1 = b_i   (o-proj, down)
//   SWIGLU  u = silu(W_gate x) * (W_up x)            (gate/up; x = RMSNorm(h) * ffn_norm)
//   QKV     x = RMSNorm(h) * attn_norm; q and k rotated by RoPE (rotate-half pairs i, i+hd/2, which
//           a tile holds together), q written for attention, k and v rounded to the cache dtype and
//           appended to the layer's KV cache at position pos-1
//   TOP2    logits of the vocab head; per-CTA top-2 (+ optional full logits for debugging)
#include "spd_internal.cuh"

namespace spd {

namespace {

constexpr int kBig = 1 << 30;
constexpr int kNCW = 8;                        // consumer warps
constexpr int kThreads = (kNCW + 1) * 32;      // + one producer warp
constexpr int kSlotsF = 16;                    // single-vector path: weight rows per stage
constexpr int kChunkF = 2048;                  // bytes of each row per stage
constexpr int kPitchF = kChunkF + 16;
constexpr int kSlotsM = 32;                    // tensor-core path: weight rows per stage
constexpr int kChunkM = 1024;
constexpr int kPitchM = kChunkM + 16;          // 16-byte pad: ldmatrix rows in distinct banks
constexpr int kStageBytes = (kSlotsF * kPitchF > kSlotsM * kPitchM) ? kSlotsF * kPitchF : kSlotsM * kPitchM;
constexpr int kStages = 4;
constexpr int kXhatFloats = kGemvMaxCols;      // staged activation (single-vector groups)
constexpr int kDynSmem = kStages * kStageBytes + kXhatFloats * 4;
constexpr int kMaxNT = 4;                      // tensor-core path: up to 4 n-tiles of 8 vectors
static_assert(kNCW * 2 * kMaxNT * 4 * 32 <= kXhatFloats, "mma reduction buffer must fit");

enum Epi { EPI_STORE = 0, EPI_RESID = 1, EPI_SWIGLU = 2, EPI_QKV = 3, EPI_TOP2 = 4 };

struct GG {
  const void* w[3];            // weight segments (QKV: wq | wk | wv) ; gate/up: w[0] gate, w[1] up
  int seg1, seg2;              // first row of segment 1 and 2
  int rows, cols;              // output rows (gate/up: rows of each weight), input columns
  short nv, nw, epi, kind;     // vectors, weights per output row, epilogue, head kind
  short mma, tr;               // tensor-core path; tile rows
  const float* x; int xrow0, xring, xstride;
  float* y; int yrow0, yring, ystride;
  const float* normw;
  float* anch; int astride;    // anchor capture (row (yrow0+v) % yring of the anchor ring)
  void* kc; void* vc;          // QKV: K / V cache of this layer, [Hkv][max_seq][hd]
  int pos0;                    // QKV: position of vector 0
  int* kvlen;                  // QKV on the target stack: kvlen[layer]
  long long cost0;             // weight elements of the launch before this group
};

struct GemvParams {
  int nparts;
  GemvPart part[2];
  int explicit_mode;
  int resolve_after_wait;      // the control block may have been written by the previous kernel
  int debug_logits;
  int has_mma;                 // bf16 weights (tensor-core path available)
  float eps;
  Dims D;
  Bufs B;
  GemvExplicit ge;
};

__device__ __forceinline__ long long rowcost(const GG& g) { return (long long)g.cols * g.nw; }

__device__ __forceinline__ int anchor_index(const Dims& D, int layer_done) {
  for (int i = 0; i < D.m; ++i)
    if (D.anchors[i] == layer_done) return i;
  return -1;
}

__device__ __forceinline__ void gg_clear(GG& o) {
  o.seg1 = o.seg2 = kBig;
  o.nw = 1; o.epi = EPI_STORE; o.kind = 0; o.mma = 0; o.nv = 1;
  o.normw = nullptr; o.anch = nullptr; o.astride = 0;
  o.kc = o.vc = nullptr; o.pos0 = 0; o.kvlen = nullptr;
  o.xrow0 = o.yrow0 = 0; o.xring = o.yring = kBig;
}

// Appends the groups of one launch part; returns the new group count.
__device__ int add_part(const GemvParams& p, const GemvPart& pt, GG* gg, int ng) {
  const Dims& D = p.D;
  const Bufs& B = p.B;
  const Launch& lc = pt.lc;
  const Act& A = lc.act;
  DevState* st = B.st;
  if (pt.op == OP_HEAD) {
    auto add = [&](const float* x, int xrow0, int xring, const void* W, const float* nw, int kind) {
      GG& o = gg[ng++];
      gg_clear(o);
      o.w[0] = o.w[1] = o.w[2] = W;
      o.rows = D.V; o.cols = D.d;
      o.x = x; o.xrow0 = xrow0; o.xring = xring; o.xstride = D.d;
      o.y = nullptr; o.normw = nw; o.epi = EPI_TOP2; o.kind = kind;
    };
    if (lc.kind == LK_DIAG) {
      if (st->a == D.n) add(B.resid, (st->t - D.n + 1) % (D.n + 1), D.n + 1, B.lm_head, B.final_norm, 0);
      if (!(st->flags & SF_TARGET_ONLY)) {
        const int R = st->t - st->pdm_len;
        if (R < 1 || R > D.n + 1) set_err(st, ERR_PDM_ROWS, 200);
        else add(A.qkv /* draft rows z */, R - 1, kBig, B.pdm_head, B.pdm_norm, 1);
      }
    } else if (lc.kind == LK_AR) {
      add(B.resid, st->t % (D.n + 1), D.n + 1, B.lm_head, B.final_norm, 0);
    } else if (lc.kind == LK_ROWS) {
      add(A.resid, lc.cnt - 1, kBig, B.lm_head, B.final_norm, 0);
    }
    return ng;
  }
  if (pt.op == OP_FC) {
    // draft rows: depth by the staircase, f by the anchor table; equal f are contiguous runs
    if (lc.kind == LK_ROWS) {
      const int f = D.ftab[D.n];
      GG& o = gg[ng++];
      gg_clear(o);
      o.w[0] = o.w[1] = o.w[2] = B.fc[f];
      o.rows = D.d; o.cols = (f + 1) * D.d; o.nv = lc.cnt;
      o.x = A.anch; o.xstride = D.m * D.d;
      o.y = A.resid; o.ystride = D.d;
      return ng;
    }
    const int t = st->t, a = st->a, R = t - st->pdm_len;
    if (R < 1 || R > D.n + 1) {
      set_err(st, ERR_PDM_ROWS, 300);
      return ng;
    }
    int prev_f = -1;
    for (int r = 0; r < R; ++r) {
      const int pos = st->pdm_len + 1 + r;
      const int depth = (t - pos < a) ? (t - pos) : D.n;
      const int f = D.ftab[depth];
      if (f != prev_f) {
        GG& o = gg[ng++];
        gg_clear(o);
        o.w[0] = o.w[1] = o.w[2] = B.fc[f];
        o.rows = D.d; o.cols = (f + 1) * D.d; o.nv = 0;
        o.x = B.anch; o.xrow0 = pos % (D.n + 1); o.xring = D.n + 1; o.xstride = D.m * D.d;
        o.y = A.resid; o.yrow0 = r; o.ystride = D.d;
        prev_f = f;
      }
      gg[ng - 1].nv++;
    }
    return ng;
  }
  RowGroup rg[kMaxGroups];
  const int nr = build_rows(lc, D, st, rg);
  const LayerW* LW = lc.stack == 0 ? B.tl : B.pl;
  const int hqd = D.hq * D.hd;
  const int esz = D.dtype == SPD_DTYPE_BF16 ? 2 : 4;
  const size_t layer_bytes = (size_t)D.hkv * D.max_seq * D.hd * esz;
  for (int i = 0; i < nr; ++i) {
    GG& o = gg[ng++];
    gg_clear(o);
    const LayerW& w = LW[rg[i].layer];
    o.nv = rg[i].nv;
    switch (pt.op) {
      case OP_QKV:
        o.w[0] = w.wq; o.w[1] = w.wk; o.w[2] = w.wv;
        o.seg1 = hqd; o.seg2 = hqd + D.hkv * D.hd; o.rows = D.qkv_rows; o.cols = D.d;
        o.x = A.resid; o.xrow0 = rg[i].rrow0; o.xring = A.resid_ring; o.xstride = D.d;
        o.normw = (const float*)w.attn_norm;
        o.y = A.qkv; o.yrow0 = rg[i].vid0; o.ystride = D.qkv_rows;
        o.epi = EPI_QKV;
        o.kc = (unsigned char*)(lc.stack == 0 ? B.kc : B.pkc) + (size_t)rg[i].layer * layer_bytes;
        o.vc = (unsigned char*)(lc.stack == 0 ? B.vc : B.pvc) + (size_t)rg[i].layer * layer_bytes;
        o.pos0 = rg[i].pos0;
        o.kvlen = (lc.stack == 0 && B.kvlen) ? B.kvlen + rg[i].layer : nullptr;
        break;
      case OP_O:
        o.w[0] = o.w[1] = o.w[2] = w.wo;
        o.rows = D.d; o.cols = hqd;
        o.x = A.attn; o.xrow0 = rg[i].vid0; o.xstride = hqd;
        o.y = A.resid; o.yrow0 = rg[i].rrow0; o.yring = A.resid_ring; o.ystride = D.d;
        o.epi = EPI_RESID;
        break;
      case OP_GATEUP:
        o.w[0] = w.wg; o.w[1] = w.wu; o.w[2] = w.wu; o.nw = 2;
        o.rows = D.ffn; o.cols = D.d;
        o.x = A.resid; o.xrow0 = rg[i].rrow0; o.xring = A.resid_ring; o.xstride = D.d;
        o.normw = (const float*)w.ffn_norm;
        o.y = A.u; o.yrow0 = rg[i].vid0; o.ystride = D.ffn;
        o.epi = EPI_SWIGLU;
        break;
      default: {  // OP_DOWN
        o.w[0] = o.w[1] = o.w[2] = w.wd;
        o.rows = D.d; o.cols = D.ffn;
        o.x = A.u; o.xrow0 = rg[i].vid0; o.xstride = D.ffn;
        o.y = A.resid; o.yrow0 = rg[i].rrow0; o.yring = A.resid_ring; o.ystride = D.d;
        o.epi = EPI_RESID;
        const int ai = (lc.stack == 0 && A.anch) ? anchor_index(D, rg[i].layer + 1) : -1;
        if (ai >= 0) { o.anch = A.anch + (size_t)ai * D.d; o.astride = D.m * D.d; }
      }
    }
  }
  return ng;
}

// Resolves every group of the launch and fixes each group's path and tile height.  Groups with
// several vectors that cannot take the tensor-core path are split into one group per vector.
__device__ int resolve_groups(const GemvParams& p, GG* gg) {
  int ng = 0;
  if (p.explicit_mode) {
    for (int g = 0; g < p.ge.G; ++g) {
      GG& o = gg[ng++];
      gg_clear(o);
      o.w[0] = o.w[1] = o.w[2] = p.ge.W[g];
      o.rows = p.ge.rows; o.cols = p.ge.cols;
      o.x = p.ge.x[g]; o.xstride = p.ge.cols;
      o.y = p.ge.y[g]; o.ystride = p.ge.rows;
      o.normw = p.ge.nw;
    }
  } else {
    for (int i = 0; i < p.nparts; ++i) ng = add_part(p, p.part[i], gg, ng);
  }
  // paths; split multi-vector groups the tensor cores cannot take
  // (a tensor-core QKV tile holds 16 rotary pairs, so it needs head_dim/2 % 16 == 0)
  int out = ng;
  for (int g = ng - 1; g >= 0; --g) {
    GG& o = gg[g];
    const bool mma_ok = p.has_mma && o.cols % 16 == 0 && (o.epi != EPI_QKV || (p.D.hd / 2) % 16 == 0);
    if (o.nv > 1 && !mma_ok) {
      const int nv = o.nv;
      if (out + nv - 1 > kMaxGroups) { set_err(p.B.st, ERR_BOUNDS, 90); return 0; }
      for (int k = out - 1; k > g; --k) gg[k + nv - 1] = gg[k];  // make room after g
      for (int v = nv - 1; v >= 0; --v) {
        GG& c = gg[g + v];
        c = o;  // o is still intact at index g until v == 0
        c.nv = 1;
        c.xrow0 = o.xrow0 + v; c.yrow0 = o.yrow0 + v; c.pos0 = o.pos0 + v;
      }
      out += nv - 1;
    }
  }
  ng = out;
  long long cost = 0;
  for (int g = 0; g < ng; ++g) {
    GG& o = gg[g];
    if (o.nv > 1 || o.cols > kXhatFloats) {
      if (!(p.has_mma && o.cols % 16 == 0) || o.nv > 8 * kMaxNT) { set_err(p.B.st, ERR_BOUNDS, 91); return 0; }
      o.mma = 1;
    }
    o.tr = (short)((o.mma ? kSlotsM : kSlotsF) / o.nw);
    o.cost0 = cost;
    cost += (long long)o.rows * rowcost(o);
  }
  return ng;
}

// Row boundary of weight-cost position X: first row of the group holding X whose cost prefix is
// >= X; rows of the rotary region of a QKV group are rounded down to whole tiles so that each tile
// holds complete (i, i+hd/2) pairs.  Monotone in X, so neighbouring shares meet exactly.
__device__ void locate(const GG* gg, int ng, long long X, int& g, int& r) {
  g = 0;
  while (g < ng && X >= gg[g].cost0 + (long long)gg[g].rows * rowcost(gg[g])) ++g;
  if (g >= ng) { g = ng; r = 0; return; }
  const long long rc = rowcost(gg[g]);
  r = (int)((X - gg[g].cost0 + rc - 1) / rc);
  if (gg[g].epi == EPI_QKV && r < gg[g].seg2) r -= r % gg[g].tr;
  if (r >= gg[g].rows) { ++g; r = 0; }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Physical weight row of virtual row `r` of a group.  In the rotary region of a QKV group a tile
// of 2P virtual rows holds rows i0..i0+P-1 and i0+hd/2..i0+hd/2+P-1 of one head (P = tile/2).
__device__ __forceinline__ int phys_row(const GG& G, int r, int hd) {
  if (G.epi != EPI_QKV || r >= G.seg2) return r;
  const int P = G.tr / 2;
  const int h = r / hd, vb = r % hd;
  const int blk = vb / G.tr, j = vb % G.tr;
  return h * hd + (j < P ? blk * P + j : hd / 2 + blk * P + (j - P));
}

__device__ __forceinline__ const unsigned char* row_src(const GG& G, int prow, int wi, int esz) {
  if (G.nw == 2) return (const unsigned char*)G.w[wi] + (size_t)prow * G.cols * esz;
  const int sg = prow < G.seg1 ? 0 : (prow < G.seg2 ? 1 : 2);
  const int off = sg == 0 ? 0 : (sg == 1 ? G.seg1 : G.seg2);
  return (const unsigned char*)G.w[sg] + (size_t)(prow - off) * G.cols * esz;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo_k, float hi_k) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo_k, hi_k);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                            uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <typename WT>
__device__ __forceinline__ void store_kv(void* base, int head, int pos, int e, const Dims& D, float v) {
  WT* p = reinterpret_cast<WT*>(base) + ((size_t)head * D.max_seq + (pos - 1)) * D.hd + e;
  *p = WTraits<WT>::from_f(v);
}

// Epilogue of one output row (or rotary pair) for vector v.  y0/y1: the two accumulations the
// caller holds (gate/up: gate and up of row r; rotary: rows r and its partner; else y1 unused).
template <typename WT>
__device__ __forceinline__ void epilogue(const GemvParams& p, const GG& G, int v, int row, float y0,
                                         float y1, bool pair, Top2* loc) {
  const Dims& D = p.D;
  if (G.epi == EPI_TOP2) {
    top2_push(loc[G.kind], y0, row);
    if (p.debug_logits) p.B.logits[(size_t)G.kind * D.V + row] = y0;
    return;
  }
  const int yr = (G.yrow0 + v) % G.yring;
  float* yrow = G.y + (size_t)yr * G.ystride;
  switch (G.epi) {
    case EPI_SWIGLU:
      yrow[row] = (y0 / (1.0f + expf(-y0))) * y1;
      break;
    case EPI_RESID: {
      const float hn = yrow[row] + y0;
      yrow[row] = hn;
      if (G.anch) G.anch[(size_t)yr * G.astride + row] = hn;
      break;
    }
    case EPI_QKV: {
      const int pos = G.pos0 + v;
      const int hd = D.hd, half = hd / 2;
      if (pair) {  // row = physical index of the first element of a rotary pair
        const int h = row / hd, i = row % hd;
        const float c = p.B.rope_cos[(size_t)(pos - 1) * half + i];
        const float s = p.B.rope_sin[(size_t)(pos - 1) * half + i];
        const float r1 = y0 * c - y1 * s;
        const float r2 = y1 * c + y0 * s;
        if (h < D.hq) {
          yrow[h * hd + i] = r1;
          yrow[h * hd + i + half] = r2;
        } else {
          store_kv<WT>(G.kc, h - D.hq, pos, i, D, r1);
          store_kv<WT>(G.kc, h - D.hq, pos, i + half, D, r2);
          if (G.kvlen && h == D.hq && i == 0) *G.kvlen = pos;
        }
      } else {  // value row
        const int vr = row - G.seg2;
        store_kv<WT>(G.vc, vr / hd, pos, vr % hd, D, y0);
      }
      break;
    }
    default:
      yrow[row] = y0;
  }
}

template <typename WT>
__global__ void __launch_bounds__(kThreads, 1) gemv_engine(const __grid_constant__ GemvParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* ring = smem;
  float* xhat = reinterpret_cast<float*>(smem + kStages * kStageBytes);
  constexpr int VEC = WTraits<WT>::kVec;
  constexpr int ESZ = sizeof(WT);
  constexpr int CWF = kChunkF / ESZ;                  // columns per single-vector chunk
  constexpr int CWM = kChunkM / 2;                    // columns per tensor-core chunk (bf16)

  __shared__ GG gg[kMaxGroups];
  __shared__ int s_ng, s_gb, s_rb, s_ge, s_re;
  __shared__ __align__(8) uint64_t full_bar[kStages];
  __shared__ __align__(8) uint64_t empty_bar[kStages];
  __shared__ float rstd_s[8 * kMaxNT];
  __shared__ float wpart[kNCW];
  __shared__ Top2 hred[kNCW][2];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  DevState* st = p.B.st;
  if (p.resolve_after_wait) pdl_wait();
  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], kNCW);
    }
    fence_mbar_init();
    const bool skip = !p.explicit_mode && (st->done || st->err);
    const int ng = skip ? 0 : resolve_groups(p, gg);
    s_ng = ng;
    long long total = ng ? gg[ng - 1].cost0 + (long long)gg[ng - 1].rows * rowcost(gg[ng - 1]) : 0;
    int gb = ng, rb = 0, ge = ng, re = 0;
    if (ng) {
      locate(gg, ng, total * blockIdx.x / gridDim.x, gb, rb);
      locate(gg, ng, total * (blockIdx.x + 1) / gridDim.x, ge, re);
    }
    s_gb = gb; s_rb = rb; s_ge = ge; s_re = re;
  }
  __syncthreads();
  const int ng = s_ng;
  const int gbeg = s_gb, rbeg = s_rb, gend = s_ge, rend = s_re;

  if (warp == kNCW) {
    // ------------------------------ producer warp ------------------------------
    const uint64_t pol = l2_evict_first_policy();
    uint32_t ctr = 0;
    bool failed = false;
    for (int g = gbeg, r = rbeg; (g < gend || (g == gend && r < rend)) && !failed;) {
      const GG& G = gg[g];
      const int last = (g == gend) ? rend : G.rows;
      const int tr = min((int)G.tr, last - r);
      const int nslot = G.mma ? kSlotsM : kSlotsF;
      const int pitch = G.mma ? kPitchM : kPitchF;
      const int cw = G.mma ? CWM : CWF;
      const int per_w = nslot / G.nw;
      for (int c0 = 0; c0 < G.cols; c0 += cw) {
        const uint32_t brow = (uint32_t)min(cw, G.cols - c0) * ESZ;
        const int s = ctr % kStages;
        if (ctr >= (uint32_t)kStages &&
            !mbar_wait_bounded(&empty_bar[s], ((ctr / kStages) - 1) & 1)) {
          if (lane == 0) set_err(st, ERR_TIMEOUT, 40);
          failed = true;
          break;
        }
        if (lane == 0) mbar_arrive_expect_tx(&full_bar[s], brow * tr * G.nw);
        __syncwarp();
        if (lane < nslot) {
          const int wi = lane / per_w, ri = lane % per_w;
          if (ri < tr) {
            const int prow = phys_row(G, r + ri, p.D.hd);
            bulk_g2s(ring + (size_t)s * kStageBytes + (size_t)lane * pitch,
                     row_src(G, prow, wi, ESZ) + (size_t)c0 * ESZ, brow, &full_bar[s], pol);
          }
        }
        ++ctr;
      }
      r += tr;
      if (r >= last) { ++g; r = 0; }
    }
    if (failed && lane == 0) {  // let the copies in flight land before leaving
      const uint32_t first = ctr > (uint32_t)kStages ? ctr - kStages : 0;
      for (uint32_t c = first; c < ctr; ++c) mbar_wait_bounded(&full_bar[c % kStages], (c / kStages) & 1);
    }
    return;
  }

  // ------------------------------ consumer warps ------------------------------
  if (!p.resolve_after_wait) pdl_wait();   // activations of the previous kernel are visible now
  pdl_trigger();
  constexpr int NCT = kNCW * 32;
  uint32_t ctr = 0;
  bool failed = false;
  Top2 loc[2];
  top2_init(loc[0]);
  top2_init(loc[1]);
  const int gq = lane >> 2, tq = lane & 3;                       // mma fragment coordinates
  const int lm_row = (lane & 7) + 8 * ((lane >> 3) & 1), lm_k = 8 * (lane >> 4);
  int last_g = -1;
  for (int g = gbeg, r = rbeg; g < gend || (g == gend && r < rend);) {
    const GG& G = gg[g];
    const int last = (g == gend) ? rend : G.rows;
    const int tr = min((int)G.tr, last - r);
    if (g != last_g) {
      // group entry: stage the (normalised) activation, or the per-vector rstd for the mma path
      named_bar(1, NCT);
      if (!G.mma) {
        const float* xr = G.x + (size_t)(G.xrow0 % G.xring) * G.xstride;
        float rstd = 1.f;
        if (G.normw) {
          float sq = 0.f;
          for (int c = tid * 4; c < G.cols; c += NCT * 4) {
            const float4 q = *reinterpret_cast<const float4*>(xr + c);
            sq += q.x * q.x; sq += q.y * q.y; sq += q.z * q.z; sq += q.w * q.w;
          }
          sq = warp_sum(sq);
          if (lane == 0) wpart[warp] = sq;
          named_bar(1, NCT);
          float tot = 0.f;
#pragma unroll
          for (int w8 = 0; w8 < kNCW; ++w8) tot += wpart[w8];
          rstd = 1.0f / sqrtf(tot / (float)G.cols + p.eps);
        }
        for (int c = tid * 4; c < G.cols; c += NCT * 4) {
          float4 q = *reinterpret_cast<const float4*>(xr + c);
          if (G.normw) {
            const float4 n4 = *reinterpret_cast<const float4*>(G.normw + c);
            q.x = q.x * rstd * n4.x; q.y = q.y * rstd * n4.y;
            q.z = q.z * rstd * n4.z; q.w = q.w * rstd * n4.w;
          }
          *reinterpret_cast<float4*>(xhat + c) = q;
        }
      } else if (G.normw) {
        for (int v = warp; v < G.nv; v += kNCW) {
          const float* xr = G.x + (size_t)((G.xrow0 + v) % G.xring) * G.xstride;
          float sq = 0.f;
          for (int c = lane * 4; c < G.cols; c += 128) {
            const float4 q = *reinterpret_cast<const float4*>(xr + c);
            sq += q.x * q.x; sq += q.y * q.y; sq += q.z * q.z; sq += q.w * q.w;
          }
          sq = warp_sum(sq);
          if (lane == 0) rstd_s[v] = 1.0f / sqrtf(sq / (float)G.cols + p.eps);
        }
      }
      named_bar(1, NCT);
      last_g = g;
    }
    if (!G.mma) {
      // ---------------- single-vector path ----------------
      float acc0 = 0.f, acc1 = 0.f;   // slots warp and warp + 8
      const bool v0 = G.nw == 2 ? warp < tr : warp < tr;
      const bool v1 = G.nw == 2 ? warp < tr : warp + 8 < tr;
      const unsigned char* sbase = ring;
      for (int c0 = 0; c0 < G.cols; c0 += CWF) {
        const int nvec = min(CWF, G.cols - c0) / VEC;
        const int s = ctr % kStages;
        if (!failed && !mbar_wait_bounded(&full_bar[s], (ctr / kStages) & 1)) {
          if (lane == 0) set_err(st, ERR_TIMEOUT, 50);
          failed = true;
        }
        if (!failed) {
          const unsigned char* sb = sbase + (size_t)s * kStageBytes;
          const unsigned char* r0p = sb + (size_t)warp * kPitchF;
          const unsigned char* r1p = sb + (size_t)(warp + 8) * kPitchF;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int k = lane + 32 * j;
            if (k < nvec) {
              float xv[VEC];
#pragma unroll
              for (int e = 0; e < VEC; e += 4) {
                const float4 q = *reinterpret_cast<const float4*>(xhat + c0 + k * VEC + e);
                xv[e] = q.x; xv[e + 1] = q.y; xv[e + 2] = q.z; xv[e + 3] = q.w;
              }
              if (v0) {
                float wf[VEC];
                WTraits<WT>::unpack(*reinterpret_cast<const uint4*>(r0p + k * 16), wf);
#pragma unroll
                for (int e = 0; e < VEC; ++e) acc0 = fmaf(wf[e], xv[e], acc0);
              }
              if (v1) {
                float wf[VEC];
                WTraits<WT>::unpack(*reinterpret_cast<const uint4*>(r1p + k * 16), wf);
#pragma unroll
                for (int e = 0; e < VEC; ++e) acc1 = fmaf(wf[e], xv[e], acc1);
              }
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[s]);
        ++ctr;
      }
      const float y0 = warp_sum(acc0), y1 = warp_sum(acc1);
      if (lane == 0 && !failed) {
        if (G.nw == 2) {
          if (v0) epilogue<WT>(p, G, 0, r + warp, y0, y1, false, loc);
        } else if (G.epi == EPI_QKV && r < G.seg2) {
          if (v0) epilogue<WT>(p, G, 0, phys_row(G, r + warp, p.D.hd), y0, y1, true, loc);
        } else {
          if (v0) epilogue<WT>(p, G, 0, r + warp, y0, 0.f, false, loc);
          if (v1) epilogue<WT>(p, G, 0, r + warp + 8, y1, 0.f, false, loc);
        }
      }
    } else {
      // ---------------- tensor-core path (bf16 weights, several vectors) ----------------
      const int nv = G.nv;
      const int NT = (nv + 7) / 8;
      const float* xrow[kMaxNT];
      float rsv[kMaxNT];
#pragma unroll
      for (int nt = 0; nt < kMaxNT; ++nt) {
        const int v = nt * 8 + gq;
        xrow[nt] = v < nv ? G.x + (size_t)((G.xrow0 + v) % G.xring) * G.xstride : nullptr;
        rsv[nt] = (v < nv && G.normw) ? rstd_s[v] : 1.f;
      }
      float acc[2][kMaxNT][4];
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < kMaxNT; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[i][j][e] = 0.f;
      for (int c0 = 0; c0 < G.cols; c0 += CWM) {
        const int ksteps = min(CWM, G.cols - c0) / 16;
        const int s = ctr % kStages;
        if (!failed && !mbar_wait_bounded(&full_bar[s], (ctr / kStages) & 1)) {
          if (lane == 0) set_err(st, ERR_TIMEOUT, 60);
          failed = true;
        }
        if (!failed) {
          const uint32_t sb = smem_u32(ring + (size_t)s * kStageBytes);
          for (int ks = warp; ks < ksteps; ks += kNCW) {
            const int col = c0 + ks * 16;
            uint32_t a[2][4];
#pragma unroll
            for (int at = 0; at < 2; ++at)
              ldmatrix_x4(sb + (uint32_t)((at * 16 + lm_row) * kPitchM + (ks * 16 + lm_k) * 2), a[at][0],
                          a[at][1], a[at][2], a[at][3]);
#pragma unroll
            for (int nt = 0; nt < kMaxNT; ++nt) {
              if (nt < NT) {
                float x0 = 0.f, x1 = 0.f, x2 = 0.f, x3 = 0.f;
                if (xrow[nt]) {
                  const int k0 = col + 2 * tq;
                  const float2 u = *reinterpret_cast<const float2*>(xrow[nt] + k0);
                  const float2 w8 = *reinterpret_cast<const float2*>(xrow[nt] + k0 + 8);
                  x0 = u.x; x1 = u.y; x2 = w8.x; x3 = w8.y;
                  if (G.normw) {
                    const float2 n0 = *reinterpret_cast<const float2*>(G.normw + k0);
                    const float2 n8 = *reinterpret_cast<const float2*>(G.normw + k0 + 8);
                    x0 = x0 * rsv[nt] * n0.x; x1 = x1 * rsv[nt] * n0.y;
                    x2 = x2 * rsv[nt] * n8.x; x3 = x3 * rsv[nt] * n8.y;
                  }
                }
                const __nv_bfloat16 h0 = __float2bfloat16_rn(x0), h1 = __float2bfloat16_rn(x1);
                const __nv_bfloat16 h2 = __float2bfloat16_rn(x2), h3 = __float2bfloat16_rn(x3);
                const uint32_t bh0 = pack_bf16x2(__bfloat162float(h0), __bfloat162float(h1));
                const uint32_t bh1 = pack_bf16x2(__bfloat162float(h2), __bfloat162float(h3));
                const uint32_t bl0 = pack_bf16x2(x0 - __bfloat162float(h0), x1 - __bfloat162float(h1));
                const uint32_t bl1 = pack_bf16x2(x2 - __bfloat162float(h2), x3 - __bfloat162float(h3));
#pragma unroll
                for (int at = 0; at < 2; ++at) {
                  mma_bf16(acc[at][nt], a[at], bh0, bh1);
                  mma_bf16(acc[at][nt], a[at], bl0, bl1);
                }
              }
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[s]);
        ++ctr;
      }
      // partial tiles of the 8 warps -> shared memory (the activation region is free here), added
      // in warp order
      float* red = xhat;  // [warp][at][nt][e][lane]
#pragma unroll
      for (int at = 0; at < 2; ++at)
#pragma unroll
        for (int nt = 0; nt < kMaxNT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (nt < NT) red[(((warp * 2 + at) * kMaxNT + nt) * 4 + e) * 32 + lane] = acc[at][nt][e];
      named_bar(1, NCT);
      auto tot = [&](int at, int m, int v) {
        const int nt = v / 8, nn = v % 8;
        const int ln = (m % 8) * 4 + nn / 2;
        const int e = (m >= 8 ? 2 : 0) + (nn & 1);
        float sum = 0.f;
#pragma unroll
        for (int w8 = 0; w8 < kNCW; ++w8) sum += red[(((w8 * 2 + at) * kMaxNT + nt) * 4 + e) * 32 + ln];
        return sum;
      };
      if (!failed) {
        if (G.nw == 2) {  // 16 rows: gate in A tile 0, up in A tile 1
          for (int idx = tid; idx < 16 * nv; idx += NCT) {
            const int m = idx / nv, v = idx % nv;
            if (m < tr) epilogue<WT>(p, G, v, r + m, tot(0, m, v), tot(1, m, v), false, loc);
          }
        } else if (G.epi == EPI_QKV && r < G.seg2) {  // 16 rotary pairs (slot m, slot m+16)
          for (int idx = tid; idx < 16 * nv; idx += NCT) {
            const int m = idx / nv, v = idx % nv;
            epilogue<WT>(p, G, v, phys_row(G, r + m, p.D.hd), tot(0, m, v), tot(1, m, v), true, loc);
          }
        } else {  // 32 rows in two A tiles
          for (int idx = tid; idx < 32 * nv; idx += NCT) {
            const int m = idx / nv, v = idx % nv;
            if (m < tr) epilogue<WT>(p, G, v, r + m, tot(m / 16, m % 16, v), 0.f, false, loc);
          }
        }
      }
      named_bar(1, NCT);  // `red` is rewritten by the next tile
    }
    r += tr;
    if (r >= last) { ++g; r = 0; }
  }
  // head: per-CTA top-2 of each kind, warps merged in order
  bool head = false;
  for (int i = 0; i < ng; ++i) head |= gg[i].epi == EPI_TOP2;
  if (head || (ng == 0 && p.nparts > 0 && p.part[0].op == OP_HEAD)) {
    if (lane == 0) { hred[warp][0] = loc[0]; hred[warp][1] = loc[1]; }
    named_bar(1, NCT);
    if (tid == 0) {
      float* hp = p.B.head_part + (size_t)blockIdx.x * 8;
      for (int k = 0; k < 2; ++k) {
        Top2 m = hred[0][k];
        for (int i = 1; i < kNCW; ++i) top2_merge(m, hred[i][k]);
        hp[k * 4 + 0] = m.v1; hp[k * 4 + 1] = __int_as_float(m.i1);
        hp[k * 4 + 2] = m.v2; hp[k * 4 + 3] = __int_as_float(m.i2);
      }
    }
  }
}

template <typename WT>
cudaError_t launch_engine(const GemvParams& p, bool pdl, cudaStream_t s) {
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(num_sms());
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kDynSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, gemv_engine<WT>, p);
}

}  // namespace

int num_sms() {
  static int sms = 0;
  if (sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 1;
  }
  return sms;
}

int gemv_head_grid(int dtype) {
  (void)dtype;
  return num_sms();  // one CTA per SM; every CTA writes its top-2 partial
}

cudaError_t gemv_setup_attributes() {
  cudaError_t e = cudaFuncSetAttribute(gemv_engine<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kDynSmem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(gemv_engine<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kDynSmem);
}

cudaError_t launch_gemv(const GemvPart* parts, int nparts, const Dims& D, const Bufs& B,
                        const LaunchCfg& cfg, bool pdl, bool resolve_after_wait, cudaStream_t s) {
  GemvParams p;
  memset(&p, 0, sizeof(p));
  p.nparts = nparts;
  for (int i = 0; i < nparts && i < 2; ++i) p.part[i] = parts[i];
  p.explicit_mode = 0;
  p.resolve_after_wait = resolve_after_wait ? 1 : 0;
  p.debug_logits = cfg.debug_logits;
  p.has_mma = D.dtype == SPD_DTYPE_BF16;
  p.eps = D.eps;
  p.D = D; p.B = B;
  return D.dtype == SPD_DTYPE_BF16 ? launch_engine<__nv_bfloat16>(p, pdl, s) : launch_engine<float>(p, pdl, s);
}

cudaError_t launch_gemv_explicit(const GemvExplicit& ge, int dtype, float eps, cudaStream_t s) {
  GemvParams p;
  memset(&p, 0, sizeof(p));
  p.explicit_mode = 1; p.resolve_after_wait = 1; p.eps = eps; p.ge = ge;
  p.has_mma = 0;
  p.D.dtype = dtype; p.D.eps = eps;
  return dtype == SPD_DTYPE_BF16 ? launch_engine<__nv_bfloat16>(p, false, s) : launch_engine<float>(p, false, s);
}

}  // namespace spd
