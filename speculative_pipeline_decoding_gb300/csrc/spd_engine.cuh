// Grouped GEMV engine for the SPD cycle: device code shared by the stand-alone GEMV kernel and the
// persistent step kernel.
//
// One launch computes y_g = W_g x_g for up to kMaxGroups groups.  Each group has its own weights,
// operator and epilogue, so one launch can carry the stage-diagonal step of the target (the token
// at depth j runs layer j*S+s, SPD summary 方法步骤详情 step 1) together with the draft module's rows
// (steps 3-4).
//
// Weight streaming: one producer warp issues TMA tensor copies (cp.async.bulk.tensor, 128-byte
// swizzle, L2 evict-first) into a 4-deep ring of 32 KB stages guarded by mbarriers; a stage holds
// 64 weight rows x 512 bytes (two 32-row bands of four 128-byte chunks), or 32 rows x 1024 bytes.
// Every weight matrix has its own tensor map, encoded once when the handle is created: 3-D (chunk,
// row, chunk index) when its rows are whole 128-byte chunks, so a band is one 16 KB copy and a
// stage two; else 2-D with 128-byte x 32-row boxes, eight copies a stage.  Issuing a copy costs the
// warp tens of nanoseconds, and an SM must start a stage every ~0.7 us to keep HBM busy, so the
// producer resolves a tile's maps and rows once per tile and issues as few copies as it can.
//
// Work split: every CTA of the persistent grid (one per SM) takes a contiguous share of the
// launch's weight bytes, cut at 32-row boundaries; tiles never straddle a group or a share.
//
// Two compute paths, eight consumer warps:
//  * single input vector (target step, plain AR, heads): warp w owns weight rows w, w+8, ..., w+56
//    of the stage, lane l the 16-byte column vector l of each 512-byte row slice (bf16: columns
//    8l..8l+7); the activation slice (RMS-normalised when the operator has a norm) comes through
//    L1 and is reused over the warp's 8 rows.  Partial sums stay in registers across stages; a row
//    ends with one xor-tree warp reduction.  A row's arithmetic depends only on its column count,
//    never on the other groups of the launch, so a token's results are bit-identical in plain AR
//    and in the SPD step.
//  * several input vectors sharing the weights (draft-module rows, prefill blocks; bf16 weights):
//    m16n8k16 bf16 tensor-core MMAs with fp32 accumulation, the weight rows as the n8 operand
//    (ldmatrix through the swizzle) and the vectors as the m16 operand.  The fp32 activations are
//    split into bf16 high and low halves (x = hi + lo keeps ~16 significant bits) and both are
//    multiplied into the accumulator.  Warp w takes the two 16-column k-steps 32w..32w+31 of every
//    stage; the eight partial tiles are added in warp order at the end of a tile.
//
// Epilogues (per group):
//   STORE   y = W x                                  (anchor FC, stand-alone operator)
//   RESID   h += W x, anchor capture when the layer index + 1 = b_i   (o-proj, down)
//   SWIGLU  u = silu(W_gate x) * (W_up x)            (gate/up; x = RMSNorm(h) * ffn_norm)
//   QKV     x = RMSNorm(h) * attn_norm; q and k rotated by RoPE (rotate-half pairs i, i+hd/2: a tile
//           holds 32 rows of a head and their 32 partners), q written for attention, k and v
//           rounded to the cache dtype and appended to the layer's KV cache at position pos-1
//   TOP2    logits of the vocab head; per-CTA top-2 (+ optional full logits for debugging)
#pragma once
#include "spd_internal.cuh"
#include "spd_tc.cuh"

namespace spd {
namespace eng {

constexpr int kBig = 1 << 30;
constexpr int kNCW = 8;                        // consumer warps
constexpr int kThreads = (kNCW + 1) * 32;      // + one producer warp
constexpr int kBoxRows = 32;                   // rows of one tensor-map box (128 bytes wide)
constexpr int kBoxBytes = kBoxRows * 128;
constexpr int kSlots = 64;                     // weight rows per stage (2 boxes high)
constexpr int kStageBytes = kSlots * 512;      // 4 boxes wide
constexpr int kStages = 4;
constexpr int kMaxMT = 2;                      // tensor-core path: up to 2 m-tiles of 16 vectors
constexpr int kCostSV = 4, kCostMma = 6;       // split cost of a weight byte: an mma.sync stage of
                                               // the draft rows takes ~1.5x a single-vector stage
                                               // streamed alongside it (measured per CTA)
// tensor-core path scratch: the warps' partial tiles of one m-tile
constexpr int kRedBytes = kNCW * 8 * 4 * 32 * 4;  // the 8 warps' partial tiles of one m-tile
constexpr int kMmaScratch = kRedBytes;

enum Epi { EPI_STORE = 0, EPI_RESID = 1, EPI_SWIGLU = 2, EPI_QKV = 3, EPI_TOP2 = 4 };

struct GG {
  const CUtensorMap* m[3];     // tensor maps of the segments (QKV: wq | wk | wv); gate/up: gate, up
  int seg1, seg2;              // first row of segment 1 and 2
  int rows, cols;              // output rows (gate/up: rows of each weight), input columns
  short nv, nw, epi, kind;     // vectors, weights per output row, epilogue, head kind
  short mma, tr;               // tensor-core path; tile height in output rows (64 / nw)
  short tc;                    // tcgen05 path (mma groups of <= 16 vectors, bf16, 3-D maps): 128-row
                               // tiles, stages of 128 rows x 2 chunks from the map at m[s] + 1
  short ks;                    // tcgen05 tiles split over ks column segments (split-K; 1: whole rows)
  int vrows;                   // rows in share space: rows, or ntiles * ks * 128 when split
  int tbase, pbase;            // split groups: first ticket of the group's tiles, first partial float
  const float* x; int xrow0, xring, xstride;
  float* y; int yrow0, yring, ystride;
  const float* normw;
  float* anch; int astride;    // anchor capture (row (yrow0+v) % yring of the anchor ring)
  void* kc; void* vc;          // QKV: K / V cache of this layer, [Hkv][max_seq][hd]
  int pos0;                    // QKV: position of vector 0
  int* kvlen;                  // QKV on the target stack: kvlen[layer]
  long long cost0;             // weight elements of the launch before this group
};

// What the group resolution and the epilogues of a launch (or of a step-kernel phase) read.
struct EngineCfg {
  int debug_logits;
  int has_mma;                 // bf16 weights (tensor-core path available)
  int has_tc;                  // tcgen05 tiles available (maps in pairs, TMEM allocated, B ring)
  int tc_nv_max;               // largest vector count of a tcgen05 tile (16 or 32: the B ring's size)
  float eps;
  Dims D;
  Bufs B;
};

// split cost of one output row: its weight elements, weighted by the path's cost per byte
constexpr int kCostTc = 6;  // a tcgen05 tile byte is weighted 1.5x a single-vector byte streamed
                            // alongside it: the best of 1.0, 1.25, 1.5 and 2 in the co-scheduled
                            // cycle of the 9B-class model (tok/s 180, 192, 199, 188)
__device__ __forceinline__ long long rowcost(const GG& g) {
  return (long long)(g.cols / g.ks) * g.nw * (g.tc ? kCostTc : (g.mma ? kCostMma : kCostSV));
}

// Split-K of tcgen05 groups: a group of whole 128-row tiles whose tiles are too few to fill the grid
// is cut into ks column segments of >= kMinSegBlocks 128-column blocks.  A unit (tile, segment)
// writes its fp32 partial tile to scratch; the last unit of a tile to finish (atomic ticket) adds the
// partials in segment order and runs the epilogue.  ks depends on the group's shape and the launch's (phase's) total work.
constexpr int kMinSegBlocks = 4;

__device__ __forceinline__ int anchor_index(const Dims& D, int layer_done) {
  for (int i = 0; i < D.m; ++i)
    if (D.anchors[i] == layer_done) return i;
  return -1;
}

__device__ __forceinline__ void gg_clear(GG& o) {
  o.seg1 = o.seg2 = kBig;
  o.nw = 1; o.epi = EPI_STORE; o.kind = 0; o.mma = 0; o.nv = 1; o.ks = 1; o.tc = 0;
  o.normw = nullptr; o.anch = nullptr; o.astride = 0;
  o.kc = o.vc = nullptr; o.pos0 = 0; o.kvlen = nullptr;
  o.xrow0 = o.yrow0 = 0; o.xring = o.yring = kBig;
}

// Appends the groups of one launch part; returns the new group count.
static __device__ int add_part(const EngineCfg& p, const GemvPart& pt, GG* gg, int ng, int cap, const View& vw) {
  const Dims& D = p.D;
  const Bufs& B = p.B;
  const Launch& lc = pt.lc;
  if (ng + (D.n + 2) > cap) {  // a part adds at most n+1 groups
    set_err(B.st, ERR_BOUNDS, 92);
    return ng;
  }
  const Act& A = lc.act;
  DevState* st = B.st;         // error flags
  const DevState* sv = vw.sv;  // control block (read)
  if (pt.op == OP_HEAD) {
    auto add = [&](const float* x, int xrow0, int xring, const CUtensorMap* W, const float* nw, int kind) {
      GG& o = gg[ng++];
      gg_clear(o);
      o.m[0] = o.m[1] = o.m[2] = W;
      o.rows = D.V; o.cols = D.d;
      o.x = x; o.xrow0 = xrow0; o.xring = xring; o.xstride = D.d;
      o.y = nullptr; o.normw = nw; o.epi = EPI_TOP2; o.kind = kind;
    };
    if (lc.kind == LK_DIAG) {
      if (sv->a == D.n) add(B.resid, (sv->t - D.n + 1) % (D.n + 1), D.n + 1, B.tm_lm, B.final_norm, 0);
      if (!(sv->flags & SF_TARGET_ONLY)) {
        const int R = sv->t - sv->pdm_len;
        if (R < 1 || R > D.n + 1) set_err(st, ERR_PDM_ROWS, 200);
        else add(A.qkv /* draft rows z */, R - 1, kBig, B.tm_pdm, B.pdm_norm, 1);
      }
    } else if (lc.kind == LK_AR) {
      add(B.resid, sv->t % (D.n + 1), D.n + 1, B.tm_lm, B.final_norm, 0);
    } else if (lc.kind == LK_ROWS) {
      add(A.resid, lc.cnt - 1, kBig, B.tm_lm, B.final_norm, 0);
    }
    return ng;
  }
  if (pt.op == OP_FC) {
    // draft rows: depth by the staircase, f by the anchor table; equal f are contiguous runs
    if (lc.kind == LK_ROWS) {
      const int f = D.ftab[D.n];
      GG& o = gg[ng++];
      gg_clear(o);
      o.m[0] = o.m[1] = o.m[2] = B.tm_fc[f];
      o.rows = D.d; o.cols = (f + 1) * D.d; o.nv = lc.cnt;
      o.x = A.anch; o.xstride = D.m * D.d;
      o.y = A.resid; o.ystride = D.d;
      return ng;
    }
    const int t = sv->t, a = sv->a, R = t - sv->pdm_len;
    if (R < 1 || R > D.n + 1) {
      set_err(st, ERR_PDM_ROWS, 300);
      return ng;
    }
    // pre-step depth t-pos of an in-flight row; one stage more when the draft module runs after the
    // step (post-step schedule); the verified prefix at n
    const int post = (sv->flags & SF_POST_STEP) ? 1 : 0;
    int prev_f = -1;
    for (int r = 0; r < R; ++r) {
      const int pos = sv->pdm_len + 1 + r;
      const int depth = (t - pos < a) ? (t - pos + post) : D.n;
      const int f = D.ftab[depth];
      if (f != prev_f) {
        GG& o = gg[ng++];
        gg_clear(o);
        o.m[0] = o.m[1] = o.m[2] = B.tm_fc[f];
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
  const int nr = build_rows(lc, D, sv, st, rg);
  const LayerW* LW = lc.stack == 0 ? vw.tl : vw.pl;
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
        o.m[0] = w.tq; o.m[1] = w.tk; o.m[2] = w.tv;
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
        o.m[0] = o.m[1] = o.m[2] = w.to;
        o.rows = D.d; o.cols = hqd;
        o.x = A.attn; o.xrow0 = rg[i].vid0; o.xstride = hqd;
        o.y = A.resid; o.yrow0 = rg[i].rrow0; o.yring = A.resid_ring; o.ystride = D.d;
        o.epi = EPI_RESID;
        break;
      case OP_GATEUP:
        o.m[0] = w.tg; o.m[1] = w.tu; o.m[2] = w.tu; o.nw = 2;
        o.rows = D.ffn; o.cols = D.d;
        o.x = A.resid; o.xrow0 = rg[i].rrow0; o.xring = A.resid_ring; o.xstride = D.d;
        o.normw = (const float*)w.ffn_norm;
        o.y = A.u; o.yrow0 = rg[i].vid0; o.ystride = D.ffn;
        o.epi = EPI_SWIGLU;
        break;
      default: {  // OP_DOWN
        o.m[0] = o.m[1] = o.m[2] = w.td;
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

// Resolves every group of a launch's parts and fixes each group's path and tile height.  Without
// tensor cores (fp32 weights) a multi-vector group becomes one group per vector.
static __device__ int finish_groups(const EngineCfg& p, GG* gg, int ng, int cap) {
  int out = ng;
  for (int g = ng - 1; g >= 0; --g) {
    GG& o = gg[g];
    if (o.nv > 1 && !p.has_mma) {
      const int nv = o.nv;
      if (out + nv - 1 > cap) { set_err(p.B.st, ERR_BOUNDS, 90); return 0; }
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
  int tickets = 0, parts = 0;
  for (int g = 0; g < ng; ++g) {
    GG& o = gg[g];
    if (o.nv > 16 * kMaxMT) { set_err(p.B.st, ERR_BOUNDS, 91); return 0; }
    o.mma = o.nv > 1;
    // tcgen05 tiles: <= 16 (32) vectors, whole 128-column stages, heads of at most 128 rows (a
    // 128-row tile holds whole heads, so RoPE pairs stay inside it)
    o.tc = (short)(p.has_tc && o.mma && o.nv <= p.tc_nv_max && o.cols % 128 == 0 && p.D.hd <= 128);
    o.tr = (short)(o.tc ? tc::kRows : kSlots / o.nw);
    o.ks = 1;
    o.vrows = o.rows;
    cost += (long long)o.rows * rowcost(o);
  }
  // a CTA's share of the launch (or phase); a tcgen05 tile costing more than one share is split so
  // that each of its units costs about half a share (the tiles of a phase that carries other work
  // usually fit, and stay whole)
  const long long share = cost / gridDim.x + 1;
  cost = 0;
  for (int g = 0; g < ng; ++g) {
    GG& o = gg[g];
    const long long tile_cost = (long long)tc::kRows * rowcost(o);
    if (o.tc && p.B.tc_part && tile_cost > share && o.rows % tc::kRows == 0 &&
        (o.epi != EPI_QKV || (o.seg1 % tc::kRows == 0 && o.seg2 % tc::kRows == 0))) {
      const int ntile = o.rows / tc::kRows, ncb = o.cols / (tc::kStageCh * tc::kChunk);
      int ks = (int)((2 * tile_cost + share - 1) / share);
      ks = min(ks, ncb / kMinSegBlocks);
      const int nvp = o.nv <= 16 ? 16 : 32;
      const int need = ntile * ks * o.nw * tc::kRows * nvp;
      if (ks > 1 && tickets + ntile <= p.B.tc_tick_cap && parts + need <= p.B.tc_part_cap) {
        o.ks = (short)ks;
        o.vrows = ntile * ks * tc::kRows;
        o.tbase = tickets;
        o.pbase = parts;
        tickets += ntile;
        parts += need;
      }
    }
    o.cost0 = cost;
    cost += (long long)o.vrows * rowcost(o);
  }
  return ng;
}

static __device__ int resolve_parts(const EngineCfg& p, const GemvPart* parts, int nparts, GG* gg, int cap,
                                    const View& vw) {
  int ng = 0;
  for (int i = 0; i < nparts; ++i) ng = add_part(p, parts[i], gg, ng, cap, vw);
  return finish_groups(p, gg, ng, cap);
}

static __device__ int resolve_explicit(const EngineCfg& p, const GemvExplicit& ge, GG* gg) {
  for (int g = 0; g < ge.G; ++g) {
    GG& o = gg[g];
    gg_clear(o);
    o.m[0] = o.m[1] = o.m[2] = ge.tm[g];
    o.rows = ge.rows; o.cols = ge.cols;
    o.x = ge.x[g]; o.xstride = ge.cols;
    o.y = ge.y[g]; o.ystride = ge.rows;
    o.normw = ge.nw;
  }
  return finish_groups(p, gg, ge.G, kMaxExplicit);
}

// Row boundary of weight-cost position X: the row of the group holding X whose cost prefix is
// nearest to X, on a 32-row box boundary (a whole 64-row tile in the rotary region of a QKV group,
// whose tiles hold complete (i, i+hd/2) pairs).  Monotone in X, so neighbouring shares meet exactly.
static __device__ void locate(const GG* gg, int ng, long long X, int& g, int& r) {
  g = 0;
  while (g < ng && X >= gg[g].cost0 + (long long)gg[g].vrows * rowcost(gg[g])) ++g;
  if (g >= ng) { g = ng; r = 0; return; }
  const long long rc = rowcost(gg[g]);
  const long long exact = (X - gg[g].cost0) / rc;
  // whole 64-row tiles in the rotary region and for tensor-core groups (a tile's stages cost the
  // same however many of its rows are used); 32-row boxes elsewhere
  const int gran = ((gg[g].epi == EPI_QKV && exact < gg[g].seg2) || gg[g].mma) ? (int)gg[g].tr : kBoxRows;
  r = (int)(((X - gg[g].cost0) + rc * gran / 2) / (rc * gran)) * gran;
  if (gg[g].ks == 1 && gg[g].epi == EPI_QKV && r > gg[g].seg2 && exact < gg[g].seg2) r = gg[g].seg2;
  if (r >= gg[g].vrows) { ++g; r = 0; }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Physical weight row of virtual row `r` of a group.  In the rotary region of a QKV group a
// 64-row tile holds rows i0..i0+31 of one head and their partners i0+hd/2..i0+hd/2+31.
__device__ __forceinline__ int phys_row(const GG& G, int r, int hd) {
  if (G.epi != EPI_QKV || r >= G.seg2) return r;
  const int h = r / hd, vb = r % hd;
  const int blk = vb / kSlots, j = vb % kSlots;
  return h * hd + (j < kBoxRows ? blk * kBoxRows + j : hd / 2 + blk * kBoxRows + (j - kBoxRows));
}

__device__ __forceinline__ void tma_box(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar,
                                        uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)), "l"(map), "r"(x), "r"(y),
      "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}

// One 3-D box: chunks z..z+3 (128 bytes each) of rows y..y+31, landing as [chunk][row][128 B].
__device__ __forceinline__ void tma_box3(void* dst, const CUtensorMap* map, int y, int z, uint64_t* bar,
                                         uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)), "l"(map), "r"(0), "r"(y), "r"(z),
      "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}

// Byte offset in a stage of the 16-byte chunk `j` (0..31 across the 512-byte row slice) of slot
// `slot` (0..63): box (slot/32, j/8), row slot%32, 128-byte swizzle (chunk ^ row % 8).
__device__ __forceinline__ uint32_t stage_off(int slot, int j) {
  const int rb = slot >> 5, rr = slot & 31;
  return (uint32_t)(((rb * 4 + (j >> 3)) * kBoxBytes) + rr * 128 + (((j & 7) ^ (rr & 7)) << 4));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo_k, float hi_k) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo_k, hi_k);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// 16-byte asynchronous global -> shared copy (completion by cp.async.wait_group)
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                            uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

// no side effects beyond its outputs: not volatile, so that independent MMAs can be interleaved
__device__ __forceinline__ void mma_bf16(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm(
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
// `pre` (or null): the inputs the epilogue reads, loaded by the caller ahead of time -- the residual
// value of the row (RESID) or the rotary cos and sin of the pair (QKV).
template <typename WT>
__device__ __forceinline__ void epilogue(const EngineCfg& p, const GG& G, int v, int row, float y0,
                                         float y1, bool pair, Top2* loc, const float* pre = nullptr) {
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
      const float hn = (pre ? pre[0] : yrow[row]) + y0;
      yrow[row] = hn;
      if (G.anch) G.anch[(size_t)yr * G.astride + row] = hn;
      break;
    }
    case EPI_QKV: {
      const int pos = G.pos0 + v;
      const int hd = D.hd, half = hd / 2;
      if (pair) {  // row = physical index of the first element of a rotary pair
        const int h = row / hd, i = row % hd;
        const float c = pre ? pre[0] : p.B.rope_cos[(size_t)(pos - 1) * half + i];
        const float s = pre ? pre[1] : p.B.rope_sin[(size_t)(pos - 1) * half + i];
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

// ------------------------------------------------------------------------------------------------
// Span streaming: one CTA's share of one launch (or one step-kernel phase).
// ------------------------------------------------------------------------------------------------

// Ring state of one role (producer warp or consumer warps); both roles walk the same stages.
struct Ring {
  unsigned char* base;    // kStages x kStageBytes, 1024-byte aligned
  uint64_t* full;
  uint64_t* empty;
  uint32_t ctr;           // stages issued (producer) or consumed (consumers) so far
  bool failed;            // a bounded wait gave up: stop waiting, keep walking
};

// This CTA's share [(gb, rb), (ge, re)) of the groups' weight bytes.
__device__ __forceinline__ void span_of(const GG* gg, int ng, int cta, int ncta, int& gb, int& rb, int& ge,
                                        int& re) {
  gb = ge = ng; rb = re = 0;
  if (!ng) return;
  const long long total = gg[ng - 1].cost0 + (long long)gg[ng - 1].vrows * rowcost(gg[ng - 1]);
  locate(gg, ng, total * cta / ncta, gb, rb);
  locate(gg, ng, total * (cta + 1) / ncta, ge, re);
}

// Output rows of the tile starting at row r (`last` = end of the share in this group): the group's
// tile height, clipped to the share and, in a QKV group, to the end of the rotary rows.
__device__ __forceinline__ int tile_rows(const GG& G, int r, int last) {
  int tr = min((int)G.tr, last - r);
  if (G.ks > 1) return tr;  // split groups: whole 128-row tiles in share space
  if (G.epi == EPI_QKV && r < G.seg2) tr = min(tr, G.seg2 - r);
  if (G.tc && G.epi == EPI_QKV && r < G.seg1) tr = min(tr, G.seg1 - r);  // one tensor map per tile
  return tr;
}

// A tcgen05 tile at share-space row r: its first physical row rr and its 128-column blocks
// [cb0, cb1) (split groups: unit r / 128 = tile * ks + segment).
__device__ __forceinline__ void tc_unit(const GG& G, int r, int& rr, int& cb0, int& cb1) {
  const int ncb = G.cols / (tc::kStageCh * tc::kChunk);
  if (G.ks > 1) {
    const int u = r / tc::kRows, seg = u % G.ks;
    rr = (u / G.ks) * tc::kRows;
    cb0 = seg * ncb / G.ks;
    cb1 = (seg + 1) * ncb / G.ks;
  } else {
    rr = r; cb0 = 0; cb1 = ncb;
  }
}

// Producer warp: one stage = the 64 weight slots of tile row `r` (tr output rows) at column c0.
// A single-vector tile of at most 32 rows (one weight per row, outside the rotary region) streams
// "wide": a stage holds its 32 rows x 1024 bytes (8 boxes across) instead of 64 rows x 512 bytes, so
// every stage carries 32 KB.  A lane still meets its column chunks in the same order.
__device__ __forceinline__ bool wide_tile(const GG& G, int r, int tr) {
  return !G.mma && G.nw == 1 && tr <= kBoxRows && !(G.epi == EPI_QKV && r < G.seg2);
}

// Where the stages of one tile come from: the tensor map and first physical row of each of its two
// 32-row boxes, how many boxes high a stage is, and whether it streams wide.  Fixed for the tile (a
// tile is one 64-slot stage high), so the producer resolves it once per tile, not once per stage.
struct TileSrc {
  const CUtensorMap* m0;
  const CUtensorMap* m1;
  int y0, y1, nrb;
  bool wide, box3;
};

__device__ __forceinline__ TileSrc tile_src(const GG& G, int r, int tr, int hd, bool box3) {
  TileSrc S;
  S.box3 = box3;
  S.wide = wide_tile(G, r, tr);
  S.nrb = G.nw == 2 ? 2 : (tr + kBoxRows - 1) / kBoxRows;
  if (G.nw == 2) {
    S.m0 = G.m[0]; S.m1 = G.m[1]; S.y0 = S.y1 = r;
  } else {
    const int p0 = phys_row(G, r, hd), p1 = phys_row(G, r + kBoxRows, hd);
    const int s0 = p0 < G.seg1 ? 0 : (p0 < G.seg2 ? 1 : 2);
    const int s1 = p1 < G.seg1 ? 0 : (p1 < G.seg2 ? 1 : 2);
    S.m0 = G.m[s0]; S.m1 = G.m[s1];
    S.y0 = p0 - (s0 == 0 ? 0 : (s0 == 1 ? G.seg1 : G.seg2));
    S.y1 = p1 - (s1 == 0 ? 0 : (s1 == 1 ? G.seg1 : G.seg2));
  }
  return S;
}

// Producer warp: one stage of a tile at column c0 (64 rows x 512 bytes, or 32 rows x 1024 bytes wide).
template <typename WT>
__device__ __forceinline__ void issue_stage(const TileSrc& S, int c0, Ring& R, DevState* st, uint64_t pol, int lane) {
  constexpr int BOXC = 128 / sizeof(WT);   // columns per box
  const int s = R.ctr % kStages;
  if (R.ctr >= (uint32_t)kStages && !mbar_wait_bounded(&R.empty[s], ((R.ctr / kStages) - 1) & 1)) {
    if (lane == 0) set_err(st, ERR_TIMEOUT, 40);
    R.failed = true;
    return;
  }
  if (lane == 0) mbar_arrive_expect_tx(&R.full[s], (uint32_t)((S.wide ? 8 : S.nrb * 4) * kBoxBytes));
  __syncwarp();
  unsigned char* dst = R.base + (size_t)s * kStageBytes;
  if (S.box3) {
    // one copy per 32-row band: bands of the two row boxes (tall), or the two 512-byte halves of a
    // wide stage's 1024 bytes; copy i lands at 16 KB x i, the same bytes as four 2-D boxes each
    const int z = c0 / BOXC;
    if (S.wide) {
      if (lane < 2) tma_box3(dst + (size_t)lane * 4 * kBoxBytes, S.m0, S.y0, z + 4 * lane, &R.full[s], pol);
    } else if (lane < S.nrb) {
      tma_box3(dst + (size_t)lane * 4 * kBoxBytes, lane ? S.m1 : S.m0, lane ? S.y1 : S.y0, z, &R.full[s], pol);
    }
  } else if (S.wide) {
    if (lane < 8)
      tma_box(R.base + (size_t)s * kStageBytes + (size_t)lane * kBoxBytes, S.m0, c0 + lane * BOXC, S.y0, &R.full[s],
              pol);
  } else if (lane < S.nrb * 4) {
    const int rbx = lane >> 2, cb = lane & 3;
    tma_box(R.base + (size_t)s * kStageBytes + (size_t)(rbx * 4 + cb) * kBoxBytes, rbx ? S.m1 : S.m0,
            c0 + cb * BOXC, rbx ? S.y1 : S.y0, &R.full[s], pol);
  }
  ++R.ctr;
}

// Producer warp: one stage of a tcgen05 tile -- 128 rows x 2 chunks (32 KB) in one 3-D copy from
// the 128-row map `mp`, landing [chunk][row][128 B].
__device__ __forceinline__ void issue_tc_stage(const CUtensorMap* mp, int y, int z, Ring& R, DevState* st,
                                               uint64_t pol, int lane) {
  const int s = R.ctr % kStages;
  if (R.ctr >= (uint32_t)kStages && !mbar_wait_bounded(&R.empty[s], ((R.ctr / kStages) - 1) & 1)) {
    if (lane == 0) set_err(st, ERR_TIMEOUT, 45);
    R.failed = true;
    return;
  }
  if (lane == 0) {
    mbar_arrive_expect_tx(&R.full[s], (uint32_t)kStageBytes);
    tma_box3(R.base + (size_t)s * kStageBytes, mp, y, z, &R.full[s], pol);
  }
  __syncwarp();
  ++R.ctr;
}

// Producer warp (all 32 lanes): issue the tensor copies of every stage of the span, tile by tile,
// column chunk by column chunk.
template <typename WT>
__device__ void produce_span(const GG* gg, int gb, int rb, int ge, int re, int hd, bool box3, Ring& R, DevState* st,
                             uint64_t pol, int lane) {
  constexpr int CW = 512 / sizeof(WT);     // columns per stage
  for (int g = gb, r = rb; (g < ge || (g == ge && r < re)) && !R.failed;) {
    const GG& G = gg[g];
    const int last = (g == ge) ? re : G.vrows;
    const int tr = tile_rows(G, r, last);
    if (G.tc) {  // tcgen05 tile: 128 physical rows, 2 chunks a stage; gate/up alternate the matrices
      int rr, cb0, cb1;
      tc_unit(G, r, rr, cb0, cb1);
      const int sg = rr < G.seg1 ? 0 : (rr < G.seg2 ? 1 : 2);
      const int y = rr - (sg == 0 ? 0 : (sg == 1 ? G.seg1 : G.seg2));
      for (int cb = cb0; cb < cb1 && !R.failed; ++cb)
        for (int h = 0; h < G.nw && !R.failed; ++h)
          issue_tc_stage(G.nw == 2 ? G.m[h] + 1 : G.m[sg] + 1, G.nw == 2 ? rr : y, cb * tc::kStageCh, R, st, pol, lane);
      r += tr;
      if (r >= last) { ++g; r = 0; }
      continue;
    }
    const TileSrc S = tile_src(G, r, tr, hd, box3);
    const int cols = G.cols, step = S.wide ? 2 * CW : CW;
    for (int c0 = 0; c0 < cols && !R.failed; c0 += step) issue_stage<WT>(S, c0, R, st, pol, lane);
    r += tr;
    if (r >= last) { ++g; r = 0; }
  }
}

// Producer warp, before it leaves after a failure: let the copies in flight land.
__device__ __forceinline__ void drain_ring(Ring& R, int lane) {
  if (R.failed && lane == 0) {
    const uint32_t first = R.ctr > (uint32_t)kStages ? R.ctr - kStages : 0;
    for (uint32_t c = first; c < R.ctr; ++c) mbar_wait_bounded(&R.full[c % kStages], (c / kStages) & 1);
  }
}

// Tensor-core path (bf16 weights, several vectors, MT m-tiles of 16 vectors): one tile of 64
// weight slots streamed column chunk by column chunk.  Warp w takes the two 16-column k-steps
// 32w..32w+31 of every chunk against all 8 n-tiles (8 weight rows each); it builds the activation
// fragments of its own k-steps in registers (normalised, split into bf16 high and low halves) from
// raw activations it prefetched one chunk ahead, so the warps never wait for each other while
// streaming.  Every weight byte is read from shared memory once (ldmatrix through the swizzle).
// At the end of the tile the 8 warps' partial tiles are added in warp order in `scratch`.
template <typename WT, int MT>
__device__ void mma_tile(const EngineCfg& p, const GG& G, int r, int tr, Ring& R, unsigned char* scratch,
                         const float* rstd_s, Top2* loc) {
  constexpr int CW = 512 / sizeof(WT);
  constexpr int NCT = kNCW * 32;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, tq = lane & 3;
  const int hd = p.D.hd;
  DevState* st = p.B.st;
  const int nv = G.nv, gcols = G.cols;
  float* red = reinterpret_cast<float*>(scratch);  // tile end: [warp][nt][e][lane]
  float acc[8][MT][4];
#pragma unroll
  for (int nt = 0; nt < 8; ++nt)
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[nt][mt][e] = 0.f;
  // this lane's vectors (mt*16 + gq, +8) and its columns of a chunk (k-step ks: 32w + 16ks + 2tq, +8)
  const float* xr[MT][2];
  float xs[MT][2];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int v = mt * 16 + gq + 8 * h;
      xr[mt][h] = (v < nv) ? G.x + (size_t)((G.xrow0 + v) % G.xring) * G.xstride : nullptr;
      xs[mt][h] = (v < nv && G.normw) ? rstd_s[v] : 1.f;
    }
  const int kw = 32 * warp + 2 * tq;
  float2 rx[MT][2][4];  // raw activations of the next chunk: [mt][ks][fragment register]
  float2 rn[2][2];      // norm weights: [ks][k half]
  auto load_raw = [&](int c0) {
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int k = c0 + kw + 16 * ks + 8 * hh;
        rn[ks][hh] = (G.normw && k < gcols) ? *reinterpret_cast<const float2*>(G.normw + k) : make_float2(1.f, 1.f);
      }
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int f = 0; f < 4; ++f) {  // a0: (v, k) a1: (v+8, k) a2: (v, k+8) a3: (v+8, k+8)
          const int k = c0 + kw + 16 * ks + 8 * (f >> 1);
          const float* xp = xr[mt][f & 1];
          rx[mt][ks][f] = (xp && k < gcols) ? *reinterpret_cast<const float2*>(xp + k) : make_float2(0.f, 0.f);
        }
    }
  };
  load_raw(0);
  // epilogue inputs of this thread's output items of m-tile 0 (the residual values, or the rotary
  // cos / sin of the pairs), loaded now so that the tile end waits for no global load
  const bool pairs = G.nw != 2 && G.epi == EPI_QKV && r < G.seg2;
  const int nitem = (G.nw == 2 || pairs) ? 32 * 16 : 64 * 16;
  float pre[4][2];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    pre[k][0] = pre[k][1] = 0.f;
    const int idx = tid + k * NCT, m = idx >> 4, v = idx & 15;
    if (MT == 1 && idx < nitem && v < nv && m < tr) {
      if (G.epi == EPI_RESID) {
        pre[k][0] = __ldcg(G.y + (size_t)((G.yrow0 + v) % G.yring) * G.ystride + r + m);
      } else if (pairs) {
        const size_t at = (size_t)(G.pos0 + v - 1) * (hd / 2) + phys_row(G, r + m, hd) % hd;
        pre[k][0] = __ldg(p.B.rope_cos + at);
        pre[k][1] = __ldg(p.B.rope_sin + at);
      }
    }
  }
  const int jb = 4 * warp + (lane >> 3);  // ldmatrix chunk of this lane (two k-steps x two halves)
  for (int c0 = 0; c0 < gcols; c0 += CW) {
    uint32_t ah[MT][2][4], al[MT][2][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int ks = 0; ks < 2; ++ks)
#pragma unroll
        for (int f = 0; f < 4; ++f) {
          const float sc = xs[mt][f & 1];
          const float2 n = rn[ks][f >> 1];
          const float x0 = rx[mt][ks][f].x * sc * n.x, x1 = rx[mt][ks][f].y * sc * n.y;
          const __nv_bfloat16 hx = __float2bfloat16_rn(x0), hy = __float2bfloat16_rn(x1);
          const float fx = __bfloat162float(hx), fy = __bfloat162float(hy);
          ah[mt][ks][f] = pack_bf16x2(fx, fy);
          al[mt][ks][f] = pack_bf16x2(x0 - fx, x1 - fy);
        }
    if (c0 + CW < gcols) load_raw(c0 + CW);  // lands while this chunk's MMAs run
    const int s = R.ctr % kStages;
    if (!R.failed && !mbar_wait_bounded(&R.full[s], (R.ctr / kStages) & 1)) {
      if (lane == 0) set_err(st, ERR_TIMEOUT, 60);
      R.failed = true;
    }
    if (!R.failed) {
      const uint32_t sb = smem_u32(R.base + (size_t)s * kStageBytes);
      // weight fragments four n-tiles at a time, then the MMAs interleaved over those four
      // independent accumulators (each accumulator still takes hi/lo x k-step in the same order)
#pragma unroll
      for (int nh = 0; nh < 8; nh += 4) {
        uint32_t bq[4][4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int nt = nh + u;
          const bool ok = G.nw == 2 ? (((nt * 8) & 31) < tr) : (nt * 8 < tr);
          if (ok) ldmatrix_x4(sb + stage_off(nt * 8 + (lane & 7), jb), bq[u][0], bq[u][1], bq[u][2], bq[u][3]);
          else bq[u][0] = bq[u][1] = bq[u][2] = bq[u][3] = 0u;
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
          for (int step = 0; step < 4; ++step) {
            const uint32_t* fa = (step & 1) ? al[mt][step >> 1] : ah[mt][step >> 1];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int nt = nh + u;
              const bool ok = G.nw == 2 ? (((nt * 8) & 31) < tr) : (nt * 8 < tr);
              if (ok) mma_bf16(acc[nt][mt], fa, bq[u][(step >> 1) * 2], bq[u][(step >> 1) * 2 + 1]);
            }
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&R.empty[s]);
    ++R.ctr;
  }
  // per m-tile: the 8 warps' partial tiles -> shared memory, added in warp order, epilogue
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
    named_bar(1, NCT);  // the previous user of `red` is done
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) red[((warp * 8 + nt) * 4 + e) * 32 + lane] = acc[nt][mt][e];
    named_bar(1, NCT);
    auto tot = [&](int slot, int vv) {
      const int nt = slot >> 3, n = slot & 7;
      const int ln = (vv & 7) * 4 + (n >> 1);
      const int e = (vv >= 8 ? 2 : 0) + (n & 1);
      float sum = 0.f;
#pragma unroll
      for (int w8 = 0; w8 < kNCW; ++w8) sum += red[((w8 * 8 + nt) * 4 + e) * 32 + ln];
      return sum;
    };
    if (!R.failed) {
      if (G.nw == 2 || pairs) {  // gate/up, or rotary pairs
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int idx = tid + k * NCT;
          const int m = idx >> 4, vv = idx & 15, v = mt * 16 + vv;
          if (v < nv && m < tr)
            epilogue<WT>(p, G, v, pairs ? phys_row(G, r + m, hd) : r + m, tot(m, vv), tot(m + 32, vv), pairs,
                         loc, (MT == 1 && pairs) ? pre[k] : nullptr);
        }
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int idx = tid + k * NCT;
          const int m = idx >> 4, vv = idx & 15, v = mt * 16 + vv;
          if (v < nv && m < tr)
            epilogue<WT>(p, G, v, r + m, tot(m, vv), 0.f, false, loc,
                         (MT == 1 && G.epi == EPI_RESID) ? pre[k] : nullptr);
        }
      }
    }
  }
  named_bar(1, NCT);  // `red` is rewritten by the next tile
}

// State of the tcgen05 path of one CTA: the B operand ring (one 8 KB slot per ring stage), the TMEM
// accumulator (64 columns: gate in 0..31, up in 32..63), the tile-completion mbarrier and its phase.
struct TcCtx {
  unsigned char* bring;   // kStages x the tile shape's B bytes, 1024-byte aligned
  uint32_t tmem;          // TMEM address of column 0
  uint64_t* done;         // arrives when every MMA of the tile has completed
  uint32_t phase;
  uint64_t* bfull;        // [kStages]: the 7 builder warps have written the slot's B (7 arrivals)
  uint32_t bphase;        // bit s: parity of bfull[s]'s next completion (kept by the issuing thread)
};

// tcgen05 tile: output rows r..r+tr-1 (physical rows; whole heads in the rotary region) of a group of
// nv <= NVP vectors (NVP = 16 or 32).  Thread 0 only issues: per stage it waits for the weights and
// for B, issues the 8 MMAs and commits them to the stage's empty barrier in place of warp 0's
// arrival, so the producer refills the slot only after the tensor core has read it.  Warps 1-7 build
// B (high and low halves of the normalised activations of the stage's 128 columns: rows v and NVP+v)
// as soon as its slot is free.  At the tile end warps 0-3 read their 32 TMEM lanes (rows) 16 vectors
// at a time and all 256 threads run the epilogues; RoPE partners (row + hd/2) are exchanged through
// `scratch`.
template <typename WT, int NVP>
__device__ void tc_tile(const EngineCfg& p, const GG& G, int r, int tr, Ring& R, TcCtx& T, unsigned char* scratch,
                        const float* rstd_s, Top2* loc, int cb0, int cb1, int unit) {
  constexpr int NCT = kNCW * 32;
  constexpr int kB = tc::Shape<NVP>::kB;
  constexpr int kBBytes = tc::Shape<NVP>::kBBytes;
  constexpr uint32_t kAcc = tc::Shape<NVP>::kAccCols;
  constexpr int kBuilders = NCT - 32;                          // warps 1-7
  constexpr int NI = (NVP * 16 + kBuilders - 1) / kBuilders;   // B items per builder thread (2 or 3)
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int hd = p.D.hd, nv = G.nv;
  DevState* st = p.B.st;
  // B of a stage is NVP x 16 items (vector, 8-column piece), both halves of each; builder b = tid - 32
  // builds items b + kBuilders i (i < NI), which share the piece (kBuilders is a multiple of 16): the
  // 8 columns 8*(b%16).. of vectors (b + kBuilders i)/16.  Rows and 1/rms are resolved once per tile.
  const int bb = tid - 32;
  const int bpc = bb & 15;
  const float* bx[NI];
  float brs[NI];
  uint32_t boff_hi[NI], boff_lo[NI];
#pragma unroll
  for (int i = 0; i < NI; ++i) {
    const int item = bb + kBuilders * i;
    const int bv = item >> 4;
    const bool use = warp != 0 && item < NVP * 16;
    bx[i] = (use && bv < nv) ? G.x + (size_t)((G.xrow0 + bv) % G.xring) * G.xstride : nullptr;
    brs[i] = (use && bv < nv && G.normw) ? rstd_s[bv] : 1.f;
    boff_hi[i] = use ? (uint32_t)((bpc >> 3) * kB * 128 + bv * 128 + (((bpc & 7) ^ (bv & 7)) << 4)) : 0xffffffffu;
    boff_lo[i] = use ? (uint32_t)((bpc >> 3) * kB * 128 + (NVP + bv) * 128 + (((bpc & 7) ^ ((NVP + bv) & 7)) << 4))
                     : 0xffffffffu;
  }
  // The stage's activations and norm weights of this thread come from L2 (each stage touches new
  // columns), so they are loaded one column block ahead into registers.  Two register sets take
  // turns; the column-block loop is unrolled by two so that each set keeps a fixed name.
  constexpr int CB = tc::kStageCh * tc::kChunk;  // columns per stage
  const int ncb = cb1;                            // blocks [cb0, cb1) of this tile (unit)
  float4 xa[NI][2], xb[NI][2], na[2], nb[2];
  auto fetch = [&](int cb, float4 (*xr)[2], float4* nr) {
    if (cb < ncb) {
      const int col = cb * CB + 8 * bpc;
#pragma unroll
      for (int i = 0; i < NI; ++i)
        if (bx[i]) {
          xr[i][0] = *reinterpret_cast<const float4*>(bx[i] + col);
          xr[i][1] = *reinterpret_cast<const float4*>(bx[i] + col + 4);
        }
      if (G.normw && bx[0]) {
        nr[0] = *reinterpret_cast<const float4*>(G.normw + col);
        nr[1] = *reinterpret_cast<const float4*>(G.normw + col + 4);
      }
    }
  };
  auto build_b = [&](unsigned char* b, const float4 (*x4)[2], const float4* n4) {
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      if (boff_hi[i] == 0xffffffffu) continue;  // no item (vectors >= nv still get zero rows)
      uint4 hi = make_uint4(0u, 0u, 0u, 0u), lo = hi;
      if (bx[i]) {
        float xv[8] = {x4[i][0].x, x4[i][0].y, x4[i][0].z, x4[i][0].w, x4[i][1].x, x4[i][1].y, x4[i][1].z, x4[i][1].w};
        if (G.normw) {
          const float nv8[8] = {n4[0].x, n4[0].y, n4[0].z, n4[0].w, n4[1].x, n4[1].y, n4[1].z, n4[1].w};
#pragma unroll
          for (int e = 0; e < 8; ++e) xv[e] = xv[e] * brs[i] * nv8[e];
        }
        uint32_t h4[4], l4[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const __nv_bfloat16 a = __float2bfloat16_rn(xv[2 * e]), c = __float2bfloat16_rn(xv[2 * e + 1]);
          const float fa = __bfloat162float(a), fc = __bfloat162float(c);
          h4[e] = pack_bf16x2(fa, fc);
          l4[e] = pack_bf16x2(xv[2 * e] - fa, xv[2 * e + 1] - fc);
        }
        hi = make_uint4(h4[0], h4[1], h4[2], h4[3]);
        lo = make_uint4(l4[0], l4[1], l4[2], l4[3]);
      }
      *reinterpret_cast<uint4*>(b + boff_hi[i]) = hi;
      *reinterpret_cast<uint4*>(b + boff_lo[i]) = lo;
    }
  };
  // Builders (warps 1-7): the nw stages (gate, up) of column block cb from set (x, n); block cb+1
  // prefetched into (xp, np).  B of a stage does not depend on its weights, so it is built as soon as
  // its slot is free -- when ring slot s was last released (its empty barrier completed for the stage
  // kStages back, which for a tensor-core stage means its MMAs are done).  A builder warp releases the
  // ring slot with its B report: the slot completes only with thread 0's commit, which follows the
  // MMAs.  The builders run up to kStages stages ahead of the tensor core.
  auto block = [&](int cb, const float4 (*x)[2], const float4* n, float4 (*xp)[2], float4* np) {
    fetch(cb + 1, xp, np);
    for (int h = 0; h < G.nw; ++h) {
      const int s = R.ctr % kStages;
      if (R.ctr >= (uint32_t)kStages && !R.failed &&
          !mbar_wait_bounded(&R.empty[s], ((R.ctr / kStages) - 1) & 1)) {
        if (lane == 0) set_err(st, ERR_TIMEOUT, 64);
        R.failed = true;
      }
      if (!R.failed) build_b(T.bring + (size_t)s * kBBytes, x, n);
      tc::fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&T.bfull[s]);
        mbar_arrive(&R.empty[s]);
      }
      ++R.ctr;
    }
  };
  const int nstages = (ncb - cb0) * G.nw;
  if (warp != 0) {
    fetch(cb0, xa, na);
    for (int cb = cb0; cb < ncb; cb += 2) {
      block(cb, xa, na, xb, nb);
      if (cb + 1 < ncb) block(cb + 1, xb, nb, xa, na);
    }
  } else if (tid == 0) {
    // the issuer: per stage the weights and B of the slot, then the MMAs (gate / up accumulators in
    // columns [0, kAcc) / [kAcc, 2 kAcc)); after a failed wait it still releases every slot
    for (int k = 0; k < nstages; ++k) {
      const int s = R.ctr % kStages, h = k % G.nw, cb = cb0 + k / G.nw;
      if (!R.failed && !mbar_wait_bounded(&R.full[s], (R.ctr / kStages) & 1)) {
        set_err(st, ERR_TIMEOUT, 61);
        R.failed = true;
      }
      const bool bok = !R.failed && mbar_wait_bounded(&T.bfull[s], (T.bphase >> s) & 1u);
      T.bphase ^= 1u << s;
      if (bok) {
        tc::fence_after();
        tc::mma_stage<NVP>(T.tmem + kAcc * (uint32_t)h, R.base + (size_t)s * kStageBytes,
                           T.bring + (size_t)s * kBBytes, cb == cb0);
        tc::commit(&R.empty[s]);  // warp 0's arrival, when the MMAs have read the stage
      } else {
        if (!R.failed) { set_err(st, ERR_TIMEOUT, 63); R.failed = true; }
        mbar_arrive(&R.empty[s]);
      }
      ++R.ctr;
    }
  } else {
    R.ctr += (uint32_t)nstages;  // lanes 1-31 of warp 0 wait at the tile end
  }
  __syncwarp();
  // tile end: every MMA done -> TMEM rows to registers -> epilogues.  The completion is committed
  // whatever happened (it arrives once the MMAs issued so far are done, at once if there are none),
  // so the barrier's phase stays in step with T.phase on the failure path too.
  if (tid == 0) tc::commit(T.done);
  bool ok = mbar_wait_bounded(T.done, T.phase);
  T.phase ^= 1u;
  if (!ok) { if (lane == 0) set_err(st, ERR_TIMEOUT, 62); R.failed = true; }
  ok = ok && !R.failed;
  tc::fence_after();
  const bool pairs = G.epi == EPI_QKV && r < G.seg2;
  const bool wok = __all_sync(0xffffffffu, ok);  // tcgen05.ld is warp-collective
  const int row = 32 * warp + lane;              // tile-local physical row (warps 0-3)
  // The tile's results go to shared memory, ya[row][v] (hi + lo of accumulator 0) and yb[row][v]
  // (accumulator 1: the up projection), then all 256 threads run the epilogues, items (row, v) with
  // consecutive rows on consecutive threads; each thread first loads every epilogue input of its
  // items (residual values, rotary cos / sin) and then computes, so the loads overlap.
  float* ya = reinterpret_cast<float*>(scratch);
  float* yb = ya + tc::kRows * NVP;
  constexpr int MAXK = tc::kRows * NVP / NCT;  // items per thread
  auto run_epilogues = [&]() {
    const int nitem = tc::kRows * nv;
    float pre[MAXK][2];
#pragma unroll
    for (int k = 0; k < MAXK; ++k) {
      const int idx = tid + k * NCT, rw = idx % tc::kRows, v = idx / tc::kRows;
      pre[k][0] = pre[k][1] = 0.f;
      if (idx < nitem && rw < tr) {
        if (G.epi == EPI_RESID) {
          pre[k][0] = __ldcg(G.y + (size_t)((G.yrow0 + v) % G.yring) * G.ystride + r + rw);
        } else if (pairs && (r + rw) % hd < hd / 2) {
          const size_t at = (size_t)(G.pos0 + v - 1) * (hd / 2) + (r + rw) % hd;
          pre[k][0] = __ldg(p.B.rope_cos + at);
          pre[k][1] = __ldg(p.B.rope_sin + at);
        }
      }
    }
#pragma unroll
    for (int k = 0; k < MAXK; ++k) {
      const int idx = tid + k * NCT, rw = idx % tc::kRows, v = idx / tc::kRows;
      if (idx >= nitem || rw >= tr) continue;
      const float y0 = ya[rw * NVP + v];
      if (pairs) {
        if ((r + rw) % hd < hd / 2)  // tiles start on a head boundary
          epilogue<WT>(p, G, v, r + rw, y0, ya[(rw + hd / 2) * NVP + v], true, loc, pre[k]);
      } else if (G.nw == 2) {
        epilogue<WT>(p, G, v, r + rw, y0, yb[rw * NVP + v], false, loc);
      } else {
        epilogue<WT>(p, G, v, r + rw, y0, 0.f, false, loc, G.epi == EPI_RESID ? pre[k] : nullptr);
      }
    }
  };
  if (G.ks > 1) {
    // split-K unit: partial tile [acc][vector][128 rows] to scratch; the last unit of the tile adds
    // the ks partials in segment order into ya / yb and runs the epilogues
    __shared__ int s_last_unit;
    const int usz = G.nw * NVP * tc::kRows;
    float* pu = p.B.tc_part + G.pbase + (size_t)unit * usz;
    if (warp < 4 && wok) {
      for (int acc = 0; acc < G.nw; ++acc)
#pragma unroll
        for (int v0 = 0; v0 < NVP; v0 += 16) {
          if (v0 >= nv) break;
          uint32_t dh[16], dl[16];
          tc::load_rows16(T.tmem + kAcc * (uint32_t)acc + v0, warp, dh);
          tc::load_rows16(T.tmem + kAcc * (uint32_t)acc + NVP + v0, warp, dl);
#pragma unroll
          for (int v = 0; v < 16; ++v)
            __stcg(pu + (size_t)(acc * NVP + v0 + v) * tc::kRows + row, __uint_as_float(dh[v]) + __uint_as_float(dl[v]));
        }
    }
    __threadfence();
    tc::fence_before();
    named_bar(1, NCT);
    if (tid == 0) {
      int* tk = p.B.tc_tick + G.tbase + unit / G.ks;
      const int old = atomicAdd(tk, 1);
      s_last_unit = old == G.ks - 1;
      if (s_last_unit) *tk = 0;  // left at zero for the next phase
    }
    named_bar(1, NCT);
    if (s_last_unit && wok) {
      __threadfence();
      const float* pt = p.B.tc_part + G.pbase + (size_t)(unit / G.ks) * G.ks * usz;
      // element e = (acc * NVP + v) * 128 + row of the tile, summed over the segments in order; four
      // elements per thread at a time with all their loads issued together
      const int nel = G.nw * NVP * tc::kRows;
      for (int e0 = tid; e0 < nel; e0 += 4 * NCT) {
        float acc4[4] = {0.f, 0.f, 0.f, 0.f};
        for (int sg = 0; sg < G.ks; ++sg) {
          float vv[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int e = e0 + q * NCT;
            vv[q] = e < nel ? __ldcg(pt + (size_t)sg * usz + e) : 0.f;
          }
#pragma unroll
          for (int q = 0; q < 4; ++q) acc4[q] += vv[q];
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int e = e0 + q * NCT;
          if (e < nel) {
            const int rw = e % tc::kRows, av = e / tc::kRows, acc = av / NVP, v = av % NVP;
            (acc ? yb : ya)[rw * NVP + v] = acc4[q];
          }
        }
      }
    }
    named_bar(1, NCT);
    if (s_last_unit && wok) run_epilogues();
    tc::fence_before();
    named_bar(1, NCT);  // TMEM and the shared buffers are rewritten by the next tile
    return;
  }
  if (warp < 4 && wok) {
#pragma unroll
    for (int v0 = 0; v0 < NVP; v0 += 16) {
      if (v0 >= nv) break;
      uint32_t dh[16], dl[16];
      tc::load_rows16(T.tmem + v0, warp, dh);
      tc::load_rows16(T.tmem + NVP + v0, warp, dl);
#pragma unroll
      for (int v = 0; v < 16; ++v) ya[row * NVP + v0 + v] = __uint_as_float(dh[v]) + __uint_as_float(dl[v]);
      if (G.nw == 2) {
        tc::load_rows16(T.tmem + kAcc + v0, warp, dh);
        tc::load_rows16(T.tmem + kAcc + NVP + v0, warp, dl);
#pragma unroll
        for (int v = 0; v < 16; ++v) yb[row * NVP + v0 + v] = __uint_as_float(dh[v]) + __uint_as_float(dl[v]);
      }
    }
  }
  named_bar(1, NCT);
  if (wok) run_epilogues();
  tc::fence_before();
  named_bar(1, NCT);  // TMEM and `scratch` are rewritten by the next tile
}

// Single-vector tile: output rows r..r+tr-1 of G, its column-chunk stages from the ring, then the
// epilogue.  The input vector comes from `xs` (staged in shared memory, already normalised) or,
// when null, from G.x through L1 (times rstd and the norm weight when the group has a norm).
template <typename WT>
__device__ void sv_tile(const EngineCfg& p, const GG& G, int r, int tr, Ring& R, const float* xs, float rstd,
                        Top2* loc) {
  constexpr int VEC = WTraits<WT>::kVec;
  constexpr int CW = 512 / sizeof(WT);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int hd = p.D.hd;
  DevState* st = p.B.st;
  // ---------------- single-vector path ----------------
  const float* xr = G.x + (size_t)(G.xrow0 % G.xring) * G.xstride;
  // the epilogue inputs of this lane's output row, loaded now: they are in registers when the
  // tile ends (the residual value, or the rotary cos / sin of the pair)
  float pre[2] = {0.f, 0.f};
  if (lane < 8 && G.nw != 2) {
    const int slot = warp + 8 * lane;
    if (G.epi == EPI_QKV && r < G.seg2) {
      if (lane < 4) {
        const int i = phys_row(G, r + slot, hd) % hd;
        const size_t at = (size_t)(G.pos0 - 1) * (hd / 2) + i;
        pre[0] = __ldg(p.B.rope_cos + at);
        pre[1] = __ldg(p.B.rope_sin + at);
      }
    } else if (G.epi == EPI_RESID && slot < tr) {
      pre[0] = __ldcg(G.y + (size_t)(G.yrow0 % G.yring) * G.ystride + r + slot);
    }
  }
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  // the lane's VEC input values at column `col` (normalised when the group has a norm), 0 beyond
  auto load_x = [&](int col, float* xv) {
    if (col < G.cols && xs) {
#pragma unroll
      for (int e = 0; e < VEC; e += 4) {
        const float4 q = *reinterpret_cast<const float4*>(xs + col + e);
        xv[e] = q.x; xv[e + 1] = q.y; xv[e + 2] = q.z; xv[e + 3] = q.w;
      }
    } else if (col < G.cols) {
#pragma unroll
      for (int e = 0; e < VEC; e += 4) {
        float4 q = *reinterpret_cast<const float4*>(xr + col + e);
        if (G.normw) {
          const float4 n4 = *reinterpret_cast<const float4*>(G.normw + col + e);
          q.x = q.x * rstd * n4.x; q.y = q.y * rstd * n4.y;
          q.z = q.z * rstd * n4.z; q.w = q.w * rstd * n4.w;
        }
        xv[e] = q.x; xv[e + 1] = q.y; xv[e + 2] = q.z; xv[e + 3] = q.w;
      }
    } else {
#pragma unroll
      for (int e = 0; e < VEC; ++e) xv[e] = 0.f;
    }
  };
  // tall stage: 64 rows x 512 bytes, warp w rows w + 8i (i < 8), lane l chunk l.  Wide stage:
  // 32 rows x 1024 bytes, warp w rows w + 8i (i < 4), lane l chunks l and l + 32 -- the same
  // chunks, in the same order, as two consecutive tall stages
  const bool wide = wide_tile(G, r, tr);
  for (int c0 = 0; c0 < G.cols; c0 += wide ? 2 * CW : CW) {
    const int s = R.ctr % kStages;
    if (!R.failed && !mbar_wait_bounded(&R.full[s], (R.ctr / kStages) & 1)) {
      if (lane == 0) set_err(st, ERR_TIMEOUT, 50);
      R.failed = true;
    }
    if (!R.failed) {
      const unsigned char* sb = R.base + (size_t)s * kStageBytes;
      uint4 wq[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {  // all eight weight chunks first (independent loads)
        const int slot = wide ? warp + 8 * (i & 3) : warp + 8 * i;
        const int j = wide ? lane + 32 * (i >> 2) : lane;
        const bool ok = wide ? slot < tr : (G.nw == 2 ? ((slot & 31) < tr) : (slot < tr));
        wq[i] = ok ? *reinterpret_cast<const uint4*>(sb + stage_off(slot, j)) : make_uint4(0, 0, 0, 0);
      }
      float xv[VEC];
      load_x(c0 + VEC * lane, xv);
      if (!wide) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          float wf[VEC];
          WTraits<WT>::unpack(wq[i], wf);
#pragma unroll
          for (int e = 0; e < VEC; ++e) acc[i] = fmaf(wf[e], xv[e], acc[i]);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float wf[VEC];
          WTraits<WT>::unpack(wq[i], wf);
#pragma unroll
          for (int e = 0; e < VEC; ++e) acc[i] = fmaf(wf[e], xv[e], acc[i]);
        }
        load_x(c0 + CW + VEC * lane, xv);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float wf[VEC];
          WTraits<WT>::unpack(wq[i + 4], wf);
#pragma unroll
          for (int e = 0; e < VEC; ++e) acc[i] = fmaf(wf[e], xv[e], acc[i]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&R.empty[s]);
    ++R.ctr;
  }
  float sums[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) sums[i] = warp_sum(acc[i]);
  if (!R.failed && lane < 8) {  // lane i finishes slot warp + 8i (and its partner slot + 32)
    float y0 = 0.f, y1 = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (k == lane) y0 = sums[k];
      if (k == lane + 4) y1 = sums[k];
    }
    const int slot = warp + 8 * lane;
    if (G.nw == 2) {
      if (lane < 4 && slot < tr) epilogue<WT>(p, G, 0, r + slot, y0, y1, false, loc);
    } else if (G.epi == EPI_QKV && r < G.seg2) {
      if (lane < 4) epilogue<WT>(p, G, 0, phys_row(G, r + slot, hd), y0, y1, true, loc, pre);
    } else if (slot < tr) {
      epilogue<WT>(p, G, 0, r + slot, y0, 0.f, false, loc, G.epi == EPI_RESID ? pre : nullptr);
    }
  }
}

// Consumer warps (named barrier 1, 256 threads): consume every stage of the span and run the
// epilogues.  `scratch` (kMmaScratch bytes) holds the tensor-core path's activation fragments and
// pair exchange, `rstd_s` one 1/rms per vector, `wpart` kNCW floats, `loc` the thread's top-2 per
// head kind.
template <typename WT, int TCMAX>
static __device__ void consume_span(const EngineCfg& p, const GG* gg, int gb, int rb, int ge, int re, Ring& R,
                             unsigned char* scratch, float* rstd_s, float* wpart, Top2* loc, TcCtx* tcx) {
  constexpr int VEC = WTraits<WT>::kVec;
  constexpr int CW = 512 / sizeof(WT);
  constexpr int NCT = kNCW * 32;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, tq = lane & 3;
  const int hd = p.D.hd;
  DevState* st = p.B.st;
  float rstd = 1.f;
  bool xs_on = false;  // single-vector group: its (normalised) input vector is staged in `scratch`
  float* xs = reinterpret_cast<float*>(scratch);
  int last_g = -1;
  for (int g = gb, r = rb; g < ge || (g == ge && r < re);) {
    const GG& G = gg[g];
    const int last = (g == ge) ? re : G.vrows;
    const int tr = tile_rows(G, r, last);
    if (g != last_g) {  // group entry: 1/rms of the input vector(s)
      named_bar(1, NCT);
      rstd = 1.f;
      xs_on = false;
      if (!G.mma) {
        const float* xr = G.x + (size_t)(G.xrow0 % G.xring) * G.xstride;
        if (G.normw) {
          float sq = 0.f;
#pragma unroll 4
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
        // the whole input vector once into shared memory (x * rstd * norm weight when normalised,
        // the product formed in the same order as on the streaming path): no per-stage loads
        if (G.cols * (int)sizeof(float) <= kMmaScratch) {
          xs_on = true;
          for (int c = tid * 4; c < G.cols; c += NCT * 4) {
            float4 q = *reinterpret_cast<const float4*>(xr + c);
            if (G.normw) {
              const float4 n4 = *reinterpret_cast<const float4*>(G.normw + c);
              q.x = q.x * rstd * n4.x; q.y = q.y * rstd * n4.y;
              q.z = q.z * rstd * n4.z; q.w = q.w * rstd * n4.w;
            }
            *reinterpret_cast<float4*>(xs + c) = q;
          }
        }
      } else if (G.normw) {
        for (int v = warp; v < G.nv; v += kNCW) {
          const float* xr = G.x + (size_t)((G.xrow0 + v) % G.xring) * G.xstride;
          float sq = 0.f;
#pragma unroll 8
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
      sv_tile<WT>(p, G, r, tr, R, xs_on ? xs : nullptr, rstd, loc);
    } else if (G.tc) {
      int rr, cb0, cb1;
      tc_unit(G, r, rr, cb0, cb1);
      const int trr = G.ks > 1 ? tc::kRows : tr;
      const int unit = r / tc::kRows;
      if constexpr (TCMAX > 16) {
        if (G.nv > 16) tc_tile<WT, 32>(p, G, rr, trr, R, *tcx, scratch, rstd_s, loc, cb0, cb1, unit);
        else tc_tile<WT, 16>(p, G, rr, trr, R, *tcx, scratch, rstd_s, loc, cb0, cb1, unit);
      } else {
        tc_tile<WT, 16>(p, G, rr, trr, R, *tcx, scratch, rstd_s, loc, cb0, cb1, unit);
      }
    } else if (G.nv <= 16) {
      mma_tile<WT, 1>(p, G, r, tr, R, scratch, rstd_s, loc);
    } else {
      mma_tile<WT, 2>(p, G, r, tr, R, scratch, rstd_s, loc);
    }
    r += tr;
    if (r >= last) { ++g; r = 0; }
  }
}

// Consumer warps: merge the threads' top-2 (lanes 0..7 of each warp hold one) into this CTA's
// head partial (8 floats: per kind v1, i1, v2, i2).  The order of a top-2 merge does not matter.
__device__ __forceinline__ void write_head_partial(const Top2* loc, Top2 (*hred)[2], float* hp) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (lane < 8) { hred[warp * 8 + lane][0] = loc[0]; hred[warp * 8 + lane][1] = loc[1]; }
  named_bar(1, kNCW * 32);
  if (tid == 0) {
    for (int k = 0; k < 2; ++k) {
      Top2 m = hred[0][k];
      for (int i = 1; i < kNCW * 8; ++i) top2_merge(m, hred[i][k]);
      hp[k * 4 + 0] = m.v1; hp[k * 4 + 1] = __int_as_float(m.i1);
      hp[k * 4 + 2] = m.v2; hp[k * 4 + 3] = __int_as_float(m.i2);
    }
  }
}

}  // namespace eng
}  // namespace spd
