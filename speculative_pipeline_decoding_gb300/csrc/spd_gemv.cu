// Grouped multi-weight GEMV engine for the SPD cycle.
//
// One launch computes y_g = W_g x_g for G groups with DISTINCT weights (the stage-diagonal step:
// the token at depth j uses layer j*S+s), or one group with several input vectors sharing the
// weights (draft-module rows, prefill blocks).  Weight rows are streamed once from HBM with 1-D
// bulk copies (cp.async.bulk, L2 evict-first) into a ring of shared-memory stages guarded by
// mbarriers; one producer warp issues the copies, eight consumer warps multiply in fp32.
//
// Work split: the rows of all groups are concatenated and every CTA of a persistent grid takes one
// contiguous, equal share (tiles of <= 4 rows never straddle a group).  A row's arithmetic depends
// only on its column count: thread k of the block owns 16-byte column vectors k, k+256, ... of
// every chunk, the chunk width is a function of the column count, and partial sums are reduced
// across lanes (xor tree) and warps (fixed order) per chunk, chunks added in order.  So a token
// gets bit-identical results whether it runs alone (plain AR) or with n-1 other tokens (SPD).
//
// Fused prologues/epilogues:
//   QKV    x = RMSNorm(h) * attn_norm          -> q|k|v rows (fp32)
//   O      x = attention output                -> h += y
//   GATEUP x = RMSNorm(h) * ffn_norm, 2 weights -> u = silu(gate) * up
//   DOWN   x = u                               -> h += y, anchor capture when layer+1 = b_i
//   FC     x = concat(h^(b_0..b_f)) (contiguous prefix of the anchor row) -> draft row z
//   HEAD   x = RMSNorm(h) * final norm        -> per-CTA top-2 of the logits (+ debug logits)
#include "spd_internal.cuh"

namespace spd {

namespace {

constexpr int kBig = 1 << 30;
constexpr int kRing = 90 * 1024;
constexpr int kStageLimit = 48 * 1024;

struct GG {
  const void* w[3];
  int seg1, seg2;
  int rows, cols, nv;
  const float* x; int xrow0, xring, xstride;
  float* y; int yrow0, yring, ystride;
  const float* normw;
  float* anch; int arow0, aring, astride;
  int row_begin;
  int kind;
};

struct GemvParams {
  int op;
  int explicit_mode;
  int mma_ok;   // bf16 weights, every column count a multiple of 16 (tensor-core path allowed)
  int max_nv;   // largest vector count a group of this launch can have
  int debug_logits;
  float eps;
  Dims D;
  Bufs B;
  Launch lc;
  GemvExplicit ge;
};

__host__ __device__ __forceinline__ int chunk_cols(int cols, int nw, int esz) {
  if (kGemvTR * nw * cols * esz <= kStageLimit) return cols;
  return 4096 / esz;  // 4 KB of each row per stage
}

__device__ __forceinline__ int anchor_index(const Dims& D, int layer_done) {
  for (int i = 0; i < D.m; ++i)
    if (D.anchors[i] == layer_done) return i;
  return -1;
}

__device__ int resolve_groups(const GemvParams& p, GG* gg) {
  const Dims& D = p.D;
  const Bufs& B = p.B;
  const Launch& lc = p.lc;
  DevState* st = B.st;
  if (p.explicit_mode) {
    for (int g = 0; g < p.ge.G; ++g) {
      GG& o = gg[g];
      o.w[0] = o.w[1] = o.w[2] = p.ge.W[g];
      o.rows = o.seg1 = o.seg2 = p.ge.rows;
      o.cols = p.ge.cols; o.nv = 1;
      o.x = p.ge.x[g]; o.xrow0 = 0; o.xring = kBig; o.xstride = p.ge.cols;
      o.y = p.ge.y[g]; o.yrow0 = 0; o.yring = kBig; o.ystride = p.ge.rows;
      o.normw = p.ge.nw; o.anch = nullptr; o.kind = 0;
    }
    return p.ge.G;
  }
  const Act& A = lc.act;
  if (p.op == OP_HEAD) {
    int ng = 0;
    auto add = [&](const float* x, int xrow0, int xring, const void* W, const float* nw, int kind) {
      GG& o = gg[ng++];
      o.w[0] = o.w[1] = o.w[2] = W;
      o.rows = o.seg1 = o.seg2 = D.V; o.cols = D.d; o.nv = 1;
      o.x = x; o.xrow0 = xrow0; o.xring = xring; o.xstride = D.d;
      o.y = nullptr; o.normw = nw; o.anch = nullptr; o.kind = kind;
    };
    if (lc.kind == LK_DIAG) {
      if (st->a == D.n) add(B.resid, (st->t - D.n + 1) % (D.n + 1), D.n + 1, B.lm_head, B.final_norm, 0);
      if (!(st->flags & SF_TARGET_ONLY)) {
        const int R = st->t - st->pdm_len;
        if (R < 1 || R > D.n + 1) {
          set_err(st, ERR_PDM_ROWS, 200);
        } else {
          add(A.qkv /* draft rows z */, R - 1, kBig, B.pdm_head, B.pdm_norm, 1);
        }
      }
    } else if (lc.kind == LK_AR) {
      add(B.resid, st->t % (D.n + 1), D.n + 1, B.lm_head, B.final_norm, 0);
    } else if (lc.kind == LK_ROWS) {
      add(A.resid, lc.cnt - 1, kBig, B.lm_head, B.final_norm, 0);
    }
    return ng;
  }
  if (p.op == OP_FC) {
    // draft rows: depth by the staircase, f by the anchor table; equal f are contiguous runs
    if (lc.kind == LK_ROWS) {
      const int f = D.ftab[D.n];
      GG& o = gg[0];
      o.w[0] = o.w[1] = o.w[2] = B.fc[f];
      o.rows = o.seg1 = o.seg2 = D.d; o.cols = (f + 1) * D.d; o.nv = lc.cnt;
      o.x = A.anch; o.xrow0 = 0; o.xring = kBig; o.xstride = D.m * D.d;
      o.y = A.resid; o.yrow0 = 0; o.yring = kBig; o.ystride = D.d;
      o.normw = nullptr; o.anch = nullptr; o.kind = 0;
      return 1;
    }
    const int t = st->t, a = st->a, R = t - st->pdm_len;
    if (R < 1 || R > D.n + 1) {
      set_err(st, ERR_PDM_ROWS, 300);
      return 0;
    }
    int ng = 0, prev_f = -1;
    for (int r = 0; r < R; ++r) {
      const int pos = st->pdm_len + 1 + r;
      const int depth = (t - pos < a) ? (t - pos) : D.n;
      const int f = D.ftab[depth];
      if (f != prev_f) {
        GG& o = gg[ng++];
        o.w[0] = o.w[1] = o.w[2] = B.fc[f];
        o.rows = o.seg1 = o.seg2 = D.d; o.cols = (f + 1) * D.d; o.nv = 0;
        o.x = B.anch; o.xrow0 = pos % (D.n + 1); o.xring = D.n + 1; o.xstride = D.m * D.d;
        o.y = A.resid; o.yrow0 = r; o.yring = kBig; o.ystride = D.d;
        o.normw = nullptr; o.anch = nullptr; o.kind = 0;
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
  for (int i = 0; i < nr; ++i) {
    GG& o = gg[i];
    const LayerW& w = LW[rg[i].layer];
    o.nv = rg[i].nv; o.anch = nullptr; o.kind = 0;
    switch (p.op) {
      case OP_QKV:
        o.w[0] = w.wq; o.w[1] = w.wk; o.w[2] = w.wv;
        o.seg1 = hqd; o.seg2 = hqd + D.hkv * D.hd; o.rows = D.qkv_rows; o.cols = D.d;
        o.x = A.resid; o.xrow0 = rg[i].rrow0; o.xring = A.resid_ring; o.xstride = D.d;
        o.normw = (const float*)w.attn_norm;
        o.y = A.qkv; o.yrow0 = rg[i].vid0; o.yring = kBig; o.ystride = D.qkv_rows;
        break;
      case OP_O:
        o.w[0] = o.w[1] = o.w[2] = w.wo;
        o.rows = o.seg1 = o.seg2 = D.d; o.cols = hqd;
        o.x = A.attn; o.xrow0 = rg[i].vid0; o.xring = kBig; o.xstride = hqd;
        o.normw = nullptr;
        o.y = A.resid; o.yrow0 = rg[i].rrow0; o.yring = A.resid_ring; o.ystride = D.d;
        break;
      case OP_GATEUP:
        o.w[0] = w.wg; o.w[1] = w.wu; o.w[2] = w.wu;
        o.rows = o.seg1 = o.seg2 = D.ffn; o.cols = D.d;
        o.x = A.resid; o.xrow0 = rg[i].rrow0; o.xring = A.resid_ring; o.xstride = D.d;
        o.normw = (const float*)w.ffn_norm;
        o.y = A.u; o.yrow0 = rg[i].vid0; o.yring = kBig; o.ystride = D.ffn;
        break;
      default: {  // OP_DOWN
        o.w[0] = o.w[1] = o.w[2] = w.wd;
        o.rows = o.seg1 = o.seg2 = D.d; o.cols = D.ffn;
        o.x = A.u; o.xrow0 = rg[i].vid0; o.xring = kBig; o.xstride = D.ffn;
        o.normw = nullptr;
        o.y = A.resid; o.yrow0 = rg[i].rrow0; o.yring = A.resid_ring; o.ystride = D.d;
        const int ai = (lc.stack == 0 && A.anch) ? anchor_index(D, rg[i].layer + 1) : -1;
        if (ai >= 0) {
          o.anch = A.anch + (size_t)ai * D.d; o.arow0 = rg[i].rrow0; o.aring = A.anch_ring;
          o.astride = D.m * D.d;
        }
      }
    }
  }
  return nr;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <int OP, typename WT, int NVB>
__global__ void __launch_bounds__(kGemvThreads, NVB == 1 ? 2 : 1)
gemv_kernel(const __grid_constant__ GemvParams p) {
  extern __shared__ __align__(128) unsigned char ring[];
  constexpr int NW = (OP == OP_GATEUP) ? 2 : 1;
  constexpr int VEC = WTraits<WT>::kVec;
  constexpr int ESZ = sizeof(WT);
  constexpr int TR = kGemvTR;
  constexpr int NRED = TR * NW * NVB;
  constexpr int NCW = kGemvConsumerWarps;
  constexpr int NCT = NCW * 32;

  __shared__ GG gg[kMaxGroups];
  __shared__ int s_ng, s_total, s_ns, s_slot;
  __shared__ __align__(8) uint64_t full_bar[kGemvMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kGemvMaxStages];
  __shared__ float red[2][NCW][NRED];
  __shared__ float tot[TR * NW * kGemvMaxNV];
  __shared__ float rstd_s[kGemvMaxNV];
  __shared__ Top2 hred[32][2];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  DevState* st = p.B.st;

  if (tid == 0) {
    const bool skip = !p.explicit_mode && (st->done || st->err);
    const int ng = skip ? 0 : resolve_groups(p, gg);
    int total = 0, slot = 16;
    for (int i = 0; i < ng; ++i) {
      gg[i].row_begin = total;
      total += gg[i].rows;
      const int cw = chunk_cols(gg[i].cols, NW, ESZ);
      slot = max(slot, TR * NW * cw * ESZ);
    }
    s_ng = ng; s_total = total; s_slot = slot;
    s_ns = min(kGemvMaxStages, kRing / slot);
    for (int i = 0; i < kGemvMaxStages; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], NCW);
    }
    fence_mbar_init();
  }
  __syncthreads();

  const int ng = s_ng;
  if (OP == OP_HEAD) {
    if (tid < 32) { top2_init(hred[tid][0]); top2_init(hred[tid][1]); }
  }
  if (ng == 0 || s_ns < 1) {
    if (OP == OP_HEAD && tid == 0) {
      float* hp = p.B.head_part + (size_t)blockIdx.x * 8;
      for (int k = 0; k < 2; ++k) {
        hp[k * 4 + 0] = -INFINITY; hp[k * 4 + 1] = __int_as_float(0x7fffffff);
        hp[k * 4 + 2] = -INFINITY; hp[k * 4 + 3] = __int_as_float(0x7fffffff);
      }
    }
    return;
  }
  const long long total = s_total;
  const int r_begin = (int)(total * blockIdx.x / gridDim.x);
  const int r_end = (int)(total * (blockIdx.x + 1) / gridDim.x);
  const int NS = s_ns;
  const int slot = s_slot;

  if (warp == NCW) {
    // ------------------------------ producer warp ------------------------------
    const uint64_t pol = l2_evict_first_policy();
    uint32_t ctr = 0;
    bool failed = false;
    int g = 0;
    for (int r = r_begin; r < r_end && !failed;) {
      while (r >= gg[g].row_begin + gg[g].rows) ++g;
      const GG& G = gg[g];
      const int rl = r - G.row_begin;
      const int tr = min(TR, min(r_end - r, G.rows - rl));
      const int cw = chunk_cols(G.cols, NW, ESZ);
      for (int c0 = 0; c0 < G.cols; c0 += cw) {
        const int w = min(cw, G.cols - c0);
        const uint32_t brow = (uint32_t)w * ESZ;
        const int s = ctr % NS;
        if (ctr >= (uint32_t)NS) {
          if (!mbar_wait_bounded(&empty_bar[s], ((ctr / NS) - 1) & 1)) {
            if (lane == 0) set_err(st, ERR_TIMEOUT, 10 + OP);
            failed = true;
            break;
          }
        }
        if (lane == 0) mbar_arrive_expect_tx(&full_bar[s], brow * tr * NW);
        __syncwarp();
        for (int idx = lane; idx < tr * NW; idx += 32) {
          const int wi = idx / tr, ri = idx % tr;
          const int row = rl + ri;
          const unsigned char* src;
          if (NW == 2) {
            src = (const unsigned char*)G.w[wi] + (size_t)row * G.cols * ESZ;
          } else {
            const int sg = row < G.seg1 ? 0 : (row < G.seg2 ? 1 : 2);
            const int off = sg == 0 ? 0 : (sg == 1 ? G.seg1 : G.seg2);
            src = (const unsigned char*)G.w[sg] + (size_t)(row - off) * G.cols * ESZ;
          }
          bulk_g2s(ring + (size_t)s * slot + (size_t)(wi * TR + ri) * brow, src + (size_t)c0 * ESZ,
                   brow, &full_bar[s], pol);
        }
        ++ctr;
      }
      r += tr;
    }
    // on failure, wait (bounded) for copies already in flight before leaving
    if (failed && lane == 0) {
      const uint32_t first = ctr > (uint32_t)NS ? ctr - NS : 0;
      for (uint32_t c = first; c < ctr; ++c) mbar_wait_bounded(&full_bar[c % NS], (c / NS) & 1);
    }
    return;
  }

  // ------------------------------ consumer warps ------------------------------
  uint32_t ctr = 0;
  bool failed = false;
  int g = 0, last_g = -1, rb = 0;
  Top2 loc[2];
  top2_init(loc[0]);
  top2_init(loc[1]);
  const int V = p.D.V;
  for (int r = r_begin; r < r_end;) {
    while (r >= gg[g].row_begin + gg[g].rows) ++g;
    const GG& G = gg[g];
    const int rl = r - G.row_begin;
    const int tr = min(TR, min(r_end - r, G.rows - rl));
    const int nv = G.nv;
    if (g != last_g) {
      if (G.normw) {
        for (int v = warp; v < nv; v += NCW) {
          const float* xr = G.x + (size_t)((G.xrow0 + v) % G.xring) * G.xstride;
          float s = 0.f;
          for (int c = lane * 4; c < G.cols; c += 128) {
            const float4 q = *reinterpret_cast<const float4*>(xr + c);
            s += q.x * q.x; s += q.y * q.y; s += q.z * q.z; s += q.w * q.w;
          }
          s = warp_sum(s);
          if (lane == 0) rstd_s[v] = 1.0f / sqrtf(s / (float)G.cols + p.eps);
        }
      }
      named_bar(1, NCT);
      last_g = g;
    }
    const int cw = chunk_cols(G.cols, NW, ESZ);
    bool first_chunk = true;
    for (int c0 = 0; c0 < G.cols; c0 += cw) {
      const int w = min(cw, G.cols - c0);
      const int brow = w * ESZ;
      const int nvec = w / VEC;
      const int s = ctr % NS;
      // a warp that gives up keeps walking the same loop (no waits, no loads, no stores) so
      // that every named barrier still sees all consumer warps
      if (!failed && !mbar_wait_bounded(&full_bar[s], (ctr / NS) & 1)) {
        if (lane == 0) set_err(st, ERR_TIMEOUT, 20 + OP);
        failed = true;
      }
      const unsigned char* sb = ring + (size_t)s * slot;
      for (int vb = 0; vb < nv; vb += NVB) {
        float acc[TR][NW][NVB];
#pragma unroll
        for (int i = 0; i < TR; ++i)
#pragma unroll
          for (int j = 0; j < NW; ++j)
#pragma unroll
            for (int v = 0; v < NVB; ++v) acc[i][j][v] = 0.f;
        for (int k = tid; k < (failed ? 0 : nvec); k += NCT) {
          const int col = c0 + k * VEC;
          float xv[NVB][VEC];
#pragma unroll
          for (int v = 0; v < NVB; ++v) {
            if (vb + v < nv) {
              const float* xr = G.x + (size_t)((G.xrow0 + vb + v) % G.xring) * G.xstride + col;
#pragma unroll
              for (int e = 0; e < VEC; e += 4) {
                const float4 q = *reinterpret_cast<const float4*>(xr + e);
                xv[v][e] = q.x; xv[v][e + 1] = q.y; xv[v][e + 2] = q.z; xv[v][e + 3] = q.w;
              }
              if (G.normw) {
                const float rs = rstd_s[vb + v];
#pragma unroll
                for (int e = 0; e < VEC; e += 4) {
                  const float4 nw4 = *reinterpret_cast<const float4*>(G.normw + col + e);
                  xv[v][e] = xv[v][e] * rs * nw4.x;
                  xv[v][e + 1] = xv[v][e + 1] * rs * nw4.y;
                  xv[v][e + 2] = xv[v][e + 2] * rs * nw4.z;
                  xv[v][e + 3] = xv[v][e + 3] * rs * nw4.w;
                }
              }
            } else {
#pragma unroll
              for (int e = 0; e < VEC; ++e) xv[v][e] = 0.f;
            }
          }
#pragma unroll
          for (int ri = 0; ri < TR; ++ri) {
            if (ri < tr) {
#pragma unroll
              for (int wi = 0; wi < NW; ++wi) {
                const uint4 q = *reinterpret_cast<const uint4*>(sb + (size_t)(wi * TR + ri) * brow + k * 16);
                float wf[VEC];
                WTraits<WT>::unpack(q, wf);
#pragma unroll
                for (int v = 0; v < NVB; ++v)
#pragma unroll
                  for (int e = 0; e < VEC; ++e) acc[ri][wi][v] = fmaf(wf[e], xv[v][e], acc[ri][wi][v]);
              }
            }
          }
        }
        // reduce across the 256 consumer threads: lanes (xor tree), then warps in order
#pragma unroll
        for (int i = 0; i < TR; ++i)
#pragma unroll
          for (int j = 0; j < NW; ++j)
#pragma unroll
            for (int v = 0; v < NVB; ++v) {
              const float sv = warp_sum(acc[i][j][v]);
              if (lane == 0) red[rb][warp][(i * NW + j) * NVB + v] = sv;
            }
        named_bar(1, NCT);
        for (int idx = tid; idx < NRED; idx += NCT) {
          float sv = 0.f;
#pragma unroll
          for (int w8 = 0; w8 < NCW; ++w8) sv += red[rb][w8][idx];
          const int v = idx % NVB, ij = idx / NVB;
          if (vb + v < nv) {
            float& tref = tot[ij * kGemvMaxNV + vb + v];
            tref = first_chunk ? sv : tref + sv;
          }
        }
        rb ^= 1;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[s]);
      ++ctr;
      first_chunk = false;
    }
    named_bar(1, NCT);
    // epilogue: one thread per (row, vector)
    for (int idx = tid; idx < (failed ? 0 : tr * nv); idx += NCT) {
      const int ri = idx / nv, v = idx % nv;
      const int row = rl + ri;
      const float y0 = tot[(ri * NW + 0) * kGemvMaxNV + v];
      if (OP == OP_HEAD) {
        top2_push(loc[G.kind], y0, row);
        if (p.debug_logits) p.B.logits[(size_t)G.kind * V + row] = y0;
      } else {
        float* yp = G.y + (size_t)((G.yrow0 + v) % G.yring) * G.ystride + row;
        if (OP == OP_GATEUP) {
          const float y1 = tot[(ri * NW + 1) * kGemvMaxNV + v];
          *yp = (y0 / (1.0f + expf(-y0))) * y1;
        } else if (OP == OP_O || OP == OP_DOWN) {
          const float hn = *yp + y0;
          *yp = hn;
          if (OP == OP_DOWN && G.anch) G.anch[(size_t)((G.arow0 + v) % G.aring) * G.astride + row] = hn;
        } else {
          *yp = y0;
        }
      }
    }
    r += tr;
  }
  if (OP == OP_HEAD) {
    named_bar(1, NCT);
    if (tid < 32) { hred[tid][0] = loc[0]; hred[tid][1] = loc[1]; }
    named_bar(1, NCT);
    if (tid == 0) {
      float* hp = p.B.head_part + (size_t)blockIdx.x * 8;
      for (int k = 0; k < 2; ++k) {
        Top2 m = hred[0][k];
        for (int i = 1; i < 32; ++i) top2_merge(m, hred[i][k]);
        hp[k * 4 + 0] = m.v1; hp[k * 4 + 1] = __int_as_float(m.i1);
        hp[k * 4 + 2] = m.v2; hp[k * 4 + 3] = __int_as_float(m.i2);
      }
    }
  }
}

// ------------------------------------------------------------------------------------------------
// Single-vector engine (one input vector per group: the stage-diagonal step, plain AR, the heads,
// the stand-alone operator).  A stage holds 32 weight rows x 2 KB (a 1024-column bf16 chunk) in a
// 3-deep, 192 KB ring, one CTA per SM.  Each consumer warp owns whole rows of the tile (rows
// w, w+8, ...): lane l multiplies the chunk's 16-byte column vectors l, l+32, ... with its slice of
// the activation held in registers and reused over the warp's rows, partial sums stay in registers
// across chunks, and a row ends with one xor-tree warp reduction.  No block-wide barrier is taken
// while streaming, so the copy engine is the only thing the consumers wait for.  A row's result
// depends only on the column count, not on the tile, the warp or the other groups of the launch.
// ------------------------------------------------------------------------------------------------
constexpr int k1Rows = 32;          // physical weight rows per stage
constexpr int k1ChunkBytes = 2048;  // bytes of each row per stage
constexpr int k1Stages = 3;
constexpr int k1Ring = k1Stages * k1Rows * k1ChunkBytes;

template <int OP, typename WT>
__global__ void __launch_bounds__(kGemvThreads, 1)
gemv1_kernel(const __grid_constant__ GemvParams p) {
  extern __shared__ __align__(128) unsigned char ring[];
  constexpr int NW = (OP == OP_GATEUP) ? 2 : 1;
  constexpr int VEC = WTraits<WT>::kVec;
  constexpr int ESZ = sizeof(WT);
  constexpr int TR = k1Rows / NW;             // output rows per tile
  constexpr int RPW = TR / 8;                 // output rows per consumer warp
  constexpr int CW = k1ChunkBytes / ESZ;      // columns per chunk
  constexpr int VPL = CW / VEC / 32;          // column vectors per lane per chunk
  constexpr int STAGE = k1Rows * k1ChunkBytes;
  constexpr int NCW = kGemvConsumerWarps;

  __shared__ GG gg[kMaxGroups];
  __shared__ int s_ng, s_total;
  __shared__ __align__(8) uint64_t full_bar[k1Stages];
  __shared__ __align__(8) uint64_t empty_bar[k1Stages];
  __shared__ Top2 hred[NCW][2];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  DevState* st = p.B.st;
  if (tid == 0) {
    const bool skip = !p.explicit_mode && (st->done || st->err);
    const int ng = skip ? 0 : resolve_groups(p, gg);
    int total = 0;
    for (int i = 0; i < ng; ++i) {
      gg[i].row_begin = total;
      total += gg[i].rows;
    }
    s_ng = ng; s_total = total;
    for (int i = 0; i < k1Stages; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], NCW);
    }
    fence_mbar_init();
  }
  __syncthreads();
  const int ng = s_ng;
  if (ng == 0) {
    if (OP == OP_HEAD && tid == 0) {
      float* hp = p.B.head_part + (size_t)blockIdx.x * 8;
      for (int k = 0; k < 2; ++k) {
        hp[k * 4 + 0] = -INFINITY; hp[k * 4 + 1] = __int_as_float(0x7fffffff);
        hp[k * 4 + 2] = -INFINITY; hp[k * 4 + 3] = __int_as_float(0x7fffffff);
      }
    }
    return;
  }
  const long long total = s_total;
  const int r_begin = (int)(total * blockIdx.x / gridDim.x);
  const int r_end = (int)(total * (blockIdx.x + 1) / gridDim.x);

  if (warp == NCW) {
    // ------------------------------ producer warp ------------------------------
    const uint64_t pol = l2_evict_first_policy();
    uint32_t ctr = 0;
    bool failed = false;
    int g = 0;
    for (int r = r_begin; r < r_end && !failed;) {
      while (r >= gg[g].row_begin + gg[g].rows) ++g;
      const GG& G = gg[g];
      const int rl = r - G.row_begin;
      const int tr = min(TR, min(r_end - r, G.rows - rl));
      for (int c0 = 0; c0 < G.cols; c0 += CW) {
        const uint32_t brow = (uint32_t)min(CW, G.cols - c0) * ESZ;
        const int s = ctr % k1Stages;
        if (ctr >= (uint32_t)k1Stages &&
            !mbar_wait_bounded(&empty_bar[s], ((ctr / k1Stages) - 1) & 1)) {
          if (lane == 0) set_err(st, ERR_TIMEOUT, 40 + OP);
          failed = true;
          break;
        }
        if (lane == 0) mbar_arrive_expect_tx(&full_bar[s], brow * tr * NW);
        __syncwarp();
        if (lane < tr * NW) {
          const int wi = lane / tr, ri = lane % tr;
          const int row = rl + ri;
          const unsigned char* src;
          if (NW == 2) {
            src = (const unsigned char*)G.w[wi] + (size_t)row * G.cols * ESZ;
          } else {
            const int sg = row < G.seg1 ? 0 : (row < G.seg2 ? 1 : 2);
            const int off = sg == 0 ? 0 : (sg == 1 ? G.seg1 : G.seg2);
            src = (const unsigned char*)G.w[sg] + (size_t)(row - off) * G.cols * ESZ;
          }
          bulk_g2s(ring + (size_t)s * STAGE + (size_t)(wi * TR + ri) * k1ChunkBytes,
                   src + (size_t)c0 * ESZ, brow, &full_bar[s], pol);
        }
        ++ctr;
      }
      r += tr;
    }
    if (failed && lane == 0) {
      const uint32_t first = ctr > (uint32_t)k1Stages ? ctr - k1Stages : 0;
      for (uint32_t c = first; c < ctr; ++c) mbar_wait_bounded(&full_bar[c % k1Stages], (c / k1Stages) & 1);
    }
    return;
  }

  // ------------------------------ consumer warps ------------------------------
  uint32_t ctr = 0;
  bool failed = false;
  int g = 0, last_g = -1;
  float rstd = 1.f;
  Top2 loc[2];
  top2_init(loc[0]);
  top2_init(loc[1]);
  const int V = p.D.V;
  for (int r = r_begin; r < r_end;) {
    while (r >= gg[g].row_begin + gg[g].rows) ++g;
    const GG& G = gg[g];
    const int rl = r - G.row_begin;
    const int tr = min(TR, min(r_end - r, G.rows - rl));
    const float* xr = G.x + (size_t)(G.xrow0 % G.xring) * G.xstride;
    if (g != last_g) {
      if (G.normw) {  // every warp forms the same rstd in the same order
        float sq = 0.f;
        for (int c = lane * 4; c < G.cols; c += 128) {
          const float4 q = *reinterpret_cast<const float4*>(xr + c);
          sq += q.x * q.x; sq += q.y * q.y; sq += q.z * q.z; sq += q.w * q.w;
        }
        sq = warp_sum(sq);
        rstd = 1.0f / sqrtf(sq / (float)G.cols + p.eps);
      }
      last_g = g;
    }
    float acc[RPW][NW];
#pragma unroll
    for (int i = 0; i < RPW; ++i)
#pragma unroll
      for (int j = 0; j < NW; ++j) acc[i][j] = 0.f;
    for (int c0 = 0; c0 < G.cols; c0 += CW) {
      const int nvec = min(CW, G.cols - c0) / VEC;
      const int s = ctr % k1Stages;
      if (!failed && !mbar_wait_bounded(&full_bar[s], (ctr / k1Stages) & 1)) {
        if (lane == 0) set_err(st, ERR_TIMEOUT, 50 + OP);
        failed = true;
      }
      if (!failed) {
        const unsigned char* sb = ring + (size_t)s * STAGE;
        float xv[VPL][VEC];
#pragma unroll
        for (int j = 0; j < VPL; ++j) {
          const int k = lane + 32 * j;
          if (k < nvec) {
            const int col = c0 + k * VEC;
#pragma unroll
            for (int e = 0; e < VEC; e += 4) {
              const float4 q = *reinterpret_cast<const float4*>(xr + col + e);
              xv[j][e] = q.x; xv[j][e + 1] = q.y; xv[j][e + 2] = q.z; xv[j][e + 3] = q.w;
            }
            if (G.normw) {
#pragma unroll
              for (int e = 0; e < VEC; e += 4) {
                const float4 nw4 = *reinterpret_cast<const float4*>(G.normw + col + e);
                xv[j][e] = xv[j][e] * rstd * nw4.x;
                xv[j][e + 1] = xv[j][e + 1] * rstd * nw4.y;
                xv[j][e + 2] = xv[j][e + 2] * rstd * nw4.z;
                xv[j][e + 3] = xv[j][e + 3] * rstd * nw4.w;
              }
            }
          }
        }
#pragma unroll
        for (int i = 0; i < RPW; ++i) {
          const int ri = warp + NCW * i;
          if (ri < tr) {
#pragma unroll
            for (int wi = 0; wi < NW; ++wi) {
              const unsigned char* rowp = sb + (size_t)(wi * TR + ri) * k1ChunkBytes;
#pragma unroll
              for (int j = 0; j < VPL; ++j) {
                const int k = lane + 32 * j;
                if (k < nvec) {
                  const uint4 q = *reinterpret_cast<const uint4*>(rowp + k * 16);
                  float wf[VEC];
                  WTraits<WT>::unpack(q, wf);
#pragma unroll
                  for (int e = 0; e < VEC; ++e) acc[i][wi] = fmaf(wf[e], xv[j][e], acc[i][wi]);
                }
              }
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[s]);
      ++ctr;
    }
    // epilogue: one warp reduction per row
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
      const int ri = warp + NCW * i;
      if (ri < tr) {
        float y[NW];
#pragma unroll
        for (int wi = 0; wi < NW; ++wi) y[wi] = warp_sum(acc[i][wi]);
        if (lane == 0 && !failed) {
          const int row = rl + ri;
          if (OP == OP_HEAD) {
            top2_push(loc[G.kind], y[0], row);
            if (p.debug_logits) p.B.logits[(size_t)G.kind * V + row] = y[0];
          } else {
            float* yp = G.y + (size_t)(G.yrow0 % G.yring) * G.ystride + row;
            if (OP == OP_GATEUP) {
              *yp = (y[0] / (1.0f + expf(-y[0]))) * y[NW - 1];
            } else if (OP == OP_O || OP == OP_DOWN) {
              const float hn = *yp + y[0];
              *yp = hn;
              if (OP == OP_DOWN && G.anch) G.anch[(size_t)(G.arow0 % G.aring) * G.astride + row] = hn;
            } else {
              *yp = y[0];
            }
          }
        }
      }
    }
    r += tr;
  }
  if (OP == OP_HEAD) {
    if (lane == 0) { hred[warp][0] = loc[0]; hred[warp][1] = loc[1]; }
    named_bar(1, NCW * 32);
    if (tid == 0) {
      float* hp = p.B.head_part + (size_t)blockIdx.x * 8;
      for (int k = 0; k < 2; ++k) {
        Top2 m = hred[0][k];
        for (int i = 1; i < NCW; ++i) top2_merge(m, hred[i][k]);
        hp[k * 4 + 0] = m.v1; hp[k * 4 + 1] = __int_as_float(m.i1);
        hp[k * 4 + 2] = m.v2; hp[k * 4 + 3] = __int_as_float(m.i2);
      }
    }
  }
}

template <int OP, typename WT>
int grid1_of() {
  static int grid = 0;
  if (grid == 0) {
    int occ = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, gemv1_kernel<OP, WT>, kGemvThreads, k1Ring);
    grid = num_sms() * (occ > 0 ? occ : 1);
  }
  return grid;
}

template <int OP, typename WT>
cudaError_t launch1(const GemvParams& p, int grid, cudaStream_t s) {
  if (grid <= 0) grid = grid1_of<OP, WT>();
  gemv1_kernel<OP, WT><<<grid, kGemvThreads, k1Ring, s>>>(p);
  return cudaGetLastError();
}

// ------------------------------------------------------------------------------------------------
// Multi-vector engine on tensor cores (bf16 weights; draft-module rows and prefill blocks, where
// up to 64 input vectors share each weight row).  y[row][v] = W[row,:] . x_v is a skinny dense
// contraction, done with mma.sync m16n8k16 (bf16 x bf16 -> fp32): the weight tile is the A operand
// (16 rows, loaded with ldmatrix from shared memory rows padded by 16 bytes so the 8 row addresses
// of a matrix fall in distinct banks), the vectors are the B operand.  The fp32 activations are
// split as x = hi + lo with hi = bf16(x), lo = bf16(x - hi), and both halves are multiplied into
// the same fp32 accumulator, which keeps about 17 significant bits of every activation.
// A tile is 16 output rows (x2 weights for gate/up); a stage carries 1536 columns of them; the 8
// consumer warps take interleaved 16-column k-steps and their partial sums are added in warp order
// once per tile.
// ------------------------------------------------------------------------------------------------
constexpr int kMColsNW = 1536;                 // columns x weights per stage
constexpr int kMStages = 3;
constexpr int kMPitchPad = 16;                 // bytes of padding per shared-memory row
constexpr int kMMaxNT = 8;                     // n-tiles of 8 vectors (64 vectors)
constexpr int kMStageBytes = 16 * (kMColsNW * 2 + 2 * kMPitchPad);
constexpr int kMRing = kMStages * kMStageBytes;

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

template <int OP, int NT>
__global__ void __launch_bounds__(kGemvThreads, 1)
gemvmma_kernel(const __grid_constant__ GemvParams p) {
  extern __shared__ __align__(128) unsigned char ring[];
  constexpr int NW = (OP == OP_GATEUP) ? 2 : 1;
  constexpr int CW = kMColsNW / NW;                  // columns per stage
  constexpr int PITCH = CW * 2 + kMPitchPad;         // bytes per shared-memory row
  constexpr int NCW = kGemvConsumerWarps;
  constexpr int NRED = NW * NT * 4;                  // accumulator floats per thread

  __shared__ GG gg[kMaxGroups];
  __shared__ int s_ng, s_total;
  __shared__ __align__(8) uint64_t full_bar[kMStages];
  __shared__ __align__(8) uint64_t empty_bar[kMStages];
  __shared__ float rstd_s[kGemvMaxNV];
  __shared__ float red[NCW][NRED][32];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  DevState* st = p.B.st;
  if (tid == 0) {
    const bool skip = st->done || st->err;
    const int ng = skip ? 0 : resolve_groups(p, gg);
    int total = 0;
    for (int i = 0; i < ng; ++i) {
      gg[i].row_begin = total;
      total += gg[i].rows;
    }
    s_ng = ng; s_total = total;
    for (int i = 0; i < kMStages; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], NCW);
    }
    fence_mbar_init();
  }
  __syncthreads();
  if (s_ng == 0) return;
  // spans of whole 16-row tiles
  const long long tiles = (s_total + 15) / 16;
  const int r_begin = (int)(tiles * blockIdx.x / gridDim.x) * 16;
  const int r_end = min(s_total, (int)(tiles * (blockIdx.x + 1) / gridDim.x) * 16);

  if (warp == NCW) {
    const uint64_t pol = l2_evict_first_policy();
    uint32_t ctr = 0;
    bool failed = false;
    int g = 0;
    for (int r = r_begin; r < r_end && !failed;) {
      while (r >= gg[g].row_begin + gg[g].rows) ++g;
      const GG& G = gg[g];
      const int rl = r - G.row_begin;
      const int tr = min(16, min(r_end - r, G.rows - rl));
      for (int c0 = 0; c0 < G.cols; c0 += CW) {
        const uint32_t brow = (uint32_t)min(CW, G.cols - c0) * 2;
        const int s = ctr % kMStages;
        if (ctr >= (uint32_t)kMStages &&
            !mbar_wait_bounded(&empty_bar[s], ((ctr / kMStages) - 1) & 1)) {
          if (lane == 0) set_err(st, ERR_TIMEOUT, 60 + OP);
          failed = true;
          break;
        }
        if (lane == 0) mbar_arrive_expect_tx(&full_bar[s], brow * tr * NW);
        __syncwarp();
        if (lane < tr * NW) {
          const int wi = lane / tr, ri = lane % tr;
          const int row = rl + ri;
          const unsigned char* src;
          if (NW == 2) {
            src = (const unsigned char*)G.w[wi] + (size_t)row * G.cols * 2;
          } else {
            const int sg = row < G.seg1 ? 0 : (row < G.seg2 ? 1 : 2);
            const int off = sg == 0 ? 0 : (sg == 1 ? G.seg1 : G.seg2);
            src = (const unsigned char*)G.w[sg] + (size_t)(row - off) * G.cols * 2;
          }
          bulk_g2s(ring + (size_t)s * kMStageBytes + (size_t)(wi * 16 + ri) * PITCH,
                   src + (size_t)c0 * 2, brow, &full_bar[s], pol);
        }
        ++ctr;
      }
      r += tr;
    }
    if (failed && lane == 0) {
      const uint32_t first = ctr > (uint32_t)kMStages ? ctr - kMStages : 0;
      for (uint32_t c = first; c < ctr; ++c) mbar_wait_bounded(&full_bar[c % kMStages], (c / kMStages) & 1);
    }
    return;
  }

  // ------------------------------ consumer warps ------------------------------
  const int gq = lane >> 2, tq = lane & 3;  // mma fragment coordinates
  // ldmatrix row address of this lane: matrix (lane/8): rows 0-7 / 8-15, k 0-7 / 8-15
  const int lm_row = (lane & 7) + 8 * ((lane >> 3) & 1);
  const int lm_k = 8 * (lane >> 4);
  uint32_t ctr = 0;
  bool failed = false;
  int g = 0, last_g = -1;
  for (int r = r_begin; r < r_end;) {
    while (r >= gg[g].row_begin + gg[g].rows) ++g;
    const GG& G = gg[g];
    const int rl = r - G.row_begin;
    const int tr = min(16, min(r_end - r, G.rows - rl));
    const int nv = G.nv;
    if (g != last_g) {
      if (G.normw) {
        for (int v = warp; v < nv; v += NCW) {
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
      named_bar(1, NCW * 32);
      last_g = g;
    }
    // this lane's B rows: vector n = nt*8 + gq
    const float* xrow[NT];
    float rsv[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int v = nt * 8 + gq;
      xrow[nt] = v < nv ? G.x + (size_t)((G.xrow0 + v) % G.xring) * G.xstride : nullptr;
      rsv[nt] = (v < nv && G.normw) ? rstd_s[v] : 1.f;
    }
    float acc[NW][NT][4];
#pragma unroll
    for (int i = 0; i < NW; ++i)
#pragma unroll
      for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[i][j][e] = 0.f;
    for (int c0 = 0; c0 < G.cols; c0 += CW) {
      const int ksteps = min(CW, G.cols - c0) / 16;
      const int s = ctr % kMStages;
      if (!failed && !mbar_wait_bounded(&full_bar[s], (ctr / kMStages) & 1)) {
        if (lane == 0) set_err(st, ERR_TIMEOUT, 70 + OP);
        failed = true;
      }
      if (!failed) {
        const uint32_t sb = smem_u32(ring + (size_t)s * kMStageBytes);
        for (int ks = warp; ks < ksteps; ks += NCW) {
          const int col = c0 + ks * 16;
          uint32_t a[NW][4];
#pragma unroll
          for (int wi = 0; wi < NW; ++wi)
            ldmatrix_x4(sb + (uint32_t)((wi * 16 + lm_row) * PITCH + (ks * 16 + lm_k) * 2), a[wi][0],
                        a[wi][1], a[wi][2], a[wi][3]);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
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
            for (int wi = 0; wi < NW; ++wi) {
              mma_bf16(acc[wi][nt], a[wi], bh0, bh1);
              mma_bf16(acc[wi][nt], a[wi], bl0, bl1);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[s]);
      ++ctr;
    }
    // add the 8 warps' partial tiles in warp order, then the epilogue
#pragma unroll
    for (int i = 0; i < NW; ++i)
#pragma unroll
      for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) red[warp][(i * NT + j) * 4 + e][lane] = acc[i][j][e];
    named_bar(1, NCW * 32);
    for (int idx = tid; idx < 16 * nv; idx += NCW * 32) {
      const int m = idx / nv, v = idx % nv;
      if (m >= tr || failed) continue;
      const int nt = v / 8, nn = v % 8;
      const int ln = (m % 8) * 4 + nn / 2;
      const int e = (m >= 8 ? 2 : 0) + (nn & 1);
      float y[NW];
#pragma unroll
      for (int wi = 0; wi < NW; ++wi) {
        float sum = 0.f;
#pragma unroll
        for (int w8 = 0; w8 < NCW; ++w8) sum += red[w8][(wi * NT + nt) * 4 + e][ln];
        y[wi] = sum;
      }
      const int row = rl + m;
      float* yp = G.y + (size_t)((G.yrow0 + v) % G.yring) * G.ystride + row;
      if (OP == OP_GATEUP) {
        *yp = (y[0] / (1.0f + expf(-y[0]))) * y[NW - 1];
      } else if (OP == OP_O || OP == OP_DOWN) {
        const float hn = *yp + y[0];
        *yp = hn;
        if (OP == OP_DOWN && G.anch) G.anch[(size_t)((G.arow0 + v) % G.aring) * G.astride + row] = hn;
      } else {
        *yp = y[0];
      }
    }
    named_bar(1, NCW * 32);  // `red` is rewritten by the next tile
    r += tr;
  }
}

template <int OP, int NT>
int gridm_of() {
  static int grid = 0;
  if (grid == 0) {
    int occ = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, gemvmma_kernel<OP, NT>, kGemvThreads, kMRing);
    grid = num_sms() * (occ > 0 ? occ : 1);
  }
  return grid;
}

template <int OP, int NT>
cudaError_t launchm_nt(const GemvParams& p, cudaStream_t s) {
  gemvmma_kernel<OP, NT><<<gridm_of<OP, NT>(), kGemvThreads, kMRing, s>>>(p);
  return cudaGetLastError();
}

// n-tiles needed for the largest vector count of the launch: 1 (<= 8), 2 (<= 16), 3 (<= 24), 4 (<= 32)
template <int OP>
cudaError_t launchm(const GemvParams& p, int max_nv, cudaStream_t s) {
  if (max_nv <= 8) return launchm_nt<OP, 1>(p, s);
  if (max_nv <= 16) return launchm_nt<OP, 2>(p, s);
  if (max_nv <= 24) return launchm_nt<OP, 3>(p, s);
  return launchm_nt<OP, 4>(p, s);
}

// persistent grid: every SM holds as many CTAs as fit (registers, shared memory)
template <int OP, typename WT, int NVB>
int grid_of() {
  static int grid = 0;
  if (grid == 0) {
    int occ = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, gemv_kernel<OP, WT, NVB>, kGemvThreads, kRing);
    grid = num_sms() * (occ > 0 ? occ : 1);
  }
  return grid;
}

template <int OP, typename WT, int NVB>
cudaError_t launch_one(const GemvParams& p, int grid, cudaStream_t s) {
  if (grid <= 0) grid = grid_of<OP, WT, NVB>();
  gemv_kernel<OP, WT, NVB><<<grid, kGemvThreads, kRing, s>>>(p);
  return cudaGetLastError();
}

template <int OP, typename WT>
cudaError_t launch_nv(const GemvParams& p, int grid, bool multi, cudaStream_t s) {
  if (!multi) return launch1<OP, WT>(p, grid, s);
  if (sizeof(WT) == 2 && p.mma_ok) return launchm<OP>(p, p.max_nv, s);
  return launch_one<OP, WT, 4>(p, grid, s);
}

template <typename WT>
cudaError_t launch_op(const GemvParams& p, int grid, bool multi, cudaStream_t s) {
  switch (p.op) {
    case OP_QKV: return launch_nv<OP_QKV, WT>(p, grid, multi, s);
    case OP_O: return launch_nv<OP_O, WT>(p, grid, multi, s);
    case OP_GATEUP: return launch_nv<OP_GATEUP, WT>(p, grid, multi, s);
    case OP_DOWN: return launch_nv<OP_DOWN, WT>(p, grid, multi, s);
    case OP_FC: return launch_nv<OP_FC, WT>(p, grid, multi, s);
    default: return launch1<OP_HEAD, WT>(p, grid, s);
  }
}

template <int OP, typename WT, int NVB>
cudaError_t set_attr_one() {
  return cudaFuncSetAttribute(gemv_kernel<OP, WT, NVB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kRing);
}
template <int OP, typename WT>
cudaError_t set_attr1() {
  return cudaFuncSetAttribute(gemv1_kernel<OP, WT>, cudaFuncAttributeMaxDynamicSharedMemorySize, k1Ring);
}
template <int OP>
cudaError_t set_attrm() {
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(gemvmma_kernel<OP, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMRing)))
    return e;
  if ((e = cudaFuncSetAttribute(gemvmma_kernel<OP, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMRing)))
    return e;
  if ((e = cudaFuncSetAttribute(gemvmma_kernel<OP, 3>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMRing)))
    return e;
  return cudaFuncSetAttribute(gemvmma_kernel<OP, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMRing);
}

template <typename WT>
cudaError_t set_attr_wt() {
  cudaError_t e = cudaSuccess;
  if (sizeof(WT) == 2) {
    if ((e = set_attrm<OP_QKV>()) || (e = set_attrm<OP_O>()) || (e = set_attrm<OP_GATEUP>()) ||
        (e = set_attrm<OP_DOWN>()) || (e = set_attrm<OP_FC>()))
      return e;
  }
#define SPD_A(op)                                              \
  if ((e = set_attr1<op, WT>()) != cudaSuccess) return e; \
  if ((e = set_attr_one<op, WT, 4>()) != cudaSuccess) return e;
  SPD_A(OP_QKV) SPD_A(OP_O) SPD_A(OP_GATEUP) SPD_A(OP_DOWN) SPD_A(OP_FC)
#undef SPD_A
  return set_attr1<OP_HEAD, WT>();
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
  return dtype == SPD_DTYPE_BF16 ? grid1_of<OP_HEAD, __nv_bfloat16>() : grid1_of<OP_HEAD, float>();
}

cudaError_t gemv_setup_attributes() {
  cudaError_t e = set_attr_wt<float>();
  if (e != cudaSuccess) return e;
  return set_attr_wt<__nv_bfloat16>();
}

cudaError_t launch_gemv(int op, const Dims& D, const Bufs& B, const Launch& lc,
                        const LaunchCfg& cfg, cudaStream_t s) {
  GemvParams p;
  memset(&p, 0, sizeof(p));
  p.op = op; p.explicit_mode = 0; p.debug_logits = cfg.debug_logits; p.eps = D.eps;
  p.D = D; p.B = B; p.lc = lc;
  const bool multi = (lc.kind == LK_PDMROWS || lc.kind == LK_ROWS) && op != OP_HEAD;
  p.max_nv = lc.kind == LK_PDMROWS ? D.n + 1 : (lc.kind == LK_ROWS ? lc.cnt : 1);
  p.mma_ok = D.dtype == SPD_DTYPE_BF16 && D.d % 16 == 0 && D.ffn % 16 == 0 && (D.hq * D.hd) % 16 == 0 &&
             p.max_nv <= 32;
  const int grid = op == OP_HEAD ? B.head_grid : 0;  // 0: the instantiation's persistent grid
  return D.dtype == SPD_DTYPE_BF16 ? launch_op<__nv_bfloat16>(p, grid, multi, s)
                                   : launch_op<float>(p, grid, multi, s);
}

cudaError_t launch_gemv_explicit(const GemvExplicit& ge, int dtype, float eps, int grid,
                                 cudaStream_t s) {
  GemvParams p;
  memset(&p, 0, sizeof(p));
  p.op = OP_QKV; p.explicit_mode = 1; p.eps = eps; p.ge = ge;
  (void)grid;
  return dtype == SPD_DTYPE_BF16 ? launch1<OP_QKV, __nv_bfloat16>(p, 0, s)
                                 : launch1<OP_QKV, float>(p, 0, s);
}

}  // namespace spd
