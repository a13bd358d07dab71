// Decode attention over per-layer KV caches: device code shared by the stand-alone attention
// kernel (prefill blocks, stand-alone operators; chunks of 128 keys) and the persistent step
// kernel (chunks of 64 keys).
//
// The query rows arrive already rotated (RoPE is applied in the QKV epilogue of the GEMV engine,
// which also appends k and v to the cache).  Work item = (query tile, kv head, key chunk).  A tile
// holds up to 8 query rows of one layer (1 row per token in the stage-diagonal step and in plain
// AR); all query heads of the grouped-query group share the K/V chunk, which is bulk-copied into
// shared memory once.  Scores use 16-dim lane slices reduced with xor shuffles, softmax is per
// chunk (max, exp, sum), and the chunk partial (o, m, l) goes to global scratch.  The last item of
// a (tile, kv head) to finish (atomic ticket, no spinning) merges the partials of each query in
// chunk order.  The number of chunks depends only on the query position, so a token's result does
// not depend on its batch.
#pragma once
#include "spd_internal.cuh"

namespace spd {
namespace att {

constexpr int kThreads = 256;   // threads taking part (named barrier 2)

struct Tile {
  int layer, nq, pos0, vid0, nch, rec_off, item_off, tick_off;
  int kn0;                   // first key the QKV step of this cycle appends for the tile's row group
  int co, old_off, new_off;  // step kernel: chunks written before this cycle; item offsets of the
                             // tile in the lists of such chunks and of the chunks holding new keys
  const unsigned char* kc;  // base of this layer's K cache (head 0, position 1)
  const unsigned char* vc;
  const float* q;           // query rows [row][qkv_rows] (rotated q at the front)
  float* out;               // attention output rows [row][hq*hd]
  float* part;              // chunk partials of this tile's launch part
  int* tick;                // merge tickets of this tile's launch part
};

// Appends the tiles of one part (a launch descriptor; rows of up to `qt` queries per tile).
static __device__ int add_tiles(const Dims& D, const Bufs& B, const Launch& lc, int qt, int ck, Tile* tiles,
                         int nt, int* items, int cap, const DevState* sv) {
  DevState* st = B.st;
  RowGroup rg[kMaxGroups];
  int nr;
  if (lc.kind == LK_EXPLICIT) {
    // caller-given positions: a row outside 1..max_seq would read keys and write partials past the
    // cache and the scratch; it gets no tile, and its output row is filled with NaN so that the
    // caller sees it (every CTA writes the same value)
    nr = 0;
    for (int r = 0; r < lc.cnt && r < kMaxGroups; ++r) {
      const int p = lc.act.pos_arr[r];
      if (p < 1 || p > D.max_seq) {
        float* o = lc.act.attn + (size_t)r * D.hq * D.hd;
        for (int i = 0; i < D.hq * D.hd; ++i) o[i] = __int_as_float(0x7fc00000);
        continue;
      }
      rg[nr].layer = 0; rg[nr].nv = 1; rg[nr].pos0 = p; rg[nr].vid0 = r; rg[nr].rrow0 = 0;
      ++nr;
    }
  } else {
    nr = build_rows(lc, D, sv, st, rg);
  }
  const int esz = D.dtype == SPD_DTYPE_BF16 ? 2 : 4;
  const size_t layer_elems = (size_t)D.hkv * D.max_seq * D.hd;
  int rec = 0, local = 0;
  for (int i = 0; i < nr; ++i) {
    for (int r0 = 0; r0 < rg[i].nv; r0 += qt) {
      if (nt >= cap) { set_err(st, ERR_BOUNDS, 400); return -1; }
      Tile& T = tiles[nt++];
      T.layer = rg[i].layer;
      T.nq = min(qt, rg[i].nv - r0);
      T.pos0 = rg[i].pos0 + r0;
      T.vid0 = rg[i].vid0 + r0;
      // every row of the group appends its key in this cycle's QKV step (one row group per layer),
      // so a tile after the group's first rows also reads keys from rows before its own
      T.kn0 = rg[i].pos0 - 1;
      const int pos_last = T.pos0 + T.nq - 1;
      T.nch = (pos_last + ck - 1) / ck;
      T.rec_off = rec;
      T.item_off = *items;
      T.tick_off = local * D.hkv;
      rec += D.hkv * T.nch * T.nq * D.gq;
      *items += D.hkv * T.nch;
      ++local;
      const void* kb;
      const void* vb;
      if (lc.kind == LK_EXPLICIT) { kb = lc.act.kc; vb = lc.act.vc; }
      else if (lc.stack == 0) { kb = B.kc; vb = B.vc; }
      else { kb = B.pkc; vb = B.pvc; }
      T.kc = (const unsigned char*)kb + (size_t)T.layer * layer_elems * esz;
      T.vc = (const unsigned char*)vb + (size_t)T.layer * layer_elems * esz;
      T.q = lc.act.qkv; T.out = lc.act.attn; T.part = lc.act.part; T.tick = lc.act.tick;
    }
  }
  return nt;
}

// Bytes of shared memory the item loop needs for chunks of `ck` keys and tiles of up to qt rows.
__host__ __device__ inline size_t smem_bytes(int hd, int gq, int esz, int qt, int ck) {
  const int qh = qt * gq;
  return (size_t)2 * ck * hd * esz + (size_t)qh * hd * 4 + (size_t)qh * ck * 4 + (size_t)2 * qh * 4;
}

// Geometry of work item `item`: tile T, kv head kh, key chunk c of `ck` keys (nk of them).
struct Item {
  int T, kh, c, nk;
};
__device__ __forceinline__ Item item_of(const Tile* tiles, int nt, int item, int ck) {
  Item it;
  it.T = 0;
  while (it.T + 1 < nt && tiles[it.T + 1].item_off <= item) ++it.T;
  const Tile& Ti = tiles[it.T];
  const int rem = item - Ti.item_off;
  it.kh = rem / Ti.nch;
  it.c = rem % Ti.nch;
  const int pos_last = Ti.pos0 + Ti.nq - 1;
  it.nk = min(ck, pos_last - it.c * ck);
  return it;
}

// One item on the 256 calling threads, its K and V chunks already in shared memory (ks, vs:
// [nk][hd] in the cache dtype): queries -> qs, scores, per-chunk softmax, unnormalised partial
// (o, m, l) to global scratch, and -- for the last item of its (tile, kv head) to finish, by an
// atomic ticket -- the merge of the partials in chunk order.  Named barrier 2.
template <typename WT, int CK>
__device__ void item_compute(const Dims& D, const Tile& Ti, const Item& it, const WT* ks, const WT* vs, float* qs,
                             float* sc, float* m_s, float* l_s, int* last_flag) {
  const int hd = D.hd, GQ = D.gq;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const float scale = 1.0f / sqrtf((float)hd);
  const int qkv_rows = D.qkv_rows;
  const int hqd = D.hq * hd;
  const int LPK = hd / 16;  // lanes per key
  const int KPW = 32 / LPK;
  const int kh = it.kh, c = it.c, nk = it.nk;
  const int QH = Ti.nq * GQ;
  const int key0 = c * CK;
  // queries (already rotated) -> shared memory
  for (int idx = tid; idx < QH * hd; idx += kThreads) {
    const int qh = idx / hd, e = idx % hd;
    const int r = qh / GQ, hg = qh % GQ;
    qs[idx] = Ti.q[(size_t)(Ti.vid0 + r) * qkv_rows + (kh * GQ + hg) * hd + e];
  }
  named_bar(2, kThreads);
  // scores
  {
    const int kl = lane / LPK, sub = lane % LPK;
    for (int kb = warp * KPW; kb < CK; kb += 8 * KPW) {
      const int kk = kb + kl;
      float kf[16];
      if (kk < nk) {
        const WT* kr = ks + (size_t)kk * hd + sub * 16;
#pragma unroll
        for (int e = 0; e < 16; e += 16 / (int)sizeof(WT)) {
          const uint4 q4 = *reinterpret_cast<const uint4*>(kr + e);
          WTraits<WT>::unpack(q4, kf + e);
        }
      } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) kf[e] = 0.f;
      }
      for (int qh = 0; qh < QH; ++qh) {
        const float* qv = qs + (size_t)qh * hd + sub * 16;
        float dot = 0.f;
#pragma unroll
        for (int e = 0; e < 16; e += 4) {
          const float4 q4 = *reinterpret_cast<const float4*>(qv + e);
          dot = fmaf(kf[e], q4.x, dot);
          dot = fmaf(kf[e + 1], q4.y, dot);
          dot = fmaf(kf[e + 2], q4.z, dot);
          dot = fmaf(kf[e + 3], q4.w, dot);
        }
        for (int o = LPK / 2; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
        if (sub == 0 && kk < nk) {
          const int pos_q = Ti.pos0 + qh / GQ;
          sc[(size_t)qh * CK + kk] = (key0 + kk < pos_q) ? dot * scale : -INFINITY;
        }
      }
    }
  }
  named_bar(2, kThreads);
  // per-chunk softmax statistics, one warp per query head
  for (int qh = warp; qh < QH; qh += 8) {
    float* srow = sc + (size_t)qh * CK;
    float m = -INFINITY;
    for (int k = lane; k < nk; k += 32) m = fmaxf(m, srow[k]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float l = 0.f;
    for (int k = lane; k < nk; k += 32) {
      const float pk = (m == -INFINITY) ? 0.f : expf(srow[k] - m);
      srow[k] = pk;
      l += pk;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    if (lane == 0) { m_s[qh] = m; l_s[qh] = l; }
  }
  named_bar(2, kThreads);
  // unnormalised chunk output -> partial record (o[hd], m, l).  With at most 128 outputs the
  // keys are split between the two thread halves (lower half first, then added in that order).
  const int nout = QH * hd;
  const bool split = 2 * nout <= kThreads;
  float* oh = qs;  // the queries are dead once the scores exist: scratch for the upper half
  for (int idx = tid; idx < (split ? 2 * nout : nout); idx += kThreads) {
    const int half = split ? idx / nout : 0;
    const int o_i = split ? idx % nout : idx;
    const int qh = o_i / hd, e = o_i % hd;
    const float* prow = sc + (size_t)qh * CK;
    const int k0 = split ? (half ? nk / 2 : 0) : 0;
    const int k1 = split ? (half ? nk : nk / 2) : nk;
    float o = 0.f;
    for (int k = k0; k < k1; ++k) o = fmaf(prow[k], WTraits<WT>::to_f(vs[(size_t)k * hd + e]), o);
    if (split && half) oh[o_i] = o;
    if (split) named_bar(3, kThreads);  // every thread reaches it once (2 * nout <= kThreads)
    if (!(split && half)) {
      if (split) o += oh[o_i];
      float* rec = Ti.part + ((size_t)Ti.rec_off + ((size_t)kh * Ti.nch + c) * QH + qh) * (hd + 2);
      rec[e] = o;
      if (e == 0) { rec[hd] = m_s[qh]; rec[hd + 1] = l_s[qh]; }
    }
  }
  if (split && tid >= 2 * nout) named_bar(3, kThreads);  // threads without an output item
  __threadfence();
  named_bar(2, kThreads);
  if (tid == 0) {
    const int old = atomicAdd(&Ti.tick[Ti.tick_off + kh], 1);
    *last_flag = (old == Ti.nch - 1);
  }
  named_bar(2, kThreads);
  if (*last_flag) {
    __threadfence();
    // merge this (tile, kv head): each query over its own chunks, in chunk order
    for (int idx = tid; idx < QH * hd; idx += kThreads) {
      const int qh = idx / hd, e = idx % hd;
      const int r = qh / GQ, hg = qh % GQ;
      const int nc = (Ti.pos0 + r + CK - 1) / CK;
      const float* base = Ti.part + ((size_t)Ti.rec_off + (size_t)kh * Ti.nch * QH + qh) * (hd + 2);
      const size_t cstride = (size_t)QH * (hd + 2);
      float M = -INFINITY;
      for (int cc = 0; cc < nc; ++cc) M = fmaxf(M, __ldcg(base + cc * cstride + hd));
      float Ls = 0.f, O = 0.f;
      for (int cc = 0; cc < nc; ++cc) {
        const float* rc = base + cc * cstride;
        const float w = expf(__ldcg(rc + hd) - M);
        Ls = fmaf(__ldcg(rc + hd + 1), w, Ls);
        O = fmaf(__ldcg(rc + e), w, O);
      }
      Ti.out[(size_t)(Ti.vid0 + r) * hqd + (kh * GQ + hg) * hd + e] = O / Ls;
    }
    if (tid == 0) Ti.tick[Ti.tick_off + kh] = 0;
  }
  named_bar(2, kThreads);  // shared buffers are reused by the next item
}

// Runs items item0, item0 + step, ... of the tiles on the 256 calling threads (threadIdx.x < 256),
// loading each item's K/V chunk itself.  `sm` (smem_bytes) and `kv_bar` (an initialised mbarrier,
// parity `phase`) belong to the caller; `fail` is a shared flag.  False if a bounded wait gave up.
template <typename WT, int CK>
static __device__ bool run_items(const Dims& D, DevState* st, const Tile* tiles, int nt, int n_items, int item0,
                                 int step, int qh_max, unsigned char* sm, uint64_t* kv_bar, uint32_t& phase,
                                 int* fail, int* last_flag) {
  constexpr int ESZ = sizeof(WT);
  const int hd = D.hd;
  const int tid = threadIdx.x;
  WT* ks = reinterpret_cast<WT*>(sm);
  WT* vs = reinterpret_cast<WT*>(sm + (size_t)CK * hd * ESZ);
  float* qs = reinterpret_cast<float*>(sm + (size_t)2 * CK * hd * ESZ);
  float* sc = qs + (size_t)qh_max * hd;
  float* m_s = sc + (size_t)qh_max * CK;
  float* l_s = m_s + qh_max;
  for (int item = item0; item < n_items; item += step) {
    const Item it = item_of(tiles, nt, item, CK);
    const Tile& Ti = tiles[it.T];
    if (tid == 0) {  // K/V chunk -> shared memory (one bulk copy each)
      const uint32_t bytes = (uint32_t)it.nk * hd * ESZ;
      const size_t off = ((size_t)it.kh * D.max_seq + it.c * CK) * hd * ESZ;
      mbar_arrive_expect_tx(kv_bar, 2 * bytes);
      const uint64_t pol = l2_evict_first_policy();
      bulk_g2s(ks, Ti.kc + off, bytes, kv_bar, pol);
      bulk_g2s(vs, Ti.vc + off, bytes, kv_bar, pol);
    }
    if (!mbar_wait_bounded(kv_bar, phase)) *fail = 1;
    phase ^= 1;
    named_bar(2, kThreads);
    if (*fail) {  // uniform decision after the barrier
      if (tid == 0) {
        set_err(st, ERR_TIMEOUT, 30);
        mbar_wait_bounded(kv_bar, phase ^ 1);  // let the copies in flight land before leaving
      }
      return false;
    }
    item_compute<WT, CK>(D, Ti, it, ks, vs, qs, sc, m_s, l_s, last_flag);
  }
  return true;
}

// ------------------------------------------------------------------------------------------------
// One warp per work item (persistent step kernel).  Item = (tile, kv head, chunk of CK = 32 keys);
// its K and V chunks sit in a ring stage ([nk][hd] each, cache dtype).  Per query head of the tile:
// lane k scores key k (a dot product over hd, reading the K row from a rotated chunk so that the
// lanes of a quarter-warp hit distinct banks), the chunk's softmax statistics come from xor-shuffle
// reductions, and lane l accumulates output dims [l*hd/32, (l+1)*hd/32) over the chunk's keys.
// The partial (o, m, l) goes to global scratch.  A warp batches the tickets of its items (one
// fence, then one atomic per (tile, kv head) it touched); the warp that takes the last ticket of a
// (tile, kv head) merges the partials of every query head in chunk order.  No block barrier.
// ------------------------------------------------------------------------------------------------
constexpr int kWarpCK = 32;

// Chunks of earlier cycles and chunks holding this cycle's keys (key kn0 onward), per tile (`ck`
// keys per chunk): fills co / old_off / new_off and returns the totals.  Only old chunks may be
// fetched before the grid barrier that ends the QKV step.
__device__ __forceinline__ void split_items(const Dims& D, Tile* tiles, int nt, int ck, int* n_old, int* n_new) {
  int o = 0, w = 0;
  for (int i = 0; i < nt; ++i) {
    Tile& T = tiles[i];
    T.co = min(T.nch, T.kn0 / ck);
    T.old_off = o;
    T.new_off = w;
    o += D.hkv * T.co;
    w += D.hkv * (T.nch - T.co);
  }
  *n_old = o;
  *n_new = w;
}

// Item `g` of the list of old (pass 0) or new (pass 1) chunks.
__device__ __forceinline__ Item item_of_pass(const Tile* tiles, int nt, int pass, int g, int ck) {
  Item it;
  it.T = 0;
  if (pass == 0) {
    while (it.T + 1 < nt && tiles[it.T + 1].old_off <= g) ++it.T;
    const Tile& T = tiles[it.T];
    const int rem = g - T.old_off;
    it.kh = rem / T.co;
    it.c = rem % T.co;
  } else {
    while (it.T + 1 < nt && tiles[it.T + 1].new_off <= g) ++it.T;
    const Tile& T = tiles[it.T];
    const int nn = T.nch - T.co;
    const int rem = g - T.new_off;
    it.kh = rem / nn;
    it.c = T.co + rem % nn;
  }
  const Tile& T = tiles[it.T];
  it.nk = min(ck, T.pos0 + T.nq - 1 - it.c * ck);
  return it;
}

// DPL consecutive elements of a K/V row in shared memory -> fp32 (DPL * sizeof(WT) bytes, aligned).
template <typename WT, int DPL>
__device__ __forceinline__ void load_row(const WT* p, float* f) {
  if constexpr (sizeof(WT) == 2 && DPL == 2) {
    const uint32_t u = *reinterpret_cast<const uint32_t*>(p);
    f[0] = bf16_lo(u); f[1] = bf16_hi(u);
  } else if constexpr (sizeof(WT) == 2 && DPL == 4) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    f[0] = bf16_lo(u.x); f[1] = bf16_hi(u.x); f[2] = bf16_lo(u.y); f[3] = bf16_hi(u.y);
  } else if constexpr (sizeof(WT) == 2 && DPL == 8) {
    WTraits<WT>::unpack(*reinterpret_cast<const uint4*>(p), f);
  } else if constexpr (DPL == 2) {
    const float2 v = *reinterpret_cast<const float2*>(p);
    f[0] = v.x; f[1] = v.y;
  } else {
#pragma unroll
    for (int e = 0; e < DPL; e += 4) {
      const float4 v = *reinterpret_cast<const float4*>(p + e);
      f[e] = v.x; f[e + 1] = v.y; f[e + 2] = v.z; f[e + 3] = v.w;
    }
  }
}

// Query head qh of tile T for kv head kh -> lane's DPL dims (rotated q, written by the QKV phase).
template <int DPL>
__device__ __forceinline__ void load_q(const Dims& D, const Tile& T, int kh, int qh, float* qv) {
  const int lane = threadIdx.x & 31;
  const int r = qh / D.gq, hg = qh % D.gq;
  const float* src = T.q + (size_t)(T.vid0 + r) * D.qkv_rows + (kh * D.gq + hg) * D.hd + lane * DPL;
  if constexpr (DPL % 4 == 0) {
#pragma unroll
    for (int e = 0; e < DPL; e += 4) {
      const float4 v = __ldcg(reinterpret_cast<const float4*>(src + e));
      qv[e] = v.x; qv[e + 1] = v.y; qv[e + 2] = v.z; qv[e + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int e = 0; e < DPL; e += 2) {
      const float2 v = __ldcg(reinterpret_cast<const float2*>(src + e));
      qv[e] = v.x; qv[e + 1] = v.y;
    }
  }
}

constexpr int kHeadsPerPass = 4;  // query heads a warp item computes together

// Query heads qh0, qh0 + qstep, ... of item `it` on the calling warp, up to four at a time: each K
// row chunk and each V row slice is read once from shared memory for all the heads of a pass, and
// the heads' dot products, softmax reductions and output sums are independent chains that overlap.
// q0[h] holds the lane's slice of query head qh0 + h*qstep (loaded ahead by the caller, first pass).
// ks / vs: the chunk's K and V rows in shared memory; qb: 4*hd floats of per-warp scratch.  Writes
// one partial (o, m, l) per query head; no ticket.  Each head's arithmetic is the same whatever
// heads share its pass.
template <typename WT, int DPL>
__device__ void warp_item(const Dims& D, const Tile& T, const Item& it, const WT* ks, const WT* vs, float* qb,
                          int qh0, int qstep, const float (*q0)[DPL]) {
  constexpr int CK = kWarpCK;
  constexpr int HP = kHeadsPerPass;
  constexpr int VEC = WTraits<WT>::kVec;  // elements per 16-byte chunk of a K row
  const int lane = threadIdx.x & 31;
  const int hd = D.hd;
  const int nchk = hd / VEC;               // 16-byte chunks per K row
  const float scale = 1.0f / sqrtf((float)hd);
  const int QH = T.nq * D.gq;
  const int kh = it.kh, c = it.c, nk = it.nk;
  const int key0 = c * CK;
  for (int g0 = qh0; g0 < QH; g0 += HP * qstep) {
    // this pass's query vectors -> shared memory (the lane's slice of each)
#pragma unroll
    for (int h = 0; h < HP; ++h) {
      const int qh = g0 + h * qstep;
      if (qh < QH) {
        float qv[DPL];
        if (g0 == qh0) {
#pragma unroll
          for (int e = 0; e < DPL; ++e) qv[e] = q0[h][e];
        } else {
          load_q<DPL>(D, T, kh, qh, qv);
        }
#pragma unroll
        for (int e = 0; e < DPL; ++e) qb[h * hd + lane * DPL + e] = qv[e];
      }
    }
    __syncwarp();
    // score of key `lane` for every head of the pass: four partial sums each (element e % 4)
    float d4[HP][4];
#pragma unroll
    for (int h = 0; h < HP; ++h) d4[h][0] = d4[h][1] = d4[h][2] = d4[h][3] = 0.f;
    if (lane < nk) {
      const WT* kr = ks + (size_t)lane * hd;
#pragma unroll 2
      for (int j = 0; j < nchk; ++j) {
        const int jj = (j + lane) % nchk;
        float kf[VEC];
        WTraits<WT>::unpack(*reinterpret_cast<const uint4*>(kr + jj * VEC), kf);
#pragma unroll
        for (int h = 0; h < HP; ++h) {
          if (g0 + h * qstep < QH) {
            const float* qv = qb + h * hd + jj * VEC;
#pragma unroll
            for (int e = 0; e < VEC; e += 4) {
              const float4 q4 = *reinterpret_cast<const float4*>(qv + e);
              d4[h][0] = fmaf(kf[e], q4.x, d4[h][0]);
              d4[h][1] = fmaf(kf[e + 1], q4.y, d4[h][1]);
              d4[h][2] = fmaf(kf[e + 2], q4.z, d4[h][2]);
              d4[h][3] = fmaf(kf[e + 3], q4.w, d4[h][3]);
            }
          }
        }
      }
    }
    float pk[HP], mh[HP], lh[HP];
#pragma unroll
    for (int h = 0; h < HP; ++h) {
      const int qh = g0 + h * qstep;
      const int pos_q = T.pos0 + (qh < QH ? qh : 0) / D.gq;
      const float dot = (d4[h][0] + d4[h][1]) + (d4[h][2] + d4[h][3]);
      const float sk = (qh < QH && lane < nk && key0 + lane < pos_q) ? dot * scale : -INFINITY;
      mh[h] = sk;
      pk[h] = sk;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
      for (int h = 0; h < HP; ++h) mh[h] = fmaxf(mh[h], __shfl_xor_sync(0xffffffffu, mh[h], o));
#pragma unroll
    for (int h = 0; h < HP; ++h) {
      pk[h] = (mh[h] == -INFINITY) ? 0.f : expf(pk[h] - mh[h]);
      lh[h] = pk[h];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
      for (int h = 0; h < HP; ++h) lh[h] += __shfl_xor_sync(0xffffffffu, lh[h], o);
    // unnormalised chunk outputs, dims lane*DPL ..; each V slice is loaded once for all heads
    float acc[HP][DPL];
#pragma unroll
    for (int h = 0; h < HP; ++h)
#pragma unroll
      for (int e = 0; e < DPL; ++e) acc[h][e] = 0.f;
#pragma unroll 4
    for (int k = 0; k < nk; ++k) {
      float vf[DPL];
      load_row<WT, DPL>(vs + (size_t)k * hd + lane * DPL, vf);
#pragma unroll
      for (int h = 0; h < HP; ++h) {
        const float pj = __shfl_sync(0xffffffffu, pk[h], k);
#pragma unroll
        for (int e = 0; e < DPL; ++e) acc[h][e] = fmaf(pj, vf[e], acc[h][e]);
      }
    }
#pragma unroll
    for (int h = 0; h < HP; ++h) {
      const int qh = g0 + h * qstep;
      if (qh < QH) {
        float* rec = T.part + ((size_t)T.rec_off + ((size_t)kh * T.nch + c) * QH + qh) * (hd + 2);
#pragma unroll
        for (int e = 0; e < DPL; ++e) rec[lane * DPL + e] = acc[h][e];
        if (lane == 0) { rec[hd] = mh[h]; rec[hd + 1] = lh[h]; }
      }
    }
    __syncwarp();  // qb is rewritten by the next pass
  }
}

// Merge of query head qh of (tile T, kv head kh) on the calling warp, once every chunk partial of
// the pair is written: O = sum_c exp(m_c - M) o_c / sum_c exp(m_c - M) l_c over the query's own nc
// chunks, M = max_c m_c.  Lane l owns dims l, l + 32, ... and adds the chunks in chunk order, so the
// arithmetic depends only on nc (the query's position) and a token's result does not depend on its
// batch.  The loads of NB consecutive chunks are issued together (the m and l loads are broadcasts),
// so a merge costs about nc / NB memory round trips.
template <int DPL>
__device__ void merge_qh(const Dims& D, const Tile& T, int kh, int qh) {
  constexpr int CK = kWarpCK;
  constexpr int NB = 32 / DPL;  // chunks per batch of loads
  const int lane = threadIdx.x & 31;
  const int hd = D.hd, GQ = D.gq;
  const int QH = T.nq * GQ;
  const int r = qh / GQ, hg = qh % GQ;
  const int nc = (T.pos0 + r + CK - 1) / CK;
  const float* base = T.part + ((size_t)T.rec_off + (size_t)kh * T.nch * QH + qh) * (hd + 2);
  const size_t cstride = (size_t)QH * (hd + 2);
  float M = -INFINITY;
  for (int cc = lane; cc < nc; cc += 32) M = fmaxf(M, __ldcg(base + cc * cstride + hd));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float Ls = 0.f, O[DPL];
#pragma unroll
  for (int e = 0; e < DPL; ++e) O[e] = 0.f;
  for (int c0 = 0; c0 < nc; c0 += NB) {
    float mm[NB], ll[NB], oo[NB][DPL];
#pragma unroll
    for (int u = 0; u < NB; ++u) {
      const float* rc = base + (size_t)min(c0 + u, nc - 1) * cstride;
      mm[u] = __ldcg(rc + hd);
      ll[u] = __ldcg(rc + hd + 1);
#pragma unroll
      for (int e = 0; e < DPL; ++e) oo[u][e] = __ldcg(rc + lane + 32 * e);
    }
#pragma unroll
    for (int u = 0; u < NB; ++u) {
      if (c0 + u < nc) {
        const float w = expf(mm[u] - M);
        Ls = fmaf(ll[u], w, Ls);
#pragma unroll
        for (int e = 0; e < DPL; ++e) O[e] = fmaf(oo[u][e], w, O[e]);
      }
    }
  }
  float* out = T.out + (size_t)(T.vid0 + r) * (D.hq * hd) + (kh * GQ + hg) * hd;
#pragma unroll
  for (int e = 0; e < DPL; ++e) out[lane + 32 * e] = O[e] / Ls;
}

}  // namespace att
}  // namespace spd
