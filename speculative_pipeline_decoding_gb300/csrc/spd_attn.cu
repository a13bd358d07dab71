// Decode attention over per-layer KV caches.
//
// The query rows arrive already rotated (RoPE is applied in the QKV epilogue of the GEMV engine,
// which also appends k and v to the cache).  Work item = (query tile, kv head, key chunk of 128
// positions).  A tile holds up to 8 query rows of one layer (1 row per token in the stage-diagonal
// step); all query heads of the grouped-query group share the K/V chunk, which is bulk-copied into
// shared memory once.  Scores use 16-dim lane slices reduced with xor shuffles, softmax is per chunk
// (max, exp, sum), and the chunk partial (o, m, l) goes to global scratch.  The last item of a
// (tile, kv head) to finish (atomic ticket, no spinning) merges the partials of each query in chunk
// order.  The number of chunks depends only on the query position, so a token's result does not
// depend on its batch.
#include "spd_internal.cuh"

namespace spd {

namespace {

struct AttnParams {
  Dims D;
  Bufs B;
  Launch lc;
  int qt;
  int qh_max;
};

struct Tile {
  int layer, nq, pos0, vid0, nch, rec_off, item_off;
  const unsigned char* kc;  // base of this layer's K cache (head 0, position 1)
  const unsigned char* vc;
};

__device__ int build_tiles(const AttnParams& p, Tile* tiles, int* n_items) {
  const Dims& D = p.D;
  const Launch& lc = p.lc;
  DevState* st = p.B.st;
  RowGroup rg[kMaxGroups];
  int nr;
  if (lc.kind == LK_EXPLICIT) {
    nr = lc.cnt;
    for (int r = 0; r < nr; ++r) {
      rg[r].layer = 0; rg[r].nv = 1; rg[r].pos0 = lc.act.pos_arr[r]; rg[r].vid0 = r; rg[r].rrow0 = 0;
    }
  } else {
    nr = build_rows(lc, D, st, rg);
  }
  const int esz = D.dtype == SPD_DTYPE_BF16 ? 2 : 4;
  const size_t layer_elems = (size_t)D.hkv * D.max_seq * D.hd;
  int nt = 0, rec = 0, items = 0;
  for (int i = 0; i < nr; ++i) {
    for (int r0 = 0; r0 < rg[i].nv; r0 += p.qt) {
      if (nt >= kMaxTiles) { set_err(st, ERR_BOUNDS, 400); *n_items = 0; return 0; }
      Tile& T = tiles[nt++];
      T.layer = rg[i].layer;
      T.nq = min(p.qt, rg[i].nv - r0);
      T.pos0 = rg[i].pos0 + r0;
      T.vid0 = rg[i].vid0 + r0;
      const int pos_last = T.pos0 + T.nq - 1;
      T.nch = (pos_last + kAttnChunk - 1) / kAttnChunk;
      T.rec_off = rec;
      T.item_off = items;
      rec += D.hkv * T.nch * T.nq * D.gq;
      items += D.hkv * T.nch;
      const void* kb;
      const void* vb;
      if (lc.kind == LK_EXPLICIT) { kb = lc.act.kc; vb = lc.act.vc; }
      else if (lc.stack == 0) { kb = p.B.kc; vb = p.B.vc; }
      else { kb = p.B.pkc; vb = p.B.pvc; }
      T.kc = (const unsigned char*)kb + (size_t)T.layer * layer_elems * esz;
      T.vc = (const unsigned char*)vb + (size_t)T.layer * layer_elems * esz;
    }
  }
  *n_items = items;
  return nt;
}

template <typename WT>
__global__ void __launch_bounds__(kAttnThreads)
attn_kernel(const __grid_constant__ AttnParams p) {
  extern __shared__ __align__(128) unsigned char sm[];
  __shared__ Tile tiles[kMaxTiles];
  __shared__ int s_nt, s_items, s_last, s_fail;
  __shared__ __align__(8) uint64_t kv_bar;
  constexpr int ESZ = sizeof(WT);
  const Dims& D = p.D;
  const int hd = D.hd, GQ = D.gq, CK = kAttnChunk;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  DevState* st = p.B.st;

  if (tid == 0) {
    const bool skip = p.lc.kind != LK_EXPLICIT && (st->done || st->err);
    int items = 0;
    s_nt = skip ? 0 : build_tiles(p, tiles, &items);
    s_items = s_nt ? items : 0;
    s_fail = 0;
    mbar_init(&kv_bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();  // q and the K/V appended by the previous kernel are visible from here on
  pdl_trigger();
  const int n_items = s_items;
  if (n_items == 0) return;

  WT* ks = reinterpret_cast<WT*>(sm);
  WT* vs = reinterpret_cast<WT*>(sm + (size_t)CK * hd * ESZ);
  float* qs = reinterpret_cast<float*>(sm + (size_t)2 * CK * hd * ESZ);
  float* sc = qs + (size_t)p.qh_max * hd;
  float* m_s = sc + (size_t)p.qh_max * CK;
  float* l_s = m_s + p.qh_max;
  const float scale = 1.0f / sqrtf((float)hd);
  const int qkv_rows = D.qkv_rows;
  const int hqd = D.hq * hd;
  float* part = p.lc.act.part;
  int* tick = p.lc.act.tick;
  const int LPK = hd / 16;  // lanes per key
  const int KPW = 32 / LPK;
  uint32_t phase = 0;

  for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    int T = 0;
    while (T + 1 < s_nt && tiles[T + 1].item_off <= item) ++T;
    const Tile& Ti = tiles[T];
    const int rem = item - Ti.item_off;
    const int kh = rem / Ti.nch, c = rem % Ti.nch;
    const int QH = Ti.nq * GQ;
    const int pos_last = Ti.pos0 + Ti.nq - 1;
    const int key0 = c * CK;
    const int nk = min(CK, pos_last - key0);
    // K/V chunk -> shared memory (one bulk copy each)
    if (tid == 0) {
      const uint32_t bytes = (uint32_t)nk * hd * ESZ;
      const size_t off = ((size_t)kh * D.max_seq + key0) * hd * ESZ;
      mbar_arrive_expect_tx(&kv_bar, 2 * bytes);
      const uint64_t pol = l2_evict_first_policy();
      bulk_g2s(ks, Ti.kc + off, bytes, &kv_bar, pol);
      bulk_g2s(vs, Ti.vc + off, bytes, &kv_bar, pol);
    }
    // queries (already rotated) -> shared memory
    for (int idx = tid; idx < QH * hd; idx += kAttnThreads) {
      const int qh = idx / hd, e = idx % hd;
      const int r = qh / GQ, hg = qh % GQ;
      qs[idx] = p.lc.act.qkv[(size_t)(Ti.vid0 + r) * qkv_rows + (kh * GQ + hg) * hd + e];
    }
    if (!mbar_wait_bounded(&kv_bar, phase)) s_fail = 1;
    phase ^= 1;
    __syncthreads();
    if (s_fail) {  // uniform decision after the barrier
      if (tid == 0) {
        set_err(st, ERR_TIMEOUT, 30);
        mbar_wait_bounded(&kv_bar, phase ^ 1);  // let the copies in flight land before leaving
      }
      break;
    }
    // scores
    {
      const int kl = lane / LPK, sub = lane % LPK;
      for (int kb = warp * KPW; kb < CK; kb += 8 * KPW) {
        const int kk = kb + kl;
        float kf[16];
        if (kk < nk) {
          const WT* kr = ks + (size_t)kk * hd + sub * 16;
#pragma unroll
          for (int e = 0; e < 16; e += 16 / ESZ) {
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
    __syncthreads();
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
    __syncthreads();
    // unnormalised chunk output -> partial record (o[hd], m, l)
    for (int idx = tid; idx < QH * hd; idx += kAttnThreads) {
      const int qh = idx / hd, e = idx % hd;
      const float* prow = sc + (size_t)qh * CK;
      float o = 0.f;
      for (int k = 0; k < nk; ++k) o = fmaf(prow[k], WTraits<WT>::to_f(vs[(size_t)k * hd + e]), o);
      float* rec = part + ((size_t)Ti.rec_off + ((size_t)kh * Ti.nch + c) * QH + qh) * (hd + 2);
      rec[e] = o;
      if (e == 0) { rec[hd] = m_s[qh]; rec[hd + 1] = l_s[qh]; }
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) {
      const int old = atomicAdd(&tick[T * D.hkv + kh], 1);
      s_last = (old == Ti.nch - 1);
    }
    __syncthreads();
    if (s_last) {
      __threadfence();
      // merge this (tile, kv head): each query over its own chunks, in chunk order
      for (int idx = tid; idx < QH * hd; idx += kAttnThreads) {
        const int qh = idx / hd, e = idx % hd;
        const int r = qh / GQ, hg = qh % GQ;
        const int nc = (Ti.pos0 + r + CK - 1) / CK;
        const float* base = part + ((size_t)Ti.rec_off + (size_t)kh * Ti.nch * QH + qh) * (hd + 2);
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
        p.lc.act.attn[(size_t)(Ti.vid0 + r) * hqd + (kh * GQ + hg) * hd + e] = O / Ls;
      }
      if (tid == 0) tick[T * D.hkv + kh] = 0;
    }
    __syncthreads();  // shared buffers are reused by the next item
  }
}

}  // namespace

size_t attn_smem_bytes(const Dims& D, bool multi) {
  const int esz = D.dtype == SPD_DTYPE_BF16 ? 2 : 4;
  const int qh = (multi ? kAttnQT : 1) * D.gq;
  return (size_t)2 * kAttnChunk * D.hd * esz + (size_t)qh * D.hd * 4 + (size_t)qh * kAttnChunk * 4 +
         (size_t)2 * qh * 4;
}

size_t attn_part_floats(int rows, int hq, int hd, int max_seq) {
  const int nch = (max_seq + kAttnChunk - 1) / kAttnChunk;
  return (size_t)rows * hq * nch * (hd + 2);
}

int attn_grid(const Dims& D, bool multi) {
  const size_t smem = attn_smem_bytes(D, multi);
  int occ = 0;
  if (D.dtype == SPD_DTYPE_BF16)
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, attn_kernel<__nv_bfloat16>, kAttnThreads, smem);
  else
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, attn_kernel<float>, kAttnThreads, smem);
  return num_sms() * (occ > 0 ? occ : 1);
}

// Raise the kernels' dynamic shared-memory limit to `need` (never lowered by a later call).
cudaError_t attn_setup_attributes(size_t need) {
  static size_t current = 0;
  if (need <= current) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(attn_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)need);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(attn_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)need);
  if (e == cudaSuccess) current = need;
  return e;
}

cudaError_t launch_attn(const Dims& D, const Bufs& B, const Launch& lc, const LaunchCfg& cfg,
                        bool pdl, cudaStream_t s) {
  AttnParams p;
  memset(&p, 0, sizeof(p));
  p.D = D; p.B = B; p.lc = lc;
  const bool multi = lc.kind == LK_PDMROWS || lc.kind == LK_ROWS;
  p.qt = multi ? kAttnQT : 1;
  p.qh_max = p.qt * D.gq;
  const size_t smem = attn_smem_bytes(D, multi);
  const int grid = multi ? cfg.attn_grid_multi : cfg.attn_grid_decode;
  cudaLaunchConfig_t lcfg;
  memset(&lcfg, 0, sizeof(lcfg));
  lcfg.gridDim = dim3(grid);
  lcfg.blockDim = dim3(kAttnThreads);
  lcfg.dynamicSmemBytes = smem;
  lcfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lcfg.attrs = attr;
  lcfg.numAttrs = pdl ? 1 : 0;
  if (D.dtype == SPD_DTYPE_BF16) return cudaLaunchKernelEx(&lcfg, attn_kernel<__nv_bfloat16>, p);
  return cudaLaunchKernelEx(&lcfg, attn_kernel<float>, p);
}

}  // namespace spd

// ------------------------------------------------------------------------------------------------
// Decode attention for callers that cannot allocate device memory.
//
// Some callers may not call cudaMalloc at all: a plugin hosted by an application that owns the
// GPU's memory budget (an inference server whose allocator reserved nearly all HBM up front), or
// code on a latency-critical path where an allocation could synchronise the device.  For them the
// split partials and the merge tickets live in one file-scope device array of fixed size that
// every GPU loading this library holds until the process exits.  Its device address is looked up
// once per device (with that device current) on the first call there; make that first call before
// any stream capture.  All calls share the array and it keeps the last call's contents: the tickets
// are cleared at the start of every call, and calls that overlap on the GPU race on the array.
// ------------------------------------------------------------------------------------------------
#include <cstdio>
#include <mutex>

namespace spd {
namespace {
constexpr size_t kStaticScratchBytes = (size_t)16 << 20;   // 16 MiB per device
constexpr size_t kStaticTicketBytes = (size_t)16 << 10;    // first 16 KiB: merge tickets
static __device__ __align__(256) unsigned char g_attn_static_scratch[kStaticScratchBytes];
std::mutex g_static_mu;
void* g_static_addr[64] = {};  // device address of the array, per device ordinal
}  // namespace

}  // namespace spd

extern "C" int spd_attention_static_scratch(const float* q, const void* k_cache, const void* v_cache,
                                            int32_t dtype, const int32_t* pos, int32_t R,
                                            int32_t n_heads, int32_t n_kv_heads, int32_t head_dim,
                                            int32_t max_seq, float* out, void* cuda_stream) {
  using namespace spd;
  char msg[256];
  if (!q || !k_cache || !v_cache || !pos || !out || R < 1 || R > kMaxAttnRows || n_kv_heads < 1 ||
      n_heads % n_kv_heads || head_dim % 16 || head_dim > 256 || max_seq < 1 ||
      (dtype != SPD_DTYPE_F32 && dtype != SPD_DTYPE_BF16))
    return spd_internal_fail(SPD_EINVAL, "spd_attention_static_scratch: bad arguments");
  const size_t tick_bytes = (size_t)kMaxTiles * n_kv_heads * sizeof(int);
  const size_t part_bytes = attn_part_floats(R, n_heads, head_dim, max_seq) * sizeof(float);
  if (tick_bytes > kStaticTicketBytes || part_bytes > kStaticScratchBytes - kStaticTicketBytes) {
    snprintf(msg, sizeof(msg),
             "spd_attention_static_scratch: needs %zu B of partials and %zu B of tickets; the static "
             "scratch holds %zu B and %zu B",
             part_bytes, tick_bytes, kStaticScratchBytes - kStaticTicketBytes, kStaticTicketBytes);
    return spd_internal_fail(SPD_EINVAL, msg);
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64)
    return spd_internal_fail(SPD_ECUDA, "spd_attention_static_scratch: no usable current device");
  void* base = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (!g_static_addr[dev]) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_attn_static_scratch);
      if (e != cudaSuccess) {
        snprintf(msg, sizeof(msg), "spd_attention_static_scratch: cudaGetSymbolAddress: %s",
                 cudaGetErrorString(e));
        return spd_internal_fail(SPD_ECUDA, msg);
      }
      g_static_addr[dev] = p;
    }
    base = g_static_addr[dev];
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(cuda_stream);
  e = cudaMemsetAsync(base, 0, tick_bytes, s);  // tickets must start at zero
  if (e != cudaSuccess) return spd_internal_fail(SPD_ECUDA, "spd_attention_static_scratch: ticket reset failed");
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
  lc.act.tick = reinterpret_cast<int*>(base);
  lc.act.part = reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(base) + kStaticTicketBytes);
  lc.act.pos_arr = pos;
  lc.act.kc = k_cache; lc.act.vc = v_cache;
  e = attn_setup_attributes(attn_smem_bytes(D, false));
  if (e != cudaSuccess) return spd_internal_fail(SPD_ECUDA, "spd_attention_static_scratch: smem attribute");
  LaunchCfg LC;
  memset(&LC, 0, sizeof(LC));
  LC.attn_grid_decode = attn_grid(D, false);
  e = launch_attn(D, B, lc, LC, false, s);
  if (e != cudaSuccess) {
    snprintf(msg, sizeof(msg), "spd_attention_static_scratch: launch: %s", cudaGetErrorString(e));
    return spd_internal_fail(SPD_ECUDA, msg);
  }
  return SPD_OK;
}

