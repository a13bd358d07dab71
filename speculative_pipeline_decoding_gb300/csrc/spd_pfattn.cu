// Causal attention of prefill blocks on the 5th-generation tensor cores (tcgen05, TMEM accumulators).
//
// A prefill block is nq <= 32 query rows at consecutive positions pos0..pos0+nq-1 of one layer; their
// keys and values are already in the layer's cache (the QKV epilogue appended them), so row i sees
// keys 1..pos0+i.  For one kv head, the queries of ng heads of its grouped-query group form a tile of
// up to 128 rows (row r = query r / ng, head r % ng of the tile's heads), the M = 128 side of the
// MMAs.  The keys are taken in chunks of 128:
//
//   S = Q K_c^T           M 128 x N 128 keys x K hd; Q as bf16 high + low halves (two MMAs per k-step,
//                         ~16 significant bits of the fp32 query), K_c straight from the cache by TMA
//   online softmax        one thread per row: S row from TMEM, scale 1/sqrt(hd), causal mask,
//                         running max m and sum l, P = exp(S - m) as bf16 high + low halves in shared
//                         memory, the O row rescaled in TMEM by exp(m_old - m_new)
//   O += P V_c            M 128 x N hd x K 128 keys; V_c as the MN-major operand (its rows are keys)
//
// S and O live in TMEM (columns 0..127 and 128..128+hd).  Long contexts are split over CTAs by key
// chunks (split-K): each split writes its unnormalised O row with m and l, and the last split of a
// tile to finish (atomic ticket) merges them in split order; a tile with one split writes O / l.
// One elected thread issues the tensor copies and the MMAs; every wait is bounded.
//
// Layout in shared memory (1024-byte aligned, 128-byte swizzle, [64-element chunk][row][128 B]):
//   Qhi, Qlo [hd/64][128 rows]   Ks [hd/64][128 keys]   Vs [hd/64][128 keys]   Phi, Plo [2][128 rows]
#include <cudaTypedefs.h>

#include <mutex>

#include "spd_internal.cuh"
#include "spd_tc.cuh"

namespace spd {
namespace pfa {

constexpr int kRows = 128;        // tile rows (M)
constexpr int kKeys = 128;        // keys per chunk
constexpr int kThreads = 128;     // one thread per tile row
constexpr uint32_t kTmemCols = 256;
constexpr int kMinChunksPerSplit = 4;

struct Params {
  CUtensorMap kmap, vmap;   // 2-D maps over the K / V caches: (element of hd, row), box 64 x 128 keys
  const float* q;           // query rows [row][q_stride] (rotated q at the front, head h at h*hd)
  float* out;               // attention rows [row][hq*hd]
  float* part;              // split partials [tile][split][128 rows][hd + 2]
  int* tick;                // merge tickets [tile] (left at zero)
  DevState* st;             // error word (may be null)
  int q_stride;
  int kv_row0;              // map row of position 1 of kv head 0 of the layer
  int max_seq;              // map rows per kv head
  int hq, hkv, hd, gq;
  int pos0, nq;             // queries at positions pos0..pos0+nq-1
  int ng, tiles_per_kv;     // heads per tile, tiles per kv head
  int nch, cps, nsplit;     // key chunks, chunks per split, splits per tile
};

__device__ __forceinline__ void tma2(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(smem_u32(dst)), "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ uint64_t desc_kmajor(const void* p) { return tc::sdesc(tc::su32(p)); }
// MN-major operand (V: rows are keys = K, 128-byte rows of 64 hd = N): the 8-key groups are 1024 B apart
// and the second 64-element half of hd is one chunk (kKeys * 128 B) further on
__device__ __forceinline__ uint64_t desc_mnmajor(const void* p, uint32_t lbo, uint32_t sbo) {
  const uint32_t a = tc::su32(p);
  return (uint64_t)((a & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
__host__ __device__ constexpr uint32_t idesc(int m, int n, int b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)b_mn_major << 16) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void st_rows(uint32_t ta, const uint32_t* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
      ::"r"(ta), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]),
        "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]),
        "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Byte offset of element (row r, column e) in a [chunk][128 rows][128 B] swizzled operand (bf16).
__device__ __forceinline__ uint32_t swz(int r, int e) {
  return (uint32_t)((e >> 6) * (kRows * 128) + r * 128 + ((((e & 63) >> 3) ^ (r & 7)) << 4) + (e & 7) * 2);
}

__device__ __forceinline__ uint32_t pack_hi_lo(float a, float b, bool lo) {
  const float ha = __bfloat162float(__float2bfloat16_rn(a)), hb = __bfloat162float(__float2bfloat16_rn(b));
  const __nv_bfloat162 p = lo ? __floats2bfloat162_rn(a - ha, b - hb) : __floats2bfloat162_rn(ha, hb);
  return *reinterpret_cast<const uint32_t*>(&p);
}

template <int HD>
__global__ void __launch_bounds__(kThreads, 1) pf_attn_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* base =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  constexpr int OPB = HD / 64 * kRows * 128;  // bytes of a 128-row operand of hd columns
  constexpr int PB = 2 * kRows * 128;         // bytes of P (128 keys)
  unsigned char* q_hi = base;
  unsigned char* q_lo = q_hi + OPB;
  unsigned char* ks = q_lo + OPB;
  unsigned char* vs = ks + OPB;
  unsigned char* p_hi = vs + OPB;
  unsigned char* p_lo = p_hi + PB;
  __shared__ __align__(8) uint64_t kbar, vbar, mbar;
  __shared__ uint32_t s_tmem;
  __shared__ int s_last;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tile = blockIdx.x / p.nsplit, split = blockIdx.x % p.nsplit;
  const int kh = tile / p.tiles_per_kv, h0 = kh * p.gq + (tile % p.tiles_per_kv) * p.ng;
  const int ng = min(p.ng, p.gq - (tile % p.tiles_per_kv) * p.ng);
  const int c0 = split * p.cps, c1 = min(p.nch, c0 + p.cps);
  const int r = tid;                                   // this thread's tile row
  const int qi = r / p.ng, g = r % p.ng;
  const bool valid = qi < p.nq && g < ng;
  const int qpos = p.pos0 + min(qi, p.nq - 1);         // padding rows see the last query's keys
  const int ky0 = p.kv_row0 + kh * p.max_seq;         // map row of position 1 of this kv head
  const float scale = 1.0f / sqrtf((float)HD);

  if (tid == 0) {
    mbar_init(&kbar, 1);
    mbar_init(&vbar, 1);
    mbar_init(&mbar, 1);
    fence_mbar_init();
  }
  // queries -> bf16 high / low halves, one row per thread (zeros for padding rows)
  {
    const float* qr = p.q + (size_t)qi * p.q_stride + (size_t)(h0 + g) * HD;
#pragma unroll 4
    for (int e = 0; e < HD; e += 8) {
      float x[8];
      if (valid) {
        const float4 a = *reinterpret_cast<const float4*>(qr + e), b = *reinterpret_cast<const float4*>(qr + e + 4);
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) x[j] = 0.f;
      }
      const uint32_t o = swz(r, e);
      *reinterpret_cast<uint4*>(q_hi + o) = make_uint4(pack_hi_lo(x[0], x[1], false), pack_hi_lo(x[2], x[3], false),
                                                       pack_hi_lo(x[4], x[5], false), pack_hi_lo(x[6], x[7], false));
      *reinterpret_cast<uint4*>(q_lo + o) = make_uint4(pack_hi_lo(x[0], x[1], true), pack_hi_lo(x[2], x[3], true),
                                                       pack_hi_lo(x[4], x[5], true), pack_hi_lo(x[6], x[7], true));
    }
  }
  tc::fence_async_smem();
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(tc::su32(&s_tmem)),
                 "r"(kTmemCols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tm_s = s_tmem, tm_o = s_tmem + kRows;
  const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;  // this warp's TMEM lanes (tcgen05.st)

  auto load_chunk = [&](unsigned char* dst, const CUtensorMap* map, int c, uint64_t* bar) {
    mbar_arrive_expect_tx(bar, (uint32_t)OPB);
#pragma unroll
    for (int hc = 0; hc < HD / 64; ++hc) tma2(dst + hc * kRows * 128, map, hc * 64, ky0 + c * kKeys, bar);
  };
  if (tid == 0 && c0 < c1) {
    load_chunk(ks, &p.kmap, c0, &kbar);
    load_chunk(vs, &p.vmap, c0, &vbar);
  }

  float m_run = -INFINITY, l_run = 0.f;
  uint32_t ph_k = 0, ph_v = 0, ph_m = 0;
  bool ok = true;
  for (int c = c0; c < c1 && ok; ++c) {
    // S = Q K_c^T (high and low halves of Q accumulate into the same columns)
    if (tid == 0) {
      ok = mbar_wait_bounded(&kbar, ph_k);
      if (ok) {
        tc::fence_after();
        constexpr uint32_t id = idesc(kRows, kKeys, 0);
#pragma unroll
        for (int half = 0; half < 2; ++half)
#pragma unroll
          for (int ksp = 0; ksp < HD / 16; ++ksp) {
            const int off = (ksp >> 2) * kRows * 128 + (ksp & 3) * 32;
            tc::mma(tm_s, desc_kmajor((half ? q_lo : q_hi) + off), desc_kmajor(ks + off), id, half > 0 || ksp > 0);
          }
      }
      tc::commit(&mbar);  // also covers the previous chunk's P V
    }
    ph_k ^= 1;
    ok = __syncthreads_and(ok && mbar_wait_bounded(&mbar, ph_m)) != 0;
    ph_m ^= 1;
    tc::fence_after();
    if (!ok) break;
    // K and V buffers are free (every MMA so far is done): next keys, this chunk's values
    if (tid == 0) {
      if (c + 1 < c1) load_chunk(ks, &p.kmap, c + 1, &kbar);
      if (c > c0) load_chunk(vs, &p.vmap, c, &vbar);
    }
    // online softmax of this thread's row
    float sv[kKeys];
#pragma unroll
    for (int j = 0; j < kKeys; j += 32) tc::load_rows(tm_s + j, warp, reinterpret_cast<uint32_t*>(sv + j));
    const int key0 = c * kKeys + 1;  // position of the chunk's first key
    float mc = -INFINITY;
#pragma unroll
    for (int j = 0; j < kKeys; ++j) {
      sv[j] = (key0 + j <= qpos) ? sv[j] * scale : -INFINITY;
      mc = fmaxf(mc, sv[j]);
    }
    const float m_new = fmaxf(m_run, mc);
    const float m_use = m_new == -INFINITY ? 0.f : m_new;
    const float corr = expf(m_run - m_use);  // 0 on the first chunk (m_run = -inf)
    float lsum = 0.f;
#pragma unroll
    for (int j = 0; j < kKeys; j += 8) {
      float pv[8];
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        pv[t] = expf(sv[j + t] - m_use);
        lsum += pv[t];
      }
      const uint32_t o = swz(r, j);
      *reinterpret_cast<uint4*>(p_hi + o) = make_uint4(pack_hi_lo(pv[0], pv[1], false), pack_hi_lo(pv[2], pv[3], false),
                                                       pack_hi_lo(pv[4], pv[5], false), pack_hi_lo(pv[6], pv[7], false));
      *reinterpret_cast<uint4*>(p_lo + o) = make_uint4(pack_hi_lo(pv[0], pv[1], true), pack_hi_lo(pv[2], pv[3], true),
                                                       pack_hi_lo(pv[4], pv[5], true), pack_hi_lo(pv[6], pv[7], true));
    }
    l_run = l_run * corr + lsum;
    m_run = m_new;
    // rescale the O row accumulated so far (warp-collective; skipped when no row of the warp moved)
    if (c > c0 && __any_sync(0xffffffffu, corr != 1.0f)) {
#pragma unroll
      for (int j = 0; j < HD; j += 32) {
        uint32_t ov[32];
        tc::load_rows(tm_o + j, warp, ov);
#pragma unroll
        for (int t = 0; t < 32; ++t) ov[t] = __float_as_uint(__uint_as_float(ov[t]) * corr);
        st_rows(tm_o + j + lane_off, ov);
      }
    }
    tc::fence_async_smem();
    tc::fence_before();
    __syncthreads();
    // O += P V_c
    if (tid == 0) {
      ok = mbar_wait_bounded(&vbar, ph_v);
      if (ok) {
        tc::fence_after();
        constexpr uint32_t id = idesc(kRows, HD, 1);
#pragma unroll
        for (int half = 0; half < 2; ++half)
#pragma unroll
          for (int ksp = 0; ksp < kKeys / 16; ++ksp) {
            const int aoff = (ksp >> 2) * kRows * 128 + (ksp & 3) * 32;
            tc::mma(tm_o, desc_kmajor((half ? p_lo : p_hi) + aoff),
                    desc_mnmajor(vs + ksp * 2048, kKeys * 128, 1024), id, c > c0 || half > 0 || ksp > 0);
          }
      }
    }
    ph_v ^= 1;
    ok = __syncthreads_or(!ok) == 0;
  }
  // every MMA done
  if (tid == 0) tc::commit(&mbar);
  ok = __syncthreads_and(ok && mbar_wait_bounded(&mbar, ph_m)) != 0;
  tc::fence_after();
  if (!ok) {
    if (tid == 0) {
      set_err(p.st, ERR_TIMEOUT, 80);
      // let the tensor copies still in flight land before the CTA leaves (bounded)
      mbar_wait_bounded(&kbar, ph_k);
      mbar_wait_bounded(&vbar, ph_v);
    }
  } else if (c0 < c1) {
    float ov[HD];
#pragma unroll
    for (int j = 0; j < HD; j += 32) tc::load_rows(tm_o + j, warp, reinterpret_cast<uint32_t*>(ov + j));
    float* orow = p.out + (size_t)qi * (p.hq * HD) + (size_t)(h0 + g) * HD;
    if (p.nsplit == 1) {
      if (valid) {
        const float inv = 1.0f / l_run;
#pragma unroll
        for (int e = 0; e < HD; e += 4)
          *reinterpret_cast<float4*>(orow + e) = make_float4(ov[e] * inv, ov[e + 1] * inv, ov[e + 2] * inv, ov[e + 3] * inv);
      }
    } else {
      float* pr = p.part + (((size_t)tile * p.nsplit + split) * kRows + r) * (HD + 2);
#pragma unroll
      for (int e = 0; e < HD; e += 2) *reinterpret_cast<float2*>(pr + e) = make_float2(ov[e], ov[e + 1]);
      *reinterpret_cast<float2*>(pr + HD) = make_float2(m_run, l_run);
      __threadfence();
      __syncthreads();
      if (tid == 0) {
        const int old = atomicAdd(p.tick + tile, 1);
        s_last = old == p.nsplit - 1;
        if (s_last) p.tick[tile] = 0;  // left at zero for the next launch
      }
      __syncthreads();
      if (s_last) {
        __threadfence();  // the other splits' partials are visible
        if (valid) {
          const float* pt = p.part + ((size_t)tile * p.nsplit * kRows + r) * (HD + 2);
          const size_t sstride = (size_t)kRows * (HD + 2);
          float mx = -INFINITY;
          for (int s = 0; s < p.nsplit; ++s) mx = fmaxf(mx, __ldcg(pt + s * sstride + HD));
          float lt = 0.f;
          for (int e = 0; e < HD; ++e) ov[e] = 0.f;
          for (int s = 0; s < p.nsplit; ++s) {  // in split order
            const float ms = __ldcg(pt + s * sstride + HD), ls = __ldcg(pt + s * sstride + HD + 1);
            const float w = ms == -INFINITY ? 0.f : expf(ms - mx);
            lt += ls * w;
#pragma unroll 8
            for (int e = 0; e < HD; ++e) ov[e] += __ldcg(pt + s * sstride + e) * w;
          }
          const float inv = 1.0f / lt;
#pragma unroll
          for (int e = 0; e < HD; e += 4)
            *reinterpret_cast<float4*>(orow + e) = make_float4(ov[e] * inv, ov[e + 1] * inv, ov[e + 2] * inv, ov[e + 3] * inv);
        }
      }
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(s_tmem), "r"(kTmemCols) : "memory");
}

}  // namespace pfa

// Dynamic shared memory of the prefill attention kernel for head size hd.
size_t pfattn_smem_bytes(int hd) { return 1024 + (size_t)4 * (hd / 64) * 128 * 128 + (size_t)2 * 2 * 128 * 128; }

bool pfattn_supported(int dtype, int hd, int nq, int gq) {
  return dtype == SPD_DTYPE_BF16 && (hd == 64 || hd == 128) && nq >= 1 && nq <= 32 && gq >= 1;
}

// Splits and partial-buffer floats of one launch (the same arithmetic as the launcher).
void pfattn_geometry(int hkv, int gq, int nq, int last_pos, int sms, int* ntiles, int* nsplit, int* cps, int* nch) {
  const int ng = 128 / nq < gq ? 128 / nq : gq;
  const int tpk = (gq + ng - 1) / ng;
  *ntiles = hkv * tpk;
  *nch = (last_pos + pfa::kKeys - 1) / pfa::kKeys;
  const int want = (*nch * *ntiles + 2 * sms - 1) / (2 * sms);  // about two CTAs per SM in all
  *cps = want > pfa::kMinChunksPerSplit ? want : pfa::kMinChunksPerSplit;
  *nsplit = (*nch + *cps - 1) / *cps;
}

size_t pfattn_part_floats(int hkv, int gq, int max_seq, int sms) {
  int nt, ns, cps, nch;
  size_t worst = 0;
  for (int nq = 1; nq <= 32; ++nq) {  // the split count grows with the tile count
    pfattn_geometry(hkv, gq, nq, max_seq, sms, &nt, &ns, &cps, &nch);
    const size_t f = (size_t)nt * ns * pfa::kRows * (128 + 2);
    if (f > worst) worst = f;
  }
  return worst;
}

cudaError_t pfattn_encode_map(CUtensorMap* out, const void* cache, long long rows, int hd) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  static std::mutex mu;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
      const cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
      if (e != cudaSuccess) return e;
      if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
      encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
  }
  const cuuint64_t gdim[2] = {(cuuint64_t)hd, (cuuint64_t)rows};
  const cuuint64_t gstride[1] = {(cuuint64_t)hd * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)pfa::kKeys};
  const cuuint32_t estride[2] = {1, 1};
  const CUresult r = encode(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(cache), gdim, gstride, box,
                            estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t pfattn_setup_attributes() {
  cudaError_t e = cudaFuncSetAttribute(pfa::pf_attn_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)pfattn_smem_bytes(128));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(pfa::pf_attn_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)pfattn_smem_bytes(64));
}

cudaError_t launch_pfattn(const PfAttnArgs& a, cudaStream_t s) {
  pfa::Params p;
  memset(&p, 0, sizeof(p));
  p.kmap = *a.kmap; p.vmap = *a.vmap;
  p.q = a.q; p.out = a.out; p.part = a.part; p.tick = a.tick; p.st = a.st;
  p.q_stride = a.q_stride; p.kv_row0 = a.kv_row0; p.max_seq = a.max_seq;
  p.hq = a.hq; p.hkv = a.hkv; p.hd = a.hd; p.gq = a.hq / a.hkv;
  p.pos0 = a.pos0; p.nq = a.nq;
  p.ng = 128 / a.nq < p.gq ? 128 / a.nq : p.gq;
  p.tiles_per_kv = (p.gq + p.ng - 1) / p.ng;
  int nt = 0;
  pfattn_geometry(a.hkv, p.gq, a.nq, a.pos0 + a.nq - 1, a.sms, &nt, &p.nsplit, &p.cps, &p.nch);
  const dim3 grid((unsigned)(nt * p.nsplit));
  if (a.hd == 128) pfa::pf_attn_kernel<128><<<grid, pfa::kThreads, pfattn_smem_bytes(128), s>>>(p);
  else pfa::pf_attn_kernel<64><<<grid, pfa::kThreads, pfattn_smem_bytes(64), s>>>(p);
  return cudaGetLastError();
}

}  // namespace spd
