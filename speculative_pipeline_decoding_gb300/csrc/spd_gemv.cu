// Stand-alone launches of the grouped GEMV engine (spd_engine.cuh): the prefill blocks, the
// per-operator path used when the step kernel is not, and the stand-alone operator
// spd_grouped_gemv.  One CTA per SM; one producer warp streams the weights with TMA tensor
// copies, eight consumer warps compute.
#include <cudaTypedefs.h>

#include <atomic>

#include "spd_engine.cuh"

namespace spd {

namespace {

using namespace eng;

// scratch: the tensor-core path's partial tiles, or the tcgen05 B ring of tiles of up to 32 vectors
constexpr int kGemvScratch = kMmaScratch > kStages * tc::Shape<32>::kBBytes ? kMmaScratch
                                                                            : kStages * tc::Shape<32>::kBBytes;
constexpr int kGemvSmem = 1024 + kStages * kStageBytes + kGemvScratch;

struct GemvParams {
  EngineCfg cfg;
  int nparts;
  GemvPart part[2];
  int explicit_mode;
  int resolve_after_wait;      // the control block may have been written by the previous kernel
  GemvExplicit ge;
};

template <typename WT>
__global__ void __launch_bounds__(kThreads, 1) gemv_engine(const __grid_constant__ GemvParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // the 128-byte swizzle wants 1024-byte aligned boxes
  unsigned char* ring =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  unsigned char* scratch = ring + kStages * kStageBytes;

  __shared__ GG gg[kMaxGroups];
  __shared__ int s_ng, s_gb, s_rb, s_ge, s_re;
  __shared__ __align__(8) uint64_t full_bar[kStages];
  __shared__ __align__(8) uint64_t empty_bar[kStages];
  __shared__ float rstd_s[16 * kMaxMT];
  __shared__ float wpart[kNCW];
  __shared__ Top2 hred[kNCW * 8][2];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  DevState* st = p.cfg.B.st;
  if (p.resolve_after_wait) pdl_wait();
  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], kNCW);
    }
    fence_mbar_init();
    int ng = 0;
    if (p.explicit_mode) ng = resolve_explicit(p.cfg, p.ge, gg);
    else if (!(st->done || st->err)) ng = resolve_parts(p.cfg, p.part, p.nparts, gg, kMaxGroups, View{st, p.cfg.B.tl, p.cfg.B.pl});
    s_ng = ng;
    span_of(gg, ng, blockIdx.x, gridDim.x, s_gb, s_rb, s_ge, s_re);
  }
  __syncthreads();
  const int ng = s_ng;
  Ring R{ring, full_bar, empty_bar, 0u, false};

  if (warp == kNCW) {  // producer warp
    produce_span<WT>(gg, s_gb, s_rb, s_ge, s_re, p.cfg.D.hd, p.cfg.D.box3 != 0, R, st, l2_evict_first_policy(), lane);
    drain_ring(R, lane);
    return;
  }
  if (!p.resolve_after_wait) pdl_wait();   // activations of the previous kernel are visible now
  pdl_trigger();
  Top2 loc[2];
  top2_init(loc[0]);
  top2_init(loc[1]);
  __shared__ uint32_t s_tmem;
  __shared__ __align__(8) uint64_t s_tc_done;
  __shared__ __align__(8) uint64_t s_tc_bfull[kStages];
  TcCtx tcx{scratch, 0u, &s_tc_done, 0u, s_tc_bfull, 0u};
  if (p.cfg.has_tc) {  // consumer warp 0 holds the TMEM accumulator columns for the launch
    if (warp == 0) tc::alloc_cols(&s_tmem, tc::kColsGemv);
    if (tid == 0) {
      mbar_init(&s_tc_done, 1);
      for (int i = 0; i < kStages; ++i) mbar_init(&s_tc_bfull[i], kNCW - 1);  // the builder warps
      fence_mbar_init();
    }
    tc::fence_before();
    named_bar(1, kNCW * 32);
    tc::fence_after();
    tcx.tmem = s_tmem;
  }
  consume_span<WT, 32>(p.cfg, gg, s_gb, s_rb, s_ge, s_re, R, scratch, rstd_s, wpart, loc, &tcx);
  if (p.cfg.has_tc) {  // every MMA this CTA issued has completed and every tcgen05.ld is done
    if (tid == 0) tc::commit(&s_tc_done);
    mbar_wait_bounded(&s_tc_done, tcx.phase);
    tc::fence_before();
    named_bar(1, kNCW * 32);
    if (warp == 0) tc::free_cols(tcx.tmem, tc::kColsGemv);
  }
  bool head = false;
  for (int i = 0; i < ng; ++i) head |= gg[i].epi == EPI_TOP2;
  if (head || (ng == 0 && p.nparts > 0 && p.part[0].op == OP_HEAD))
    write_head_partial(loc, hred, p.cfg.B.head_part + (size_t)blockIdx.x * 8);
}

template <typename WT>
cudaError_t launch_engine(const GemvParams& p, bool pdl, cudaStream_t s) {
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(num_sms());
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kGemvSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, gemv_engine<WT>, p);
}

}  // namespace

// SM count of the current device, looked up once per device ordinal (atomics: host threads may make
// their first calls concurrently; a repeated lookup stores the same value).
int num_sms() {
  static std::atomic<int> sms[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) dev = 0;
  if (dev >= 64) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 1;
  }
  int n = sms[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
    sms[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

int gemv_head_grid(int dtype) {
  (void)dtype;
  return num_sms();  // one CTA per SM; every CTA writes its top-2 partial
}

cudaError_t gemv_setup_attributes() {
  cudaError_t e = cudaFuncSetAttribute(gemv_engine<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kGemvSmem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(gemv_engine<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kGemvSmem);
}

cudaError_t launch_gemv(const GemvPart* parts, int nparts, const Dims& D, const Bufs& B,
                        const LaunchCfg& cfg, bool pdl, bool resolve_after_wait, cudaStream_t s) {
  GemvParams p;
  memset(&p, 0, sizeof(p));
  p.nparts = nparts;
  for (int i = 0; i < nparts && i < 2; ++i) p.part[i] = parts[i];
  p.explicit_mode = 0;
  p.resolve_after_wait = resolve_after_wait ? 1 : 0;
  p.cfg.debug_logits = cfg.debug_logits;
  p.cfg.has_mma = D.dtype == SPD_DTYPE_BF16;
  p.cfg.has_tc = D.tc;
  p.cfg.tc_nv_max = 32;
  p.cfg.eps = D.eps;
  p.cfg.D = D; p.cfg.B = B;
  return D.dtype == SPD_DTYPE_BF16 ? launch_engine<__nv_bfloat16>(p, pdl, s) : launch_engine<float>(p, pdl, s);
}

cudaError_t launch_gemv_explicit(const GemvExplicit& ge, int dtype, float eps, cudaStream_t s) {
  GemvParams p;
  memset(&p, 0, sizeof(p));
  p.explicit_mode = 1; p.resolve_after_wait = 1; p.ge = ge;
  p.cfg.eps = eps; p.cfg.has_mma = 0;
  p.cfg.D.dtype = dtype; p.cfg.D.eps = eps; p.cfg.D.box3 = box3_cols(ge.cols, dtype);
  return dtype == SPD_DTYPE_BF16 ? launch_engine<__nv_bfloat16>(p, false, s) : launch_engine<float>(p, false, s);
}

cudaError_t gemv_encode_map(CUtensorMap* out, const void* W, int rows, int cols, int dtype, bool box3) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (!encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    const cudaError_t e =
        cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  if (box3 && !box3_cols(cols, dtype)) return cudaErrorInvalidValue;
  const int esz = dtype == SPD_DTYPE_BF16 ? 2 : 4;
  const cuuint32_t ce = (cuuint32_t)(128 / esz);  // elements of one 128-byte chunk
  const CUtensorMapDataType ty = dtype == SPD_DTYPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  CUresult r;
  if (box3) {
    // (element in chunk, row, chunk): the chunk stride (128 B) is below the row stride, which the
    // tiled mode accepts; every coordinate in range addresses inside the matrix
    const cuuint64_t gdim[3] = {ce, (cuuint64_t)rows, (cuuint64_t)(cols / ce)};
    const cuuint64_t gstride[2] = {(cuuint64_t)cols * esz, 128};
    const cuuint32_t box[3] = {ce, (cuuint32_t)kBoxRows, 4};
    const cuuint32_t estride[3] = {1, 1, 1};
    r = encode(out, ty, 3, const_cast<void*>(W), gdim, gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    const cuuint64_t gdim[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t gstride[1] = {(cuuint64_t)cols * esz};
    const cuuint32_t box[2] = {ce, (cuuint32_t)kBoxRows};
    const cuuint32_t estride[2] = {1, 1};
    r = encode(out, ty, 2, const_cast<void*>(W), gdim, gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t gemv_encode_tc_map(CUtensorMap* out, const void* W, int rows, int cols) {
  CUtensorMap probe;
  cudaError_t e = gemv_encode_map(&probe, W, rows, cols, SPD_DTYPE_BF16, true);  // resolves the encoder
  if (e != cudaSuccess) return e;
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (!encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  const cuuint64_t gdim[3] = {64, (cuuint64_t)rows, (cuuint64_t)(cols / 64)};
  const cuuint64_t gstride[2] = {(cuuint64_t)cols * 2, 128};
  const cuuint32_t box[3] = {64, (cuuint32_t)tc::kRows, (cuuint32_t)tc::kStageCh};
  const cuuint32_t estride[3] = {1, 1, 1};
  const CUresult r = encode(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(W), gdim, gstride, box, estride,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace spd
