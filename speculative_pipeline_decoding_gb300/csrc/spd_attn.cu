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
// Stand-alone launches of decode attention (device code in spd_attn.cuh): prefill blocks, the
// per-operator path used when the step kernel is not, and the stand-alone operators.  Chunks of
// 128 keys; every CTA of the grid takes items blockIdx.x, blockIdx.x + gridDim.x, ...
#include <mutex>

#include "spd_attn.cuh"

namespace spd {

namespace {

struct AttnParams {
  Dims D;
  Bufs B;
  Launch lc;
  int qt;
  int qh_max;
};

template <typename WT>
__global__ void __launch_bounds__(kAttnThreads) attn_kernel(const __grid_constant__ AttnParams p) {
  extern __shared__ __align__(128) unsigned char sm[];
  __shared__ att::Tile tiles[kMaxTiles];
  __shared__ int s_nt, s_items, s_last, s_fail;
  __shared__ __align__(8) uint64_t kv_bar;
  DevState* st = p.B.st;
  if (threadIdx.x == 0) {
    const bool skip = p.lc.kind != LK_EXPLICIT && (st->done || st->err);
    int items = 0;
    const int nt = skip ? 0 : att::add_tiles(p.D, p.B, p.lc, p.qt, kAttnChunk, tiles, 0, &items, kMaxTiles, p.B.st);
    s_nt = nt > 0 ? nt : 0;
    s_items = nt > 0 ? items : 0;
    s_fail = 0;
    mbar_init(&kv_bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();  // q and the K/V appended by the previous kernel are visible from here on
  pdl_trigger();
  if (s_items == 0) return;
  uint32_t phase = 0;
  att::run_items<WT, kAttnChunk>(p.D, st, tiles, s_nt, s_items, blockIdx.x, gridDim.x, p.qh_max, sm, &kv_bar,
                                 phase, &s_fail, &s_last);
}

}  // namespace

size_t attn_smem_bytes(const Dims& D, bool multi) {
  return att::smem_bytes(D.hd, D.gq, D.dtype == SPD_DTYPE_BF16 ? 2 : 4, multi ? kAttnQT : 1, kAttnChunk);
}

size_t attn_part_floats(int rows, int hq, int hd, int max_seq, int ck) {
  const int nch = (max_seq + ck - 1) / ck;
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

// Raise the kernels' dynamic shared-memory limit on the current device to `need` (never lowered by a
// later call).  The limit belongs to one device, so the raised value is kept per device ordinal,
// under a mutex (host threads may make their first calls concurrently).
cudaError_t attn_setup_attributes(size_t need) {
  static std::mutex mu;
  static size_t current[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (dev >= 0 && dev < 64 && need <= current[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(attn_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)need);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(attn_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)need);
  if (e == cudaSuccess && dev >= 0 && dev < 64) current[dev] = need;
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

