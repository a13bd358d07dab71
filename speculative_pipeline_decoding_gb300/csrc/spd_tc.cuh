// Draft-module tiles on the 5th-generation tensor cores (tcgen05, TMEM accumulators): the device
// layer the GEMV engine would use for groups of several vectors sharing a weight.
//
// Shapes: A = 128 weight rows x K (bf16, K-major, 128-byte swizzle: [chunk][128 rows][128 B] per
// stage of two 64-element chunks, one 3-D TMA copy), B = 32 rows x K: rows 0..15 the bf16 high
// halves of up to 16 activation vectors, rows 16..31 their low halves (x - hi), built by the
// consumer warps per stage.  D = A B^T, fp32 in TMEM: lane = weight row (0..127), column = B row
// (0..31); y[row][v] = D[row][v] + D[row][16 + v].  Gate / up tiles keep two accumulators
// (columns 0..31 and 32..63).
//
// Ownership: consumer warp 0 of the CTA allocates kCols TMEM columns before the first tile and
// frees them after the last (after every warp's last tcgen05.ld).  One elected thread issues the
// MMAs and the commits; completion arrives on mbarriers.
#pragma once
#include <cuda_bf16.h>
#include <stdint.h>

namespace spd {
namespace tc {

constexpr int kRows = 128;     // M: weight rows of a tile
constexpr int kChunk = 64;     // bf16 elements of a 128-byte chunk
constexpr int kStageCh = 2;    // chunks per 32 KB stage
// A tile serves up to NVP vectors (16 or 32): B has 2*NVP rows (NVP high halves, NVP low halves),
// the accumulator 2*NVP TMEM columns (gate / up tiles: two accumulators).
template <int NVP> struct Shape {
  static constexpr int kB = 2 * NVP;                          // N: B rows
  static constexpr int kBBytes = kStageCh * kB * 128;         // B bytes per stage (8 or 16 KB)
  static constexpr uint32_t kAccCols = 2 * NVP;               // TMEM columns of one accumulator
};
constexpr uint32_t kColsStep = 64;    // TMEM columns the step kernel allocates (16 vectors, gate + up)
constexpr uint32_t kColsGemv = 128;   // ... the stand-alone engine (32 vectors, gate + up)

__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// shared-memory matrix descriptor, K-major operand with the 128-byte swizzle: start address >> 4,
// leading byte offset 16 B (unused for this layout), stride byte offset 1024 B (one 8-row group of
// 128-byte rows), descriptor version 1, layout type 2 (128-byte swizzle)
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// instruction descriptor of kind::f16: fp32 D, bf16 A and B, both K-major, N >> 3, M >> 4
__host__ __device__ constexpr uint32_t idesc_bf16(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void alloc_cols(uint32_t* smem_dst, uint32_t ncols) {  // whole warp
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(smem_dst)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void free_cols(uint32_t taddr, uint32_t ncols) {  // whole warp
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// generic-proxy shared-memory writes (the B operand) -> visible to the tensor core
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void mma(uint32_t d_tmem, uint64_t da, uint64_t db, uint32_t id, bool accumulate) {
  asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
               " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
               "l"(da), "l"(db), "r"(id), "r"((uint32_t)accumulate)
               : "memory");
}
// completion of every MMA this thread issued so far arrives once on `bar`
__device__ __forceinline__ void commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(su32(bar))
               : "memory");
}

// One stage: A (kStageCh chunks x 128 rows) at `a`, B (kStageCh chunks x 2*NVP rows) at `b`, both
// 1024-byte aligned; 4 MMAs of K = 16 per chunk, advancing 32 bytes inside the swizzle atom.
template <int NVP>
__device__ __forceinline__ void mma_stage(uint32_t d_tmem, const unsigned char* a, const unsigned char* b,
                                          bool first) {
  constexpr int kB = Shape<NVP>::kB;
  constexpr uint32_t id = idesc_bf16(kRows, kB);
#pragma unroll
  for (int ch = 0; ch < kStageCh; ++ch)
#pragma unroll
    for (int ks = 0; ks < kChunk / 16; ++ks)
      mma(d_tmem, sdesc(su32(a) + ch * kRows * 128 + ks * 32), sdesc(su32(b) + ch * kB * 128 + ks * 32), id,
          !(first && ch == 0 && ks == 0));
}

// The warp's 32 TMEM lanes (rows 32*(warp%4) .. +31), 16 columns, into v[0..15] (fp32 bits).
__device__ __forceinline__ void load_rows16(uint32_t tmem, int warp, uint32_t* v) {
  const uint32_t ta = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(ta));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// The warp's 32 TMEM lanes (rows 32*(warp%4) .. +31), 32 columns, into v[0..31] (fp32 bits).
__device__ __forceinline__ void load_rows(uint32_t tmem, int warp, uint32_t* v) {
  const uint32_t ta = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
        "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
        "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(ta));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

}  // namespace tc
}  // namespace spd
