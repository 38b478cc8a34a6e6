// 5th-generation tensor-core (tcgen05) helpers: TMEM allocation, shared-memory
// matrix descriptors for the core-matrix tiles of kda_mma.cuh, split-bf16
// products issued by one thread, and accumulator reads whose register layout
// equals the mma.sync m16n8 accumulator fragment.
//
// Tile layout (kda_mma.cuh Op): 8 x 8 bf16 core matrices of 128 bytes, core
// (rb, cb) of an R x Kc tile at byte (rb * Kc / 8 + cb) * 128.  Used as a
// K-major operand (rows = M or N, columns = K) the descriptor strides are
// LBO = 128 (next core along K) and SBO = Kc / 8 * 128 (next 8-row group);
// used as an MN-major operand (rows = K, columns = M or N) they swap:
// LBO = Kc / 8 * 128, SBO = 128.  An M = 64 accumulator occupies TMEM lanes
// 32 q .. 32 q + 15 for rows 16 q .. 16 q + 15, and the 16x256b load gives
// warp q exactly the m16n8 fragments of those rows.
#pragma once
#include "kda_mma.cuh"

namespace kda {
namespace tc {
using mma::Op;
using mma::smem_u32;

// Warp-wide: allocate `ncols` TMEM columns (a power of two >= 32), address to *slot.
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(smem_u32(slot)), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t base, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(base), "r"(ncols) : "memory");
}
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }

__device__ __forceinline__ uint64_t desc(const void* start, uint32_t lbo, uint32_t sbo) {
  const uint32_t a = smem_u32(start);
  uint64_t d = (uint64_t)((a >> 4) & 0x3FFF);
  d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version; base offset 0, no swizzle
  return d;
}
// Operand view of a tile: rows/columns offset (multiples of 8) and major-ness.
//   K-major: element (mn, k) = X[r0 + mn][c0 + k];  MN-major: element (mn, k) = X[r0 + k][c0 + mn].
struct View {
  const __nv_bfloat16* hi;
  const __nv_bfloat16* lo;  // nullptr: exact in bf16
  int Kc;                   // columns of the stored tile
  int r0, c0;
  bool mn;                  // MN-major
};
__device__ __forceinline__ View kmaj(const Op& t, int r0 = 0, int c0 = 0) { return View{t.hi, t.lo, t.K, r0, c0, false}; }
__device__ __forceinline__ View mnmaj(const Op& t, int r0 = 0, int c0 = 0) { return View{t.hi, t.lo, t.K, r0, c0, true}; }

// Descriptor of K-step ks (16 wide) of a view, for the hi or lo tile.
__device__ __forceinline__ uint64_t vdesc(const View& v, const __nv_bfloat16* base, int ks) {
  const uint32_t rowg = (uint32_t)(v.Kc / 8) * 128u;  // bytes per 8-row group
  if (!v.mn) {
    const char* p = (const char*)base + (v.r0 / 8) * rowg + (v.c0 / 8 + 2 * ks) * 128;
    return desc(p, 128, rowg);
  }
  const char* p = (const char*)base + (v.r0 / 8 + 2 * ks) * rowg + (v.c0 / 8) * 128;
  return desc(p, rowg, 128);
}

__device__ __forceinline__ uint32_t idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
  uint32_t d = 0;
  d |= 1u << 4;   // D f32
  d |= 1u << 7;   // A bf16
  d |= 1u << 10;  // B bf16
  d |= (uint32_t)a_mn << 15;
  d |= (uint32_t)b_mn << 16;
  d |= (uint32_t)(N >> 3) << 17;
  d |= (uint32_t)(M >> 4) << 24;
  return d;
}

__device__ __forceinline__ void mma_issue(uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\ntcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(id), "r"(accumulate)
      : "memory");
}

// Descriptor increment of one K-step (16 columns = two core matrices along
// K) of a view, in the descriptor's 16-byte address units.
__device__ __forceinline__ uint64_t vstep(const View& v) {
  return v.mn ? (uint64_t)(2 * (v.Kc / 8) * 128 / 16) : (uint64_t)(2 * 128 / 16);
}

// D (M = 64 rows, N columns at TMEM address d) = (or +=, when acc) A B over
// ksteps x 16, every operand split into bf16 hi + lo: hi*hi + hi*lo + lo*hi
// (a null lo is exact and skips its product).  One thread issues.  The
// descriptors are built once and stepped along K by adding to their start
// address field (a shared-memory address stays below 2^18 bytes, so the
// 14-bit field never carries).
__device__ __forceinline__ void gemm_split(uint32_t d, const View& A, const View& B, int N, int ksteps, bool acc) {
  const uint32_t id = idesc_bf16(64, N, A.mn, B.mn);
  const uint64_t sa = vstep(A), sb = vstep(B);
  uint64_t ah = vdesc(A, A.hi, 0), bh = vdesc(B, B.hi, 0);
  uint64_t al = A.lo ? vdesc(A, A.lo, 0) : 0, bl = B.lo ? vdesc(B, B.lo, 0) : 0;
  for (int ks = 0; ks < ksteps; ks++) {
    mma_issue(d, ah, bh, id, (acc || ks > 0) ? 1u : 0u);
    if (B.lo) mma_issue(d, ah, bl, id, 1u);
    if (A.lo) mma_issue(d, al, bh, id, 1u);
    ah += sa;
    bh += sb;
    al += sa;
    bl += sb;
  }
}

// Every previously issued MMA of this thread arrives on `bar` when complete.
__device__ __forceinline__ void commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(smem_u32(bar))
               : "memory");
}

// The 16 x 8 NT tile at rows 16 q .. (q = warp % 4), columns c0 .. of an M = 64
// accumulator, as m16n8 fragments v[j] (columns c0 + 8 j ..).
template <int NT>
__device__ __forceinline__ void ld_frag(uint32_t tbase, int c0, float (&v)[NT][4]);
template <>
__device__ __forceinline__ void ld_frag<1>(uint32_t tbase, int c0, float (&v)[1][4]) {
  const uint32_t a = tbase + ((uint32_t)(32 * ((threadIdx.x >> 5) & 3)) << 16) + (uint32_t)c0;
  uint32_t r[4];
  asm volatile("tcgen05.ld.sync.aligned.16x256b.x1.b32 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(a));
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
  for (int e = 0; e < 4; e++) v[0][e] = __uint_as_float(r[e]);
}
template <>
__device__ __forceinline__ void ld_frag<2>(uint32_t tbase, int c0, float (&v)[2][4]) {
  const uint32_t a = tbase + ((uint32_t)(32 * ((threadIdx.x >> 5) & 3)) << 16) + (uint32_t)c0;
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.16x256b.x2.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(a));
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
  for (int j = 0; j < 2; j++)
#pragma unroll
    for (int e = 0; e < 4; e++) v[j][e] = __uint_as_float(r[4 * j + e]);
}
template <>
__device__ __forceinline__ void ld_frag<4>(uint32_t tbase, int c0, float (&v)[4][4]) {
  const uint32_t a = tbase + ((uint32_t)(32 * ((threadIdx.x >> 5) & 3)) << 16) + (uint32_t)c0;
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(a));
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
  for (int j = 0; j < 4; j++)
#pragma unroll
    for (int e = 0; e < 4; e++) v[j][e] = __uint_as_float(r[4 * j + e]);
}

}  // namespace tc
}  // namespace kda
