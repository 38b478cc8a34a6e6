// Warp-level tensor-core helpers (mma.sync m16n8k8, tf32 operands, fp32
// accumulate) and cp.async staging used by the dk=32 / dv=64 kernels.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace kda {
namespace mma {

__device__ __forceinline__ uint32_t tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ void mma_tf32(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// acc[j] (a 16 x 8 tile, j < NT) += sum_k fa(m, k) * fb(k, j, c) for k in
// [0, 8 * ksteps), m < 16, c < 8.  One warp.  Accumulator element e of tile
// j sits at row gq + 8 * (e >> 1), column 2 * tq + (e & 1), where
// gq = lane / 4 and tq = lane % 4.
// SPLIT carries each operand as a tf32 head plus a tf32 remainder and
// accumulates hi*hi + hi*lo + lo*hi (about 21 significant bits).  AX / BX
// declare the A / B operand exactly representable in tf32 (a bf16 input):
// its remainder is zero, so the product with it is skipped.
template <int NT, bool SPLIT = false, bool AX = false, bool BX = false, class FA, class FB>
__device__ __forceinline__ void rows16(float (&acc)[NT][4], int ksteps, FA fa, FB fb) {
  const int lane = threadIdx.x & 31, gq = lane >> 2, tq = lane & 3;
  for (int ks = 0; ks < ksteps; ks++) {
    const int kk = ks * 8 + tq;
    const float fa0 = fa(gq, kk), fa1 = fa(gq + 8, kk), fa2 = fa(gq, kk + 4), fa3 = fa(gq + 8, kk + 4);
    const uint32_t a0 = tf32(fa0), a1 = tf32(fa1), a2 = tf32(fa2), a3 = tf32(fa3);
    uint32_t l0 = 0, l1 = 0, l2 = 0, l3 = 0;
    if (SPLIT && !AX) {
      l0 = tf32(fa0 - __uint_as_float(a0));
      l1 = tf32(fa1 - __uint_as_float(a1));
      l2 = tf32(fa2 - __uint_as_float(a2));
      l3 = tf32(fa3 - __uint_as_float(a3));
    }
#pragma unroll
    for (int j = 0; j < NT; j++) {
      const float fb0 = fb(kk, j, gq), fb1 = fb(kk + 4, j, gq);
      const uint32_t b0 = tf32(fb0), b1 = tf32(fb1);
      mma_tf32(acc[j], a0, a1, a2, a3, b0, b1);
      if (SPLIT && !BX) {
        const uint32_t h0 = tf32(fb0 - __uint_as_float(b0)), h1 = tf32(fb1 - __uint_as_float(b1));
        mma_tf32(acc[j], a0, a1, a2, a3, h0, h1);
      }
      if (SPLIT && !AX) mma_tf32(acc[j], l0, l1, l2, l3, b0, b1);
    }
  }
}

template <int NT>
__device__ __forceinline__ void zero(float (&acc)[NT][4]) {
#pragma unroll
  for (int j = 0; j < NT; j++)
#pragma unroll
    for (int e = 0; e < 4; e++) acc[j][e] = 0.f;
}

// Visits every accumulator element as fn(row < 16, col < 8 * NT, value&).
template <int NT, class F>
__device__ __forceinline__ void each(float (&acc)[NT][4], F fn) {
  const int lane = threadIdx.x & 31, gq = lane >> 2, tq = lane & 3;
#pragma unroll
  for (int j = 0; j < NT; j++)
#pragma unroll
    for (int e = 0; e < 4; e++) fn(gq + 8 * (e >> 1), j * 8 + 2 * tq + (e & 1), acc[j][e]);
}

// ------------------------------------------------------------ cp.async
__device__ __forceinline__ void cp16(void* smem, const void* gmem) {
  uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem));
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::); }
__device__ __forceinline__ void cp_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::); }

}  // namespace mma
}  // namespace kda
