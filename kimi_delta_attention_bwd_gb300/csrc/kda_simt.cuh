// CTA-wide fp32 products of the general (SIMT) kernels: C x N outputs of
// sum_k A(m, k) B(k, n), with the operands staged through shared memory in
// KS-wide slabs so that every global read is coalesced and every shared
// read is a broadcast or a conflict-free 16-byte load.
#pragma once
#include "kda_internal.cuh"

namespace kda {

constexpr int KS = 32;         // k slab of a staged product
constexpr int APAD = C + 4;    // row stride of the A slab [KS][C]

// Floats of shared memory the two slabs of an N-column product take.
constexpr int mm_slab_floats(int nmax) { return KS * APAD + KS * (nmax + 4); }

// Thread layout of an N-column product on NTH threads: NG = N / 4 column
// groups of four, RPT rows per thread; threads at or past ACT are idle.
template <int N, int NTH>
struct MmShape {
  static constexpr int NG = N / 4;
  static constexpr int ACT = NG * C < NTH ? NG * C : NTH;
  static constexpr int RPT = C * NG / ACT;
  static_assert(N % 4 == 0 && ACT % NG == 0 && (C * NG) % ACT == 0, "product shape");
};

// acc (this thread's RPT x 4 outputs: rows RPT (tid / NG) + q, columns
// 4 (tid % NG) + e) += sum over k < K of fa(m, k) fb(k, n).  AK: A's k index
// is contiguous in memory (else m); BN: B's n index is contiguous (else k);
// these pick the staging order.  as / bs: mm_slab_floats(N) floats of shared
// memory (as first).  Every thread of the CTA must call it; it starts with a
// barrier (the slabs' previous readers, and the operands' writers, are done)
// and ends without one.
template <int N, int K, int NTH, bool AK, bool BN, class FA, class FB>
__device__ __forceinline__ void cta_mm(float (&acc)[MmShape<N, NTH>::RPT][4], float* sm_slab, FA fa, FB fb) {
  using S = MmShape<N, NTH>;
  constexpr int BS = N + 4;
  static_assert(K % KS == 0, "k must be a multiple of the slab");
  float* as = sm_slab;
  float* bs = sm_slab + KS * APAD;
  const int tid = threadIdx.x, ng = tid % S::NG, m0 = (tid / S::NG) * S::RPT;
  for (int k0 = 0; k0 < K; k0 += KS) {
    __syncthreads();
    for (int e = tid; e < C * KS; e += NTH) {
      const int m = AK ? e / KS : e % C, k = AK ? e % KS : e / C;
      as[k * APAD + m] = fa(m, k0 + k);
    }
    for (int e = tid; e < KS * N; e += NTH) {
      const int k = BN ? e / N : e % KS, n = BN ? e % N : e / KS;
      bs[k * BS + n] = fb(k0 + k, n);
    }
    __syncthreads();
    if (tid < S::ACT) {
#pragma unroll 8
      for (int k = 0; k < KS; k++) {
        const float4 b = *reinterpret_cast<const float4*>(bs + k * BS + 4 * ng);
#pragma unroll
        for (int q = 0; q < S::RPT; q++) {
          const float a = as[k * APAD + m0 + q];
          acc[q][0] = fmaf(a, b.x, acc[q][0]);
          acc[q][1] = fmaf(a, b.y, acc[q][1]);
          acc[q][2] = fmaf(a, b.z, acc[q][2]);
          acc[q][3] = fmaf(a, b.w, acc[q][3]);
        }
      }
    }
  }
}

// Calls out(m, n, acc[q][e]) for every output this thread holds.
template <int N, int NTH, class F>
__device__ __forceinline__ void mm_out(const float (&acc)[MmShape<N, NTH>::RPT][4], F out) {
  using S = MmShape<N, NTH>;
  const int tid = threadIdx.x;
  if (tid >= S::ACT) return;
  const int ng = tid % S::NG, m0 = (tid / S::NG) * S::RPT;
#pragma unroll
  for (int q = 0; q < S::RPT; q++)
#pragma unroll
    for (int e = 0; e < 4; e++) out(m0 + q, 4 * ng + e, acc[q][e]);
}

template <int N, int NTH>
__device__ __forceinline__ void mm_zero(float (&acc)[MmShape<N, NTH>::RPT][4]) {
#pragma unroll
  for (int q = 0; q < MmShape<N, NTH>::RPT; q++) acc[q][0] = acc[q][1] = acc[q][2] = acc[q][3] = 0.f;
}

}  // namespace kda
