// CTA-wide fp32-accurate products of the general kernels: M x N outputs of
// sum_k A(m, k) B(k, n), with the operands staged through shared memory in
// KS-wide slabs so that every global read is coalesced and every shared
// read is a broadcast or conflict-free; on the tensor cores (split tf32) for
// the per-chunk kernels, fp32 FMA for the scans.  Also the blocked inverse
// of the unit lower chunk factor and an L2 prefetch helper.
#pragma once
#include "kda_internal.cuh"
#include "kda_mma.cuh"

namespace kda {

constexpr int KS = 32;         // k slab of a staged product
constexpr float LOG2E_S = 1.4426950408889634f;  // the general kernels keep G in log2 units

// Thread layout of an M x N product on NTH threads: NG = N / 4 column groups
// of four, RPT rows per thread; threads at or past ACT are idle.
template <int M, int N, int NTH>
struct MmShape {
  static constexpr int NG = N / 4;
  static constexpr int ACT = NG * M < NTH ? NG * M : NTH;
  static constexpr int RPT = M * NG / ACT;
  static_assert(N % 4 == 0 && ACT % NG == 0 && (M * NG) % ACT == 0, "product shape");
};
template <int M, int N, int NTH>
using MmAcc = float[MmShape<M, N, NTH>::RPT][4];

// acc[q][e] += sum over k < KS of as[k][m0 + q] b(k)[4 ng + e], with b's row
// k at bs + k * ldb (16-byte aligned, ldb a multiple of 4).
template <int M, int N, int NTH>
__device__ __forceinline__ void slab_fma(MmAcc<M, N, NTH>& acc, const float* as, const float* bs, int ldb) {
  using S = MmShape<M, N, NTH>;
  const int tid = threadIdx.x;
  if (tid >= S::ACT) return;
  const int ng = tid % S::NG, m0 = (tid / S::NG) * S::RPT;
#pragma unroll 8
  for (int k = 0; k < KS; k++) {
    const float4 b = *reinterpret_cast<const float4*>(bs + k * ldb + 4 * ng);
#pragma unroll
    for (int q = 0; q < S::RPT; q++) {
      const float a = as[k * (M + 1) + m0 + q];
      acc[q][0] = fmaf(a, b.x, acc[q][0]);
      acc[q][1] = fmaf(a, b.y, acc[q][1]);
      acc[q][2] = fmaf(a, b.z, acc[q][2]);
      acc[q][3] = fmaf(a, b.w, acc[q][3]);
    }
  }
}

// acc (this thread's RPT x 4 outputs: rows RPT (tid / NG) + q, columns
// 4 (tid % NG) + e) += sum over k < K of fa(m, k) b(k, n), with B already in
// shared memory: row k of B at b + k * ldb
// (16-byte aligned, ldb a multiple of 4); only A is staged (slab: at least
// KS (M + 1) floats).  Every A element this thread stages, over all K / KS
// slabs, is loaded into registers first, so that the product waits for one
// memory latency rather than one per slab.
template <int M, int N, int K, int NTH, bool AK, class FA>
__device__ __forceinline__ void cta_mm_sb(MmAcc<M, N, NTH>& acc, float* slab, FA fa, const float* b, int ldb) {
  static_assert(K % KS == 0 && (M * KS) % NTH == 0, "k must be a multiple of the slab, the slab of the threads");
  constexpr int NS = K / KS, PER = M * KS / NTH;
  float pre[NS][PER];
#pragma unroll
  for (int sl = 0; sl < NS; sl++)
#pragma unroll
    for (int u = 0; u < PER; u++) {
      const int e = threadIdx.x + u * NTH;
      const int m = AK ? e / KS : e % M, k = AK ? e % KS : e / M;
      pre[sl][u] = fa(m, sl * KS + k);
    }
#pragma unroll
  for (int sl = 0; sl < NS; sl++) {
    __syncthreads();
#pragma unroll
    for (int u = 0; u < PER; u++) {
      const int e = threadIdx.x + u * NTH;
      const int m = AK ? e / KS : e % M, k = AK ? e % KS : e / M;
      slab[k * (M + 1) + m] = pre[sl][u];
    }
    __syncthreads();
    slab_fma<M, N, NTH>(acc, slab, b + sl * KS * ldb, ldb);
  }
}

// T = (I + A)^-1 for the strictly lower C x C matrix A (row-major), written
// transposed: tt[c * C + r] = T[r][c], zero above the diagonal.  In 16 x 16
// blocks: the four diagonal blocks by forward substitution (one warp each,
// lane = column, the column in registers), then the blocks below them by
// block distance, T_IJ = -T_II sum over K in [J, I) of A_IK T_KJ; each
// thread's sum over k starts at a lane-dependent offset so that the
// transposed reads fall in distinct banks.  x: 768 floats of scratch.  Every
// thread of the CTA calls it (NTH >= 768); A must be visible on entry (a
// barrier after it was written), and the result is on exit.
template <int NTH>
__device__ __forceinline__ void unit_lower_inverse_t(const float* A, float* tt, float* x) {
  static_assert(C == 64 && NTH >= 768, "blocked inverse layout");
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int idx = tid; idx < C * C; idx += NTH) {  // the blocks above the diagonal
    const int c = idx / C, r = idx % C;
    if ((r >> 4) < (c >> 4)) tt[idx] = 0.f;
  }
  if (warp < 4 && lane < 16) {
    const int I = warp, c = lane;
    const float* Ab = A + 16 * I * C + 16 * I;
    float t[16];
#pragma unroll
    for (int r = 0; r < 16; r++) {
      float v = (r == c) ? 1.f : 0.f;
#pragma unroll
      for (int s2 = 0; s2 < r; s2++) v = fmaf(-Ab[r * C + s2], t[s2], v);
      t[r] = v;
    }
#pragma unroll
    for (int r = 0; r < 16; r++) tt[(16 * I + c) * C + 16 * I + r] = t[r];
  }
  __syncthreads();
  for (int dl = 1; dl < 4; dl++) {
    const int nb = 4 - dl, span = 16 * dl;
    const int J = tid >> 8, I = J + dl, r = (tid >> 4) & 15, c = tid & 15;
    if (tid < nb * 256) {  // X_IJ = sum_K A_IK T_KJ
      float v = 0.f;
      for (int kk = 0; kk < span; kk++) {
        const int k = 16 * J + (kk + c) % span;
        v = fmaf(A[(16 * I + r) * C + k], tt[(16 * J + c) * C + k], v);
      }
      x[tid] = v;
    }
    __syncthreads();
    if (tid < nb * 256) {  // T_IJ = -T_II X_IJ
      float v = 0.f;
#pragma unroll
      for (int k = 0; k < 16; k++) v = fmaf(tt[(16 * I + k) * C + 16 * I + r], x[J * 256 + k * 16 + c], v);
      tt[(16 * J + c) * C + 16 * I + r] = -v;
    }
    __syncthreads();
  }
}

// Threads of the CTA prefetch n floats from p into L2 (one request per
// 128-byte line).
template <int NTH>
__device__ __forceinline__ void prefetch_span(const float* p, int n) {
  for (int o = threadIdx.x * 32; o < n; o += NTH * 32) asm volatile("prefetch.global.L2 [%0];" ::"l"(p + o));
}

// ---- the same products on the tensor cores (mma.sync m16n8k8, tf32 operands
// split into a head and a remainder, hi*hi + hi*lo + lo*hi: about 21
// significant bits, the accuracy of the fp32 loop above).  Warp w owns the
// 16 x 8 output tiles w, w + NW, ...; the slabs hold each operand's head and
// remainder with rows padded to 8 (mod 32) words, so that fragment loads
// are conflict-free.
template <int M, int N, int NTH>
struct TcShape {
  static constexpr int NW = NTH / 32, TN = N / 8, T = (M / 16) * TN, TPW = (T + NW - 1) / NW;
  static constexpr int AP = M + 8, BP = N + 8;
  static_assert(M % 16 == 0 && N % 8 == 0 && AP % 32 == 8 && BP % 32 == 8, "tile shape");
};
template <int M, int N, int NTH>
using TcAcc = float[TcShape<M, N, NTH>::TPW][4];

// Words of shared memory the tensor-core slabs of products with up to mmax
// rows and nmax columns take.
constexpr int tc_slab_floats(int mmax, int nmax) { return 2 * KS * (mmax + 8) + 2 * KS * (nmax + 8); }

// Index (k, x) of element e < KS X of a slab: for an operand whose k index
// is contiguous in memory, lanes take 4 consecutive k of 8 consecutive x
// (16-byte global runs, and stores to distinct banks of the 8 (mod 32)
// padded rows); otherwise lanes take consecutive x.
template <int X, bool KC>
__device__ __forceinline__ void slab_index(int e, int& k, int& x) {
  if (KC) {
    const int q = e >> 5, ln = e & 31;
    k = (ln & 3) + 4 * (q % (KS / 4));
    x = (ln >> 2) + 8 * (q / (KS / 4));
  } else {
    k = e / X;
    x = e % X;
  }
}

// acc += sum over k < K of fa(m, k) fb(k, n) on the tensor cores, both
// operands staged; AK / BN: A's k / B's n index is contiguous in memory.
// Slab k0 + KS is loaded into registers while slab k0 is multiplied.  slab:
// tc_slab_floats(M, N) words.  Every thread of the CTA must call it; it
// starts with a barrier (the slab's previous readers, and the operands'
// writers, are done) and ends without one.
template <int M, int N, int K, int NTH, bool AK, bool BN, class FA, class FB>
__device__ __forceinline__ void cta_mma(TcAcc<M, N, NTH>& acc, float* slab, FA fa, FB fb) {
  using S = TcShape<M, N, NTH>;
  static_assert(K % KS == 0 && (M * KS) % NTH == 0 && (N * KS) % NTH == 0, "k a multiple of the slab, slabs of the threads");
  static_assert(!AK || M % 8 == 0, "row groups");
  constexpr int PA = M * KS / NTH, PB = N * KS / NTH;
  uint32_t* ah = reinterpret_cast<uint32_t*>(slab);
  uint32_t* al = ah + KS * S::AP;
  uint32_t* bh = al + KS * S::AP;
  uint32_t* bl = bh + KS * S::BP;
  float ra[PA], rb[PB];
  auto load = [&](int k0) {
#pragma unroll
    for (int u = 0; u < PA; u++) {
      int k, m;
      slab_index<M, AK>(threadIdx.x + u * NTH, k, m);
      ra[u] = fa(m, k0 + k);
    }
#pragma unroll
    for (int u = 0; u < PB; u++) {
      int k, n;
      slab_index<N, !BN>(threadIdx.x + u * NTH, k, n);
      rb[u] = fb(k0 + k, n);
    }
  };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  load(0);
  for (int k0 = 0; k0 < K; k0 += KS) {
    __syncthreads();
#pragma unroll
    for (int u = 0; u < PA; u++) {
      int k, m;
      slab_index<M, AK>(threadIdx.x + u * NTH, k, m);
      mma::split_tf32(ra[u], ah[k * S::AP + m], al[k * S::AP + m]);
    }
#pragma unroll
    for (int u = 0; u < PB; u++) {
      int k, n;
      slab_index<N, !BN>(threadIdx.x + u * NTH, k, n);
      mma::split_tf32(rb[u], bh[k * S::BP + n], bl[k * S::BP + n]);
    }
    __syncthreads();
    if (k0 + KS < K) load(k0 + KS);
#pragma unroll
    for (int k8 = 0; k8 < KS; k8 += 8) {
#pragma unroll
      for (int j = 0; j < S::TPW; j++) {
        const int tile = warp + j * S::NW;
        if (tile < S::T) {
          const int m0 = 16 * (tile / S::TN) + g, n0 = 8 * (tile % S::TN) + g;
          const int r0 = (k8 + t) * S::AP + m0, r1 = r0 + 4 * S::AP;
          const int c0 = (k8 + t) * S::BP + n0, c1 = c0 + 4 * S::BP;
          const uint32_t a0 = ah[r0], a1 = ah[r0 + 8], a2 = ah[r1], a3 = ah[r1 + 8];
          const uint32_t b0 = bh[c0], b1 = bh[c1];
          mma::mma_tf32(acc[j], a0, a1, a2, a3, b0, b1);
          mma::mma_tf32(acc[j], a0, a1, a2, a3, bl[c0], bl[c1]);
          mma::mma_tf32(acc[j], al[r0], al[r0 + 8], al[r1], al[r1 + 8], b0, b1);
        }
      }
    }
  }
}

// Calls out(m, n, v) for every output of the warp's tiles held by this lane.
template <int M, int N, int NTH, class F>
__device__ __forceinline__ void tc_out(const TcAcc<M, N, NTH>& acc, F out) {
  using S = TcShape<M, N, NTH>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int j = 0; j < S::TPW; j++) {
    const int tile = warp + j * S::NW;
    if (tile < S::T) {
      const int m0 = 16 * (tile / S::TN) + g, n0 = 8 * (tile % S::TN) + 2 * t;
      out(m0, n0, acc[j][0]);
      out(m0, n0 + 1, acc[j][1]);
      out(m0 + 8, n0, acc[j][2]);
      out(m0 + 8, n0 + 1, acc[j][3]);
    }
  }
}

template <int M, int N, int NTH>
__device__ __forceinline__ void tc_zero(TcAcc<M, N, NTH>& acc) {
#pragma unroll
  for (int j = 0; j < TcShape<M, N, NTH>::TPW; j++) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
}

// Calls out(m, n, acc[q][e]) for every output this thread holds.
template <int M, int N, int NTH, class F>
__device__ __forceinline__ void mm_out(const MmAcc<M, N, NTH>& acc, F out) {
  using S = MmShape<M, N, NTH>;
  const int tid = threadIdx.x;
  if (tid >= S::ACT) return;
  const int ng = tid % S::NG, m0 = (tid / S::NG) * S::RPT;
#pragma unroll
  for (int q = 0; q < S::RPT; q++)
#pragma unroll
    for (int e = 0; e < 4; e++) out(m0 + q, 4 * ng + e, acc[q][e]);
}

template <int M, int N, int NTH>
__device__ __forceinline__ void mm_zero(MmAcc<M, N, NTH>& acc) {
#pragma unroll
  for (int q = 0; q < MmShape<M, N, NTH>::RPT; q++) acc[q][0] = acc[q][1] = acc[q][2] = acc[q][3] = 0.f;
}

}  // namespace kda
