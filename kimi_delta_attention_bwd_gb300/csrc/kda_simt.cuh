// CTA-wide fp32-accurate products of the general kernels: M x N outputs of
// sum_k A(m, k) B(k, n), with the operands staged through shared memory in
// KS-wide slabs so that every global read is coalesced and every shared
// read is a broadcast or conflict-free; on the 5th-generation tensor cores
// (split bf16, tcgen05) for the per-chunk kernels, fp32 FMA for the scans.
// Also the blocked inverse of the unit lower chunk factor and an L2 prefetch
// helper.
#pragma once
#include "kda_internal.cuh"
#include "kda_mma.cuh"
#include "kda_tc.cuh"

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

// ---- the per-chunk products on the 5th-generation tensor cores.  Each KS-wide
// slab of both operands is staged as bf16 head and remainder tiles (x = hi +
// lo, hi*hi + hi*lo + lo*hi: the neglected lo*lo term is below 2^-16 of the
// product) in the core-matrix layout of kda_mma.cuh, A with rows m and B with
// rows n (both K-major); one thread issues the slab's tcgen05 MMAs into a TMEM
// accumulator of M = 64 rows and N fp32 columns and commits them to the
// slab buffer's mbarrier.  All of a product's operand loads are issued before
// its first slab is stored.  Two slab buffers; a buffer is restaged once the
// MMAs that read it have completed.
struct Tc5 {
  uint32_t tmem;          // accumulator base: 64 rows, TC5_COLS columns
  uint64_t* bar;          // [2] MMA completion of each slab buffer
  __nv_bfloat16* buf;     // [2][(64 + NMAX) * KS * 2] slab buffers, 128-byte aligned
  int* err;               // set to -7 when a wait on the tensor core runs out
  uint32_t ph[2];         // phase of each buffer's barrier
  bool busy[2];           // MMAs issued on the buffer and not yet waited for
  int next;               // buffer of the next slab
};
constexpr int TC5_COLS = 128;  // N <= 128
// Shared words the slab buffers of products with up to nmax columns take (with
// the slack that aligns them).
constexpr int tc5_slab_floats(int nmax) { return (64 + nmax) * KS * 2 + 32; }
__device__ __forceinline__ __nv_bfloat16* tc5_align(float* p) {
  return reinterpret_cast<__nv_bfloat16*>((reinterpret_cast<uintptr_t>(p) + 127) & ~(uintptr_t)127);
}
__device__ __forceinline__ void tc5_wait(Tc5& t, int bi) {
  if (t.busy[bi]) {
    if (!mma::mbar_wait(&t.bar[bi], t.ph[bi]) && threadIdx.x == 0) atomicExch(t.err, -7);
    t.ph[bi] ^= 1u;
    t.busy[bi] = false;
  }
}
// D (TMEM) = (or +=, when accumulate) sum over k < K of fa(m, k) fb(k, n), M = 64.
// AK / BN: A's k / B's n index is contiguous in memory (pairs of k are read
// together).  Every thread of the CTA must call it; it ends with the MMAs
// complete (tc5_out may read the accumulator) and without a barrier.  The
// operands' writers must be separated from the call by a barrier.
template <int N, int K, int NTH, int NMAX, bool AK, bool BN, class FA, class FB>
__device__ __forceinline__ void cta_tc(Tc5& t, bool accumulate, FA fa, FB fb) {
  constexpr int M = 64, NS = K / KS, QA = M * KS / 2, QB = N * KS / 2;  // bf16 pairs of a slab
  constexpr int PA = (QA + NTH - 1) / NTH, PB = (QB + NTH - 1) / NTH, BUF = (64 + NMAX) * KS * 2;
  static_assert(N % 8 == 0 && N <= NMAX && NMAX <= TC5_COLS && K % KS == 0 && KS % 16 == 0, "product shape");
  auto ia = [](int p, int& m, int& k) {
    if (AK) { m = p / (KS / 2); k = 2 * (p % (KS / 2)); } else { m = p % M; k = 2 * (p / M); }
  };
  auto ib = [](int p, int& n, int& k) {
    if (BN) { n = p % N; k = 2 * (p / N); } else { n = p / (KS / 2); k = 2 * (p % (KS / 2)); }
  };
  // every slab's operands are loaded into registers first, so that the product
  // waits for one memory latency rather than one per slab
  float2 ra[NS][PA], rb[NS][PB];
#pragma unroll
  for (int s = 0; s < NS; s++) {
#pragma unroll
    for (int u = 0; u < PA; u++) {
      const int p = threadIdx.x + u * NTH;
      int m, k;
      ia(p, m, k);
      if (p < QA) ra[s][u] = make_float2(fa(m, s * KS + k), fa(m, s * KS + k + 1));
    }
#pragma unroll
    for (int u = 0; u < PB; u++) {
      const int p = threadIdx.x + u * NTH;
      int n, k;
      ib(p, n, k);
      if (p < QB) rb[s][u] = make_float2(fb(s * KS + k, n), fb(s * KS + k + 1, n));
    }
  }
#pragma unroll
  for (int s = 0; s < NS; s++) {
    const int bi = t.next;
    t.next ^= 1;
    tc5_wait(t, bi);  // the MMAs that last read this buffer are done
    __nv_bfloat16* A = t.buf + bi * BUF;
    __nv_bfloat16* B = A + 2 * M * KS;
    const mma::Op OA{A, A + M * KS, KS}, OB{B, B + N * KS, KS};
#pragma unroll
    for (int u = 0; u < PA; u++) {
      const int p = threadIdx.x + u * NTH;
      int m, k;
      ia(p, m, k);
      if (p < QA) mma::op_store2(OA, m, k, ra[s][u].x, ra[s][u].y);
    }
#pragma unroll
    for (int u = 0; u < PB; u++) {
      const int p = threadIdx.x + u * NTH;
      int n, k;
      ib(p, n, k);
      if (p < QB) mma::op_store2(OB, n, k, rb[s][u].x, rb[s][u].y);
    }
    mma::fence_async_smem();  // the staged tiles are visible to the tensor core
    tc::fence_before();
    __syncthreads();
    if (threadIdx.x == 0) {
      tc::fence_after();
      tc::gemm_split(t.tmem, tc::kmaj(OA), tc::kmaj(OB), N, KS / 16, accumulate || s > 0);
      tc::commit(&t.bar[bi]);
    }
    t.busy[bi] = true;
  }
  tc5_wait(t, 0);
  tc5_wait(t, 1);
  tc::fence_after();
}
// Calls out(m, n, v) for every accumulator element: warp w reads rows
// 16 (w % 4) .. (its TMEM lane quarter) of the 8-column groups w / 4,
// w / 4 + NTH / 128, ...  Ends with the reads complete (the next cta_tc may
// overwrite the accumulator after its barrier).
template <int N, int NTH, class F>
__device__ __forceinline__ void tc5_out(const Tc5& t, F out) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, q = warp & 3, gq = lane >> 2, tq = lane & 3;
  for (int g = warp >> 2; g < N / 8; g += NTH / 128) {
    float v[1][4];
    tc::ld_frag<1>(t.tmem, 8 * g, v);
    const int m0 = 16 * q + gq, n0 = 8 * g + 2 * tq;
    out(m0, n0, v[0][0]);
    out(m0, n0 + 1, v[0][1]);
    out(m0 + 8, n0, v[0][2]);
    out(m0 + 8, n0 + 1, v[0][3]);
  }
  tc::fence_before();
}
// Allocates the accumulator and initialises the barriers (every thread; warp 0
// allocates).  slot / bar: shared memory.
__device__ __forceinline__ Tc5 tc5_setup(uint32_t* slot, uint64_t* bar, float* slab, int* err) {
  if (threadIdx.x < 32) tc::tmem_alloc(slot, TC5_COLS);
  if (threadIdx.x == 0) {
    mma::mbar_init(&bar[0], 1);
    mma::mbar_init(&bar[1], 1);
    mma::mbar_init_fence();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  Tc5 t;
  t.tmem = *slot;
  t.bar = bar;
  t.buf = tc5_align(slab);
  t.err = err;
  t.ph[0] = t.ph[1] = 0u;
  t.busy[0] = t.busy[1] = false;
  t.next = 0;
  return t;
}
// Frees the accumulator (every thread; after the last tc5_out).
__device__ __forceinline__ void tc5_release(const Tc5& t) {
  tc::fence_before();
  __syncthreads();
  if (threadIdx.x < 32) tc::tmem_dealloc(t.tmem, TC5_COLS);
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
