// Warp-level tensor-core helpers (mma.sync: tf32 m16n8k8 and bf16 m16n8k16,
// fp32 accumulate), split-operand tiles and cp.async staging used by the
// dk=32 / dv=64 kernels.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>
#include <cuda_bf16.h>

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

// Split-tf32 helpers of the pairwise decay terms (3 products each, ~21 bits).
__device__ __forceinline__ void split_tf32(float x, uint32_t& hi, uint32_t& lo) {
  hi = tf32(x);
  lo = tf32(x - __uint_as_float(hi));
}

// acc1 += A1 B and acc2 += A2 B (16 x 8 NT tiles over K = 8 ksteps): two A
// operands share each B fragment.  fb(k, j, n) gives B(k, 8 j + n).
template <int NT, class FA1, class FA2, class FB>
__device__ __forceinline__ void rows16_2a(float (&acc1)[NT][4], float (&acc2)[NT][4], int ksteps, FA1 fa1, FA2 fa2,
                                          FB fb) {
  const int lane = threadIdx.x & 31, gq = lane >> 2, tq = lane & 3;
  for (int ks = 0; ks < ksteps; ks++) {
    const int kk = ks * 8 + tq;
    uint32_t a[4], al[4], c[4], cl[4];
    split_tf32(fa1(gq, kk), a[0], al[0]);
    split_tf32(fa1(gq + 8, kk), a[1], al[1]);
    split_tf32(fa1(gq, kk + 4), a[2], al[2]);
    split_tf32(fa1(gq + 8, kk + 4), a[3], al[3]);
    split_tf32(fa2(gq, kk), c[0], cl[0]);
    split_tf32(fa2(gq + 8, kk), c[1], cl[1]);
    split_tf32(fa2(gq, kk + 4), c[2], cl[2]);
    split_tf32(fa2(gq + 8, kk + 4), c[3], cl[3]);
#pragma unroll
    for (int j = 0; j < NT; j++) {
      uint32_t b0, b0l, b1, b1l;
      split_tf32(fb(kk, j, gq), b0, b0l);
      split_tf32(fb(kk + 4, j, gq), b1, b1l);
      mma_tf32(acc1[j], a[0], a[1], a[2], a[3], b0, b1);
      mma_tf32(acc1[j], a[0], a[1], a[2], a[3], b0l, b1l);
      mma_tf32(acc1[j], al[0], al[1], al[2], al[3], b0, b1);
      mma_tf32(acc2[j], c[0], c[1], c[2], c[3], b0, b1);
      mma_tf32(acc2[j], c[0], c[1], c[2], c[3], b0l, b1l);
      mma_tf32(acc2[j], cl[0], cl[1], cl[2], cl[3], b0, b1);
    }
  }
}

// acc += A1 B1 + A2 B2 (16 x 8 NT tiles over K = 8 ksteps); fb(k, j, n)
// returns the pair (B1(k, 8 j + n), B2(k, 8 j + n)).
template <int NT, class FA1, class FA2, class FB>
__device__ __forceinline__ void rows16_ab(float (&acc)[NT][4], int ksteps, FA1 fa1, FA2 fa2, FB fb) {
  const int lane = threadIdx.x & 31, gq = lane >> 2, tq = lane & 3;
  for (int ks = 0; ks < ksteps; ks++) {
    const int kk = ks * 8 + tq;
    uint32_t a[4], al[4], c[4], cl[4];
    split_tf32(fa1(gq, kk), a[0], al[0]);
    split_tf32(fa1(gq + 8, kk), a[1], al[1]);
    split_tf32(fa1(gq, kk + 4), a[2], al[2]);
    split_tf32(fa1(gq + 8, kk + 4), a[3], al[3]);
    split_tf32(fa2(gq, kk), c[0], cl[0]);
    split_tf32(fa2(gq + 8, kk), c[1], cl[1]);
    split_tf32(fa2(gq, kk + 4), c[2], cl[2]);
    split_tf32(fa2(gq + 8, kk + 4), c[3], cl[3]);
#pragma unroll
    for (int j = 0; j < NT; j++) {
      const float2 v0 = fb(kk, j, gq), v1 = fb(kk + 4, j, gq);
      uint32_t b0, b0l, b1, b1l, d0, d0l, d1, d1l;
      split_tf32(v0.x, b0, b0l);
      split_tf32(v1.x, b1, b1l);
      split_tf32(v0.y, d0, d0l);
      split_tf32(v1.y, d1, d1l);
      mma_tf32(acc[j], a[0], a[1], a[2], a[3], b0, b1);
      mma_tf32(acc[j], a[0], a[1], a[2], a[3], b0l, b1l);
      mma_tf32(acc[j], al[0], al[1], al[2], al[3], b0, b1);
      mma_tf32(acc[j], c[0], c[1], c[2], c[3], d0, d1);
      mma_tf32(acc[j], c[0], c[1], c[2], c[3], d0l, d1l);
      mma_tf32(acc[j], cl[0], cl[1], cl[2], cl[3], d0, d1);
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

// ------------------------------------------------------------ bf16 split operands
// An operand tile of R rows x K columns (K a multiple of 8) kept as two bf16
// arrays, hi = RN(x) and lo = RN(x - hi), in the canonical K-major core-matrix
// layout: 8 rows x 8 elements per 128-byte core matrix, core (rb, kb) at
// index rb * (K / 8) + kb.  The same storage serves an operand and its
// transpose (ldmatrix with and without .trans).  lo == nullptr marks a tile
// whose values are exact in bf16 (its remainder is zero).
struct Op {
  __nv_bfloat16* hi;
  __nv_bfloat16* lo;
  int K;
};

__device__ __forceinline__ int opix(int r, int k, int K) {
  return ((((r >> 3) * (K >> 3)) + (k >> 3)) << 6) + ((r & 7) << 3) + (k & 7);
}

__device__ __forceinline__ void op_store2(const Op& o, int r, int k, float x0, float x1) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  const float2 hf = __bfloat1622float2(h);
  const int i = opix(r, k, o.K);
  *reinterpret_cast<__nv_bfloat162*>(o.hi + i) = h;
  if (o.lo) *reinterpret_cast<__nv_bfloat162*>(o.lo + i) = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
}

__device__ __forceinline__ void op_store1(const Op& o, int r, int k, float x) {
  const __nv_bfloat16 h = __float2bfloat16_rn(x);
  const int i = opix(r, k, o.K);
  o.hi[i] = h;
  if (o.lo) o.lo[i] = __float2bfloat16_rn(x - __bfloat162float(h));
}

__device__ __forceinline__ float op_get(const Op& o, int r, int k) {
  const int i = opix(r, k, o.K);
  return __bfloat162float(o.hi[i]) + (o.lo ? __bfloat162float(o.lo[i]) : 0.f);
}

__device__ __forceinline__ void ldsm4(uint32_t (&r)[4], const void* p) {
  const uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(a));
}
__device__ __forceinline__ void ldsm4t(uint32_t (&r)[4], const void* p) {
  const uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(a));
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// A fragment (16 x 16) at logical A(m0.., k0..).  AT: A(m, k) = X[k][m].
template <bool AT>
__device__ __forceinline__ void frag_a(uint32_t (&r)[4], const __nv_bfloat16* X, int K, int m0, int k0) {
  const int lane = threadIdx.x & 31, mi = lane >> 3, l7 = lane & 7;
  if (!AT) ldsm4(r, X + opix(m0 + l7 + 8 * (mi & 1), k0 + 8 * (mi >> 1), K));
  else ldsm4t(r, X + opix(k0 + l7 + 8 * (mi >> 1), m0 + 8 * (mi & 1), K));
}

// B fragments (16 x 16: two n8 tiles) at logical B(k0.., n0..).  BT: B(k, n) = X[k][n],
// else B(k, n) = X[n][k].  r[0..1] feed tile n0, r[2..3] tile n0 + 8.
template <bool BT>
__device__ __forceinline__ void frag_b(uint32_t (&r)[4], const __nv_bfloat16* X, int K, int k0, int n0) {
  const int lane = threadIdx.x & 31, mi = lane >> 3, l7 = lane & 7;
  if (!BT) ldsm4(r, X + opix(n0 + l7 + 8 * (mi >> 1), k0 + 8 * (mi & 1), K));
  else ldsm4t(r, X + opix(k0 + l7 + 8 * (mi & 1), n0 + 8 * (mi >> 1), K));
}

// acc[2p + t] (16 x 8 tiles, columns n0 + 16 p + 8 t) += A(m0.., k) B(k, n0..)
// over ksteps blocks of 16 along k (A from ka0, B from kb0), with each
// operand split into bf16 hi + lo and hi*hi + hi*lo + lo*hi accumulated
// (about 16 significant bits).  An operand whose lo is null is exact.
template <int NP, bool AT, bool BT>
__device__ __forceinline__ void gemm3(float (&acc)[2 * NP][4], const Op& A, int m0, int ka0, const Op& B, int n0,
                                      int kb0, int ksteps) {
  for (int ks = 0; ks < ksteps; ks++) {
    uint32_t ah[4], al[4], bh[NP][4], bl[NP][4];
    frag_a<AT>(ah, A.hi, A.K, m0, ka0 + 16 * ks);
    if (A.lo) frag_a<AT>(al, A.lo, A.K, m0, ka0 + 16 * ks);
#pragma unroll
    for (int p = 0; p < NP; p++) {
      frag_b<BT>(bh[p], B.hi, B.K, kb0 + 16 * ks, n0 + 16 * p);
      if (B.lo) frag_b<BT>(bl[p], B.lo, B.K, kb0 + 16 * ks, n0 + 16 * p);
    }
    // consecutive products go to different accumulators
#pragma unroll
    for (int p = 0; p < NP; p++) {
      mma_bf16(acc[2 * p], ah, bh[p][0], bh[p][1]);
      mma_bf16(acc[2 * p + 1], ah, bh[p][2], bh[p][3]);
    }
    if (B.lo) {
#pragma unroll
      for (int p = 0; p < NP; p++) {
        mma_bf16(acc[2 * p], ah, bl[p][0], bl[p][1]);
        mma_bf16(acc[2 * p + 1], ah, bl[p][2], bl[p][3]);
      }
    }
    if (A.lo) {
#pragma unroll
      for (int p = 0; p < NP; p++) {
        mma_bf16(acc[2 * p], al, bh[p][0], bh[p][1]);
        mma_bf16(acc[2 * p + 1], al, bh[p][2], bh[p][3]);
      }
    }
  }
}

// ------------------------------------------------------------ cp.async
__device__ __forceinline__ void cp16(void* smem, const void* gmem) {
  uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem));
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::); }
__device__ __forceinline__ void cp_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::); }


// ------------------------------------------------------------ bulk copies
// One-instruction copies of contiguous tiles between global and shared memory
// (cp.async.bulk, the Tensor Memory Accelerator's 1-D form).  Loads complete
// on an mbarrier; stores are tracked by bulk groups.  Addresses and sizes are
// multiples of 16 bytes.
__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_init_fence() { asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory"); }
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ uint32_t mbar_try(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done;
}
// Bound of every wait on an mbarrier: a phase that has not completed after
// WAIT_POLLS polls (each try_wait may suspend the thread briefly) never will,
// so the wait gives up and the kernel flags the error.  A bound on the global
// clock instead measured 1 to 2% slower on the per-chunk kernels, which wait
// several times per CTA.
constexpr int WAIT_POLLS = 1 << 18;  // about 1 s: a failed poll suspends the thread about 4 us (measured)
// Polls phase `parity` of the barrier; returns false after WAIT_POLLS polls
// (the caller flags the error).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done = 0;
  for (int it = 0; it < WAIT_POLLS && !done; it++) done = mbar_try(bar, parity);
  return done != 0;
}
__device__ __forceinline__ void bulk_s2g(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;\n" ::"l"(dst), "r"(smem_u32(src)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;\n" ::: "memory"); }
// The shared-memory sources of every committed bulk store have been read.
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory"); }
// L2 prefetches: the 128-byte line holding p, and a contiguous region (bulk).
__device__ __forceinline__ void prefetch_l2(const void* p) { asm volatile("prefetch.global.L2 [%0];\n" ::"l"(p)); }
__device__ __forceinline__ void bulk_prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(p), "r"(bytes) : "memory");
}
// A 2-D tile of a tensor map (TMA, cp.async.bulk.tensor) into shared memory,
// completing on an mbarrier: box element (x0 + i, y0 + j) of the map lands at
// dst + (j * box_x + i) elements.  x0 times the element size must be a multiple
// of 16 bytes; coordinates past the tensor read as zero.
__device__ __forceinline__ void tma_load_2d(void* dst, const void* map, int x0, int y0, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n" ::"r"(
          smem_u32(dst)),
      "l"(map), "r"(x0), "r"(y0), "r"(smem_u32(bar))
      : "memory");
}
// Orders this thread's generic-proxy shared-memory accesses before later bulk copies.
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }

// ------------------------------------------------------------ thread-block clusters
// Distributed shared memory between the CTAs of a cluster: an address of this
// CTA's shared memory mapped to the same variable in CTA `rank` of the
// cluster, asynchronous remote stores that signal the peer's mbarrier, and the
// cluster-wide barrier.  A CTA must not exit while a peer may still access
// its shared memory: kernels that exchange end with cluster_sync().
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_map(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
// Asynchronous store of two floats into a peer CTA's shared memory that
// completes 8 bytes of the transaction count of the peer's mbarrier `bar_addr`
// when the data has landed: the receiver's barrier phase (armed with
// mbar_expect_tx for the bytes it expects) completes with the data visible,
// and the sender needs no release fence.  (A release-ordered remote arrival
// would first wait for every global store the sending thread still has in
// flight, about a microsecond under load.)
__device__ __forceinline__ void st_async_f32x2(uint32_t addr, float a, float b, uint32_t bar_addr) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];\n" ::"r"(addr),
               "f"(a), "f"(b), "r"(bar_addr)
               : "memory");
}
// mbar_wait with acquire at cluster scope, for phases completed by a peer
// CTA's asynchronous stores.  Bounded like mbar_wait.
__device__ __forceinline__ uint32_t mbar_try_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n.reg .pred p;\nmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, "
      "p;\n}\n"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done;
}
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t done = 0;
  for (int it = 0; it < WAIT_POLLS && !done; it++) done = mbar_try_cluster(bar, parity);
  return done != 0;
}
// Every thread of every CTA of the cluster (warp-convergent).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}

}  // namespace mma
}  // namespace kda
