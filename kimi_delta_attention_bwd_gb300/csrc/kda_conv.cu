// Varlen short causal depthwise convolution (kernel 4) with SiLU, the step
// before the KDA path on the concatenated q | k | v channels ("Pure KDA 300M"
// guide, Overview: short-conv kernel size 4, depthwise on the concatenated QKV;
// the guide's troubleshooting uses FLA's causal_conv1d on [B, T, D] directly;
// torchtitan PR "[kimi k3] Support sample packing in KDA": per-document reset):
//   z_t = sum_j w_j x_{t-3+j}   (x before the document start is 0),   y_t = silu(z_t)
// and its backward dz = dy silu'(z), dx_t = sum_j w_j dz_{t+3-j} (same document),
// dw_j = sum_t dz_t x_{t-3+j}.  Token-major [Ntok, C] rows stream through once;
// a thread owns 16 bytes of channels over a run of tokens and slides its
// window in registers.
#include "kda_internal.cuh"
#include "kda_mma.cuh"
#include "../../include/kda.h"

namespace kda {
namespace {
using mma::bulk_g2s;
using mma::mbar_expect_tx;
using mma::mbar_init;
using mma::mbar_init_fence;
using mma::mbar_wait;

constexpr int KW = 4;     // kernel width
constexpr int TBF = 16;   // tokens per thread, forward (more warps in flight; halo reads hit L2)
constexpr int TBB = 64;   // tokens per thread, backward (fewer weight-gradient partials)
constexpr int CTHR = 128;

template <typename T>
struct V16 {
  static constexpr int N = 16 / sizeof(T);
};
__device__ __forceinline__ void vld(const float* p, float (&v)[4]) {
  const float4 f = __ldg(reinterpret_cast<const float4*>(p));
  v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
}
__device__ __forceinline__ void vst(__nv_bfloat16* p, const float (&v)[8]) {
  uint4 u;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
  for (int e = 0; e < 4; e++) h[e] = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
  *reinterpret_cast<uint4*>(p) = u;
}
__device__ __forceinline__ void vst(float* p, const float (&v)[4]) {
  *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
}
// 8-byte variants (four bf16 channels) for the backward, whose per-thread state
// (taps, weight-gradient sums, two windows) grows with the channel count.
__device__ __forceinline__ void vld(const __nv_bfloat16* p, float (&v)[4]) {
  const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
}
__device__ __forceinline__ void vst(__nv_bfloat16* p, const float (&v)[4]) {
  uint2 u;
  *reinterpret_cast<__nv_bfloat162*>(&u.x) = __floats2bfloat162_rn(v[0], v[1]);
  *reinterpret_cast<__nv_bfloat162*>(&u.y) = __floats2bfloat162_rn(v[2], v[3]);
  *reinterpret_cast<uint2*>(p) = u;
}

// Raw loads (16 or 8 bytes) and their unpacking: a thread loads a batch of
// rows before it uses any, so its loads are in flight together.
__device__ __forceinline__ uint4 raw16(const void* p) { return __ldg(reinterpret_cast<const uint4*>(p)); }
__device__ __forceinline__ uint2 raw8(const void* p) { return __ldg(reinterpret_cast<const uint2*>(p)); }
__device__ __forceinline__ void unpack(const uint4& u, float (&v)[8]) {  // 8 bf16
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int e = 0; e < 4; e++) {
    const float2 f = __bfloat1622float2(h[e]);
    v[2 * e] = f.x;
    v[2 * e + 1] = f.y;
  }
}
__device__ __forceinline__ void unpack(const uint4& u, float (&v)[4]) {  // 4 fp32
  v[0] = __uint_as_float(u.x); v[1] = __uint_as_float(u.y); v[2] = __uint_as_float(u.z); v[3] = __uint_as_float(u.w);
}
__device__ __forceinline__ void unpack(const uint2& u, float (&v)[4]) {  // 4 bf16
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
}
template <typename T> struct Raw4;  // the raw type of 4 channels
template <> struct Raw4<__nv_bfloat16> {
  using type = uint2;
  static __device__ __forceinline__ uint2 ld(const __nv_bfloat16* p) { return raw8(p); }
};
template <> struct Raw4<float> {
  using type = uint4;
  static __device__ __forceinline__ uint4 ld(const float* p) { return raw16(p); }
};
constexpr int LB = 4;  // rows per load batch

// Document of token t: the largest d < n_docs with cu[d] <= t (cu non-decreasing
// from 0; without cu, rows of row_len tokens).  Returns its start, and its end
// in *end.
__device__ __forceinline__ int64_t doc_of(const int32_t* cu, int n_docs, int64_t n_tok, int64_t t, int& d,
                                          int64_t& end, int64_t row_len) {
  if (!cu) {
    d = (int)(t / row_len);
    const int64_t st = (int64_t)d * row_len;
    end = st + row_len < n_tok ? st + row_len : n_tok;
    return st;
  }
  int lo = 0, hi = n_docs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cu[mid] <= t) lo = mid;
    else hi = mid - 1;
  }
  d = lo;
  end = d + 1 <= n_docs ? cu[d + 1] : n_tok;
  return cu[d];
}
// Advance (d, start, end) to the document of token t >= end.
__device__ __forceinline__ void next_doc(const int32_t* cu, int n_docs, int64_t n_tok, int64_t t, int& d,
                                         int64_t& start, int64_t& end, int64_t row_len) {
  if (!cu) {
    start = doc_of(cu, n_docs, n_tok, t, d, end, row_len);
    return;
  }
  while (d + 1 < n_docs && cu[d + 1] <= t) d++;
  start = cu[d];
  end = d + 1 <= n_docs ? cu[d + 1] : n_tok;
}

__device__ __forceinline__ float silu(float z) { return z * sigmoid_fast(z); }
__device__ __forceinline__ float dsilu(float z) {
  const float s = sigmoid_fast(z);
  return s * (1.0f + z * (1.0f - s));
}

// Forward.  A CTA covers TBF tokens x (CTHR x 16 bytes) of channels: its input
// rows t0 - 3 .. t1 - 1 are copied into shared memory first, one 1-D bulk copy
// per row (all in flight together, completion on an mbarrier), then each
// thread slides its window down its 16-byte column.  Should the bounded wait
// run out, the thread reads its rows from global memory instead.
template <typename T>
__global__ void __launch_bounds__(CTHR) conv_fwd_kernel(int64_t n_tok, int C, int act, const int32_t* __restrict__ cu,
                                                       int n_docs, const T* __restrict__ x,
                                                       const float* __restrict__ w, T* __restrict__ y) {
  constexpr int N = V16<T>::N;
  extern __shared__ __align__(16) unsigned char csm[];  // (TBF + KW - 1) rows x CTHR x 16 bytes, then the barrier
  uint64_t* bar = reinterpret_cast<uint64_t*>(csm + (TBF + KW - 1) * CTHR * 16);
  const int cblk = blockIdx.x * CTHR * N, cw = min(CTHR * N, C - cblk);  // the CTA's channels
  const int64_t t0 = (int64_t)blockIdx.y * TBF, t1 = t0 + TBF < n_tok ? t0 + TBF : n_tok;
  const int64_t rb = t0 - (KW - 1), r0 = rb > 0 ? rb : 0;  // row slot of token p: p - rb
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    mbar_init_fence();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    mbar_expect_tx(bar, (uint32_t)((t1 - r0) * cw * sizeof(T)));
    for (int64_t p = r0; p < t1; p++)
      bulk_g2s(csm + (p - rb) * CTHR * 16, x + p * C + cblk, (uint32_t)(cw * sizeof(T)), bar);
  }
  const int cv = threadIdx.x, c0 = cblk + cv * N;
  const bool active = cv * N < cw;
  float wv[N][KW];
#pragma unroll
  for (int e = 0; e < N; e++) {  // the thread's N x 4 taps are contiguous
    float4 t4 = make_float4(0.f, 0.f, 0.f, 0.f);
    if (active) t4 = __ldg(reinterpret_cast<const float4*>(w + (c0 + e) * KW));
    wv[e][0] = t4.x; wv[e][1] = t4.y; wv[e][2] = t4.z; wv[e][3] = t4.w;
  }
  int d;
  int64_t end;
  int64_t start = doc_of(cu, n_docs, n_tok, t0, d, end, n_tok);
  const bool staged = mbar_wait(bar, 0);
  auto row = [&](int64_t p) -> uint4 {  // this thread's 16 bytes of token p
    return staged ? *reinterpret_cast<const uint4*>(csm + (p - rb) * CTHR * 16 + cv * 16) : raw16(x + p * C + c0);
  };
  if (active) {
    float win[KW - 1][N];  // x_{t-3}, x_{t-2}, x_{t-1}
#pragma unroll
    for (int k = 0; k < KW - 1; k++) {
      const int64_t p = rb + k;
      if (p >= start && p >= 0) unpack(row(p), win[k]);
      else {
#pragma unroll
        for (int e = 0; e < N; e++) win[k][e] = 0.f;
      }
    }
    for (int64_t t = t0; t < t1; t++) {
      if (t >= end) {  // a new document: the window restarts from zero
        next_doc(cu, n_docs, n_tok, t, d, start, end, n_tok);
#pragma unroll
        for (int k2 = 0; k2 < KW - 1; k2++)
#pragma unroll
          for (int e = 0; e < N; e++) win[k2][e] = 0.f;
      }
      float xt[N], out[N];
      unpack(row(t), xt);
#pragma unroll
      for (int e = 0; e < N; e++) {
        const float z = wv[e][0] * win[0][e] + wv[e][1] * win[1][e] + wv[e][2] * win[2][e] + wv[e][3] * xt[e];
        out[e] = act ? silu(z) : z;
        win[0][e] = win[1][e];
        win[1][e] = win[2][e];
        win[2][e] = xt[e];
      }
      vst(y + t * C + c0, out);
    }
  }
  if (!staged) mbar_wait(bar, 0);  // the copies land before the CTA's shared memory is released
}

// Backward.  At step u the thread forms dz_u (from x_{u-3..u}) and emits
// dx_{u-3} from dz_{u-3..u}; a token's document start is kept for the last
// four positions so that no window reaches across a document boundary.
constexpr int NB = 4;  // channels per thread in the backward

// T: the type of x and dx; TY: the type of dy (the fused KDA backward hands
// over fp32 gradients).  Without cu, documents are rows of row_len tokens.
template <typename T, typename TY = T>
__global__ void __launch_bounds__(CTHR) conv_bwd_kernel(int64_t n_tok, int C, int act, const int32_t* __restrict__ cu,
                                                       int n_docs, int64_t row_len, const T* __restrict__ x,
                                                       const float* __restrict__ w, const TY* __restrict__ dy,
                                                       T* __restrict__ dx, float* __restrict__ part) {
  constexpr int N = NB;
  const int cv = blockIdx.x * CTHR + threadIdx.x;
  if (cv >= C / N) return;
  const int c0 = cv * N;
  const int64_t t0 = (int64_t)blockIdx.y * TBB, t1 = t0 + TBB < n_tok ? t0 + TBB : n_tok;
  float wv[N][KW], dwa[N][KW];
#pragma unroll
  for (int e = 0; e < N; e++) {
    const float4 t4 = __ldg(reinterpret_cast<const float4*>(w + (c0 + e) * KW));
    wv[e][0] = t4.x; wv[e][1] = t4.y; wv[e][2] = t4.z; wv[e][3] = t4.w;
#pragma unroll
    for (int j = 0; j < KW; j++) dwa[e][j] = 0.f;
  }
  int d;
  int64_t end;
  int64_t start = doc_of(cu, n_docs, n_tok, t0, d, end, row_len);
  float xw[KW - 1][N];  // x_{u-3..u-1}
  float dzw[KW - 1][N];  // dz_{u-3..u-1}
  int64_t dsw[KW];       // document starts of u-3 .. u
#pragma unroll
  for (int k = 0; k < KW - 1; k++) {
    const int64_t p = t0 - (KW - 1) + k;
    if (p >= start && p >= 0) vld(x + p * C + c0, xw[k]);
    else {
#pragma unroll
      for (int e = 0; e < N; e++) xw[k][e] = 0.f;
    }
#pragma unroll
    for (int e = 0; e < N; e++) dzw[k][e] = 0.f;
    dsw[k] = start;  // positions before t0 only pair with dz of tokens >= t0 through dx_{< t0}: never emitted
  }
  using R = typename Raw4<T>::type;
  using RY = typename Raw4<TY>::type;
  const int64_t u1 = t1 + (KW - 1);  // dx of the last token needs dz up to t1 + 2
  for (int64_t ub = t0; ub < u1; ub += LB) {
  R rx[LB];  // the batch's rows of x and dy, loaded before any is used
  RY rdy[LB];
#pragma unroll
  for (int k = 0; k < LB; k++) {
    rx[k] = R{};
    rdy[k] = RY{};
    if (ub + k < u1 && ub + k < n_tok) {
      rx[k] = Raw4<T>::ld(x + (ub + k) * C + c0);
      rdy[k] = Raw4<TY>::ld(dy + (ub + k) * C + c0);
    }
  }
#pragma unroll
  for (int kb = 0; kb < LB; kb++) {
    const int64_t u = ub + kb;
    if (u >= u1) break;
    float dzu[N];
    const bool live = u < n_tok;
    if (live) {
      if (u >= end) {
        next_doc(cu, n_docs, n_tok, u, d, start, end, row_len);
#pragma unroll
        for (int k = 0; k < KW - 1; k++)
#pragma unroll
          for (int e = 0; e < N; e++) xw[k][e] = 0.f;
      }
      float xu[N], dyu[N];
      unpack(rx[kb], xu);
      unpack(rdy[kb], dyu);
#pragma unroll
      for (int e = 0; e < N; e++) {
        const float z = wv[e][0] * xw[0][e] + wv[e][1] * xw[1][e] + wv[e][2] * xw[2][e] + wv[e][3] * xu[e];
        dzu[e] = act ? dyu[e] * dsilu(z) : dyu[e];
        if (u < t1) {  // each output token's weight gradient is counted by exactly one tile
          dwa[e][0] += dzu[e] * xw[0][e];
          dwa[e][1] += dzu[e] * xw[1][e];
          dwa[e][2] += dzu[e] * xw[2][e];
          dwa[e][3] += dzu[e] * xu[e];
        }
        xw[0][e] = xw[1][e];
        xw[1][e] = xw[2][e];
        xw[2][e] = xu[e];
      }
    } else {
#pragma unroll
      for (int e = 0; e < N; e++) dzu[e] = 0.f;
    }
    dsw[KW - 1] = live ? start : -1;
    // dx_{u-3} = sum_j w_j dz_{u-j}, over the tokens u-3 .. u of its document
    const int64_t p = u - (KW - 1);
    if (p >= t0 && p < t1) {
      float o[N];
#pragma unroll
      for (int e = 0; e < N; e++) {
        float acc = wv[e][3] * dzw[0][e];  // j = 3 pairs dz_p with x_p
        if (dsw[1] == dsw[0]) acc += wv[e][2] * dzw[1][e];
        if (dsw[2] == dsw[0]) acc += wv[e][1] * dzw[2][e];
        if (dsw[3] == dsw[0]) acc += wv[e][0] * dzu[e];
        o[e] = acc;
      }
      vst(dx + p * C + c0, o);
    }
#pragma unroll
    for (int e = 0; e < N; e++) {
      dzw[0][e] = dzw[1][e];
      dzw[1][e] = dzw[2][e];
      dzw[2][e] = dzu[e];
    }
    dsw[0] = dsw[1];
    dsw[1] = dsw[2];
    dsw[2] = dsw[3];
  }
  }
  float* pp = part + ((int64_t)blockIdx.y * C + c0) * KW;
#pragma unroll
  for (int e = 0; e < N; e++)
#pragma unroll
    for (int j = 0; j < KW; j++) pp[e * KW + j] = dwa[e][j];
}

bool a16(const void* p) { return (uintptr_t)p % 16 == 0; }

kda_status check(int64_t n_tok, int C, int dtype, int act, const int32_t* cu, int n_docs) {
  if (n_tok <= 0 || n_tok > ((int64_t)1 << 31) || C <= 0 || C > (1 << 20)) return KDA_ERR_INVALID_ARG;
  if (dtype != KDA_BF16 && dtype != KDA_F32) return KDA_ERR_INVALID_ARG;
  if (act != 0 && act != 1) return KDA_ERR_INVALID_ARG;
  if (C % (dtype == KDA_BF16 ? 8 : 4) != 0) return KDA_ERR_ALIGNMENT;
  if (cu && (n_docs <= 0 || (uintptr_t)cu % 4 != 0)) return KDA_ERR_INVALID_ARG;
  return KDA_OK;
}

}  // namespace
}  // namespace kda

using namespace kda;

extern "C" KDA_API size_t kda_short_conv_workspace_size(int64_t n_tok, int C) {
  if (n_tok <= 0 || C <= 0) return 0;
  return (size_t)((n_tok + TBB - 1) / TBB) * C * KW * sizeof(float);
}

extern "C" KDA_API kda_status kda_short_conv_fwd(int64_t n_tok, int C, int dtype, int activation,
                                                 const int32_t* cu_seqlens, int n_docs, const void* x,
                                                 const float* w, void* y, cudaStream_t st) {
  kda_status s = check(n_tok, C, dtype, activation, cu_seqlens, n_docs);
  if (s != KDA_OK) return s;
  if (!x || !w || !y) return KDA_ERR_INVALID_ARG;
  if (!a16(x) || !a16(y) || !a16(w)) return KDA_ERR_ALIGNMENT;
  const int nvec = C / (dtype == KDA_BF16 ? 8 : 4);
  const dim3 grid((nvec + CTHR - 1) / CTHR, (unsigned)((n_tok + TBF - 1) / TBF));
  if (grid.y > 2147483647u) return KDA_ERR_INVALID_ARG;
  const size_t smem = (TBF + KW - 1) * CTHR * 16 + sizeof(uint64_t);
  prof_begin(K_CONV_FWD, st);
  if (dtype == KDA_BF16)
    conv_fwd_kernel<__nv_bfloat16><<<grid, CTHR, smem, st>>>(n_tok, C, activation, cu_seqlens, n_docs,
                                                           (const __nv_bfloat16*)x, w, (__nv_bfloat16*)y);
  else
    conv_fwd_kernel<float><<<grid, CTHR, smem, st>>>(n_tok, C, activation, cu_seqlens, n_docs, (const float*)x, w,
                                                   (float*)y);
  prof_end(K_CONV_FWD, st);
  return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

extern "C" KDA_API kda_status kda_short_conv_bwd(int64_t n_tok, int C, int dtype, int activation,
                                                 const int32_t* cu_seqlens, int n_docs, const void* x,
                                                 const float* w, const void* dy, void* dx, float* dw,
                                                 void* workspace, size_t workspace_bytes, cudaStream_t st) {
  kda_status s = check(n_tok, C, dtype, activation, cu_seqlens, n_docs);
  if (s != KDA_OK) return s;
  if (!x || !w || !dy || !dx || !dw) return KDA_ERR_INVALID_ARG;
  if (!a16(x) || !a16(dy) || !a16(dx) || !a16(w) || (uintptr_t)dw % 4 != 0) return KDA_ERR_ALIGNMENT;
  if (!workspace || workspace_bytes < kda_short_conv_workspace_size(n_tok, C)) return KDA_ERR_WORKSPACE;
  if ((uintptr_t)workspace % 16 != 0) return KDA_ERR_ALIGNMENT;
  const int nvec = C / NB;
  const int n_tiles = (int)((n_tok + TBB - 1) / TBB);
  const dim3 grid((nvec + CTHR - 1) / CTHR, (unsigned)n_tiles);
  float* part = (float*)workspace;
  prof_begin(K_CONV_BWD, st);
  if (dtype == KDA_BF16)
    conv_bwd_kernel<__nv_bfloat16><<<grid, CTHR, 0, st>>>(n_tok, C, activation, cu_seqlens, n_docs, n_tok,
                                                           (const __nv_bfloat16*)x, w, (const __nv_bfloat16*)dy,
                                                           (__nv_bfloat16*)dx, part);
  else
    conv_bwd_kernel<float><<<grid, CTHR, 0, st>>>(n_tok, C, activation, cu_seqlens, n_docs, n_tok, (const float*)x,
                                                   w, (const float*)dy, (float*)dx, part);
  prof_end(K_CONV_BWD, st);
  if (cudaGetLastError() != cudaSuccess) return KDA_ERR_CUDA;
  prof_begin(K_CONV_RED, st);
  const cudaError_t e = launch_sum_rows(part, n_tiles, C * KW, dw, st);
  prof_end(K_CONV_RED, st);
  return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

namespace kda {
// The fused convolution's backward (kda_bwd_conv): dx (bf16) and dw from x
// (bf16) and the fp32 gradients of the convolution's silu outputs that the
// KDA backward kernels wrote; documents are cu's, or rows of row_len tokens.
// part: kda_short_conv_workspace_size(n_tok, C) bytes.
cudaError_t launch_conv_bwd_fused(int64_t n_tok, int C, const int32_t* cu, int n_docs, int64_t row_len,
                                  const __nv_bfloat16* x, const float* w, const float* dy, __nv_bfloat16* dx,
                                  float* part, float* dw, cudaStream_t st) {
  const int n_tiles = (int)((n_tok + TBB - 1) / TBB);
  const dim3 grid((C / NB + CTHR - 1) / CTHR, (unsigned)n_tiles);
  prof_begin(K_CONV_BWD, st);
  conv_bwd_kernel<__nv_bfloat16, float><<<grid, CTHR, 0, st>>>(n_tok, C, 1, cu, n_docs, row_len, x, w, dy, dx, part);
  prof_end(K_CONV_BWD, st);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  prof_begin(K_CONV_RED, st);
  e = launch_sum_rows(part, n_tiles, C * KW, dw, st);
  prof_end(K_CONV_RED, st);
  return e;
}
}  // namespace kda
