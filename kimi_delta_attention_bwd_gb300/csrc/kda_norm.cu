// Gated RMSNorm output epilogue: per token and head over the value dim dv,
//   r = 1 / sqrt(mean_j x_j^2 + eps),  y_j = x_j r w_j sigmoid(g_j)
// ("Pure KDA 300M" guide, Overview: per-head output gate, RMSNorm eps 1e-6;
// openkimi README, "What is implemented": fused RMSNorm plus sigmoid gate on
// the KDA output), and its backward
//   s = sigmoid(g), xh = x r, dg = dy xh w s (1 - s), a = dy w s,
//   dx = r (a - xh mean(a xh)),  dw = sum over rows of dy xh s.
// Each row is split over DV * size / 16 lanes with 16-byte loads (several rows
// per warp); the rows are HBM-streamed once.  The weight gradient is
// reduced per CTA over a fixed contiguous range of rows, then over the CTAs
// in order (deterministic).
#include "kda_internal.cuh"
#include "../../include/kda.h"

namespace kda {
namespace {

constexpr int NTHR = 256;
constexpr int MAXBLK = 1024;  // CTAs of the backward (partials of dw)

// 16 bytes per lane: EPL elements; LPR lanes per row; RPW rows per warp.
template <int DV, typename T>
struct Shape {
  static constexpr int EPL = 16 / sizeof(T);
  static constexpr int LPR = DV / EPL;
  static constexpr int RPW = 32 / LPR;
  static constexpr int RPC = RPW * (NTHR / 32);  // rows per CTA pass
};

__device__ __forceinline__ void ld16(const __nv_bfloat16* p, float (&v)[8]) {
  const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int e = 0; e < 4; e++) {
    const float2 f = __bfloat1622float2(h[e]);
    v[2 * e] = f.x;
    v[2 * e + 1] = f.y;
  }
}
__device__ __forceinline__ void ld16(const float* p, float (&v)[4]) {
  const float4 f = __ldg(reinterpret_cast<const float4*>(p));
  v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
}
__device__ __forceinline__ void st16(__nv_bfloat16* p, const float (&v)[8]) {
  uint4 u;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
  for (int e = 0; e < 4; e++) h[e] = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
  *reinterpret_cast<uint4*>(p) = u;
}
__device__ __forceinline__ void st16(float* p, const float (&v)[4]) {
  *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
}
// Sum over the LPR lanes of one row (aligned groups of a warp).
template <int LPR>
__device__ __forceinline__ float row_sum(float x) {
#pragma unroll
  for (int o = LPR / 2; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

template <int DV, typename T>
__global__ void __launch_bounds__(NTHR) norm_gate_fwd_kernel(int64_t n, float eps, const T* __restrict__ x,
                                                             const T* __restrict__ g, const float* __restrict__ w,
                                                             T* __restrict__ y) {
  typedef Shape<DV, T> S;
  constexpr int EPL = S::EPL, LPR = S::LPR;
  const int lane = threadIdx.x & 31, sub = lane / LPR, c0 = (lane % LPR) * EPL;
  const int64_t row = ((int64_t)blockIdx.x * (NTHR / 32) + (threadIdx.x >> 5)) * S::RPW + sub;
  const bool ok = row < n;  // the whole group of a row agrees; shuffles stay warp-wide
  float xv[EPL], gv[EPL], yv[EPL];
  if (ok) {
    ld16(x + row * DV + c0, xv);
    ld16(g + row * DV + c0, gv);
  } else {
#pragma unroll
    for (int e = 0; e < EPL; e++) xv[e] = gv[e] = 0.f;
  }
  float ss = 0.f;
#pragma unroll
  for (int e = 0; e < EPL; e++) ss += xv[e] * xv[e];
  ss = row_sum<LPR>(ss);
  const float r = 1.0f / sqrtf(ss / DV + eps);
#pragma unroll
  for (int e = 0; e < EPL; e++) yv[e] = xv[e] * r * w[c0 + e] * sigmoid_fast(gv[e]);
  if (ok) st16(y + row * DV + c0, yv);
}

template <int DV, typename T>
__global__ void __launch_bounds__(NTHR) norm_gate_bwd_kernel(int64_t n, int64_t per_blk, float eps,
                                                             const T* __restrict__ x, const T* __restrict__ g,
                                                             const float* __restrict__ w, const T* __restrict__ dy,
                                                             T* __restrict__ dx, T* __restrict__ dg,
                                                             float* __restrict__ part) {
  typedef Shape<DV, T> S;
  constexpr int EPL = S::EPL, LPR = S::LPR, NWP = NTHR / 32;
  __shared__ float red[NWP * S::RPW][DV];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, sub = lane / LPR, c0 = (lane % LPR) * EPL;
  const int64_t r0 = (int64_t)blockIdx.x * per_blk, r1 = r0 + per_blk < n ? r0 + per_blk : n;
  float wv[EPL], dwacc[EPL];
#pragma unroll
  for (int e = 0; e < EPL; e++) { wv[e] = w[c0 + e]; dwacc[e] = 0.f; }
#pragma unroll 2
  for (int64_t base = r0; base < r1; base += S::RPC) {  // uniform trip count over the CTA
    const int64_t row = base + warp * S::RPW + sub;
    const bool ok = row < r1;
    float xv[EPL], gv[EPL], dyv[EPL], a[EPL], xh[EPL], o1[EPL], o2[EPL];
    if (ok) {
      ld16(x + row * DV + c0, xv);
      ld16(g + row * DV + c0, gv);
      ld16(dy + row * DV + c0, dyv);
    } else {
#pragma unroll
      for (int e = 0; e < EPL; e++) xv[e] = gv[e] = dyv[e] = 0.f;
    }
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < EPL; e++) ss += xv[e] * xv[e];
    ss = row_sum<LPR>(ss);
    const float r = 1.0f / sqrtf(ss / DV + eps);
    float m = 0.f;
#pragma unroll
    for (int e = 0; e < EPL; e++) {
      const float s = sigmoid_fast(gv[e]);
      xh[e] = xv[e] * r;
      a[e] = dyv[e] * wv[e] * s;
      o2[e] = dyv[e] * xh[e] * wv[e] * s * (1.0f - s);  // dg
      dwacc[e] += dyv[e] * xh[e] * s;
      m += a[e] * xh[e];
    }
    m = row_sum<LPR>(m) / DV;
#pragma unroll
    for (int e = 0; e < EPL; e++) o1[e] = r * (a[e] - xh[e] * m);  // dx
    if (ok) {
      st16(dx + row * DV + c0, o1);
      st16(dg + row * DV + c0, o2);
    }
  }
#pragma unroll
  for (int e = 0; e < EPL; e++) red[warp * S::RPW + sub][c0 + e] = dwacc[e];
  __syncthreads();
  for (int j = threadIdx.x; j < DV; j += NTHR) {  // fixed order over the row slots
    float s = 0.f;
    for (int q = 0; q < NWP * S::RPW; q++) s += red[q][j];
    part[(int64_t)blockIdx.x * DV + j] = s;
  }
}

}  // namespace

// out[c] = sum_r part[r][c] over r = 0 .. nrows - 1, in a fixed order: a CTA
// owns 32 columns; its 8 row groups each sum every 8th row with four
// independent partial sums, then the groups are added in order.
__global__ void __launch_bounds__(256) sum_rows_kernel(const float* __restrict__ part, int nrows, int ncols,
                                                       float* __restrict__ out) {
  __shared__ float red[8][32];
  const int cx = threadIdx.x & 31, gy = threadIdx.x >> 5, c = blockIdx.x * 32 + cx;
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
  if (c < ncols) {
    int r = gy;
    for (; r + 24 < nrows; r += 32) {
      a0 += part[(int64_t)r * ncols + c];
      a1 += part[(int64_t)(r + 8) * ncols + c];
      a2 += part[(int64_t)(r + 16) * ncols + c];
      a3 += part[(int64_t)(r + 24) * ncols + c];
    }
    for (; r < nrows; r += 8) a0 += part[(int64_t)r * ncols + c];
  }
  red[gy][cx] = (a0 + a1) + (a2 + a3);
  __syncthreads();
  if (gy == 0 && c < ncols) {
    float s = 0.f;
    for (int g = 0; g < 8; g++) s += red[g][cx];
    out[c] = s;
  }
}

cudaError_t launch_sum_rows(const float* part, int nrows, int ncols, float* out, cudaStream_t st) {
  sum_rows_kernel<<<(ncols + 31) / 32, 256, 0, st>>>(part, nrows, ncols, out);
  return cudaGetLastError();
}

namespace {

int bwd_blocks(int64_t n) {
  const int64_t want = (n + 31) / 32;  // at least 32 rows per CTA
  return (int)(want < MAXBLK ? want : MAXBLK);
}

template <int DV, typename T>
unsigned fwd_grid(int64_t n) {
  return (unsigned)((n + Shape<DV, T>::RPC - 1) / Shape<DV, T>::RPC);
}

bool aligned16(const void* p) { return (uintptr_t)p % 16 == 0; }

}  // namespace
}  // namespace kda

using namespace kda;

extern "C" KDA_API size_t kda_norm_gate_workspace_size(int64_t n_rows, int dv) {
  if (n_rows <= 0 || (dv != 64 && dv != 128)) return 0;
  return (size_t)bwd_blocks(n_rows) * dv * sizeof(float);
}

extern "C" KDA_API kda_status kda_norm_gate_fwd(int64_t n_rows, int dv, int dtype, float eps, const void* x,
                                                const void* g, const float* w, void* y, cudaStream_t st) {
  if (n_rows <= 0 || n_rows > ((int64_t)1 << 34)) return KDA_ERR_INVALID_ARG;
  if (dtype != KDA_BF16 && dtype != KDA_F32) return KDA_ERR_INVALID_ARG;
  if (dv != 64 && dv != 128) return KDA_ERR_UNSUPPORTED;
  if (!x || !g || !w || !y) return KDA_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(g) || !aligned16(w) || !aligned16(y)) return KDA_ERR_ALIGNMENT;
  const float e = eps > 0.f ? eps : 1e-6f;
  prof_begin(K_NORM_FWD, st);
  typedef __nv_bfloat16 B;
  if (dtype == KDA_BF16) {
    if (dv == 64)
      norm_gate_fwd_kernel<64, B><<<fwd_grid<64, B>(n_rows), NTHR, 0, st>>>(n_rows, e, (const B*)x, (const B*)g, w, (B*)y);
    else
      norm_gate_fwd_kernel<128, B><<<fwd_grid<128, B>(n_rows), NTHR, 0, st>>>(n_rows, e, (const B*)x, (const B*)g, w,
                                                                               (B*)y);
  } else {
    if (dv == 64)
      norm_gate_fwd_kernel<64, float><<<fwd_grid<64, float>(n_rows), NTHR, 0, st>>>(n_rows, e, (const float*)x,
                                                                                     (const float*)g, w, (float*)y);
    else
      norm_gate_fwd_kernel<128, float><<<fwd_grid<128, float>(n_rows), NTHR, 0, st>>>(n_rows, e, (const float*)x,
                                                                                       (const float*)g, w, (float*)y);
  }
  prof_end(K_NORM_FWD, st);
  return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

extern "C" KDA_API kda_status kda_norm_gate_bwd(int64_t n_rows, int dv, int dtype, float eps, const void* x,
                                                const void* g, const float* w, const void* dy, void* dx, void* dg,
                                                float* dw, void* workspace, size_t workspace_bytes,
                                                cudaStream_t st) {
  if (n_rows <= 0 || n_rows > ((int64_t)1 << 34)) return KDA_ERR_INVALID_ARG;
  if (dtype != KDA_BF16 && dtype != KDA_F32) return KDA_ERR_INVALID_ARG;
  if (dv != 64 && dv != 128) return KDA_ERR_UNSUPPORTED;
  if (!x || !g || !w || !dy || !dx || !dg || !dw) return KDA_ERR_INVALID_ARG;
  const void* ptrs[] = {x, g, w, dy, dx, dg, dw};
  for (const void* p : ptrs)
    if (!aligned16(p)) return KDA_ERR_ALIGNMENT;
  if (!workspace || workspace_bytes < kda_norm_gate_workspace_size(n_rows, dv)) return KDA_ERR_WORKSPACE;
  if (!aligned16(workspace)) return KDA_ERR_ALIGNMENT;
  const float e = eps > 0.f ? eps : 1e-6f;
  const int nblk = bwd_blocks(n_rows);
  const int64_t per = (n_rows + nblk - 1) / nblk;
  float* part = (float*)workspace;
  prof_begin(K_NORM_BWD, st);
  typedef __nv_bfloat16 B;
  if (dtype == KDA_BF16) {
    if (dv == 64)
      norm_gate_bwd_kernel<64, B><<<nblk, NTHR, 0, st>>>(n_rows, per, e, (const B*)x, (const B*)g, w, (const B*)dy,
                                                         (B*)dx, (B*)dg, part);
    else
      norm_gate_bwd_kernel<128, B><<<nblk, NTHR, 0, st>>>(n_rows, per, e, (const B*)x, (const B*)g, w, (const B*)dy,
                                                          (B*)dx, (B*)dg, part);
  } else {
    if (dv == 64)
      norm_gate_bwd_kernel<64, float><<<nblk, NTHR, 0, st>>>(n_rows, per, e, (const float*)x, (const float*)g, w,
                                                             (const float*)dy, (float*)dx, (float*)dg, part);
    else
      norm_gate_bwd_kernel<128, float><<<nblk, NTHR, 0, st>>>(n_rows, per, e, (const float*)x, (const float*)g, w,
                                                              (const float*)dy, (float*)dx, (float*)dg, part);
  }
  prof_end(K_NORM_BWD, st);
  if (cudaGetLastError() != cudaSuccess) return KDA_ERR_CUDA;
  prof_begin(K_NORM_RED, st);
  const cudaError_t e2 = launch_sum_rows(part, nblk, dv, dw, st);
  prof_end(K_NORM_RED, st);
  return e2 == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}
