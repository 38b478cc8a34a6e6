// Single-token recurrent step (decode): for every sequence and head, one
// token of the recurrence applied to a state held in HBM,
//   S <- (I - beta k^ k^T) Diag(exp g) S + beta k^ v^T,   o = scale S^T q^
// computed as D = Diag(exp g) S,  u = D^T k^,  S' = D + k^ (beta (v - u))^T,
// o = scale S'^T q^.  The state is read once and written once (fp32), so the
// step is bound by HBM bandwidth.  The "Pure KDA 300M" guide fixes the
// recurrence (Overview); inference-only forward backends are the use the
// openkimi README's discussion of FlashKDA names ("forward-only and
// inference-only").
#include "kda_internal.cuh"
#include "../../include/kda.h"

namespace kda {
namespace {

constexpr int DTH = 256;

// One CTA per (sequence, head).  Thread t: value column t % DV, key rows of
// group t / DV (DK / (DTH / DV) consecutive rows).
template <int DK, int DV, typename T>
__global__ void __launch_bounds__(DTH) decode_kernel(int H, int gate, float scale, const T* __restrict__ q,
                                                     const T* __restrict__ k, const T* __restrict__ v,
                                                     const T* __restrict__ f, const T* __restrict__ b,
                                                     const float* __restrict__ A_log,
                                                     const float* __restrict__ dt_bias, float* __restrict__ state,
                                                     T* __restrict__ o) {
  constexpr int RG = DTH / DV, RPT = DK / RG;
  __shared__ float qh[DK], kh[DK], dec[DK], vv[DV];
  __shared__ float red[RG][DV];
  __shared__ float bet;
  const int sh = blockIdx.x, h = sh % H, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (warp == 0) {  // q^, k^ and the decay exp(g) over the key channels
    constexpr int PL = DK / 32;
    float qv[PL], kv[PL], sq = 0.f, sk = 0.f;
#pragma unroll
    for (int e = 0; e < PL; e++) {
      const int i = lane + 32 * e;
      qv[e] = ldf(q + (size_t)sh * DK + i);
      kv[e] = ldf(k + (size_t)sh * DK + i);
      sq += qv[e] * qv[e];
      sk += kv[e] * kv[e];
    }
    sq = warp_sum(sq);
    sk = warp_sum(sk);
    const float iq = 1.0f / sqrtf(sq + L2_EPS), ik = 1.0f / sqrtf(sk + L2_EPS), a = expf(A_log[h]);
#pragma unroll
    for (int e = 0; e < PL; e++) {
      const int i = lane + 32 * e;
      qh[i] = qv[e] * iq;
      kh[i] = kv[e] * ik;
      dec[i] = gate ? expf(-a * softplus_f(ldf(f + sh) + dt_bias[h]))
                    : expf(-a * softplus_f(ldf(f + (size_t)sh * DK + i) + dt_bias[h * DK + i]));
    }
  } else if (warp == 1) {
    for (int j = lane; j < DV; j += 32) vv[j] = ldf(v + (size_t)sh * DV + j);
    if (lane == 0) bet = sigmoid_f(ldf(b + sh));
  }
  __syncthreads();
  const int j = tid % DV, rg = tid / DV, i0 = rg * RPT;
  float* S = state + (size_t)sh * DK * DV;
  float s[RPT];
  float u = 0.f;
#pragma unroll
  for (int e = 0; e < RPT; e++) {
    s[e] = dec[i0 + e] * S[(size_t)(i0 + e) * DV + j];
    u += kh[i0 + e] * s[e];
  }
  red[rg][j] = u;
  __syncthreads();
  u = 0.f;
#pragma unroll
  for (int g2 = 0; g2 < RG; g2++) u += red[g2][j];
  const float wj = bet * (vv[j] - u);
  float oo = 0.f;
#pragma unroll
  for (int e = 0; e < RPT; e++) {
    s[e] += kh[i0 + e] * wj;
    S[(size_t)(i0 + e) * DV + j] = s[e];
    oo += qh[i0 + e] * s[e];
  }
  __syncthreads();  // every read of red is done
  red[rg][j] = oo;
  __syncthreads();
  if (rg == 0) {
    oo = 0.f;
#pragma unroll
    for (int g2 = 0; g2 < RG; g2++) oo += red[g2][j];
    stf(o + (size_t)sh * DV + j, scale * oo);
  }
}

template <int DK, int DV>
cudaError_t launch_decode(int dtype, int gate, int n, int H, float scale, const void* q, const void* k, const void* v,
                          const void* f, const void* b, const float* A_log, const float* dt_bias, float* state,
                          void* o, cudaStream_t st) {
  prof_begin(K_DECODE, st);
  if (dtype == KDA_BF16) {
    typedef __nv_bfloat16 T;
    decode_kernel<DK, DV, T><<<n * H, DTH, 0, st>>>(H, gate, scale, (const T*)q, (const T*)k, (const T*)v, (const T*)f,
                                                    (const T*)b, A_log, dt_bias, state, (T*)o);
  } else {
    decode_kernel<DK, DV, float><<<n * H, DTH, 0, st>>>(H, gate, scale, (const float*)q, (const float*)k, (const float*)v,
                                                        (const float*)f, (const float*)b, A_log, dt_bias, state,
                                                        (float*)o);
  }
  prof_end(K_DECODE, st);
  return cudaGetLastError();
}

}  // namespace
}  // namespace kda

extern "C" KDA_API kda_status kda_decode(int n_seq, int H, int dk, int dv, int dtype, int gate, float scale,
                                         const void* q,
                                         const void* k, const void* v, const void* f, const void* b,
                                         const float* A_log, const float* dt_bias, float* state, void* o,
                                         cudaStream_t stream) {
  using namespace kda;
  if (n_seq <= 0 || H <= 0 || H > 4096 || (int64_t)n_seq * H > ((int64_t)1 << 30)) return KDA_ERR_INVALID_ARG;
  if (dtype != KDA_BF16 && dtype != KDA_F32) return KDA_ERR_INVALID_ARG;
  if (gate != KDA_GATE_CHANNEL && gate != KDA_GATE_SCALAR) return KDA_ERR_INVALID_ARG;
  if (!q || !k || !v || !f || !b || !A_log || !dt_bias || !state || !o) return KDA_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, f, b, A_log, dt_bias, state, o};
  for (const void* x : ptrs)
    if ((uintptr_t)x % 16 != 0) return KDA_ERR_ALIGNMENT;
  const float sc = scale > 0.f ? scale : 1.0f / sqrtf((float)dk);
  cudaError_t e;
  if (dk == 32 && dv == 64) e = launch_decode<32, 64>(dtype, gate, n_seq, H, sc, q, k, v, f, b, A_log, dt_bias, state, o, stream);
  else if (dk == 64 && dv == 64) e = launch_decode<64, 64>(dtype, gate, n_seq, H, sc, q, k, v, f, b, A_log, dt_bias, state, o, stream);
  else if (dk == 64 && dv == 128) e = launch_decode<64, 128>(dtype, gate, n_seq, H, sc, q, k, v, f, b, A_log, dt_bias, state, o, stream);
  else if (dk == 128 && dv == 128) e = launch_decode<128, 128>(dtype, gate, n_seq, H, sc, q, k, v, f, b, A_log, dt_bias, state, o, stream);
  else return KDA_ERR_UNSUPPORTED;
  return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}
