// Forward kernels of the KDA chunked gated delta rule.
//
// Chunk algebra (per document, head and 64-token chunk with entry state S;
// G = in-chunk inclusive cumulative log-decay, Gamma = exp(G)):
//   A  = strict_lower( diag(beta) (K^ K^T with ratios exp(G_r - G_s)) )
//   T  = (I + A)^-1,  W = T diag(beta) (K^ * Gamma),  U = T diag(beta) V
//   E  = U - W S                    (the per-token corrections e_r)
//   O  = scale (Q^ * Gamma) S + scale inclusive_lower(Q^ K^T ratios) E
//   S' = Diag(Gamma_last) S + (K^ * exp(G_last - G))^T E
// This is the recurrence of the "Pure KDA 300M" guide (Overview) and of the
// openkimi KDA oracle unrolled over one chunk; every decay ratio used is
// exp of a non-positive number, so nothing can overflow.
#include "kda_simt.cuh"

namespace kda {

constexpr int NT = 32;        // dv columns per scan CTA
constexpr int LDS = NT + 4;   // row stride of the scans' [rows][NT] tiles (16-byte rows)
constexpr int GTH = 1024;     // threads of the per-chunk kernels
constexpr int STH = 256;      // threads of the scan kernels

// One CTA per (chunk, head): the gate/norm prologue and the intra-chunk
// factors W, U, P, QG, KD, gamma, written to the workspace.
template <typename TI, int DK, int DV>
__global__ void __launch_bounds__(GTH) fwd_intra_kernel(Dims d, FwdIO io, Ws w) {
  const int j = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  if (j >= *w.n_chunks) return;
  const int L = w.chunk_len[j];
  if (L <= 0) return;
  const int t0 = w.chunk_tok0[j];
  const int H = d.H;
  const int64_t ch = (int64_t)j * H + h;

  extern __shared__ float sm[];
  float* qh = sm;               // [C][DK]
  float* kh = qh + C * DK;      // [C][DK]
  float* G = kh + C * DK;       // [C][DK] in-chunk cumulative log-decay, log2 units
  float* vv = G + C * DK;       // [C][DV]
  float* Am = vv + C * DV;      // [C][C]
  float* Tt = Am + C * C;       // [C][C] T transposed
  float* bet = Tt + C * C;      // [C]
  float* slab = bet + C;        // staged-product slabs

  const TI* q = (const TI*)io.q;
  const TI* k = (const TI*)io.k;
  const TI* f = (const TI*)io.f;
  const TI* v = (const TI*)io.v;
  const TI* b = (const TI*)io.b;
  const float a = expf(io.A_log[h]);

  for (int idx = tid; idx < C * DK; idx += blockDim.x) {
    int r = idx / DK, i = idx % DK;
    float qv = 0.f, kv = 0.f, gv = 0.f;
    if (r < L) {
      int64_t off = ((int64_t)(t0 + r) * H + h) * DK + i;
      qv = ldf(q + off);
      kv = ldf(k + off);
      gv = d.gate ? -a * softplus_f(ldf(f + ((int64_t)(t0 + r) * H + h)) + io.dt_bias[h])
                  : -a * softplus_f(ldf(f + off) + io.dt_bias[h * DK + i]);
    }
    qh[idx] = qv; kh[idx] = kv; G[idx] = gv;
  }
  for (int idx = tid; idx < C * DV; idx += blockDim.x) {
    int r = idx / DV, jj = idx % DV;
    vv[idx] = r < L ? ldf(v + ((int64_t)(t0 + r) * H + h) * DV + jj) : 0.f;
  }
  for (int r = tid; r < C; r += blockDim.x)
    bet[r] = r < L ? sigmoid_f(ldf(b + (int64_t)(t0 + r) * H + h)) : 0.f;
  __syncthreads();

  // L2 norms (one warp per row) and the in-chunk cumulative log-decay.
  const int warp = tid >> 5, lane = tid & 31, nw = blockDim.x >> 5;
  for (int r = warp; r < C; r += nw) {
    float sq = 0.f, sk = 0.f;
    for (int i = lane; i < DK; i += 32) { sq += qh[r * DK + i] * qh[r * DK + i]; sk += kh[r * DK + i] * kh[r * DK + i]; }
    sq = warp_sum(sq); sk = warp_sum(sk);
    float iq = 1.0f / sqrtf(sq + L2_EPS), ik = 1.0f / sqrtf(sk + L2_EPS);
    for (int i = lane; i < DK; i += 32) { qh[r * DK + i] *= iq; kh[r * DK + i] *= ik; }
  }
  for (int i = tid; i < DK; i += blockDim.x) {
    float acc = 0.f;
    for (int r = 0; r < C; r++) { acc += G[r * DK + i]; G[r * DK + i] = acc * LOG2E_S; }  // G log2(e)
  }
  __syncthreads();

  // A (strict lower, beta-scaled) and P (inclusive lower, scale-scaled): the
  // C (C + 1) / 2 pairs s <= r, one per thread, each lane walking the key
  // channels in a rotated order (conflict-free reads); then the upper parts.
  float* Pg = w.P + ch * C * C;
  for (int idx = tid; idx < C * C; idx += blockDim.x) {
    const int r = idx / C, s = idx % C;
    if (s > r) {
      Am[idx] = 0.f;
      Pg[idx] = 0.f;
    }
  }
  for (int p = tid; p < C * (C + 1) / 2; p += blockDim.x) {
    int r = (int)((sqrtf(8.f * (float)p + 1.f) - 1.f) * 0.5f);  // p = r (r + 1) / 2 + s, s <= r
    while (r * (r + 1) / 2 > p) r--;
    while ((r + 1) * (r + 2) / 2 <= p) r++;
    const int s = p - r * (r + 1) / 2;
    float accA = 0.f, accP = 0.f;
    for (int i0 = 0; i0 < DK; i0++) {
      const int i = (i0 + lane) & (DK - 1);
      const float ks = kh[s * DK + i] * ex2(G[r * DK + i] - G[s * DK + i]);
      accP += qh[r * DK + i] * ks;
      accA += kh[r * DK + i] * ks;
    }
    Am[r * C + s] = s < r ? bet[r] * accA : 0.f;
    Pg[r * C + s] = d.scale * accP;
  }
  __syncthreads();

  // T = (I + A)^-1, held transposed (Tt[c][r] = T[r][c])
  unit_lower_inverse_t<GTH>(Am, Tt, slab);

  float* Wg = w.W + ch * C * DK;
  float* QGg = w.QG + ch * C * DK;
  float* KDg = w.KD + ch * C * DK;
  const float* Glast = G + (L - 1) * DK;
  float* xk = qh;  // XK = diag(beta) (K^ * Gamma) over Q^ once QG is out
  for (int idx = tid; idx < C * DK; idx += blockDim.x) {
    const int r = idx / DK, i = idx % DK;
    const float Gr = G[idx], eG = ex2(Gr);
    QGg[idx] = d.scale * qh[idx] * eG;
    KDg[idx] = kh[idx] * ex2(Glast[i] - Gr);
    xk[idx] = bet[r] * kh[idx] * eG;
  }
  for (int i = tid; i < DK; i += blockDim.x) w.gam[ch * DK + i] = ex2(Glast[i]);
  // W = T XK and U = T diag(beta) V (T unit lower, its upper part zero) on the
  // tensor cores: the accumulator in TMEM, the slab buffers over the inverse's
  // scratch; tc5_setup's barrier also orders the XK writes above before the
  // product reads them
  constexpr int NX = (DK > DV ? DK : DV) > C ? (DK > DV ? DK : DV) : C;
  __shared__ uint32_t t5slot;
  __shared__ uint64_t t5bar[2];
  Tc5 t5 = tc5_setup(&t5slot, t5bar, slab, w.err);
  cta_tc<DK, C, GTH, NX, false, true>(t5, false, [&](int m, int k) { return Tt[k * C + m]; },
                                      [&](int k, int n) { return xk[k * DK + n]; });
  tc5_out<DK, GTH>(t5, [&](int m, int n, float v) { Wg[m * DK + n] = v; });
  float* Ug = w.U + ch * C * DV;
  cta_tc<DV, C, GTH, NX, false, true>(t5, false, [&](int m, int k) { return Tt[k * C + m]; },
                                      [&](int k, int n) { return bet[k] * vv[k * DV + n]; });
  tc5_out<DV, GTH>(t5, [&](int m, int n, float v) { Ug[m * DV + n] = v; });
  tc5_release(t5);
}


// One CTA per (document, head, NT value columns): walks the document's
// chunks in order carrying the fp32 state slice S[:, cols] in shared memory;
// each step's products read the chunk's factors through the staged slab.
template <typename TI, int DK, int DV>
__global__ void __launch_bounds__(STH) fwd_scan_kernel(Dims d, FwdIO io, Ws w) {
  // one CTA per (document, head, column slice), slices fastest, then heads,
  // then the documents in the chunk table's longest-first order
  constexpr int NSL = DV / NT;
  const int lin = blockIdx.x, c0col = (lin % NSL) * NT, h = (lin / NSL) % d.H, tid = threadIdx.x;
  const int doc = w.doc_order[lin / (NSL * d.H)];
  if (*w.err != 0) return;
  const int H = d.H;
  extern __shared__ __align__(16) float sm[];
  float* S = sm;               // [DK][LDS] the carried state slice
  float* E = S + DK * LDS;     // [C][LDS]
  float* slab = E + C * LDS;   // A slab of the staged products
  TI* o = (TI*)io.o;
  const int64_t dh = ((int64_t)doc * H + h) * DK * DV;

  for (int idx = tid; idx < DK * NT; idx += STH) {
    const int i = idx / NT, jj = idx % NT;
    S[i * LDS + jj] = io.h0 ? io.h0[dh + i * DV + c0col + jj] : 0.f;
  }
  const int cb = w.doc_chunk0[doc], ce = w.doc_chunk0[doc + 1];
  for (int c = cb; c < ce; c++) {
    const int64_t ch = (int64_t)c * H + h;
    const int L = w.chunk_len[c], t0 = w.chunk_tok0[c];
    const float* W = w.W + ch * C * DK;
    __syncthreads();  // the previous step's state is complete
    if (c + 1 < ce) {  // the next chunk's factors into L2 while this one runs
      const int64_t nx = ch + H;
      prefetch_span<STH>(w.W + nx * C * DK, C * DK);
      prefetch_span<STH>(w.QG + nx * C * DK, C * DK);
      prefetch_span<STH>(w.KD + nx * C * DK, C * DK);
      prefetch_span<STH>(w.P + nx * C * C, C * C);
      if (tid < C) asm volatile("prefetch.global.L2 [%0];" ::"l"(w.U + (nx * C + tid) * DV + c0col));
    }
    if (io.save)
      for (int idx = tid; idx < DK * NT; idx += STH) {
        const int i = idx / NT, jj = idx % NT;
        w.Sent[(ch * DK + i) * DV + c0col + jj] = S[i * LDS + jj];
      }
    {  // E = U[:, cols] - W S
      MmAcc<C, NT, STH> acc;
      mm_zero<C, NT, STH>(acc);
      cta_mm_sb<C, NT, DK, STH, true>(acc, slab, [&](int m, int k) { return W[m * DK + k]; }, S, LDS);
      mm_out<C, NT, STH>(acc, [&](int m, int n, float v) { E[m * LDS + n] = w.U[(ch * C + m) * DV + c0col + n] - v; });
    }
    {  // O = QG S + P E (rows < L)
      const float* QG = w.QG + ch * C * DK;
      const float* P = w.P + ch * C * C;
      MmAcc<C, NT, STH> acc;
      mm_zero<C, NT, STH>(acc);
      cta_mm_sb<C, NT, DK, STH, true>(acc, slab, [&](int m, int k) { return QG[m * DK + k]; }, S, LDS);
      cta_mm_sb<C, NT, C, STH, true>(acc, slab, [&](int m, int k) { return P[m * C + k]; }, E, LDS);
      mm_out<C, NT, STH>(acc, [&](int m, int n, float v) {
        if (m < L) stf(o + ((int64_t)(t0 + m) * H + h) * DV + c0col + n, v);
      });
    }
    {  // S' = Diag(gamma) S + KD^T E (each thread rewrites only the entries it owns)
      const float* KD = w.KD + ch * C * DK;
      const float* gm = w.gam + ch * DK;
      MmAcc<DK, NT, STH> acc;
      mm_zero<DK, NT, STH>(acc);
      cta_mm_sb<DK, NT, C, STH, false>(acc, slab, [&](int m, int k) { return KD[k * DK + m]; }, E, LDS);
      mm_out<DK, NT, STH>(acc, [&](int m, int n, float v) { S[m * LDS + n] = gm[m] * S[m * LDS + n] + v; });
    }
  }
  __syncthreads();
  if (io.h_final)
    for (int idx = tid; idx < DK * NT; idx += STH) {
      const int i = idx / NT, jj = idx % NT;
      io.h_final[dh + i * DV + c0col + jj] = S[i * LDS + jj];
    }
}

template <typename TI, int DK, int DV>
static cudaError_t fwd_intra_launch(const Dims& d, const FwdIO& io, const Ws& w, cudaStream_t st) {
  constexpr int NMAX = DK > DV ? DK : DV;
  size_t smem = sizeof(float) * (3 * C * DK + C * DV + 2 * C * C + C + tc5_slab_floats(NMAX > C ? NMAX : C));
  cudaError_t e = cudaFuncSetAttribute(fwd_intra_kernel<TI, DK, DV>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(d.nc_max, d.H);
  prof_begin(K_FWD_INTRA, st);
  fwd_intra_kernel<TI, DK, DV><<<grid, GTH, smem, st>>>(d, io, w);
  prof_end(K_FWD_INTRA, st);
  return cudaGetLastError();
}

template <typename TI, int DK, int DV>
static cudaError_t fwd_scan_launch(const Dims& d, const FwdIO& io, const Ws& w, cudaStream_t st) {
  size_t smem = sizeof(float) * ((DK + C) * LDS + KS * ((DK > C ? DK : C) + 1));
  cudaError_t e = cudaFuncSetAttribute(fwd_scan_kernel<TI, DK, DV>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)d.n_docs * d.H * (DV / NT));
  prof_begin(K_FWD_SCAN, st);
  fwd_scan_kernel<TI, DK, DV><<<grid, STH, smem, st>>>(d, io, w);
  prof_end(K_FWD_SCAN, st);
  return cudaGetLastError();
}

#define KDA_DISPATCH(FN, ...)                                                              \
  do {                                                                                     \
    if (dtype == 0) {                                                                      \
      if (d.dk == 32 && d.dv == 64) return FN<__nv_bfloat16, 32, 64>(__VA_ARGS__);         \
      if (d.dk == 64 && d.dv == 64) return FN<__nv_bfloat16, 64, 64>(__VA_ARGS__);         \
      if (d.dk == 64 && d.dv == 128) return FN<__nv_bfloat16, 64, 128>(__VA_ARGS__);       \
      if (d.dk == 128 && d.dv == 128) return FN<__nv_bfloat16, 128, 128>(__VA_ARGS__);     \
    } else {                                                                               \
      if (d.dk == 32 && d.dv == 64) return FN<float, 32, 64>(__VA_ARGS__);                 \
      if (d.dk == 64 && d.dv == 64) return FN<float, 64, 64>(__VA_ARGS__);                 \
      if (d.dk == 64 && d.dv == 128) return FN<float, 64, 128>(__VA_ARGS__);               \
      if (d.dk == 128 && d.dv == 128) return FN<float, 128, 128>(__VA_ARGS__);             \
    }                                                                                      \
    return cudaErrorInvalidValue;                                                          \
  } while (0)

cudaError_t launch_fwd_intra(int dtype, const Dims& d, const FwdIO& io, const Ws& w, cudaStream_t st) {
  KDA_DISPATCH(fwd_intra_launch, d, io, w, st);
}
cudaError_t launch_fwd_scan(int dtype, const Dims& d, const FwdIO& io, const Ws& w, cudaStream_t st) {
  KDA_DISPATCH(fwd_scan_launch, d, io, w, st);
}

}  // namespace kda
