// Backward kernels of the KDA chunked gated delta rule.
//
// With E = U - W S, O = QG S + P E and S' = Diag(gamma) S + KD^T E per chunk
// (QG and P carry the output scale), the reverse pass is
//   dE = P^T dO + KD dS'                 (per chunk, from the state gradient)
//   dS = Diag(gamma) dS' + QG^T dO - W^T dE
// carried backwards over a document's chunks (bwd_scan), followed by the
// local gradients of every chunk through T = (I + A)^-1, the decay ratios,
// the cumulative gate, the softplus gate, the sigmoid and the L2 norms
// (bwd_intra), and a fixed-order reduction of the per-head parameter
// gradients (bwd_reduce).  Derivation: reverse-mode differentiation of the
// recurrence of the "Pure KDA 300M" guide (Overview), chunked as in the
// forward kernels.
#include "kda_simt.cuh"

namespace kda {

constexpr int NT = 32;        // dv columns per scan CTA
constexpr int LDS = NT + 4;   // row stride of the scans' [rows][NT] tiles (16-byte rows)
constexpr int GTH = 1024;     // threads of the per-chunk kernels
constexpr int STH = 256;      // threads of the scan kernels

// One CTA per (document, head, NT value columns): walks the document's
// chunks backwards carrying the state-gradient slice dS[:, cols] in shared
// memory; each step's products read the chunk's factors through the staged
// slab.
template <typename TI, int DK, int DV>
__global__ void __launch_bounds__(STH) bwd_scan_kernel(Dims d, BwdIO io, Ws w) {
  // one CTA per (document, head, column slice), slices fastest, then heads,
  // then the documents in the chunk table's longest-first order
  constexpr int NSL = DV / NT;
  const int lin = blockIdx.x, c0col = (lin % NSL) * NT, h = (lin / NSL) % d.H, tid = threadIdx.x;
  const int doc = w.doc_order[lin / (NSL * d.H)];
  if (!saved_ok(d, w.tag, w.err)) return;
  const int H = d.H;
  extern __shared__ __align__(16) float sm[];
  float* dS = sm;                // [DK][LDS] the carried state gradient
  float* dOt = dS + DK * LDS;    // [C][LDS]  dO rows of the chunk (zero past L)
  float* dEt = dOt + C * LDS;    // [C][LDS]
  float* slab = dEt + C * LDS;   // A slab of the staged products
  const TI* dO = (const TI*)io.dO;
  const int64_t dh = ((int64_t)doc * H + h) * DK * DV;

  for (int idx = tid; idx < DK * NT; idx += STH) {
    const int i = idx / NT, jj = idx % NT;
    dS[i * LDS + jj] = io.dh_final ? io.dh_final[dh + i * DV + c0col + jj] : 0.f;
  }
  const int cb = w.doc_chunk0[doc], ce = w.doc_chunk0[doc + 1];
  for (int c = ce - 1; c >= cb; c--) {
    const int64_t ch = (int64_t)c * H + h;
    const int L = w.chunk_len[c], t0 = w.chunk_tok0[c];
    __syncthreads();  // the previous step's dS and its readers are done
    if (c > cb) {  // the previous chunk's factors and dO rows into L2 while this one runs
      const int64_t nx = ch - H;
      prefetch_span<STH>(w.P + nx * C * C, C * C);
      prefetch_span<STH>(w.KD + nx * C * DK, C * DK);
      prefetch_span<STH>(w.QG + nx * C * DK, C * DK);
      prefetch_span<STH>(w.W + nx * C * DK, C * DK);
      const int Ln = w.chunk_len[c - 1], tn = w.chunk_tok0[c - 1];
      if (tid < Ln) asm volatile("prefetch.global.L2 [%0];" ::"l"(dO + ((int64_t)(tn + tid) * H + h) * DV + c0col));
    }
    for (int idx = tid; idx < DK * NT; idx += STH) {
      const int i = idx / NT, jj = idx % NT;
      w.dSn[(ch * DK + i) * DV + c0col + jj] = dS[i * LDS + jj];
    }
    for (int idx = tid; idx < C * NT; idx += STH) {
      const int r = idx / NT, jj = idx % NT;
      dOt[r * LDS + jj] = r < L ? ldf(dO + ((int64_t)(t0 + r) * H + h) * DV + c0col + jj) : 0.f;
    }
    {  // dE = P^T dO + KD dS' (to the workspace for the per-chunk kernel, and to dEt)
      const float* P = w.P + ch * C * C;
      const float* KD = w.KD + ch * C * DK;
      MmAcc<C, NT, STH> acc;
      mm_zero<C, NT, STH>(acc);
      cta_mm_sb<C, NT, C, STH, false>(acc, slab, [&](int m, int k) { return P[k * C + m]; }, dOt, LDS);
      cta_mm_sb<C, NT, DK, STH, true>(acc, slab, [&](int m, int k) { return KD[m * DK + k]; }, dS, LDS);
      mm_out<C, NT, STH>(acc, [&](int m, int n, float v) {
        dEt[m * LDS + n] = v;
        w.dE[(ch * C + m) * DV + c0col + n] = v;
      });
    }
    {  // dS = Diag(gamma) dS' + QG^T dO - W^T dE (each thread rewrites only the entries it owns)
      const float* QG = w.QG + ch * C * DK;
      const float* W = w.W + ch * C * DK;
      const float* gm = w.gam + ch * DK;
      MmAcc<DK, NT, STH> acc;
      mm_zero<DK, NT, STH>(acc);
      cta_mm_sb<DK, NT, C, STH, false>(acc, slab, [&](int m, int k) { return QG[k * DK + m]; }, dOt, LDS);
      cta_mm_sb<DK, NT, C, STH, false>(acc, slab, [&](int m, int k) { return -W[k * DK + m]; }, dEt, LDS);
      mm_out<DK, NT, STH>(acc, [&](int m, int n, float v) { dS[m * LDS + n] = gm[m] * dS[m * LDS + n] + v; });
    }
  }
  __syncthreads();
  if (io.dh0)
    for (int idx = tid; idx < DK * NT; idx += STH) {
      const int i = idx / NT, jj = idx % NT;
      io.dh0[dh + i * DV + c0col + jj] = dS[i * LDS + jj];
    }
}

__device__ __forceinline__ float block_sum(float x, float* red) {
  x = warp_sum(x);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  __syncthreads();
  if (lane == 0) red[warp] = x;
  __syncthreads();
  float r = 0.f;
  if (threadIdx.x == 0) {
    for (int i = 0; i < nw; i++) r += red[i];
    red[0] = r;
  }
  __syncthreads();
  return red[0];
}

// One CTA per (chunk, head): all local gradients of the chunk.
template <typename TI, int DK, int DV>
__global__ void __launch_bounds__(GTH) bwd_intra_kernel(Dims d, BwdIO io, Ws w) {
  const int j = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  if (!saved_ok(d, w.tag, w.err)) return;
  if (j >= *w.n_chunks) return;
  const int L = w.chunk_len[j];
  if (L <= 0) return;
  const int t0 = w.chunk_tok0[j];
  const int H = d.H;
  const int64_t ch = (int64_t)j * H + h;
  const float scale = d.scale;

  extern __shared__ float sm[];
  float* qh = sm;               // [C][DK]
  float* kh = qh + C * DK;      // [C][DK]
  float* G = kh + C * DK;       // [C][DK] in-chunk cumulative log-decay, log2 units
  float* Ap = G + C * DK;       // [C][C] unscaled strict-lower K^K^T with ratios
  float* Tt = Ap + C * C;       // [C][C] T transposed
  float* dAm = Tt + C * C;      // [C][C]
  float* dPm = dAm + C * C;     // [C][C]
  float* bet = dPm + C * C;     // [C]
  float* nq = bet + C;          // [C]
  float* nk = nq + C;           // [C]
  float* dbet = nk + C;         // [C]
  float* omb = dbet + C;        // [C]  1 - beta, as sigmoid(-b) (exact near beta = 1)
  float* dgam = omb + C;        // [DK]
  float* red = dgam + DK;       // [32]
  float* slab = red + 32;       // staged-product slabs

  // this chunk's saved state, state gradient and factors into L2 while the prologue runs
  prefetch_span<GTH>(w.Sent + ch * DK * DV, DK * DV);
  prefetch_span<GTH>(w.dSn + ch * DK * DV, DK * DV);
  prefetch_span<GTH>(w.W + ch * C * DK, C * DK);
  prefetch_span<GTH>(w.U + ch * C * DV, C * DV);
  prefetch_span<GTH>(w.dE + ch * C * DV, C * DV);

  float* scr = w.scr + ch * w.scr_per_ch;
  float* E = scr;               // [C][DV]
  float* YU = E + C * DV;       // [C][DV]
  float* dQG = YU + C * DV;     // [C][DK]  gradient of Q^ * Gamma (unscaled)
  float* dKd = dQG + C * DK;    // [C][DK]
  float* dW = dKd + C * DK;     // [C][DK]
  float* YW = dW + C * DK;      // [C][DK]
  float* dqh = YW + C * DK;     // [C][DK]
  float* dkh = dqh + C * DK;    // [C][DK]
  float* dG = dkh + C * DK;     // [C][DK]

  const TI* q = (const TI*)io.q;
  const TI* k = (const TI*)io.k;
  const TI* f = (const TI*)io.f;
  const TI* v = (const TI*)io.v;
  const TI* b = (const TI*)io.b;
  const TI* dO = (const TI*)io.dO;
  const float a = expf(io.A_log[h]);
  const float* Sg = w.Sent + ch * DK * DV;
  const float* dSg = w.dSn + ch * DK * DV;
  const float* dEg = w.dE + ch * C * DV;
  const float* Wg = w.W + ch * C * DK;
  const float* Ug = w.U + ch * C * DV;

  // ---- prologue (same arithmetic as the forward)
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
  for (int r = tid; r < C; r += blockDim.x) {
    float br = r < L ? ldf(b + (int64_t)(t0 + r) * H + h) : 0.f;
    bet[r] = r < L ? sigmoid_f(br) : 0.f;
    omb[r] = sigmoid_f(-br);
    dbet[r] = 0.f;
  }
  __syncthreads();
  const int warp = tid >> 5, lane = tid & 31, nw = blockDim.x >> 5;
  for (int r = warp; r < C; r += nw) {
    float sq = 0.f, sk = 0.f;
    for (int i = lane; i < DK; i += 32) { sq += qh[r * DK + i] * qh[r * DK + i]; sk += kh[r * DK + i] * kh[r * DK + i]; }
    sq = warp_sum(sq); sk = warp_sum(sk);
    float nqr = sqrtf(sq + L2_EPS), nkr = sqrtf(sk + L2_EPS);
    float iq = 1.0f / nqr, ik = 1.0f / nkr;
    for (int i = lane; i < DK; i += 32) { qh[r * DK + i] *= iq; kh[r * DK + i] *= ik; }
    if (lane == 0) { nq[r] = nqr; nk[r] = nkr; }
  }
  for (int i = tid; i < DK; i += blockDim.x) {
    float acc = 0.f;
    for (int r = 0; r < C; r++) { acc += G[r * DK + i]; G[r * DK + i] = acc * LOG2E_S; }  // G log2(e)
  }
  __syncthreads();

  // ---- intra-chunk factors (same arithmetic as the forward; A' only, dP comes
  //      from dO): the C (C - 1) / 2 strictly lower pairs (r, s), one per
  //      thread, each lane walking the key channels in a rotated order
  //      (conflict-free reads); then the rest of Ap and dAm
  for (int idx = tid; idx < C * C; idx += blockDim.x) {
    const int r = idx / C, s = idx % C;
    if (s >= r) Ap[idx] = dAm[idx] = 0.f;
  }
  for (int p = tid; p < C * (C - 1) / 2; p += blockDim.x) {
    int r = (int)((1.f + sqrtf(1.f + 8.f * (float)p)) * 0.5f);  // p = r (r - 1) / 2 + s, s < r
    while (r * (r - 1) / 2 > p) r--;
    while ((r + 1) * r / 2 <= p) r++;
    const int s = p - r * (r - 1) / 2;
    float accA = 0.f;
    for (int i0 = 0; i0 < DK; i0++) {
      const int i = (i0 + lane) & (DK - 1);
      accA += kh[r * DK + i] * kh[s * DK + i] * ex2(G[r * DK + i] - G[s * DK + i]);
    }
    Ap[r * C + s] = accA;
    dAm[r * C + s] = bet[r] * accA;  // A = diag(beta) Ap, used for the solve
  }
  __syncthreads();
  // T = (I + A)^-1, held transposed (Tt[c][r] = T[r][c])
  unit_lower_inverse_t<GTH>(dAm, Tt, slab);
  // the products below on the tensor cores: the accumulator in TMEM, the slab
  // buffers over the inverse's scratch (done: the inverse ends with a barrier)
  constexpr int NX = (DK > DV ? DK : DV) > C ? (DK > DV ? DK : DV) : C;
  __shared__ uint32_t t5slot;
  __shared__ uint64_t t5bar[2];
  Tc5 t5 = tc5_setup(&t5slot, t5bar, slab, w.err);

  // ---- E = U - W S (scratch), dgamma; then with the value columns as k:
  //      dQG = scale dO S^T, dW = -dE S^T, dKd = E dS'^T (products staged
  //      through shared memory, every global read coalesced; each product's
  //      operands were written before a barrier of an earlier product)
  cta_tc<DV, DK, GTH, NX, true, true>(t5, false, [&](int m, int k) { return Wg[m * DK + k]; },
                                      [&](int k, int n) { return Sg[k * DV + n]; });
  tc5_out<DV, GTH>(t5, [&](int m, int n, float v) { E[m * DV + n] = Ug[m * DV + n] - v; });
  for (int i = warp; i < DK; i += nw) {
    float acc = 0.f;
    for (int jj = lane; jj < DV; jj += 32) acc += dSg[i * DV + jj] * Sg[i * DV + jj];
    acc = warp_sum(acc);
    if (lane == 0) dgam[i] = acc;
  }
  const TI* dOc = dO + ((int64_t)t0 * H + h) * DV;  // row r of the chunk at dOc + r H dv
  auto fdO = [&](int m, int k) { return m < L ? ldf(dOc + (int64_t)m * H * DV + k) : 0.f; };
  cta_tc<DK, DV, GTH, NX, true, false>(t5, false, fdO, [&](int k, int n) { return Sg[n * DV + k]; });
  tc5_out<DK, GTH>(t5, [&](int m, int n, float v) { dQG[m * DK + n] = scale * v; });
  cta_tc<DK, DV, GTH, NX, true, false>(t5, false, [&](int m, int k) { return dEg[m * DV + k]; },
                                       [&](int k, int n) { return Sg[n * DV + k]; });
  tc5_out<DK, GTH>(t5, [&](int m, int n, float v) { dW[m * DK + n] = -v; });
  cta_tc<DK, DV, GTH, NX, true, false>(t5, false, [&](int m, int k) { return E[m * DV + k]; },
                                       [&](int k, int n) { return dSg[n * DV + k]; });
  tc5_out<DK, GTH>(t5, [&](int m, int n, float v) { dKd[m * DK + n] = v; });

  // ---- dP = scale dO E^T (inclusive lower, rows < L), YW = T^T dW, YU = T^T dE
  cta_tc<C, DV, GTH, NX, true, false>(t5, false, fdO, [&](int k, int n) { return E[n * DV + k]; });
  tc5_out<C, GTH>(t5, [&](int m, int n, float v) { dPm[m * C + n] = n <= m && m < L ? scale * v : 0.f; });
  cta_tc<DK, C, GTH, NX, true, true>(t5, false, [&](int m, int k) { return Tt[m * C + k]; },
                                     [&](int k, int n) { return dW[k * DK + n]; });
  tc5_out<DK, GTH>(t5, [&](int m, int n, float v) { YW[m * DK + n] = v; });
  cta_tc<DV, C, GTH, NX, true, true>(t5, false, [&](int m, int k) { return Tt[m * C + k]; },
                                     [&](int k, int n) { return dEg[k * DV + n]; });
  tc5_out<DV, GTH>(t5, [&](int m, int n, float v) { YU[m * DV + n] = v; });
  __syncthreads();

  // ---- dv = beta YU;  dbeta from U and W;  dA = -(YU U^T + YW W^T) strict lower
  TI* dvo = (TI*)io.dv;
  for (int idx = tid; idx < C * DV; idx += blockDim.x) {
    int r = idx / DV, jj = idx % DV;
    if (r < L) stf(dvo + ((int64_t)(t0 + r) * H + h) * DV + jj, bet[r] * YU[idx]);
  }
  for (int r = warp; r < L; r += nw) {
    float acc = 0.f;
    for (int jj = lane; jj < DV; jj += 32) acc += YU[r * DV + jj] * ldf(v + ((int64_t)(t0 + r) * H + h) * DV + jj);
    for (int i = lane; i < DK; i += 32) acc += YW[r * DK + i] * kh[r * DK + i] * ex2(G[r * DK + i]);
    acc = warp_sum(acc);
    if (lane == 0) dbet[r] += acc;
  }
  cta_tc<C, DV, GTH, NX, true, false>(t5, false, [&](int m, int k) { return YU[m * DV + k]; },
                                      [&](int k, int n) { return Ug[n * DV + k]; });
  cta_tc<C, DK, GTH, NX, true, false>(t5, true, [&](int m, int k) { return YW[m * DK + k]; },
                                      [&](int k, int n) { return Wg[n * DK + k]; });
  tc5_out<C, GTH>(t5, [&](int m, int n, float v) { dAm[m * C + n] = n < m ? -v : 0.f; });
  tc5_release(t5);
  __syncthreads();
  for (int r = warp; r < L; r += nw) {
    float acc = 0.f;
    for (int s = lane; s < r; s += 32) acc += dAm[r * C + s] * Ap[r * C + s];
    acc = warp_sum(acc);
    if (lane == 0) dbet[r] += acc;
  }
  __syncthreads();
  for (int idx = tid; idx < C * C; idx += blockDim.x) dAm[idx] *= bet[idx / C];  // gradient of Ap
  __syncthreads();

  // ---- pairwise decay-ratio terms and the elementwise ones -> dqh, dkh, dG
  for (int idx = tid; idx < C * DK; idx += blockDim.x) {
    int r = idx / DK, i = idx % DK;
    float Gr = G[idx];
    float prow = 0.f, arow = 0.f, col = 0.f;
    for (int s = 0; s <= r; s++) {
      float e = ex2(Gr - G[s * DK + i]);
      prow += dPm[r * C + s] * kh[s * DK + i] * e;
      arow += dAm[r * C + s] * kh[s * DK + i] * e;   // dAm is 0 on the diagonal
    }
    for (int rr = r; rr < C; rr++) {
      float e = ex2(G[rr * DK + i] - Gr);
      col += dPm[rr * C + r] * qh[rr * DK + i] * e + dAm[rr * C + r] * kh[rr * DK + i] * e;
    }
    float Gam = ex2(Gr);
    float KDr = kh[idx] * ex2(G[(L - 1) * DK + i] - Gr);
    float dkg = bet[r] * YW[idx];  // gradient of K^ * Gamma
    dqh[idx] = prow + dQG[idx] * Gam;
    dkh[idx] = arow + col + dkg * Gam + dKd[idx] * ex2(G[(L - 1) * DK + i] - Gr);
    dG[idx] = qh[idx] * prow + kh[idx] * arow - kh[idx] * col + dQG[idx] * qh[idx] * Gam
              + dkg * kh[idx] * Gam - dKd[idx] * KDr;
  }
  __syncthreads();

  // ---- per channel: G_last terms, reverse cumsum -> dg, gate backward, partials.
  //      Channel i's rows split into NSEG segments of RPS rows, one thread each:
  //      segment totals first, then each segment adds the totals after it (a
  //      fixed order, so the sums are deterministic) and walks its own rows
  constexpr int NSEG = GTH / DK, RPS = C / NSEG;
  static_assert(NSEG * DK == GTH && NSEG * RPS == C, "gate segments");
  float* segd = slab;              // [NSEG][DK] segment totals of dG
  float* sege = segd + NSEG * DK;  // [NSEG][DK] segment totals of the G_last terms
  float* segp = sege + NSEG * DK;  // [NSEG][DK] segment partials of ddt_bias
  TI* dfo = (TI*)io.df;
  const int gi = tid % DK, gseg = tid / DK, r0 = gseg * RPS;
  const float Glast = G[(L - 1) * DK + gi];
  {
    float sd = 0.f, se = 0.f;
#pragma unroll
    for (int u = 0; u < RPS; u++) {
      const int r = r0 + u;
      if (r < L) {
        sd += dG[r * DK + gi];
        se += dKd[r * DK + gi] * kh[r * DK + gi] * ex2(Glast - G[r * DK + gi]);
      }
    }
    segd[gseg * DK + gi] = sd;
    sege[gseg * DK + gi] = se;
  }
  __syncthreads();
  float pA_local = 0.f;
  {
    float acc = dgam[gi] * ex2(Glast);  // dG at row L-1 gets the G_last terms
    for (int sg = 0; sg < NSEG; sg++) acc += sege[sg * DK + gi];
    for (int sg = NSEG - 1; sg > gseg; sg--) acc += segd[sg * DK + gi];
    float pdt = 0.f;
#pragma unroll
    for (int u = RPS - 1; u >= 0; u--) {
      const int r = r0 + u;
      if (r < L) {
        acc += dG[r * DK + gi];
        const int64_t off = ((int64_t)(t0 + r) * H + h) * DK + gi;
        const float x = d.gate ? ldf(f + ((int64_t)(t0 + r) * H + h)) + io.dt_bias[h] : ldf(f + off) + io.dt_bias[h * DK + gi];
        const float g = -a * softplus_f(x);
        const float dx = acc * (-a) * sigmoid_f(x);
        if (d.gate) dG[r * DK + gi] = dx;  // summed over the channels below
        else stf(dfo + off, dx);
        pdt += dx;
        pA_local += acc * g;
      }
    }
    segp[gseg * DK + gi] = pdt;
  }
  __syncthreads();
  for (int i = tid; i < DK; i += blockDim.x) {
    float p = 0.f;
    for (int sg = 0; sg < NSEG; sg++) p += segp[sg * DK + i];
    w.pdt[ch * DK + i] = p;
  }
  float tot = block_sum(pA_local, red);
  if (tid == 0) w.pA[ch] = tot;
  if (d.gate) {  // scalar gate: df of a token is the sum over its channels (fixed order)
    __syncthreads();
    for (int r = warp; r < L; r += nw) {
      float sdx = 0.f;
      for (int i = lane; i < DK; i += 32) sdx += dG[r * DK + i];
      sdx = warp_sum(sdx);
      if (lane == 0) stf(dfo + (int64_t)(t0 + r) * H + h, sdx);
    }
  }

  // ---- L2-norm backward and db
  TI* dqo = (TI*)io.dq;
  TI* dko = (TI*)io.dk;
  TI* dbo = (TI*)io.db;
  for (int r = warp; r < L; r += nw) {
    float pq = 0.f, pk = 0.f;
    for (int i = lane; i < DK; i += 32) { pq += qh[r * DK + i] * dqh[r * DK + i]; pk += kh[r * DK + i] * dkh[r * DK + i]; }
    pq = warp_sum(pq); pk = warp_sum(pk);
    for (int i = lane; i < DK; i += 32) {
      int64_t off = ((int64_t)(t0 + r) * H + h) * DK + i;
      stf(dqo + off, (dqh[r * DK + i] - qh[r * DK + i] * pq) / nq[r]);
      stf(dko + off, (dkh[r * DK + i] - kh[r * DK + i] * pk) / nk[r]);
    }
    if (lane == 0) stf(dbo + (int64_t)(t0 + r) * H + h, dbet[r] * bet[r] * omb[r]);
  }
}

// dA_log[h] and ddt_bias[h, :] summed over chunks in a fixed order: 32
// groups of 32 threads, group g owning chunks g, g + 32, ... of a block of 32
// channels with four independent partial sums, then the groups in order.
// The scalar gate sums ddt_bias over the channels too.
constexpr int RTH = 1024, RG = RTH / 32;
__global__ void __launch_bounds__(RTH) bwd_reduce_kernel(Dims d, BwdIO io, Ws w) {
  const int h = blockIdx.x, tid = threadIdx.x, grp = tid >> 5, lane = tid & 31, H = d.H, dk = d.dk;
  __shared__ float red[RTH];
  pdl_wait();  // the per-chunk partials of the kernel before
  if (!saved_ok(d, w.tag, w.err)) return;
  if (h == H) {  // (fused gated norm, dv = 64) dw: the (document, head) partials in a fixed order
    constexpr int NG = RTH / 64;
    const int j = tid % 64, g = tid / 64, rows = d.n_docs * H;
    float acc = 0.f;
    for (int r = g; r < rows; r += NG) acc += w.pdw[(int64_t)r * 64 + j];
    red[tid] = acc;
    __syncthreads();
    if (tid < 64) {
      float t = 0.f;
      for (int g2 = 0; g2 < NG; g2++) t += red[g2 * 64 + tid];
      io.dw[tid] = t;
    }
    return;
  }
  const int nc = *w.n_chunks;
  {  // per thread, then a fixed shuffle tree per warp, then the warps in order
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    int c = tid;
    for (; c + 3 * RTH < nc; c += 4 * RTH)
#pragma unroll
      for (int u = 0; u < 4; u++) acc[u] += w.pA[(int64_t)(c + u * RTH) * H + h];
    for (; c < nc; c += RTH) acc[0] += w.pA[(int64_t)c * H + h];
    const float x = warp_sum((acc[0] + acc[1]) + (acc[2] + acc[3]));
    if (lane == 0) red[grp] = x;
    __syncthreads();
    if (tid == 0) {
      float t = 0.f;
      for (int g = 0; g < RG; g++) t += red[g];
      io.dA_log[h] = t;
    }
  }
  float gsum = 0.f;
  for (int i0 = 0; i0 < dk; i0 += 32) {
    __syncthreads();
    const int i = i0 + lane;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    if (i < dk) {
      int c = grp;
      for (; c + 3 * RG < nc; c += 4 * RG)
#pragma unroll
        for (int u = 0; u < 4; u++) acc[u] += w.pdt[((int64_t)(c + u * RG) * H + h) * dk + i];
      for (; c < nc; c += RG) acc[0] += w.pdt[((int64_t)c * H + h) * dk + i];
    }
    red[tid] = (acc[0] + acc[1]) + (acc[2] + acc[3]);
    __syncthreads();
    if (grp == 0) {
      float t = 0.f;
      for (int g = 0; g < RG; g++) t += red[g * 32 + lane];
      if (!d.gate && i < dk) io.ddt_bias[h * dk + i] = t;
      if (d.gate) {
        t = warp_sum(i < dk ? t : 0.f);
        gsum += t;
      }
    }
  }
  if (d.gate && tid == 0) io.ddt_bias[h] = gsum;
}

template <typename TI, int DK, int DV>
static cudaError_t bwd_scan_launch(const Dims& d, const BwdIO& io, const Ws& w, cudaStream_t st) {
  size_t smem = sizeof(float) * ((DK + 2 * C) * LDS + KS * ((DK > C ? DK : C) + 1));
  cudaError_t e = cudaFuncSetAttribute(bwd_scan_kernel<TI, DK, DV>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)d.n_docs * d.H * (DV / NT));
  prof_begin(K_BWD_SCAN, st);
  bwd_scan_kernel<TI, DK, DV><<<grid, STH, smem, st>>>(d, io, w);
  prof_end(K_BWD_SCAN, st);
  return cudaGetLastError();
}

template <typename TI, int DK, int DV>
static cudaError_t bwd_intra_launch(const Dims& d, const BwdIO& io, const Ws& w, cudaStream_t st) {
  constexpr int NMAX = DK > DV ? DK : DV;
  size_t smem = sizeof(float) * (3 * C * DK + 4 * C * C + 5 * C + DK + 32 + tc5_slab_floats(NMAX > C ? NMAX : C));
  cudaError_t e = cudaFuncSetAttribute(bwd_intra_kernel<TI, DK, DV>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(d.nc_max, d.H);
  prof_begin(K_BWD_INTRA, st);
  bwd_intra_kernel<TI, DK, DV><<<grid, GTH, smem, st>>>(d, io, w);
  prof_end(K_BWD_INTRA, st);
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

cudaError_t launch_bwd_scan(int dtype, const Dims& d, const BwdIO& io, const Ws& w, cudaStream_t st) {
  KDA_DISPATCH(bwd_scan_launch, d, io, w, st);
}
cudaError_t launch_bwd_intra(int dtype, const Dims& d, const BwdIO& io, const Ws& w, cudaStream_t st) {
  KDA_DISPATCH(bwd_intra_launch, d, io, w, st);
}
cudaError_t launch_bwd_reduce(const Dims& d, const BwdIO& io, const Ws& w, cudaStream_t st) {
  prof_begin(K_BWD_REDUCE, st);
  const bool dw = d.fast && d.norm;  // one more block sums the fused norm's dw partials
  const cudaError_t e = launch_pdl(bwd_reduce_kernel, dim3(d.H + (dw ? 1 : 0)), dim3(RTH), 0, st, d, io, w);
  prof_end(K_BWD_REDUCE, st);
  return e;
}

}  // namespace kda
