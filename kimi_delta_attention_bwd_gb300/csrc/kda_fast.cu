// Tensor-core path for the 300M-layer head shape (dk = 32, dv = 64, bf16 io).
//
// Per 64-token chunk (G = in-chunk cumulative log-decay):
//   A  = strict_lower(diag(beta) (K^ K^T with ratios exp(G_r - G_s)))
//   P  = inclusive_lower(Q^ K^T with the same ratios)
//   T  = (I + A)^-1,  W = T diag(beta) (K^ exp G),  U = T diag(beta) V
//   E  = U - W S,  O = scale (Q^ exp G) S + scale P E
//   S <- Diag(exp G_last) S + (K^ exp(G_last - G))^T E
// Forward: fwd_chunk forms, for every chunk and head in parallel, the
// state-independent products M = Diag(gamma) - KD^T W, KU = KD^T U,
// QW = QG - P W and PU = P U; fwd_state then carries S' = M S + KU and writes
// O = QW S + PU, one CTA per document, head and 32 value columns.
// The ratios never appear as exp of a positive number: rows and columns are
// split in 16-token sub-blocks; block (I, J <= I) is
//   (X_I exp(G - G_first(I))) (K_J exp(G_first(I) - G))^T
// where the left factor is <= 1, the right one is <= 1 off the diagonal and
// <= exp(80) on it when the block's decay span is at most 80 nats; a wider
// diagonal block is evaluated pairwise and exactly.
// Precision: with single tf32 (or bf16) operands the gate gradient df misses
// max|err|/rms <= 1e-2 (0.18 measured at the 300M shape).  Large products
// therefore split each operand into a bf16 head and a bf16 remainder and
// accumulate three products in fp32 (mma.sync m16n8k16, ~16 significant
// bits); the pairwise decay terms of the gate gradient, whose row and column
// sums cancel in the cumulative sum, split into tf32 head + remainder
// (m16n8k8, ~21 bits).
//
// Backward: a reverse scan over each document's chunks carries dS with
//   dS_in = M^T dS_out + QW^T dO
// (M and QW per chunk come from the forward), then one CTA per chunk
// recomputes the chunk and forms every local gradient on chip.
#include "kda_internal.cuh"
#include "kda_mma.cuh"
#include "kda_tc.cuh"

#include <cudaTypedefs.h>  // PFN_cuTensorMapEncodeTiled

#include <type_traits>

namespace kda {
namespace fast {
using namespace mma;
typedef __nv_bfloat16 bf16;

constexpr int DK = 32, DV = 64;
constexpr int SQ = DK + 4;  // row stride of [C][DK] operands read along rows
constexpr int SV = DV + 8;  // row stride of [C][DV] operands
constexpr int SC = C + 4;   // row stride of [C][C] matrices
constexpr int NBLK = 10;    // lower 16 x 16 blocks of a C x C matrix, block I (I + 1) / 2 + J
constexpr int PB = 20;      // row stride of a 16 x 16 fp32 block (shared memory and the hand-over arrays)
constexpr int NTH = 256, NW = 8;
constexpr uint32_t TCOLS = 256;  // TMEM columns of a tensor-core CTA (two per SM share the 512)
constexpr float SPAN_MAX = 80.f;
// The per-chunk kernels keep G in log2 units (G2 = G log2(e)) so that every
// decay factor exp(G_a - G_b) is one exp2f of a difference.
constexpr float LOG2E = 1.4426950408889634f;
constexpr float SPAN2 = SPAN_MAX * LOG2E;
// Every tensor-core product runs with split operands (see the header).
constexpr bool SF = true;  // forward chain products

__device__ __forceinline__ int pidx(int I, int J) { return I * (I - 1) / 2 + J; }

// The chain operands of a chunk-head in one block, [KU0 | PU0 | M | QW | KU1 |
// PU1] (byte offsets below; KU, PU per 32-column half in fragment order, M, QW
// split bf16): either half's fwd_state stage (its KU and PU with the shared M
// and QW) and bwd_scan's M | QW are each one contiguous copy.
constexpr int CB_KU0 = 0, CB_PU0 = 4 * DK * 32, CB_M = CB_PU0 + 4 * C * 32, CB_QW = CB_M + 4 * DK * DK,
              CB_KU1 = CB_QW + 4 * C * DK, CB_PU1 = CB_KU1 + 4 * DK * 32, CB_BYTES = CB_PU1 + 4 * C * 32;
constexpr int CB_STAGE = CB_KU1 - CB_KU0;  // one half's stage: 24 KB from CB_KU0 (half 0) or CB_M (half 1)
static_assert(CB_BYTES == 4 * (DK * DK + C * DK + DK * DV + C * DV) && CB_BYTES - CB_M == CB_STAGE,
              "chain block layout");
__device__ __forceinline__ unsigned char* chblk(const Ws& w, int64_t ch) { return w.chb + ch * CB_BYTES; }
__device__ __forceinline__ float bfl(bf16 x) { return __bfloat162float(x); }

// Arrays of the intra-chunk recomputation shared by the forward and backward.
struct Intra {
  float *qh, *kh, *gg;     // [C][SQ]  q^, k^, G
  float *lq, *lk, *rr;     // [C][SQ]  q^ e^{G-Gb}, k^ e^{G-Gb}, k^ e^{Ge-G}
  float *bet, *inq, *ink, *braw;  // [C]
  float *gl, *gam;         // [DK]
  float *gb, *ge, *dd, *ei;  // [4][DK], [4][DK], [6][DK], [4][DK]
  float* tot;              // [NW][DK]
  int* spanok;             // [4]
};

// Stage layout of one chunk's raw inputs: q, k, f [C][DK], v [C][DV] (bf16).
constexpr int STAGE_ELEMS = 3 * C * DK + C * DV;

__device__ __forceinline__ void stage_chunk(bf16* st, const FwdIO& io, int H, int h, int t0, int L, bool gdn) {
  const bf16* q = (const bf16*)io.q;
  const bf16* k = (const bf16*)io.k;
  const bf16* f = (const bf16*)io.f;
  const bf16* v = (const bf16*)io.v;
  for (int idx = threadIdx.x; idx < C * 4; idx += NTH) {  // 4 x 16 B per dk row
    int r = idx >> 2, p = idx & 3;
    if (r < L) {
      size_t g = ((size_t)(t0 + r) * H + h) * DK + p * 8;
      cp16(st + r * DK + p * 8, q + g);
      cp16(st + C * DK + r * DK + p * 8, k + g);
      if (!gdn) cp16(st + 2 * C * DK + r * DK + p * 8, f + g);
    }
  }
  for (int idx = threadIdx.x; idx < C * 8; idx += NTH) {  // 8 x 16 B per dv row
    int r = idx >> 3, p = idx & 7;
    if (r < L) cp16(st + 3 * C * DK + r * DV + p * 8, v + ((size_t)(t0 + r) * H + h) * DV + p * 8);
  }
  cp_commit();
}

__device__ __forceinline__ void unpack8(const uint4& u, float* x) {
  const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int e = 0; e < 4; e++) {
    float2 f = __bfloat1622float2(p[e]);
    x[2 * e] = f.x;
    x[2 * e + 1] = f.y;
  }
}

// q^, k^ (L2-normalised), G (in-chunk inclusive cumulative log-decay), beta
// from the staged chunk.  Thread t owns row t / 4 and
// key channels 8 (t % 4) .. + 7 (value columns 16 (t % 4) .. + 15).  Rows
// >= L are zero (G continues flat).  vraw returns the thread's raw v.
// fg (scalar gate): f of this head, one value per token at stride H from token
// t0; dtb then points at the head's single dt_bias.
__device__ void prologue(const Intra& c, const bf16* st, int L, float a, const float* dtb, uint4 (&vraw)[2],
                         const bf16* fg, int t0, int H) {
  const int tid = threadIdx.x, r = tid >> 2, q4 = tid & 3, lane = tid & 31, warp = tid >> 5;
  float qv[8], kv[8], gv[8];
  const bool in = r < L;
  if (in) {
    unpack8(*reinterpret_cast<const uint4*>(st + r * DK + 8 * q4), qv);
    unpack8(*reinterpret_cast<const uint4*>(st + C * DK + r * DK + 8 * q4), kv);
    if (fg) {
      const float g = -a * softplus_fast(bfl(fg[(size_t)(t0 + r) * H]) + dtb[0]);
#pragma unroll
      for (int e = 0; e < 8; e++) gv[e] = g;
    } else {
      unpack8(*reinterpret_cast<const uint4*>(st + 2 * C * DK + r * DK + 8 * q4), gv);
#pragma unroll
      for (int e = 0; e < 8; e++) gv[e] = -a * softplus_fast(gv[e] + dtb[8 * q4 + e]);
    }
    vraw[0] = *reinterpret_cast<const uint4*>(st + 3 * C * DK + r * DV + 16 * q4);
    vraw[1] = *reinterpret_cast<const uint4*>(st + 3 * C * DK + r * DV + 16 * q4 + 8);
  } else {
#pragma unroll
    for (int e = 0; e < 8; e++) qv[e] = kv[e] = gv[e] = 0.f;
    vraw[0] = vraw[1] = make_uint4(0u, 0u, 0u, 0u);
  }
  float sq = 0.f, sk = 0.f;
#pragma unroll
  for (int e = 0; e < 8; e++) { sq += qv[e] * qv[e]; sk += kv[e] * kv[e]; }
  sq += __shfl_xor_sync(0xffffffffu, sq, 1);
  sq += __shfl_xor_sync(0xffffffffu, sq, 2);
  sk += __shfl_xor_sync(0xffffffffu, sk, 1);
  sk += __shfl_xor_sync(0xffffffffu, sk, 2);
  const float iq = 1.0f / sqrtf(sq + L2_EPS), ik = 1.0f / sqrtf(sk + L2_EPS);
  if (q4 == 0) {
    c.inq[r] = iq;
    c.ink[r] = ik;
    c.bet[r] = in ? sigmoid_fast(c.braw[r]) : 0.f;
  }
#pragma unroll
  for (int e = 0; e < 8; e++) {
    c.qh[r * SQ + 8 * q4 + e] = qv[e] * iq;
    c.kh[r * SQ + 8 * q4 + e] = kv[e] * ik;
  }
  // cumulative sum of g over rows: within a warp (8 rows) by shuffles among
  // lanes of equal t % 4, then across warps through smem
#pragma unroll
  for (int e = 0; e < 8; e++) {
    float x = gv[e];
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      float y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    gv[e] = x;
  }
  if (lane >= 28)
#pragma unroll
    for (int e = 0; e < 8; e++) c.tot[warp * DK + 8 * q4 + e] = gv[e];
  __syncthreads();
#pragma unroll
  for (int e = 0; e < 8; e++) {
    float off = 0.f;
    for (int w2 = 0; w2 < warp; w2++) off += c.tot[w2 * DK + 8 * q4 + e];
    c.gg[r * SQ + 8 * q4 + e] = gv[e] + off;
  }
  __syncthreads();
}

// Sub-block references (G at each 16-row block start and end), span guards,
// the per-pair channel factors and the chunk-end gate.
__device__ void refs(const Intra& c, int L) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (warp < 4) {
    const int I = warp;
    float b = c.gg[(16 * I) * SQ + lane], e = c.gg[(16 * I + 15) * SQ + lane];
    float span = b - e;
    bool ok = span <= SPAN_MAX;
    c.gb[I * DK + lane] = b;
    c.ge[I * DK + lane] = e;
    c.ei[I * DK + lane] = expf(fminf(span, SPAN_MAX));
    unsigned all = __all_sync(0xffffffffu, ok);
    if (lane == 0) c.spanok[I] = all ? 1 : 0;
  } else if (warp < 6) {  // 6 pairs I > J over two warps
    for (int p = warp - 4; p < 6; p += 2) {
      int I = p < 1 ? 1 : p < 3 ? 2 : 3, J = p - pidx(I, 0);
      c.dd[p * DK + lane] = expf(c.gg[(16 * I) * SQ + lane] - c.gg[(16 * J + 15) * SQ + lane]);
    }
  } else if (warp == 6) {
    float g = c.gg[(L - 1) * SQ + lane];
    c.gl[lane] = g;
    c.gam[lane] = expf(g);
  }
  __syncthreads();
}

// Factor arrays: lq, lk (in place of q^, k^ in the forward) and rr stay fp32
// for the decay-ratio blocks; QG = scale q^ e^G (skipped when QG.hi is
// null), KD = k^ e^{Gl - G} and XK = beta k^ e^G go to split-bf16 tiles.
__device__ void factors_fwd(const Intra& c, int L, float scale, const Op& QG, const Op& KD, const Op& XK) {
  const int tid = threadIdx.x;
  refs(c, L);
  for (int idx = tid; idx < C * DK / 2; idx += NTH) {
    const int r = idx / (DK / 2), i = 2 * (idx % (DK / 2)), I = r >> 4;
    float qg2[2], kd2[2], xk2[2];
#pragma unroll
    for (int e = 0; e < 2; e++) {
      const float G = c.gg[r * SQ + i + e];
      const float eL = expf(G - c.gb[I * DK + i + e]), eR = expf(c.ge[I * DK + i + e] - G);
      const float Gm = expf(G), kdf = expf(c.gl[i + e] - G);
      const float q = c.qh[r * SQ + i + e], k = c.kh[r * SQ + i + e];
      qg2[e] = scale * q * Gm;
      kd2[e] = k * kdf;
      xk2[e] = c.bet[r] * k * Gm;
      c.rr[r * SQ + i + e] = k * eR;
      c.lq[r * SQ + i + e] = q * eL;
      c.lk[r * SQ + i + e] = k * eL;
    }
    if (QG.hi) op_store2(QG, r, i, qg2[0], qg2[1]);
    op_store2(KD, r, i, kd2[0], kd2[1]);
    op_store2(XK, r, i, xk2[0], xk2[1]);
  }
  __syncthreads();
}

// Exact pairwise value sum_i x_ri k_si exp(G_ri - G_si) from the raw inputs
// (the diagonal-block fallback when the in-block decay span exceeds 80).
__device__ __forceinline__ float pair_exact(const bf16* X, float ix, const bf16* Kr, float ik, const float* Gr,
                                            const float* Gs) {
  float acc = 0.f;
  for (int i = 0; i < DK; i++) acc += (bfl(X[i]) * ix) * (bfl(Kr[i]) * ik) * expf(Gr[i] - Gs[i]);
  return acc;
}

// pair_exact with G in log2 units.
__device__ __forceinline__ float pair_exact2(const bf16* X, float ix, const bf16* Kr, float ik, const float* Gr,
                                             const float* Gs) {
  float acc = 0.f;
  for (int i = 0; i < DK; i++) acc += (bfl(X[i]) * ix) * (bfl(Kr[i]) * ik) * ex2(Gr[i] - Gs[i]);
  return acc;
}

// A (strict lower) and P (inclusive lower).  am gets beta_r A' (BETA) or A';
// pm gets pscale * P'.  Upper blocks are never read and are left untouched.
template <bool BETA, bool SPL = false>
__device__ void ap(const Intra& c, float* am, float* pm, float pscale, const bf16* qraw, const bf16* kraw, int H,
                   int h, int t0, int L, const Op* pop = nullptr) {
  const int warp = threadIdx.x >> 5;
  for (int task = warp; task < 20; task += NW) {
    const int blk = task >> 1, isP = task & 1;
    const int I = blk < 1 ? 0 : blk < 3 ? 1 : blk < 6 ? 2 : 3;
    const int J = blk - I * (I + 1) / 2;
    float acc[2][4];
    zero(acc);
    const float* X = isP ? c.lq : c.lk;
    if (J < I || c.spanok[I]) {
      const float* scl = J < I ? c.dd + pidx(I, J) * DK : c.ei + I * DK;
      rows16<2, SPL>(acc, DK / 8, [&](int m, int k) { return X[(16 * I + m) * SQ + k]; },
                [&](int k, int j, int n) { return c.rr[(16 * J + 8 * j + n) * SQ + k] * scl[k]; });
    } else {
      each(acc, [&](int m, int n, float& v) {
        int r = 16 * I + m, s = 16 * I + n;
        if (s <= r && r < L) {  // rows past the chunk end are not read
          const bf16* xr = (isP ? qraw : kraw) + ((size_t)(t0 + r) * H + h) * DK;
          const bf16* ks = kraw + ((size_t)(t0 + s) * H + h) * DK;
          v = pair_exact(xr, isP ? c.inq[r] : c.ink[r], ks, c.ink[s], c.gg + r * SQ, c.gg + s * SQ);
        }
      });
    }
    if (isP && pop) {  // P as a split-bf16 operand tile
      const int lane = threadIdx.x & 31, gq = lane >> 2, tq = lane & 3;
#pragma unroll
      for (int jt = 0; jt < 2; jt++)
#pragma unroll
        for (int hh = 0; hh < 2; hh++) {
          const int r = 16 * I + gq + 8 * hh, s0 = 16 * J + 8 * jt + 2 * tq;
          op_store2(*pop, r, s0, s0 <= r ? pscale * acc[jt][2 * hh] : 0.f,
                    s0 + 1 <= r ? pscale * acc[jt][2 * hh + 1] : 0.f);
        }
    } else {
      each(acc, [&](int m, int n, float& v) {
        int r = 16 * I + m, s = 16 * J + n;
        if (isP) pm[r * SC + s] = s <= r ? pscale * v : 0.f;
        else am[r * SC + s] = s < r ? (BETA ? c.bet[r] * v : v) : 0.f;
      });
    }
  }
  __syncthreads();
}

// T = (I + A)^-1 for unit-lower A (A = beta_r am_rs when !BETA).  The 16x16
// diagonal blocks by forward substitution (one lane per column), then block
// rows I = 1..3 on the tensor cores:  Y = A[I, <I] T[<I, <I],  T[I, <I] = -T_II Y.
template <bool BETA>
__device__ void solve(const float* am, float* tm, float* yy, const float* bet) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  auto A = [&](int r, int s) { return BETA ? am[r * SC + s] : bet[r] * am[r * SC + s]; };
  if (warp < 2) {
    const int I = 2 * warp + (lane >> 4), cidx = lane & 15;
    float tc[16];
#pragma unroll
    for (int r = 0; r < 16; r++) {
      float v0 = (r == cidx) ? 1.f : 0.f, v1 = 0.f;
#pragma unroll
      for (int s = 0; s + 1 < r; s += 2) {
        v0 = fmaf(-A(16 * I + r, 16 * I + s), tc[s], v0);
        v1 = fmaf(-A(16 * I + r, 16 * I + s + 1), tc[s + 1], v1);
      }
      if (r & 1) v0 = fmaf(-A(16 * I + r, 16 * I + r - 1), tc[r - 1], v0);
      tc[r] = v0 + v1;
    }
#pragma unroll
    for (int r = 0; r < 16; r++) tm[(16 * I + r) * SC + 16 * I + cidx] = tc[r];
  }
  __syncthreads();
  for (int I = 1; I < 4; I++) {
    if (warp < 2 * I) {  // Y tile w: columns 8w.. of block J = w / 2; k over blocks J..I-1
      const int J = warp >> 1, k0 = 16 * J;
      float acc[1][4];
      zero(acc);
      rows16<1, true>(acc, 2 * (I - J), [&](int m, int k) { return A(16 * I + m, k0 + k); },
                      [&](int k, int j, int n) { return tm[(k0 + k) * SC + 8 * warp + n]; });
      each(acc, [&](int m, int col, float& v) { yy[m * C + 8 * warp + col] = v; });
    }
    __syncthreads();
    if (warp < 2 * I) {
      float acc[1][4];
      zero(acc);
      rows16<1, true>(acc, 2, [&](int m, int k) { return tm[(16 * I + m) * SC + 16 * I + k]; },
                      [&](int k, int j, int n) { return yy[k * C + 8 * warp + n]; });
      each(acc, [&](int m, int col, float& v) { tm[(16 * I + m) * SC + 8 * warp + col] = -v; });
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------------ forward
// The fused forward (kda_fwd_noalloc): one CTA per (document, head) walks the
// document's chunks with S in shared memory and needs no scratch beyond the
// chunk table.  It saves nothing for the backward.
struct FwdSm {
  bf16 stage[STAGE_ELEMS];
  float qh[C * SQ], kh[C * SQ], gg[C * SQ], rr[C * SQ];  // q^ / k^ become lq / lk
  float am[C * SC];   // A (fp32) for the solve, then the split-bf16 T operand
  float tm[C * SC];   // T (fp32)
  float uf[C * SV];   // U (fp32)
  float ss[DK * SV];  // state S (fp32)
  float yy[16 * C];
  bf16 oqg[2 * C * DK], okd[2 * C * DK], oxk[2 * C * DK], ow[2 * C * DK];
  bf16 oxv[2 * C * DV];  // beta v, then E
  bf16 op[2 * C * C];    // P (scaled)
  bf16 os[2 * DK * DV];  // S
  float tot[NW * DK];
  float bet[C], inq[C], ink[C], braw[C];
  float gl[DK], gam[DK], gb[4 * DK], ge[4 * DK], dd[6 * DK], ei[4 * DK];
  int spanok[4];
};

__global__ void __launch_bounds__(NTH, 1) fwd_chain_kernel(Dims d, FwdIO io, Ws w) {
  extern __shared__ __align__(128) unsigned char smraw[];
  FwdSm& sm = *reinterpret_cast<FwdSm*>(smraw);
  const int doc = blockIdx.x, h = blockIdx.y, tid = threadIdx.x, warp = tid >> 5;
  const int lane = tid & 31, gq = lane >> 2, tq = lane & 3;
  if (*w.err != 0) return;
  const int H = d.H;
  const int cb = w.doc_chunk0[doc], ce = w.doc_chunk0[doc + 1];
  const float a = expf(io.A_log[h]);
  const bool gdn = d.gate != 0;
  const float* dtb = io.dt_bias + h * (gdn ? 1 : DK);
  const bf16* fg = gdn ? (const bf16*)io.f + h : nullptr;
  const bf16* braw = (const bf16*)io.b;
  Intra c{sm.qh, sm.kh, sm.gg, sm.qh, sm.kh, sm.rr, sm.bet, sm.inq, sm.ink,
          sm.braw, sm.gl, sm.gam, sm.gb, sm.ge, sm.dd, sm.ei, sm.tot, sm.spanok};
  const Op QG{sm.oqg, sm.oqg + C * DK, DK}, KD{sm.okd, sm.okd + C * DK, DK}, XK{sm.oxk, sm.oxk + C * DK, DK};
  const Op W{sm.ow, sm.ow + C * DK, DK}, XV{sm.oxv, sm.oxv + C * DV, DV}, E = XV;
  const Op P{sm.op, sm.op + C * C, C}, S{sm.os, sm.os + DK * DV, DV};
  const Op T{reinterpret_cast<bf16*>(sm.am), reinterpret_cast<bf16*>(sm.am) + C * C, C};

  for (int idx = tid; idx < DK * DV / 2; idx += NTH) {
    const int i = idx / (DV / 2), j = 2 * (idx % (DV / 2));
    float s0 = 0.f, s1 = 0.f;
    if (io.h0) {
      const float* hp = io.h0 + (((int64_t)doc * H + h) * DK + i) * DV + j;
      s0 = hp[0];
      s1 = hp[1];
    }
    sm.ss[i * SV + j] = s0;
    sm.ss[i * SV + j + 1] = s1;
    op_store2(S, i, j, s0, s1);
  }
  float bnext = 0.f;
  if (cb < ce) {
    const int L0 = w.chunk_len[cb], t00 = w.chunk_tok0[cb];
    stage_chunk(sm.stage, io, H, h, t00, L0, gdn);
    if (tid < L0) bnext = bfl(braw[(size_t)(t00 + tid) * H + h]);
  }
  for (int ci = cb; ci < ce; ci++) {
    const int L = w.chunk_len[ci], t0 = w.chunk_tok0[ci];
    cp_wait_all();
    if (tid < C) sm.braw[tid] = bnext;
    __syncthreads();
    uint4 vraw[2];
    prologue(c, sm.stage, L, a, dtb, vraw, fg, t0, H);
    {  // beta v -> XV (thread: row tid / 4, columns 16 (tid % 4) ..)
      const int r = tid >> 2, q4 = tid & 3;
      const float br = r < L ? sm.bet[r] : 0.f;
      float vv[16];
      unpack8(vraw[0], vv);
      unpack8(vraw[1], vv + 8);
#pragma unroll
      for (int e = 0; e < 16; e += 2) op_store2(XV, r, 16 * q4 + e, br * vv[e], br * vv[e + 1]);
    }
    if (ci + 1 < ce) {  // stage the next chunk while this one computes
      const int L1 = w.chunk_len[ci + 1], t01 = w.chunk_tok0[ci + 1];
      stage_chunk(sm.stage, io, H, h, t01, L1, gdn);
      bnext = tid < L1 ? bfl(braw[(size_t)(t01 + tid) * H + h]) : 0.f;
    }
    factors_fwd(c, L, d.scale, QG, KD, XK);
    ap<true, SF>(c, sm.am, nullptr, d.scale, (const bf16*)io.q, (const bf16*)io.k, H, h, t0, L, &P);
    solve<true>(sm.am, sm.tm, sm.yy, sm.bet);
    for (int idx = tid; idx < C * C / 2; idx += NTH) {  // T -> split-bf16 operand (over A's storage)
      const int r = idx / (C / 2), s2 = 2 * (idx % (C / 2));
      op_store2(T, r, s2, sm.tm[r * SC + s2], sm.tm[r * SC + s2 + 1]);
    }
    __syncthreads();
    {  // W | U = T [XK | XV]  (T lower block-triangular: k < 16 (I + 1))
      const int I = warp & 3, half = warp >> 2;
      if (half == 0) {
        float aw[4][4], au[2][4];
        zero(aw);
        zero(au);
        gemm3<2, false, true>(aw, T, 16 * I, 0, XK, 0, 0, I + 1);
        gemm3<1, false, true>(au, T, 16 * I, 0, XV, 0, 0, I + 1);
#pragma unroll
        for (int jt = 0; jt < 4; jt++)
#pragma unroll
          for (int hh = 0; hh < 2; hh++)
            op_store2(W, 16 * I + gq + 8 * hh, 8 * jt + 2 * tq, aw[jt][2 * hh], aw[jt][2 * hh + 1]);
        each(au, [&](int m, int col, float& v) { sm.uf[(16 * I + m) * SV + col] = v; });
      } else {
        float au[6][4];
        zero(au);
        gemm3<3, false, true>(au, T, 16 * I, 0, XV, 16, 0, I + 1);
        each(au, [&](int m, int col, float& v) { sm.uf[(16 * I + m) * SV + 16 + col] = v; });
      }
    }
    __syncthreads();
    {  // E = U - W S  (into XV's storage)
      const int I = warp & 3, half = warp >> 2;
      float acc[4][4];
      zero(acc);
      gemm3<2, false, true>(acc, W, 16 * I, 0, S, 32 * half, 0, DK / 16);
#pragma unroll
      for (int jt = 0; jt < 4; jt++)
#pragma unroll
        for (int hh = 0; hh < 2; hh++) {
          const int r = 16 * I + gq + 8 * hh, col = 32 * half + 8 * jt + 2 * tq;
          op_store2(E, r, col, sm.uf[r * SV + col] - acc[jt][2 * hh], sm.uf[r * SV + col + 1] - acc[jt][2 * hh + 1]);
        }
    }
    __syncthreads();
    {  // O = QG S + P E  -> o
      const int I = warp & 3, half = warp >> 2;
      float acc[4][4];
      zero(acc);
      gemm3<2, false, true>(acc, QG, 16 * I, 0, S, 32 * half, 0, DK / 16);
      gemm3<2, false, true>(acc, P, 16 * I, 0, E, 32 * half, 0, I + 1);
      bf16* o = (bf16*)io.o;
#pragma unroll
      for (int j = 0; j < 4; j++)
#pragma unroll
        for (int hh = 0; hh < 2; hh++) {
          int r = 16 * I + gq + 8 * hh;
          if (r < L) {
            int col = 32 * half + 8 * j + 2 * tq;
            *reinterpret_cast<__nv_bfloat162*>(o + ((size_t)(t0 + r) * H + h) * DV + col) =
                __floats2bfloat162_rn(acc[j][2 * hh], acc[j][2 * hh + 1]);
          }
        }
    }
    float snew[2][4];
    const int mI = warp & 1, jq = warp >> 1;
    {  // S' = gamma S + KD^T E (registers until every reader of S is done)
      zero(snew);
      gemm3<1, true, true>(snew, KD, 16 * mI, 0, E, 16 * jq, 0, C / 16);
      each(snew, [&](int m, int col, float& v) {
        int i = 16 * mI + m;
        v += sm.gam[i] * sm.ss[i * SV + 16 * jq + col];
      });
    }
    __syncthreads();
#pragma unroll
    for (int jt = 0; jt < 2; jt++)
#pragma unroll
      for (int hh = 0; hh < 2; hh++) {
        const int i = 16 * mI + gq + 8 * hh, col = 16 * jq + 8 * jt + 2 * tq;
        sm.ss[i * SV + col] = snew[jt][2 * hh];
        sm.ss[i * SV + col + 1] = snew[jt][2 * hh + 1];
        op_store2(S, i, col, snew[jt][2 * hh], snew[jt][2 * hh + 1]);
      }
    __syncthreads();
  }
  __syncthreads();  // other threads wrote ss (for an empty document: the initial state just above)
  if (io.h_final)
    for (int idx = tid; idx < DK * DV; idx += NTH) {
      int i = idx / DV, j = idx % DV;
      io.h_final[(((int64_t)doc * H + h) * DK + i) * DV + j] = sm.ss[i * SV + j];
    }
}

// ------------------------------------------------------------------ forward
// The forward runs in two kernels.  fwd_chunk (one CTA per chunk-head, all in
// parallel) forms everything that does not depend on the carried state:
//   M  = Diag(gamma) - KD^T W   [dk x dk]      KU = KD^T U   [dk x dv]
//   QW = QG - P W               [C x dk]       PU = P U      [C x dv]
// so that the chunk's state update and output are
//   S' = M S + KU,   O = QW S + PU.
// fwd_state then carries S through each document's chunks and writes O.

// Rows of the decay-ratio right operands: R_I holds k^_s exp(G_first(I) - G_s)
// for the 16 (I + 1) rows s of blocks J <= I, stacked from row 8 I (I + 1).
__device__ __forceinline__ int roff(int I) { return 8 * I * (I + 1); }

// ---- fwd_chunk's solve, T = (I + A)^-1, by merging block inverses: a
// unit-lower [[I + A_a, 0], [A_ba, I + A_b]] has the inverse
// [[T_a, 0], [-T_b A_ba T_a, T_b]].  The four 16 x 16 diagonal inverses come
// from forward substitution (one warp each, inside the A / P step), merge into
// the two 32 x 32 ones and those into T: four rounds of small products instead
// of a row-by-row sweep.

// Diagonal inverse I is kept in an upper block of the A array (never written
// by the A / P step): (0, 1), (0, 2), (0, 3), (1, 3).
__device__ __forceinline__ int tdoff(int I) { return I < 3 ? 16 * (I + 1) : 16 * SC + 48; }

// Forward substitution of diagonal block I of A (beta-scaled, fp32, stride
// SC) by one warp, lane c % 16 owning column c; T_II to td (stride SC).
__device__ __forceinline__ void diag_inverse(const float* am, float* td, int I) {
  const int lane = threadIdx.x & 31, cidx = lane & 15;
  const float* Ab = am + (16 * I) * SC + 16 * I;
  float tc[16];
#pragma unroll
  for (int r = 0; r < 16; r++) {
    float v0 = (r == cidx) ? 1.f : 0.f, v1 = 0.f;
#pragma unroll
    for (int s = 0; s + 1 < r; s += 2) {
      v0 = fmaf(-Ab[r * SC + s], tc[s], v0);
      v1 = fmaf(-Ab[r * SC + s + 1], tc[s + 1], v1);
    }
    if (r & 1) v0 = fmaf(-Ab[r * SC + r - 1], tc[r - 1], v0);
    tc[r] = v0 + v1;
  }
  if (lane < 16)
#pragma unroll
    for (int r = 0; r < 16; r++) td[r * SC + cidx] = tc[r];
}

// (x0, x1) as bf16 pairs: hi = bf16(x), lo = bf16(x - hi).
__device__ __forceinline__ void split_bf2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  const float2 hf = __bfloat1622float2(h);
  const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

// acc (a 16 x 8 m16n8 fragment) = sum over k < 16 KS of fl(m, k) fr(k, n) in
// split bf16 (hi*hi + hi*lo + lo*hi, about 16 bits, the precision of the
// split tiles the products' results are stored in); all operand loads are
// issued before the products.
template <int KS, class FL, class FR>
__device__ __forceinline__ void tile_bf16s(float (&acc)[4], FL fl, FR fr) {
  const int lane = threadIdx.x & 31, gq = lane >> 2, tq = lane & 3;
  uint32_t ah[KS][4], al[KS][4], bh[KS][2], bl[KS][2];
#pragma unroll
  for (int ks = 0; ks < KS; ks++) {
    const int k0 = 16 * ks + 2 * tq;
    split_bf2(fl(gq, k0), fl(gq, k0 + 1), ah[ks][0], al[ks][0]);
    split_bf2(fl(gq + 8, k0), fl(gq + 8, k0 + 1), ah[ks][1], al[ks][1]);
    split_bf2(fl(gq, k0 + 8), fl(gq, k0 + 9), ah[ks][2], al[ks][2]);
    split_bf2(fl(gq + 8, k0 + 8), fl(gq + 8, k0 + 9), ah[ks][3], al[ks][3]);
    split_bf2(fr(k0, gq), fr(k0 + 1, gq), bh[ks][0], bl[ks][0]);
    split_bf2(fr(k0 + 8, gq), fr(k0 + 9, gq), bh[ks][1], bl[ks][1]);
  }
  acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
#pragma unroll
  for (int ks = 0; ks < KS; ks++) {
    mma_bf16(acc, ah[ks], bh[ks][0], bh[ks][1]);
    mma_bf16(acc, ah[ks], bl[ks][0], bl[ks][1]);
    mma_bf16(acc, al[ks], bh[ks][0], bh[ks][1]);
  }
}
template <class F>
__device__ __forceinline__ void tile_store(const float (&acc)[4], F fn) {
  const int lane = threadIdx.x & 31, gq = lane >> 2, tq = lane & 3;
  fn(gq, 2 * tq, acc[0]);
  fn(gq, 2 * tq + 1, acc[1]);
  fn(gq + 8, 2 * tq, acc[2]);
  fn(gq + 8, 2 * tq + 1, acc[3]);
}

constexpr int YS = 40;  // row stride of the merge scratch [32][YS]

// The merges after the diagonal inverses (in the td blocks of am): T's lower
// blocks assembled in tm (fp32, stride SC); yy is scratch.  Ends with a barrier.
__device__ void solve_merge(const float* am, float* tm, float* yy) {
  const int tid = threadIdx.x, warp = tid >> 5;
  if (warp < 4) {  // X_10 = A_10 T_00 and X_32 = A_32 T_22
    const int p = warp >> 1, n0 = 8 * (warp & 1);
    const float* Al = am + (16 + 32 * p) * SC + 32 * p;
    const float* Tr = am + tdoff(2 * p) + n0;
    float acc[4];
    tile_bf16s<1>(acc, [&](int m, int k) { return Al[m * SC + k]; }, [&](int k, int n) { return Tr[k * SC + n]; });
    tile_store(acc, [&](int m, int n, float v) { yy[(16 * p + m) * YS + n0 + n] = v; });
  } else {  // the diagonal inverses into T
    for (int idx = tid - 128; idx < 4 * 256; idx += 128) {
      const int I = idx >> 8, r = (idx >> 4) & 15, c = idx & 15;
      tm[(16 * I + r) * SC + 16 * I + c] = am[tdoff(I) + r * SC + c];
    }
  }
  __syncthreads();
  if (warp < 4) {  // T_10 = -T_11 X_10 and T_32 = -T_33 X_32
    const int p = warp >> 1, n0 = 8 * (warp & 1);
    const float* Tl = am + tdoff(2 * p + 1);
    float acc[4];
    tile_bf16s<1>(acc, [&](int m, int k) { return Tl[m * SC + k]; },
                 [&](int k, int n) { return yy[(16 * p + k) * YS + n0 + n]; });
    float* out = tm + (16 + 32 * p) * SC + 32 * p + n0;
    tile_store(acc, [&](int m, int n, float v) { out[m * SC + n] = -v; });
  }
  __syncthreads();
  const int rb = warp >> 2, n0 = 8 * (warp & 3);  // one 16 x 8 tile of a 32 x 32 block per warp
  {  // Y = A[32.., ..32) T[..32, ..32): columns 16.. of the lower T need k >= 16 only
    const float* Al = am + (32 + 16 * rb) * SC;
    float acc[4];
    if (n0 < 16)
      tile_bf16s<2>(acc, [&](int m, int k) { return Al[m * SC + k]; }, [&](int k, int n) { return tm[k * SC + n0 + n]; });
    else
      tile_bf16s<1>(acc, [&](int m, int k) { return Al[m * SC + 16 + k]; },
                   [&](int k, int n) { return tm[(16 + k) * SC + n0 + n]; });
    tile_store(acc, [&](int m, int n, float v) { yy[(16 * rb + m) * YS + n0 + n] = v; });
  }
  __syncthreads();
  {  // T[32.., ..32) = -T[32.., 32..) Y: rows 32..47 of the lower T need k < 16 only
    const float* Tl = tm + (32 + 16 * rb) * SC + 32;
    float acc[4];
    if (rb == 0)
      tile_bf16s<1>(acc, [&](int m, int k) { return Tl[m * SC + k]; }, [&](int k, int n) { return yy[k * YS + n0 + n]; });
    else
      tile_bf16s<2>(acc, [&](int m, int k) { return Tl[m * SC + k]; }, [&](int k, int n) { return yy[k * YS + n0 + n]; });
    float* out = tm + (32 + 16 * rb) * SC + n0;
    tile_store(acc, [&](int m, int n, float v) { out[m * SC + n] = -v; });
  }
  __syncthreads();
}

// Shared memory of fwd_chunk (about 104 KB: two CTAs per SM).  bf16 arrays
// are split operand tiles; regions are reused as noted.
struct ChunkSm {
  float gg[C * SQ];    // G2 = G log2(e) (fp32); QG (split) once the A / P blocks are done
  bf16 x[18432];       // LQ | LK | R  ->  T (fp32) + Y scratch  ->  [W | U];  KD in the last 8 KB
  float am[C * SC];    // beta_r A (fp32), then T (split)
  bf16 op[2 * C * C];  // P (scaled, split)
  bf16 y[2 * C * DK + 2 * C * DV];  // [XK | XV] (XK = beta k^ e^G, XV = beta v)  ->  W | U for the save
  float bet[C], inq[C], ink[C];
  float gam[DK];
  float tot[NW * DK];
  int spanok[4];
  uint64_t bar;    // tensor-core rounds
  uint32_t tslot;  // TMEM base address
};

// The six upper 16 x 16 blocks of a C x C split tile set to zero (the backward
// reads whole tiles with the tensor core).
__device__ __forceinline__ void zero_upper(const Op& t) {
  for (int idx = threadIdx.x; idx < 6 * 16 * 8; idx += NTH) {
    const int u = idx >> 7, rem = idx & 127;
    const int bI = u < 3 ? 0 : u < 5 ? 1 : 2, bJ = u < 3 ? u + 1 : u < 5 ? u - 1 : 3;
    op_store2(t, 16 * bI + (rem >> 3), 16 * bJ + 2 * (rem & 7), 0.f, 0.f);
  }
}

// The per-chunk kernels run on a 1-D grid, heads fastest: CTA n is chunk n / H
// of head n % H, so the H heads of a chunk, whose rows share the token-major
// 128-byte lines, run together.  ahead_of gives the chunk-head that fwd_chunk
// runs d.ahead CTAs (half a wave) after CTA (j, h), from registers only; false
// past the last chunk.  Its table row is loaded with the CTA's own (rows past
// the last chunk have length 0), and prefetching its inputs into L2 turns the
// later CTA's cold DRAM reads into L2 hits.
__device__ __forceinline__ bool ahead_of(const Dims& d, int j, int h, int& j2, int& h2) {
  const int64_t nxt = (int64_t)j * d.H + h + d.ahead;
  j2 = (int)(nxt / d.H);
  h2 = (int)(nxt % d.H);
  return d.ahead > 0 && j2 < d.nc_max;
}
// A thread's 8 consecutive channel values rotated by q4 pairs in place:
// v'[2 p + b] = v[2 ((p + q4) & 3) + b].  Stored by store8_rot, the 32 lanes of
// a warp (8 rows x 4 channel groups, one core matrix each) then write 32
// different banks instead of 8.
__device__ __forceinline__ void rot_pairs(float (&v)[8], int q4) {
  float t[8];
#pragma unroll
  for (int i = 0; i < 8; i++) t[i] = (q4 & 1) ? v[(i + 2) & 7] : v[i];
#pragma unroll
  for (int i = 0; i < 8; i++) v[i] = (q4 & 2) ? t[(i + 4) & 7] : t[i];
}
__device__ __forceinline__ void store8_rot(const Op& t, int r, int c0, const float (&v)[8], int q4) {
#pragma unroll
  for (int p = 0; p < 4; p++) op_store2(t, r, c0 + 2 * ((p + q4) & 3), v[2 * p], v[2 * p + 1]);
}
// Adds to g[e] (channel 8 q4 + e of this thread's row) the totals of the rows
// of the earlier warps (tot: each warp's last-row inclusive sums, [NW][DK]),
// in warp order: lane c forms channel c's prefix and shuffles hand each
// thread its eight.
__device__ __forceinline__ void add_warp_prefix(float (&g)[8], const float* tot, int warp, int lane, int q4) {
  float pre = 0.f;
#pragma unroll
  for (int w2 = 0; w2 < NW - 1; w2++)
    if (w2 < warp) pre += tot[w2 * DK + lane];
#pragma unroll
  for (int e = 0; e < 8; e++) g[e] += __shfl_sync(0xffffffffu, pre, 8 * q4 + e);
}
// Row r, channels 8 q4 .. 8 q4 + 7 of a [C][SQ] fp32 array (two 16-byte stores).
__device__ __forceinline__ void store_row8(float* gg, int r, int q4, const float (&g)[8]) {
  float4* p = reinterpret_cast<float4*>(gg + r * SQ + 8 * q4);
  p[0] = make_float4(g[0], g[1], g[2], g[3]);
  p[1] = make_float4(g[4], g[5], g[6], g[7]);
}
// Thread tid < L prefetches row tid of a [tokens][H][n] bf16 tensor (n * 2 <= 128 bytes).
__device__ __forceinline__ void prefetch_rows(const void* base, int n, int t0, int L, int H, int h) {
  if ((int)threadIdx.x < L) prefetch_l2((const bf16*)base + ((size_t)(t0 + threadIdx.x) * H + h) * n);
}

// Stores a 16 x (8 NT) accumulator tile at (r0, c0) of a split operand tile
// (global or shared), mapping each value through fn(r, c, v).
template <int NT, class F>
__device__ __forceinline__ void store_acc_op(const float (&acc)[NT][4], const Op& g, int r0, int c0, F fn) {
  const int lane = threadIdx.x & 31, gq = lane >> 2, tq = lane & 3;
#pragma unroll
  for (int jt = 0; jt < NT; jt++)
#pragma unroll
    for (int hh = 0; hh < 2; hh++) {
      const int r = r0 + gq + 8 * hh, c = c0 + 8 * jt + 2 * tq;
      op_store2(g, r, c, fn(r, c, acc[jt][2 * hh]), fn(r, c + 1, acc[jt][2 * hh + 1]));
    }
}

// Stores a 16 x (8 NT) accumulator tile to a row-major fp32 matrix with
// leading dimension ld at (r0, c0), mapping each value through fn(r, c, v).
template <int NT, class F>
__device__ __forceinline__ void store_acc(const float (&acc)[NT][4], float* g, int ld, int r0, int c0, F fn) {
  const int lane = threadIdx.x & 31, gq = lane >> 2, tq = lane & 3;
#pragma unroll
  for (int jt = 0; jt < NT; jt++)
#pragma unroll
    for (int hh = 0; hh < 2; hh++) {
      const int r = r0 + gq + 8 * hh, c = c0 + 8 * jt + 2 * tq;
      *reinterpret_cast<float2*>(g + (size_t)r * ld + c) =
          make_float2(fn(r, c, acc[jt][2 * hh]), fn(r, c + 1, acc[jt][2 * hh + 1]));
    }
}

// ---- the short convolution fused into the prologues ("Pure KDA 300M" guide,
// Overview: short-conv kernel size 4, depthwise on the concatenated QKV;
// torchtitan PR "[kimi k3] Support sample packing in KDA": the window resets
// at each document start):  u_t,c = silu(sum_j w_c,j x_{t-3+j,c}), with x of
// tokens before the document start taken as 0.  Every kernel that needs q, k
// or v recomputes them from x with these helpers, in the same order of
// operations, so the forward and the backward see the same bits.
__device__ __forceinline__ float silu_f(float z) { return z * sigmoid_fast(z); }
// N consecutive channels (N a multiple of 8) of token t: x points at channel 0
// of them in token 0's row, rows ld elements apart; wc at their taps [N][4];
// tokens below tmin read as zero.
template <int N>
__device__ __forceinline__ void conv_load(float* out, const bf16* x, int ld, int t, int tmin, const float* wc) {
#pragma unroll
  for (int e8 = 0; e8 < N; e8 += 8) {
    uint4 raw[4];  // the window's four rows, issued together; rows before tmin read as 0
#pragma unroll
    for (int jt = 0; jt < 4; jt++) {
      const int tt = t - 3 + jt;
      raw[jt] = tt >= tmin ? __ldg(reinterpret_cast<const uint4*>(x + (size_t)tt * ld + e8)) : make_uint4(0u, 0u, 0u, 0u);
    }
    // element e of a row's 8 bf16 (exact widening: the bf16 bits are the fp32's top half)
    auto xe = [&](int jt, int e) {
      const uint32_t wd = e < 2 ? raw[jt].x : e < 4 ? raw[jt].y : e < 6 ? raw[jt].z : raw[jt].w;
      return __uint_as_float((e & 1) ? (wd & 0xffff0000u) : (wd << 16));
    };
#pragma unroll
    for (int e = 0; e < 8; e++) {
      const float4 w4 = __ldg(reinterpret_cast<const float4*>(wc + 4 * (e8 + e)));  // taps of one channel
      float z = fmaf(w4.x, xe(0, e), 0.f);
      z = fmaf(w4.y, xe(1, e), z);
      z = fmaf(w4.z, xe(2, e), z);
      z = fmaf(w4.w, xe(3, e), z);
      out[e8 + e] = silu_f(z);
    }
  }
}
// One channel (the exact wide-span fallback's operands): conv_load's value,
// with the same operations in the same order (a token before tmin gives a
// zero term, which leaves z unchanged exactly as the skipped row does).
__device__ __forceinline__ float conv_one(const bf16* x, int ld, int t, int tmin, const float* wc) {
  const float4 w4 = __ldg(reinterpret_cast<const float4*>(wc));
  auto xa = [&](int jt) { const int tt = t - 3 + jt; return tt >= tmin ? bfl(x[(size_t)tt * ld]) : 0.f; };
  float z = fmaf(w4.x, xa(0), 0.f);
  z = fmaf(w4.y, xa(1), z);
  z = fmaf(w4.z, xa(2), z);
  z = fmaf(w4.w, xa(3), z);
  return silu_f(z);
}
// The exact diagonal-block value of pair_exact2 with q / k recomputed through
// the convolution (X: the q or k block, Kx: the k block, channel 0 of head h).
__device__ __forceinline__ float pair_exact2_conv(const bf16* X, const float* wX, float ix, const bf16* Kx,
                                                  const float* wK, float ik, int ld, int tr, int ts, int tmin,
                                                  const float* Gr, const float* Gs) {
  float acc = 0.f;
  for (int i = 0; i < DK; i++)
    acc += (conv_one(X + i, ld, tr, tmin, wX + 4 * i) * ix) * (conv_one(Kx + i, ld, ts, tmin, wK + 4 * i) * ik) *
           ex2(Gr[i] - Gs[i]);
  return acc;
}
// First token whose x is read for chunk j starting at t0: the 3 tokens before
// t0 belong to the chunk's document when the chunk before it does.
__device__ __forceinline__ int conv_tmin(const Ws& w, int j, int t0) {
  return (j > 0 && w.chunk_doc[j - 1] == w.chunk_doc[j]) ? t0 - 3 : t0;
}

static_assert(offsetof(ChunkSm, x) % 16 == 0 && offsetof(ChunkSm, am) % 16 == 0 && offsetof(ChunkSm, op) % 16 == 0 &&
                  offsetof(ChunkSm, y) % 16 == 0,
              "operand tiles need 16-byte rows");

template <bool CONV>
__global__ void __launch_bounds__(NTH, 2) fwd_chunk_kernel(Dims d, FwdIO io, Ws w) {
  extern __shared__ __align__(128) unsigned char smraw[];
  ChunkSm& sm = *reinterpret_cast<ChunkSm*>(smraw);
  const int j = (int)(blockIdx.x / (unsigned)d.H), h = (int)(blockIdx.x % (unsigned)d.H), tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Equal rows (d.rows): chunk j is chunk j % nr of row j / nr, so this kernel reads no table and
  // runs alongside the chunk-table kernel; it waits for that grid before it ends, so that the
  // kernels after it find the table complete.  Otherwise it waits for the table first.
  const bool rows = d.rows != 0;
  if (!rows) pdl_wait();  // the chunk table of the kernel before
  pdl_release();          // fwd_state may launch (it waits for this grid)
  int j2, h2;
  const bool pf = ahead_of(d, j, h, j2, h2);
  int err = 0, L, t0, L2 = 0, t2 = 0;
  if (rows) {
    const int nr = (d.T + C - 1) / C;
    auto at = [&](int jj, int& len, int& tok) {
      const int c = jj % nr;
      tok = (jj / nr) * d.T + c * C;
      len = min(C, d.T - c * C);
    };
    at(j, L, t0);
    if (pf) at(j2, L2, t2);
  } else {
    err = *w.err;
    L = w.chunk_len[j];
    t0 = w.chunk_tok0[j];  // one round trip
    L2 = pf ? w.chunk_len[j2] : 0;
    t2 = pf ? w.chunk_tok0[j2] : 0;
  }
  struct TableWait {  // (equal rows) wait for the chunk-table grid on every way out
    bool on;
    __device__ ~TableWait() {
      if (on) pdl_wait();
    }
  } table_wait{rows};
  if (err != 0 || L <= 0) return;
  const int H = d.H;
  const int64_t ch = (int64_t)j * H + h;
  const float a = expf(io.A_log[h]), scale = d.scale;
  const bool gdn = d.gate != 0;
  const float* dtb = io.dt_bias + h * (gdn ? 1 : DK);
  const bf16* qraw = (const bf16*)io.q;
  const bf16* kraw = (const bf16*)io.k;
  if (warp == 0) tc::tmem_alloc(&sm.tslot, TCOLS);  // published by the first barrier below
  // The raw inputs are loaded straight into the registers of the thread that uses them (a
  // tensor-map staging through shared memory measured 1.8% slower here: one more barrier and
  // a shared-memory round trip for data no other thread reads).
  if (tid == 0) {
    mbar_init(&sm.bar, 1);
    mbar_init_fence();
  }
  if (L2 > 0) {
    if constexpr (CONV) {  // rows of the q, k, v blocks of x
      if ((int)threadIdx.x < L2) {
        const size_t o2 = (size_t)(t2 + threadIdx.x) * io.ld;
        prefetch_l2(qraw + o2 + h2 * DK);
        prefetch_l2(kraw + o2 + h2 * DK);
        prefetch_l2((const bf16*)io.v + o2 + h2 * DV);
      }
    } else {
      prefetch_rows(io.q, DK, t2, L2, H, h2);
      prefetch_rows(io.k, DK, t2, L2, H, h2);
      prefetch_rows(io.v, DV, t2, L2, H, h2);
    }
    prefetch_rows(io.f, gdn ? 1 : DK, t2, L2, H, h2);
    prefetch_rows(io.b, 1, t2, L2, H, h2);
  }
  const int tmin = !CONV ? t0 : rows ? (j % ((d.T + C - 1) / C) > 0 ? t0 - 3 : t0) : conv_tmin(w, j, t0);

  const Op LQ{sm.x, sm.x + 2048, DK}, LK{sm.x + 4096, sm.x + 6144, DK}, R{sm.x + 8192, sm.x + 13312, DK};
  // [XK | XV] and [W | U] are single 96-column tiles (one tensor-core operand
  // each); W and U for the backward are copied apart over XKV once it is read
  const Op WU{sm.x, sm.x + 6144, DK + DV}, KD{sm.x + 14336, sm.x + 16384, DK};
  const Op XKV{sm.y, sm.y + 6144, DK + DV}, Ws{sm.y, sm.y + 2048, DK}, Us{sm.y + 4096, sm.y + 8192, DV};
  const Op P{sm.op, sm.op + C * C, C};
  const Op T{reinterpret_cast<bf16*>(sm.am), reinterpret_cast<bf16*>(sm.am) + C * C, C};
  bf16* qgb = reinterpret_cast<bf16*>(sm.gg);
  const Op QG{qgb, qgb + C * DK, DK};
  float* tm = reinterpret_cast<float*>(sm.x);  // [C][SC]
  float* yy = tm + C * SC;                     // [32][YS], below KD
  static_assert((C * SC + 32 * YS) * 4 <= 14336 * 2, "solve scratch overlaps KD");

  // ---- prologue in registers: thread = row r (tid / 4), key channels 8 (tid % 4) ..,
  //      value columns 16 (tid % 4) ..; rows >= L are zero with G flat
  const int r = tid >> 2, q4 = tid & 3, I = r >> 4;
  const bool in = r < L;
  float qv[8], kv[8], gv[8], vv[16], braw = 0.f;
  if (in) {
    const size_t row = (size_t)(t0 + r) * H + h;
    if constexpr (CONV) {  // (v is convolved where beta v is stored, below)
      conv_load<8>(qv, qraw + h * DK + 8 * q4, io.ld, t0 + r, tmin, io.cwq + 4 * (h * DK + 8 * q4));
      conv_load<8>(kv, kraw + h * DK + 8 * q4, io.ld, t0 + r, tmin, io.cwk + 4 * (h * DK + 8 * q4));
    } else {
      unpack8(__ldg(reinterpret_cast<const uint4*>(qraw + row * DK + 8 * q4)), qv);
      unpack8(__ldg(reinterpret_cast<const uint4*>(kraw + row * DK + 8 * q4)), kv);
      const uint4* vp = reinterpret_cast<const uint4*>((const bf16*)io.v + row * DV + 16 * q4);
      unpack8(__ldg(vp), vv);
      unpack8(__ldg(vp + 1), vv + 8);
    }
    if (!gdn) unpack8(__ldg(reinterpret_cast<const uint4*>((const bf16*)io.f + row * DK + 8 * q4)), gv);
    braw = bfl(((const bf16*)io.b)[row]);
    if (gdn) {
      const float g = -a * LOG2E * softplus_fast(bfl(((const bf16*)io.f)[row]) + dtb[0]);
#pragma unroll
      for (int e = 0; e < 8; e++) gv[e] = g;
    } else {
#pragma unroll
      for (int e = 0; e < 8; e++) gv[e] = -a * LOG2E * softplus_fast(gv[e] + dtb[8 * q4 + e]);
    }
  } else {
#pragma unroll
    for (int e = 0; e < 8; e++) qv[e] = kv[e] = gv[e] = 0.f;
#pragma unroll
    for (int e = 0; e < 16; e++) vv[e] = 0.f;
  }
  if (tid < 4) sm.spanok[tid] = 1;
  float sq = 0.f, sk = 0.f;
#pragma unroll
  for (int e = 0; e < 8; e++) { sq += qv[e] * qv[e]; sk += kv[e] * kv[e]; }
  sq += __shfl_xor_sync(0xffffffffu, sq, 1);
  sq += __shfl_xor_sync(0xffffffffu, sq, 2);
  sk += __shfl_xor_sync(0xffffffffu, sk, 1);
  sk += __shfl_xor_sync(0xffffffffu, sk, 2);
  const float iq = 1.0f / sqrtf(sq + L2_EPS), ik = 1.0f / sqrtf(sk + L2_EPS);
  const float beta = in ? sigmoid_fast(braw) : 0.f;
  if (q4 == 0) {
    sm.bet[r] = beta;
    sm.inq[r] = iq;
    sm.ink[r] = ik;
  }
#pragma unroll
  for (int hv = 0; hv < 2; hv++) {  // XV = beta v (its region is free from the start)
    float xv[8];
    if constexpr (CONV) {
      if (in)
        conv_load<8>(xv, (const bf16*)io.v + h * DV + 16 * q4 + 8 * hv, io.ld, t0 + r, tmin,
                     io.cwv + 4 * (h * DV + 16 * q4 + 8 * hv));
#pragma unroll
      for (int e = 0; e < 8; e++) xv[e] = in ? beta * xv[e] : 0.f;
    } else {
#pragma unroll
      for (int e = 0; e < 8; e++) xv[e] = beta * vv[8 * hv + e];
    }
    rot_pairs(xv, q4);
    store8_rot(XKV, r, DK + 16 * q4 + 8 * hv, xv, q4);
  }
#pragma unroll
  for (int e = 0; e < 8; e++) { qv[e] *= iq; kv[e] *= ik; }
  // cumulative sum of g over rows: shuffles among lanes of equal tid % 4, then warp offsets
#pragma unroll
  for (int e = 0; e < 8; e++) {
    float x = gv[e];
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      const float y2 = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y2;
    }
    gv[e] = x;
  }
  if (lane >= 28)
#pragma unroll
    for (int e = 0; e < 8; e++) sm.tot[warp * DK + 8 * q4 + e] = gv[e];
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tb = sm.tslot;
  add_warp_prefix(gv, sm.tot, warp, lane, q4);
  store_row8(sm.gg, r, q4, gv);
  __syncthreads();

  // ---- factors: LQ, LK, R (decay-ratio operands), XK, XV; QG and KD stay in
  //      registers until their storage frees up
  float qg[8], kd[8];
  {
    float gbv[8], xk[8];
    bool wide = false;
#pragma unroll
    for (int e = 0; e < 8; e++) {
      gbv[e] = sm.gg[(16 * I) * SQ + 8 * q4 + e];
      const float gl = sm.gg[(L - 1) * SQ + 8 * q4 + e];
      const float eG = ex2(gv[e]);
      qg[e] = scale * qv[e] * eG;
      kd[e] = kv[e] * ex2(gl - gv[e]);
      xk[e] = beta * kv[e] * eG;
      if (r == 0) sm.gam[8 * q4 + e] = ex2(gl);
      wide |= (r & 15) == 15 && gbv[e] - gv[e] > SPAN2;
    }
    if (wide) sm.spanok[I] = 0;
    {
      float lq[8], lk[8];
#pragma unroll
      for (int e = 0; e < 8; e++) {
        const float l = ex2(gv[e] - gbv[e]);
        lq[e] = qv[e] * l;
        lk[e] = kv[e] * l;
      }
      rot_pairs(lq, q4);
      rot_pairs(lk, q4);
      rot_pairs(xk, q4);
      store8_rot(LQ, r, 8 * q4, lq, q4);
      store8_rot(LK, r, 8 * q4, lk, q4);
      store8_rot(XKV, r, 8 * q4, xk, q4);
      rot_pairs(qg, q4);  // stored after the A / P blocks
      rot_pairs(kd, q4);
    }
    for (int I2 = I; I2 < 4; I2++) {
      float rv[8];
#pragma unroll
      for (int e = 0; e < 8; e++) rv[e] = kv[e] * ex2(fminf(sm.gg[(16 * I2) * SQ + 8 * q4 + e] - gv[e], SPAN2));
      rot_pairs(rv, q4);
      store8_rot(R, roff(I2) + r, 8 * q4, rv, q4);
    }
  }
  __syncthreads();

  // ---- A (beta_r-scaled, strict lower, fp32) and P (scale, inclusive lower, split):
  //      20 block tasks; a diagonal block whose decay span exceeds 80 is exact
  //      tasks 4..7 (warps 4..7) are the diagonal A blocks, which their warp then inverts
  for (int task = warp; task < 20; task += NW) {
    int blk, isP;
    if (task >= 4 && task < 8) {
      blk = (task - 4) * (task - 1) / 2;  // block (I, I), I = task - 4
      isP = 0;
    } else {
      const int u = task < 4 ? task : task - 4;  // P blocks 0..9, then A blocks 1, 3, 4, 6, 7, 8
      const int i = u - 10;
      isP = u < 10;
      blk = isP ? u : i < 2 ? 2 * i + 1 : i < 3 ? 4 : i + 3;
    }
    const int bI = blk < 1 ? 0 : blk < 3 ? 1 : blk < 6 ? 2 : 3, bJ = blk - bI * (bI + 1) / 2;
    float acc[2][4];
    zero(acc);
    if (bJ < bI || sm.spanok[bI]) {
      gemm3<1, false, false>(acc, isP ? LQ : LK, 16 * bI, 0, R, roff(bI) + 16 * bJ, 0, DK / 16);
    } else {
      each(acc, [&](int m, int n, float& v) {
        const int rr = 16 * bI + m, s = 16 * bI + n;
        if (s <= rr && rr < L) {
          if constexpr (CONV) {
            v = pair_exact2_conv((isP ? qraw : kraw) + h * DK, (isP ? io.cwq : io.cwk) + 4 * h * DK,
                                 isP ? sm.inq[rr] : sm.ink[rr], kraw + h * DK, io.cwk + 4 * h * DK, sm.ink[s], io.ld,
                                 t0 + rr, t0 + s, tmin, sm.gg + rr * SQ, sm.gg + s * SQ);
          } else {
            const bf16* xr = (isP ? qraw : kraw) + ((size_t)(t0 + rr) * H + h) * DK;
            const bf16* ks = kraw + ((size_t)(t0 + s) * H + h) * DK;
            v = pair_exact2(xr, isP ? sm.inq[rr] : sm.ink[rr], ks, sm.ink[s], sm.gg + rr * SQ, sm.gg + s * SQ);
          }
        }
      });
    }
    if (isP) {
      const int gq = lane >> 2, tq = lane & 3;
#pragma unroll
      for (int jt = 0; jt < 2; jt++)
#pragma unroll
        for (int hh = 0; hh < 2; hh++) {
          const int rr = 16 * bI + gq + 8 * hh, s0 = 16 * bJ + 8 * jt + 2 * tq;
          op_store2(P, rr, s0, s0 <= rr ? scale * acc[jt][2 * hh] : 0.f,
                    s0 + 1 <= rr ? scale * acc[jt][2 * hh + 1] : 0.f);
        }
    } else {
      each(acc, [&](int m, int n, float& v) {
        const int rr = 16 * bI + m, s = 16 * bJ + n;
        sm.am[rr * SC + s] = s < rr ? sm.bet[rr] * v : 0.f;
        if (io.save) w.sA[(ch * NBLK + blk) * 16 * PB + m * PB + n] = s < rr ? v : 0.f;  // A' for dbeta
      });
    }
  }
  if (warp >= 4) {  // the diagonal A block this warp computed first
    __syncwarp();
    diag_inverse(sm.am, sm.am + tdoff(warp - 4), warp - 4);
  }
  zero_upper(P);  // the tensor core reads whole tiles
  fence_async_smem();
  __syncthreads();
  if (io.save && tid == 0) {  // P for the backward (its tile is not written again)
    bulk_s2g(w.sP + ch * 2 * C * C, P.hi, 4 * C * C);
    bulk_commit();
  }
  // QG over G, KD in the tail of the x region (both free now)
  store8_rot(QG, r, 8 * q4, qg, q4);  // rotated in the factors step
  store8_rot(KD, r, 8 * q4, kd, q4);
  solve_merge(sm.am, tm, yy);
  for (int idx = tid; idx < C * C / 2; idx += NTH) {  // T -> split operand over A (upper blocks zero)
    const int core = idx >> 5, ln = idx & 31;  // a warp writes one whole core matrix
    const int rr = 8 * (core >> 3) + (ln >> 2), s2 = 8 * (core & 7) + 2 * (ln & 3);
    const bool low = (s2 >> 4) <= (rr >> 4);
    op_store2(T, rr, s2, low ? tm[rr * SC + s2] : 0.f, low ? tm[rr * SC + s2 + 1] : 0.f);
  }
  fence_async_smem();
  tc::fence_before();
  __syncthreads();
  if (io.save && tid == 0) {  // T for the backward (its tile is not written again)
    bulk_s2g(w.sT + ch * 2 * C * C, T.hi, 4 * C * C);
    bulk_commit();
  }
  // tensor-core rounds: one thread issues, completion on sm.bar, then every warp
  // reads the m16n8 fragments of its 16 rows.  TMEM columns: W 0 | U 32; then
  // M' 0 | KU' 32 (rows 32.. unused) and QW' 96 | PU 128
  uint32_t mph = 0;
  auto round_done = [&]() -> bool {  // uniform over the CTA
    const bool ok = mbar_wait(&sm.bar, mph);
    mph ^= 1;
    tc::fence_after();
    return !__syncthreads_or(!ok);
  };
  auto bail = [&]() {
    mbar_wait(&sm.bar, mph ^ 1);
    tc::fence_before();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tb, TCOLS);
    if (tid == 0) atomicExch(w.err, -7);
  };
  if (tid == 0) {  // W | U = T [XK | XV]
    tc::fence_after();
    tc::gemm_split(tb + 0, tc::kmaj(T), tc::mnmaj(XKV), DK + DV, C / 16, false);
    tc::commit(&sm.bar);
  }
  if (!round_done()) { bail(); return; }
  {
    const int wI = warp & 3, hk = warp >> 2, gq = lane >> 2, tq = lane & 3;
    float aw[2][4], au[4][4];
    tc::ld_frag<2>(tb + 0, 16 * hk, aw);
    tc::ld_frag<4>(tb + 32, 32 * hk, au);
#pragma unroll
    for (int jt = 0; jt < 2; jt++)
#pragma unroll
      for (int hh = 0; hh < 2; hh++) {
        const int rr = 16 * wI + gq + 8 * hh, c = 16 * hk + 8 * jt + 2 * tq;
        op_store2(WU, rr, c, aw[jt][2 * hh], aw[jt][2 * hh + 1]);
        if (io.save) op_store2(Ws, rr, c, aw[jt][2 * hh], aw[jt][2 * hh + 1]);
      }
#pragma unroll
    for (int jt = 0; jt < 4; jt++)
#pragma unroll
      for (int hh = 0; hh < 2; hh++) {
        const int rr = 16 * wI + gq + 8 * hh, c = 32 * hk + 8 * jt + 2 * tq;
        op_store2(WU, rr, DK + c, au[jt][2 * hh], au[jt][2 * hh + 1]);
        if (io.save) op_store2(Us, rr, c, au[jt][2 * hh], au[jt][2 * hh + 1]);
      }
  }
  fence_async_smem();
  tc::fence_before();
  __syncthreads();
  if (io.save && tid == 0) {  // W and U for the backward
    bulk_s2g(w.sW + ch * 2 * C * DK, Ws.hi, 4 * C * DK);
    bulk_s2g(w.sU + ch * 2 * C * DV, Us.hi, 4 * C * DV);
    bulk_commit();
  }
  // outputs, straight from the fragments to global: PU and KU (fp32), QW and M
  // (split)
  if (tid == 0) {  // [QW' | PU] = P [W | U], [M' | KU'] = KD^T [W | U] (KD^T: rows 32.. unused)
    tc::fence_after();
    tc::gemm_split(tb + 96, tc::kmaj(P), tc::mnmaj(WU), DK + DV, C / 16, false);
    tc::gemm_split(tb + 0, tc::mnmaj(KD), tc::mnmaj(WU), DK + DV, C / 16, false);
    tc::commit(&sm.bar);
  }
  if (!round_done()) { bail(); return; }
  {
    const int wI = warp & 3, hk = warp >> 2;
    bf16* qwg = reinterpret_cast<bf16*>(chblk(w, ch) + CB_QW);
    bf16* mg = reinterpret_cast<bf16*>(chblk(w, ch) + CB_M);
    const Op QWg{qwg, qwg + C * DK, DK}, Mg{mg, mg + DK * DK, DK};
    float pu[4][4], qw[2][4];
    tc::ld_frag<4>(tb + 128, 32 * hk, pu);
    tc::ld_frag<2>(tb + 96, 16 * hk, qw);
    // PU and KU per 32-column half (warp column hk), each half contiguous so that the chain CTA
    // of a half loads it in one copy, and in fragment order: fragment jt of lane l of warp row wI
    // (4 values) at float4 (4 wI + jt) x 32 + l, so a warp's store and the chain warp's read of
    // one fragment cover 512 contiguous bytes
    float4* pud = reinterpret_cast<float4*>(chblk(w, ch) + (hk ? CB_PU1 : CB_PU0)) + wI * 128 + lane;
#pragma unroll
    for (int jt = 0; jt < 4; jt++) pud[32 * jt] = make_float4(pu[jt][0], pu[jt][1], pu[jt][2], pu[jt][3]);
    store_acc_op(qw, QWg, 16 * wI, 16 * hk, [&](int rr, int c, float v) { return op_get(QG, rr, c) - v; });
    if (wI < 2) {  // rows i < dk of the KD^T products
      float ku[4][4], mm[2][4];
      tc::ld_frag<4>(tb + 32, 32 * hk, ku);
      tc::ld_frag<2>(tb + 0, 16 * hk, mm);
      float4* kud = reinterpret_cast<float4*>(chblk(w, ch) + (hk ? CB_KU1 : CB_KU0)) + wI * 128 + lane;
#pragma unroll
      for (int jt = 0; jt < 4; jt++) kud[32 * jt] = make_float4(ku[jt][0], ku[jt][1], ku[jt][2], ku[jt][3]);
      store_acc_op(mm, Mg, 16 * wI, 16 * hk, [&](int i, int jc, float v) { return (i == jc ? sm.gam[i] : 0.f) - v; });
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tb, TCOLS);
  if (tid == 0) bulk_wait_read();  // the saves' shared-memory reads are done (the writes complete with the grid)
}

// ------------------------------------------------------------ state chains
// Both chains are affine recurrences over a document's chunks,
//   forward:   S_{c+1} = M_c S_c + KU_c,        O_c = QW_c S_c + PU_c
//   backward:  dS_c    = M_c^T dS_{c+1} + QW_c^T dO_c
// (from h0 / dh_final; the last state is h_final / dh0).  Value columns are
// independent: one CTA of four warps per (document, head, 32 value columns)
// carries a 32 x 32 slice as a split-bf16 operand tile in shared memory and
// streams the chunk's operands through a three-stage ring of 1-D bulk copies
// (one thread issues, completion on the stage's mbarrier; the backward's dO
// rows, strided in the input, by cp.async).  Only the
// state product is on the chain; the output (forward) and QW^T dO (backward)
// take the same step's other warps' slack.  Each step also stores the carried
// state (S entering the chunk, dS leaving it) as a split operand tile for the
// per-chunk kernels.  The fp32 state rounds to ~16 bits only as an operand;
// h_final and dh0 are the fp32 accumulators.
constexpr int NSC = 32;   // value columns per chain CTA
constexpr int NSTG = 3;   // stages of the fused-norm chains
constexpr int FSTG = 4;   // stages of fwd_state (plain)
constexpr int BSTG = 4;   // stages of bwd_scan (plain)
constexpr int CTH = 128;  // chain threads

// A document's chunks are consecutive C-token pieces from its first token
// (how the chunk table is built), so a chain derives chunk c's first token and
// length from the document's first token and length, loaded once, instead of
// loading table rows inside its step loop (a dependent global load on the
// step's path).
struct DocSpan {
  int tok0 = 0, len = 0;
  __device__ int t0(int c) const { return tok0 + C * c; }
  __device__ int L(int c) const { return min(C, len - C * c); }
};
__device__ __forceinline__ DocSpan doc_span(const Ws& w, int cb, int n) {
  DocSpan sp;
  if (n > 0) {
    sp.tok0 = w.chunk_tok0[cb];
    sp.len = w.chunk_tok0[cb + n - 1] + w.chunk_len[cb + n - 1] - sp.tok0;
  }
  return sp;
}

// Copies the 32 x NSC slice tile (K = NSC) into columns col0.. of the chunk's
// full 32 x dv state tile (K = dv) in global memory: whole 8 x 8 core matrices.
// t: the copying thread's index among CTH threads.
__device__ __forceinline__ void slice_to_global(bf16* g, const bf16* s, int col0, int t) {
  for (int idx = t; idx < 2 * 16 * 8; idx += CTH) {  // (hi|lo) x 16 cores x 8 uint4
    const int part = idx >> 7, core = (idx >> 3) & 15, q = idx & 7;
    const int rb = core >> 2, kb = core & 3;
    const uint4 v = *reinterpret_cast<const uint4*>(s + part * DK * NSC + (rb * (NSC / 8) + kb) * 64 + q * 8);
    *reinterpret_cast<uint4*>(g + part * DK * DV + (rb * (DV / 8) + (col0 >> 3) + kb) * 64 + q * 8) = v;
  }
}

// The state chains' grids (fwd_seg, fwd_state, bwd_seg, bwd_scan) with split
// chains (Dims::seg): one dimension, CTA i = (rank, head, column half) with
// the half fastest (the two halves of a chunk read the same M and QW), ranks
// in the segment table's dispatch order (heaviest units first).  Without seg:
// (document, head, half) as blockIdx.
struct ChainCta {
  int unit, h, half;
};
__device__ __forceinline__ ChainCta chain_cta(const Dims& d, const Ws& w) {
  ChainCta c{(int)blockIdx.x, (int)blockIdx.y, (int)blockIdx.z};
  if (d.seg) {
    const int i = (int)blockIdx.x, rank = i / (2 * d.H);
    c.half = i & 1;
    c.h = (i >> 1) % d.H;
    c.unit = rank < *w.n_units ? w.uorder[rank] : -1;
  }
  return c;
}

// S <- Phi_t S + B_t for t = 0 .. count - 1 in fp32, composite t at comp + t
// cstride (Phi [DK][DK], then B [DK][DV] of which columns col0 .. are this
// CTA's).  fs: S [DK][NSC], holding the initial state and then the result;
// fp, fb: scratch of DK x DK and DK x NSC floats (shared memory).  NT threads,
// each owning E consecutive entries of a row of S; composite t + 1's loads
// are in flight during product t.  Ends with a barrier.
template <int NT>
__device__ void fold_composites(float* fs, float* fp, float* fb, const float* comp, int64_t cstride, int count,
                                int col0) {
  constexpr int E = DK * NSC / NT, Q = E / 4;
  static_assert(E % 4 == 0 && NSC % E == 0, "whole float4s of one row per thread");
  const int tid = threadIdx.x, i = tid / (NSC / E), c = E * (tid % (NSC / E));
  float4 pv[Q], bv[Q];
  auto load = [&](const float* cp) {
#pragma unroll
    for (int q = 0; q < Q; q++) {
      pv[q] = reinterpret_cast<const float4*>(cp + E * tid)[q];
      bv[q] = reinterpret_cast<const float4*>(cp + DK * DK + i * DV + col0 + c)[q];
    }
  };
  load(comp);
  for (int t = 0; t < count; t++) {
#pragma unroll
    for (int q = 0; q < Q; q++) {
      reinterpret_cast<float4*>(fp + E * tid)[q] = pv[q];
      reinterpret_cast<float4*>(fb + i * NSC + c)[q] = bv[q];
    }
    __syncthreads();  // S, Phi_t and B_t are visible
    if (t + 1 < count) load(comp + (t + 1) * cstride);
    float a[E];
#pragma unroll
    for (int e = 0; e < E; e++) a[e] = fb[i * NSC + c + e];
#pragma unroll 4
    for (int k = 0; k < DK; k++) {
      const float pk = fp[i * DK + k];
#pragma unroll
      for (int e = 0; e < E; e++) a[e] = fmaf(pk, fs[k * NSC + c + e], a[e]);
    }
    __syncthreads();  // every read of S, Phi_t and B_t is done
#pragma unroll
    for (int e = 0; e < E; e++) fs[i * NSC + c + e] = a[e];
  }
  __syncthreads();
}

template <bool NORM>
struct FChainStage {  // one copy of this half's part of the chain block: KU, PU, M, QW (half 0)
  __align__(128) unsigned char raw[CB_STAGE];  // or M, QW, KU, PU (half 1)
  bf16 g[NORM ? C * NSC : 8];  // (NORM) the gate's columns of this half for the step's chunk, [C][NSC], by TMA
};
// Row partials exchanged by the two column-half CTAs of a (document, head)
// when the gated RMSNorm is fused into a chain: the peer CTA stores its
// partials for step s into part[s % NX] of this CTA's shared memory by
// asynchronous stores, each completing its 8 bytes of bar[s % NX]'s
// transaction count.  One thread of this CTA arms each phase (one arrival
// expecting the slot's XBYTES): for steps 0 .. NX - 1 at the start, for step
// s + NX right after its own wait for step s succeeded.  The forward sends
// step s's partials before it reads step s - 1's, and a CTA's send of step m
// only waits (through its own barrier) for the peer's partials of step m - 2:
// while this CTA has not read step j's, the peer may have sent up to j + 3,
// so four slots, and the peer cannot send step s + NX before every thread
// here has passed its wait for step s (so an early arming never completes a
// phase under a thread still waiting).  (The backward sends and reads the
// same step's.)
constexpr int NX = 4;
constexpr uint32_t XBYTES = C * 8;  // one slot: a float2 per row
struct Xchg {
  float2 part[NX][C];
  uint64_t bar[NX];
};
struct __align__(16) FChainNorm {  // (fused norm) one step's rows handed from the output to the carry warps
  float u[2][C * NSC];         // u = o w sigmoid(g), [C][NSC] with 8-column groups swizzled by row
  float own[2][C];             // this CTA's half of each row's sum of o^2
};
template <bool NORM>
struct FChainSm {
  FChainStage<NORM> st[NORM ? NSTG : FSTG];
  bf16 S[2][2 * DK * NSC];          // the carried state (split), double-buffered
  uint64_t bar[NORM ? NSTG : FSTG];  // stage completion
  Xchg x;                           // fused norm only
  FChainNorm nr[NORM ? 1 : 0];
};
static_assert(offsetof(FChainSm<true>, nr) % 16 == 0, "the u tiles are read as float4");
// Column c of row r of a u tile: 8-column groups XOR-permuted by r % 4, so the
// output warps' fragment stores (8 rows x 4 column pairs per instruction) and
// the carry warps' 8-column reads spread over the banks.
__device__ __forceinline__ int uswz(int r, int c) { return r * NSC + (c ^ (8 * (r & 3))); }
static_assert(sizeof(FChainStage<false>) % 128 == 0 && sizeof(FChainStage<true>) % 128 == 0 &&
                  offsetof(FChainStage<true>, g) % 128 == 0,
              "bulk and tensor copy targets need 128-byte alignment");

// fwd_state: warps 0..3 carry the state (S' = M S + KU into the other buffer
// of the double-buffered tile), then store the entering state and issue the
// stage copy of a later step; warps 4..7 write the output O = QW S + PU, on
// the same step's state; one barrier per step.
// NORM: the gated RMSNorm epilogue ("Pure KDA 300M" guide, Overview: per-head
// output gate and RMSNorm, eps 1e-6), y = o r w sigmoid(g) with
// r = 1 / sqrt(mean_j o_j^2 + eps) over the dv columns of a row, is fused into
// the chain.  A row's 64 columns are split over the two CTAs of the
// (document, head); launched as a cluster of those two CTAs.  At step s the
// output warps send their rows' partial sums of o^2 into the peer's shared
// memory, write o (io dtype) when io.o is set and, with io.save, o in fp32 for
// the fused backward (a bf16 copy would make its dg depend on a rounding), and
// hand u = o w sigmoid(g) and their own partials to the carry warps, which at
// step s + 1, after their state update, wait (bounded) for the peer's
// partials of step s and write y = u r.  (The carry warps' part of a step is
// the shorter one; the output warps' product and stores set the step time.)
// A CTA of a cluster never leaves before the final cluster barrier: errors
// skip the remaining steps instead of returning.
template <bool NORM>
__global__ void __launch_bounds__(2 * CTH) fwd_state_kernel(Dims d, FwdIO io, Ws w, const __grid_constant__ NMaps nmap) {
  extern __shared__ __align__(128) unsigned char smraw[];
  FChainSm<NORM>& sm = *reinterpret_cast<FChainSm<NORM>*>(smraw);
  constexpr int NS = NORM ? NSTG : FSTG;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int lane = tid & 31, gq = lane >> 2, tq = lane & 3;
  pdl_wait();  // fwd_chunk's products (and with d.seg, fwd_seg's composites)
  const int err0 = *w.err;
  if (!NORM && err0 != 0) return;
  const int H = d.H;
  const ChainCta cc = chain_cta(d, w);
  const int h = cc.h, zc = cc.half, col0 = zc * NSC;
  // this CTA's run of chunks: a whole document, or with d.seg one unit of the segment table
  // (segment sg of its document, chunks c0 ..; `last`: the run ends the document)
  int doc = cc.unit, cb, n, sg = 0;
  bool last = true;
  if (d.seg && err0 != 0) {  // (NORM) the table may be stale: no steps, to the cluster barriers
    doc = 0;
    cb = n = 0;
  } else if (d.seg) {
    if (cc.unit < 0) return;  // (NORM: both CTAs of the cluster, the same rank)
    const int4 un = w.useg[cc.unit];
    doc = un.x;
    sg = un.w;
    cb = w.doc_chunk0[doc] + un.y;
    n = un.z;
    last = un.y + n == w.doc_chunk0[doc + 1] - w.doc_chunk0[doc];
  } else {
    cb = w.doc_chunk0[doc];
    n = err0 != 0 ? 0 : w.doc_chunk0[doc + 1] - cb;
  }
  const DocSpan sp = doc_span(w, cb, n);
  const int64_t dh = ((int64_t)doc * H + h) * DK * DV;
  const Op S0{sm.S[0], sm.S[0] + DK * NSC, NSC}, S1{sm.S[1], sm.S[1] + DK * NSC, NSC};
  for (int idx = tid; sg == 0 && idx < DK * NSC / 2; idx += 2 * CTH) {  // (a later segment's is folded below)
    const int i = idx / (NSC / 2), jc = 2 * (idx % (NSC / 2));
    float2 v = make_float2(0.f, 0.f);
    if (io.h0) v = *reinterpret_cast<const float2*>(io.h0 + dh + i * DV + col0 + jc);
    op_store2(S0, i, jc, v.x, v.y);
  }
  if (tid == 0) {
    for (int s2 = 0; s2 < NS; s2++) mbar_init(&sm.bar[s2], 1);
    if (NORM) {
      for (int x2 = 0; x2 < NX; x2++) mbar_init(&sm.x.bar[x2], 1);  // one local arming per phase + the peer's bytes
    }
    mbar_init_fence();
    if (NORM)
      for (int x2 = 0; x2 < NX; x2++) mbar_expect_tx(&sm.x.bar[x2], XBYTES);  // steps 0 .. NX - 1
  }
  __syncthreads();  // the barriers are initialised before any thread waits on them
  uint32_t xpart = 0, xbar = 0;  // the peer's exchange slots, mapped into the cluster window
  float nwv[4][2];               // (output warps, NORM) the norm weight of this thread's columns
  if constexpr (NORM) {
    cluster_sync();  // ... and before the peer arrives on them
    const uint32_t peer = cluster_rank() ^ 1u;
    xpart = cluster_map(&sm.x.part[0][0], peer);
    xbar = cluster_map(&sm.x.bar[0], peer);
#pragma unroll
    for (int jj = 0; jj < 4; jj++)
#pragma unroll
      for (int c1 = 0; c1 < 2; c1++) nwv[jj][c1] = io.nw[col0 + 8 * jj + 2 * tq + c1];
  }
  bool xfail = false;  // (carry warps) the peer's partials did not arrive in bound
  bool bad = false;
  // (NORM, carry warps) the rows of step k: thread = row tid / 2, columns 16 (tid % 2) ..
  auto finish_rows = [&](int k) {
    const int row = tid >> 1, hf = tid & 1, slot = k % NX, ub = k & 1;
    if (!mbar_wait_cluster(&sm.x.bar[slot], (k / NX) & 1)) {
      xfail = true;  // bails at the next step's barrier (or skips the end state)
      return;
    }
    if (tid == 0) mbar_expect_tx(&sm.x.bar[slot], XBYTES);  // armed for step k + NX
    const int L = sp.L(k), t0 = sp.t0(k);
    if (row < L) {
      const float tot = sm.nr[0].own[ub][row] + sm.x.part[slot][row].x;
      const float rr = 1.0f / sqrtf(tot * (1.0f / DV) + io.neps);
      bf16* yp = (bf16*)io.y + ((size_t)(t0 + row) * d.H + h) * DV + col0 + 16 * hf;
#pragma unroll
      for (int lg = 0; lg < 2; lg++) {
        const float4* up = reinterpret_cast<const float4*>(sm.nr[0].u[ub] + uswz(row, 16 * hf + 8 * lg));
        const float4 a = up[0], b = up[1];
        uint4 o4;
        __nv_bfloat162* o2 = reinterpret_cast<__nv_bfloat162*>(&o4);
        o2[0] = __floats2bfloat162_rn(a.x * rr, a.y * rr);
        o2[1] = __floats2bfloat162_rn(a.z * rr, a.w * rr);
        o2[2] = __floats2bfloat162_rn(b.x * rr, b.y * rr);
        o2[3] = __floats2bfloat162_rn(b.z * rr, b.w * rr);
        *reinterpret_cast<uint4*>(yp + 8 * lg) = o4;
      }
    }
  };
  // the stage of `step`: one copy (with the gate tile: two), issued by carry thread 0 once its part of
  // the step before is done (the output warps' part is the longer one)
  const int oKU = zc ? CB_KU1 - CB_M : 0, oPU = oKU + (CB_PU0 - CB_KU0);
  const int oM = zc ? 0 : CB_M - CB_KU0, oQW = oM + (CB_QW - CB_M);
  auto prefetch = [&](int step) {
    if (step < n && tid == 0) {
      const int slot = step % NS;
      const int64_t ch = (int64_t)(cb + step) * H + h;
      mbar_expect_tx(&sm.bar[slot], (uint32_t)(CB_STAGE + (NORM ? 2 * C * NSC : 0) + d.tx_extra));
      bulk_g2s(sm.st[slot].raw, chblk(w, ch) + (zc ? CB_M : CB_KU0), CB_STAGE, &sm.bar[slot]);
      if (NORM)  // the gate rows of the chunk (rows past its end are not used)
        tma_load_2d(sm.st[slot].g, &nmap.g, h * DV + col0, sp.t0(step), &sm.bar[slot]);
    }
  };
  for (int s = 0; s < NS - 1; s++) prefetch(s);
  if (sg > 0) {
    // entry state of segment sg: the composites of the document's earlier segments (the units
    // cc.unit - sg ..) folded onto the initial state.  Scratch: the ring's last slot, whose first
    // copy is issued in step 0 (after this).
    float* fs = reinterpret_cast<float*>(sm.st[NS - 1].raw);
    float* fp = fs + DK * NSC;
    float* fb = fp + DK * DK;
    for (int idx = tid; idx < DK * NSC; idx += 2 * CTH) {
      const int r = idx / NSC, c = idx % NSC;
      fs[idx] = io.h0 ? io.h0[dh + r * DV + col0 + c] : 0.f;
    }
    fold_composites<2 * CTH>(fs, fp, fb, w.segc + ((int64_t)(cc.unit - sg) * H + h) * DK * (DK + DV),
                             (int64_t)H * DK * (DK + DV), sg, col0);
    for (int idx = tid; idx < DK * NSC / 2; idx += 2 * CTH) {
      const int r = idx / (NSC / 2), jc = 2 * (idx % (NSC / 2));
      op_store2(S0, r, jc, fs[r * NSC + jc], fs[r * NSC + jc + 1]);
    }
  }
  const bool carry = warp < 4;
  const int wq = warp & 3, mI = wq & 1, jn = wq >> 1;
  float snew[2][4];  // (carry warps) tile of the updated state: rows 16 mI .., columns 16 jn ..
  zero(snew);
  bf16* o = (bf16*)io.o;
  for (int step = 0; step < n; step++) {
    const FChainStage<NORM>& s = sm.st[step % NS];
    const int ci = cb + step;
    if (__syncthreads_or(!mbar_wait(&sm.bar[step % NS], (step / NS) & 1) || xfail)) {  // a wait ran out
      for (int k2 = step; k2 < n && k2 < step + NS - 1; k2++) mbar_wait(&sm.bar[k2 % NS], (k2 / NS) & 1);
      if (tid == 0) atomicExch(w.err, -7);
      bad = true;
      break;
    }  // this step's stage and state are visible; the other state buffer is free
    bf16* smp = reinterpret_cast<bf16*>(const_cast<unsigned char*>(s.raw) + oM);
    bf16* sqp = reinterpret_cast<bf16*>(const_cast<unsigned char*>(s.raw) + oQW);
    const float* sku = reinterpret_cast<const float*>(s.raw + oKU);
    const float* spu = reinterpret_cast<const float*>(s.raw + oPU);
    const Op Mo{smp, smp + DK * DK, DK};
    const Op QWo{sqp, sqp + C * DK, DK};
    const Op& Sc = (step & 1) ? S1 : S0;
    if (carry) {
      const Op& Sn = (step & 1) ? S0 : S1;
      zero(snew);
      gemm3<1, false, true>(snew, Mo, 16 * mI, 0, Sc, 16 * jn, 0, DK / 16);
      // KU in fragment order: this lane's values of columns 16 jn .. are fragments 2 jn, 2 jn + 1
      const float4* kup = reinterpret_cast<const float4*>(sku) + (4 * mI + 2 * jn) * 32 + lane;
#pragma unroll
      for (int jj = 0; jj < 2; jj++) {
        const float4 k4 = kup[32 * jj];
        snew[jj][0] += k4.x;
        snew[jj][1] += k4.y;
        snew[jj][2] += k4.z;
        snew[jj][3] += k4.w;
#pragma unroll
        for (int hh = 0; hh < 2; hh++)
          op_store2(Sn, 16 * mI + gq + 8 * hh, 16 * jn + 8 * jj + 2 * tq, snew[jj][2 * hh], snew[jj][2 * hh + 1]);
      }
      if (io.save) slice_to_global(w.sS + ((int64_t)ci * H + h) * 2 * DK * DV, Sc.hi, col0, tid);  // for bwd_grad
      if constexpr (NORM)
        if (step > 0) finish_rows(step - 1);  // the previous step's y, off the state's path
      prefetch(step + NS - 1);  // into the slot of step - 1, free since the barrier
    } else {
      const int L = sp.L(step), t0 = sp.t0(step);
      float oo[4][4];
      zero(oo);
      gemm3<2, false, true>(oo, QWo, 16 * wq, 0, Sc, 0, 0, DK / 16);
      const float4* pup = reinterpret_cast<const float4*>(spu) + 4 * wq * 32 + lane;  // fragment order
      if constexpr (!NORM) {
#pragma unroll
        for (int jj = 0; jj < 4; jj++) {
          const float4 p4 = pup[32 * jj];
          const int r = 16 * wq + gq, c = 8 * jj + 2 * tq;
          if (r < L)
            *reinterpret_cast<__nv_bfloat162*>(o + ((size_t)(t0 + r) * H + h) * DV + col0 + c) =
                __floats2bfloat162_rn(oo[jj][0] + p4.x, oo[jj][1] + p4.y);
          if (r + 8 < L)
            *reinterpret_cast<__nv_bfloat162*>(o + ((size_t)(t0 + r + 8) * H + h) * DV + col0 + c) =
                __floats2bfloat162_rn(oo[jj][2] + p4.z, oo[jj][3] + p4.w);
        }
      } else {
        // o of rows r = 16 wq + gq and r + 8 (columns 8 jj + 2 tq + {0, 1}); rows past the
        // chunk end are zero (their QW and PU rows are).  The row partials go to the peer now.
        const int r = 16 * wq + gq, slot = step % NX, ub = step & 1;
#pragma unroll
        for (int jj = 0; jj < 4; jj++) {
          const float4 p4 = pup[32 * jj];
          oo[jj][0] += p4.x;
          oo[jj][1] += p4.y;
          oo[jj][2] += p4.z;
          oo[jj][3] += p4.w;
        }
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int jj = 0; jj < 4; jj++) {
          s0 += oo[jj][0] * oo[jj][0] + oo[jj][1] * oo[jj][1];
          s1 += oo[jj][2] * oo[jj][2] + oo[jj][3] * oo[jj][3];
        }
        s0 += __shfl_xor_sync(0xffffffffu, s0, 1);
        s0 += __shfl_xor_sync(0xffffffffu, s0, 2);
        s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
        s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
        if (tq == 0) {  // rows r and r + 8 into the peer's slot, each completing 8 of its barrier's bytes
          st_async_f32x2(xpart + (uint32_t)((slot * C + r) * 8), s0, 0.f, xbar + (uint32_t)(slot * 8));
          st_async_f32x2(xpart + (uint32_t)((slot * C + r + 8) * 8), s1, 0.f, xbar + (uint32_t)(slot * 8));
          sm.nr[0].own[ub][r] = s0;
          sm.nr[0].own[ub][r + 8] = s1;
        }
        float* ut = sm.nr[0].u[ub];
#pragma unroll
        for (int jj = 0; jj < 4; jj++) {
          const int c = 8 * jj + 2 * tq;  // the gate tile arrived with the stage
          const float2 g0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(s.g + r * NSC + c));
          const float2 g1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(s.g + (r + 8) * NSC + c));
          *reinterpret_cast<float2*>(ut + uswz(r, c)) =
              make_float2(oo[jj][0] * nwv[jj][0] * sigmoid_fast(g0.x), oo[jj][1] * nwv[jj][1] * sigmoid_fast(g0.y));
          *reinterpret_cast<float2*>(ut + uswz(r + 8, c)) =
              make_float2(oo[jj][2] * nwv[jj][0] * sigmoid_fast(g1.x), oo[jj][3] * nwv[jj][1] * sigmoid_fast(g1.y));
          bf16* op = (bf16*)io.o;
          if (r < L) {
            const size_t i = ((size_t)(t0 + r) * H + h) * DV + col0 + c;
            if (op) *reinterpret_cast<__nv_bfloat162*>(op + i) = __floats2bfloat162_rn(oo[jj][0], oo[jj][1]);
            if (io.save) *reinterpret_cast<float2*>(w.nO + i) = make_float2(oo[jj][0], oo[jj][1]);
          }
          if (r + 8 < L) {
            const size_t i = ((size_t)(t0 + r + 8) * H + h) * DV + col0 + c;
            if (op) *reinterpret_cast<__nv_bfloat162*>(op + i) = __floats2bfloat162_rn(oo[jj][2], oo[jj][3]);
            if (io.save) *reinterpret_cast<float2*>(w.nO + i) = make_float2(oo[jj][2], oo[jj][3]);
          }
        }
      }
    }
  }
  if constexpr (NORM) {
    __syncthreads();  // the output warps' last u tile and partials are written
    if (!bad && n > 0 && carry) finish_rows(n - 1);  // the last step's rows
  }
  if (NORM && __syncthreads_or(xfail) && !bad) {  // the last step's exchange ran out
    if (tid == 0) atomicExch(w.err, -7);
    bad = true;
  }
  if (io.h_final && !bad && err0 == 0 && last) {
    if (n > 0) {
      if (carry)
#pragma unroll
        for (int jj = 0; jj < 2; jj++)
#pragma unroll
          for (int hh = 0; hh < 2; hh++) {
            const int i = 16 * mI + gq + 8 * hh, c = 16 * jn + 8 * jj + 2 * tq;
            *reinterpret_cast<float2*>(io.h_final + dh + i * DV + col0 + c) =
                make_float2(snew[jj][2 * hh], snew[jj][2 * hh + 1]);
          }
    } else {
      for (int idx = tid; idx < DK * NSC; idx += 2 * CTH) {
        const int i = idx / NSC, jc = idx % NSC;
        io.h_final[dh + i * DV + col0 + jc] = io.h0 ? io.h0[dh + i * DV + col0 + jc] : 0.f;
      }
    }
  }
  if constexpr (NORM) cluster_sync();  // the peer no longer touches this CTA's shared memory
}

// fwd_seg: the composites of split forward chains (Dims::seg).  One CTA of
// four warps per (unit, head, 32 value columns) whose unit is a segment before
// its document's last: X = [Phi | B] (32 x 64; Phi the product of the
// segment's M_c, B the state it reaches from zero) by X <- M_c X + [0 | KU_c]
// from [I | 0], with fwd_state's split-bf16 products and double-buffered split
// tile, and a four-stage ring of M and this half's KU (bulk copies, bounded
// waits).  Phi is the same for both halves; half 0 stores it.
constexpr int SSTG = 4;
struct SegStage {
  bf16 M[2 * DK * DK];  // M (split)
  float ku[DK * NSC];   // KU of this half, in fragment order
};
struct SegSm {
  SegStage st[SSTG];
  bf16 X[2][2 * DK * 2 * NSC];  // [Phi | B] (split), double-buffered
  uint64_t bar[SSTG];
};
static_assert(sizeof(SegStage) % 16 == 0 && offsetof(SegStage, ku) % 16 == 0 && offsetof(SegSm, X) % 16 == 0,
              "bulk copy targets and operand tiles need 16-byte alignment");

__global__ void __launch_bounds__(CTH) fwd_seg_kernel(Dims d, FwdIO io, Ws w) {
  (void)io;
  extern __shared__ __align__(128) unsigned char smraw[];
  SegSm& sm = *reinterpret_cast<SegSm*>(smraw);
  const int tid = threadIdx.x, warp = tid >> 5;
  const int lane = tid & 31, gq = lane >> 2, tq = lane & 3;
  pdl_wait();     // fwd_chunk's chain operands
  pdl_release();  // fwd_state may launch: it waits for this grid before reading the composites
  if (*w.err != 0) return;
  const ChainCta cc = chain_cta(d, w);
  const int u = cc.unit, h = cc.h, half = cc.half;
  if (u < 0) return;
  const int4 un = w.useg[u];  // (document, first chunk in it, chunks, segment)
  const int c0d = w.doc_chunk0[un.x], n = un.z;
  if (un.y + n == w.doc_chunk0[un.x + 1] - c0d) return;  // the document's last segment is not composed
  const int H = d.H, cb = c0d + un.y;
  constexpr int XK = 2 * NSC;  // columns of X
  const Op X0{sm.X[0], sm.X[0] + DK * XK, XK}, X1{sm.X[1], sm.X[1] + DK * XK, XK};
  for (int idx = tid; idx < DK * XK / 2; idx += CTH) {  // [I | 0]
    const int i = idx / (XK / 2), jc = 2 * (idx % (XK / 2));
    op_store2(X0, i, jc, i == jc ? 1.f : 0.f, i == jc + 1 ? 1.f : 0.f);
  }
  if (tid == 0) {
    for (int s2 = 0; s2 < SSTG; s2++) mbar_init(&sm.bar[s2], 1);
    mbar_init_fence();
  }
  __syncthreads();  // the barriers are initialised before any thread waits on them
  auto prefetch = [&](int step) {
    if (step < n && tid == 0) {
      const int slot = step % SSTG;
      const int64_t ch = (int64_t)(cb + step) * H + h;
      mbar_expect_tx(&sm.bar[slot], (uint32_t)(4 * DK * DK + 4 * DK * NSC + d.tx_extra));
      bulk_g2s(sm.st[slot].M, chblk(w, ch) + CB_M, 4 * DK * DK, &sm.bar[slot]);
      bulk_g2s(sm.st[slot].ku, chblk(w, ch) + (half ? CB_KU1 : CB_KU0), 4 * DK * NSC, &sm.bar[slot]);
    }
  };
  for (int s = 0; s < SSTG - 1; s++) prefetch(s);
  const int mI = warp & 1, jn = warp >> 1;  // this warp's tile of X: rows 16 mI .., columns 32 jn ..
  float xn[4][4];
  zero(xn);
  for (int step = 0; step < n; step++) {
    const SegStage& st = sm.st[step % SSTG];
    if (__syncthreads_or(!mbar_wait(&sm.bar[step % SSTG], (step / SSTG) & 1))) {  // a wait ran out
      for (int k2 = step; k2 < n && k2 < step + SSTG - 1; k2++) mbar_wait(&sm.bar[k2 % SSTG], (k2 / SSTG) & 1);
      if (tid == 0) atomicExch(w.err, -7);
      return;
    }  // this step's stage and X are visible; the other X buffer and the slot of step - 1 are free
    prefetch(step + SSTG - 1);
    const Op Mo{const_cast<bf16*>(st.M), const_cast<bf16*>(st.M) + DK * DK, DK};
    const Op& Xc = (step & 1) ? X1 : X0;
    const Op& Xn = (step & 1) ? X0 : X1;
    zero(xn);
    gemm3<2, false, true>(xn, Mo, 16 * mI, 0, Xc, 32 * jn, 0, DK / 16);
    if (jn == 1) {  // + KU: fragment jt of this lane's row block in KU's fragment order
      const float4* kup = reinterpret_cast<const float4*>(st.ku) + 4 * mI * 32 + lane;
#pragma unroll
      for (int jt = 0; jt < 4; jt++) {
        const float4 k4 = kup[32 * jt];
        xn[jt][0] += k4.x;
        xn[jt][1] += k4.y;
        xn[jt][2] += k4.z;
        xn[jt][3] += k4.w;
      }
    }
#pragma unroll
    for (int jt = 0; jt < 4; jt++)
#pragma unroll
      for (int hh = 0; hh < 2; hh++)
        op_store2(Xn, 16 * mI + gq + 8 * hh, 32 * jn + 8 * jt + 2 * tq, xn[jt][2 * hh], xn[jt][2 * hh + 1]);
  }
  float* out = w.segc + ((int64_t)u * H + h) * DK * (DK + DV);  // Phi [DK][DK], then B [DK][DV]
  if (jn == 0 && half != 0) return;
#pragma unroll
  for (int jt = 0; jt < 4; jt++)
#pragma unroll
    for (int hh = 0; hh < 2; hh++) {
      const int r = 16 * mI + gq + 8 * hh, c = 8 * jt + 2 * tq;
      float* dst = jn == 0 ? out + r * DK + c : out + DK * DK + r * DV + half * NSC + c;
      *reinterpret_cast<float2*>(dst) = make_float2(xn[jt][2 * hh], xn[jt][2 * hh + 1]);
    }
}

struct BChainStage {
  bf16 M[2 * DK * DK];  // M (split)
  bf16 QW[2 * C * DK];  // QW (split)
  bf16 dO[C * NSC];     // columns col0.. of dO (exact bf16, operand layout)
};
struct BChainSm {
  BChainStage st[BSTG];
  bf16 dS[2 * DK * NSC];  // the carried state gradient (split)
  uint64_t bar[BSTG];     // completion of the stage's M and QW
};
static_assert(sizeof(BChainStage) % 16 == 0 && offsetof(BChainStage, QW) == 4 * DK * DK &&
                  offsetof(BChainStage, dO) == CB_KU1 - CB_M,
              "M | QW arrive in one copy");

// bwd_scan: the reverse chain dS = M^T dS' + QW^T dO, one CTA of four warps
// per (document, head, 32 value columns).
__global__ void __launch_bounds__(CTH) bwd_scan_kernel(Dims d, BwdIO io, Ws w) {
  extern __shared__ __align__(128) unsigned char smraw[];
  BChainSm& sm = *reinterpret_cast<BChainSm*>(smraw);
  const int tid = threadIdx.x, warp = tid >> 5;
  const int lane = tid & 31, gq = lane >> 2, tq = lane & 3;
  pdl_release();  // bwd_grad may launch: it waits for this grid before reading dS
  if (!saved_ok(d, w.tag, w.err)) return;
  const int H = d.H;
  const ChainCta cc = chain_cta(d, w);
  if (cc.unit < 0) return;
  const int h = cc.h, col0 = cc.half * NSC;
  // this CTA's run of chunks, taken from the last: a whole document, or with d.seg one unit of the
  // segment table (segment sg; `later` segments of the document follow it, all of n chunks but
  // the document's last)
  int doc = cc.unit, cb, n, sg = 0, later = 0;
  if (d.seg) {
    const int4 un = w.useg[cc.unit];
    doc = un.x;
    sg = un.w;
    n = un.z;
    cb = w.doc_chunk0[doc] + un.y;
    const int rest = w.doc_chunk0[doc + 1] - cb - n;
    later = rest > 0 ? (rest + n - 1) / n : 0;
  } else {
    cb = w.doc_chunk0[doc];
    n = w.doc_chunk0[doc + 1] - cb;
  }
  const int ce = cb + n;
  const DocSpan sp = doc_span(w, cb, n);
  const int64_t dh = ((int64_t)doc * H + h) * DK * DV;
  const Op dS{sm.dS, sm.dS + DK * NSC, NSC};
  for (int idx = tid; later == 0 && idx < DK * NSC / 2; idx += CTH) {  // (an earlier segment's is folded below)
    const int i = idx / (NSC / 2), jc = 2 * (idx % (NSC / 2));
    float2 v = make_float2(0.f, 0.f);
    if (io.dh_final) v = *reinterpret_cast<const float2*>(io.dh_final + dh + i * DV + col0 + jc);
    op_store2(dS, i, jc, v.x, v.y);
  }
  const bf16* dOg = (const bf16*)io.dO;
  if (tid == 0) {
    for (int s2 = 0; s2 < BSTG; s2++) mbar_init(&sm.bar[s2], 1);
    mbar_init_fence();
  }
  __syncthreads();  // the barriers are initialised before any thread waits on them
  auto prefetch = [&](int step) {  // always commits a cp.async group (empty past the end)
    if (step < n) {
      const int slot = step % BSTG;
      BChainStage& s = sm.st[slot];
      const int ci = ce - 1 - step, L = sp.L(n - 1 - step), t0 = sp.t0(n - 1 - step);
      const int64_t ch = (int64_t)ci * H + h;
      if (tid == 0) {  // M | QW, adjacent in the chain block and in the stage
        mbar_expect_tx(&sm.bar[slot], CB_KU1 - CB_M);
        bulk_g2s(s.M, chblk(w, ch) + CB_M, CB_KU1 - CB_M, &sm.bar[slot]);
      }
      for (int idx = tid; idx < C * NSC / 8; idx += CTH) {
        const int r = idx / (NSC / 8), p = idx % (NSC / 8);
        bf16* dst = s.dO + opix(r, 8 * p, NSC);
        if (r < L) cp16(dst, dOg + ((size_t)(t0 + r) * H + h) * DV + col0 + 8 * p);
        else *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    cp_commit();
  };
  for (int s = 0; s < BSTG - 1; s++) prefetch(s);
  if (later > 0) {
    // the gradient leaving segment sg: the composites of the document's later segments (the units
    // cc.unit + later down to cc.unit + 1) folded onto dS_final.  Scratch: the ring's last slot,
    // whose first copies are issued in step 0 (after this).
    float* fs = reinterpret_cast<float*>(&sm.st[BSTG - 1]);
    float* fp = fs + DK * NSC;
    float* fb = fp + DK * DK;
    for (int idx = tid; idx < DK * NSC; idx += CTH) {
      const int r = idx / NSC, c = idx % NSC;
      fs[idx] = io.dh_final ? io.dh_final[dh + r * DV + col0 + c] : 0.f;
    }
    fold_composites<CTH>(fs, fp, fb, w.segc + ((int64_t)(cc.unit + later) * H + h) * DK * (DK + DV),
                         -(int64_t)H * DK * (DK + DV), later, col0);
    for (int idx = tid; idx < DK * NSC / 2; idx += CTH) {
      const int r = idx / (NSC / 2), jc = 2 * (idx % (NSC / 2));
      op_store2(dS, r, jc, fs[r * NSC + jc], fs[r * NSC + jc + 1]);
    }
  }
  float acc[2][4];  // this warp's tile of the carried gradient: rows 16 (warp & 1) .., columns 16 (warp >> 1) ..
  zero(acc);
  const int mI = warp & 1, jn = warp >> 1;
  for (int step = 0; step < n; step++) {
    const BChainStage& s = sm.st[step % BSTG];
    const int ci = ce - 1 - step;
    asm volatile("cp.async.wait_group %0;\n" ::"n"(BSTG - 2));
    if (__syncthreads_or(!mbar_wait(&sm.bar[step % BSTG], (step / BSTG) & 1))) {  // a stage did not arrive in bound
      for (int k2 = step; k2 < n && k2 < step + BSTG - 1; k2++) mbar_wait(&sm.bar[k2 % BSTG], (k2 / BSTG) & 1);
      cp_wait_all();
      if (tid == 0) atomicExch(w.err, -7);
      return;
    }  // this step's stage and the last state update are visible
    prefetch(step + BSTG - 1);
    const Op Mo{const_cast<bf16*>(s.M), const_cast<bf16*>(s.M) + DK * DK, DK};
    const Op QWo{const_cast<bf16*>(s.QW), const_cast<bf16*>(s.QW) + C * DK, DK};
    const Op dOo{const_cast<bf16*>(s.dO), nullptr, NSC};
    float ax[2][4];
    zero(acc);
    zero(ax);
    gemm3<1, true, true>(ax, QWo, 16 * mI, 0, dOo, 16 * jn, 0, C / 16);
    gemm3<1, true, true>(acc, Mo, 16 * mI, 0, dS, 16 * jn, 0, DK / 16);
    slice_to_global(w.sdS + ((int64_t)ci * H + h) * 2 * DK * DV, sm.dS, col0, threadIdx.x);
#pragma unroll
    for (int jj = 0; jj < 2; jj++)
#pragma unroll
      for (int e = 0; e < 4; e++) acc[jj][e] += ax[jj][e];
    __syncthreads();  // every read of the state tile is done
#pragma unroll
    for (int jj = 0; jj < 2; jj++)
#pragma unroll
      for (int hh = 0; hh < 2; hh++)
        op_store2(dS, 16 * mI + gq + 8 * hh, 16 * jn + 8 * jj + 2 * tq, acc[jj][2 * hh], acc[jj][2 * hh + 1]);
  }
  cp_wait_all();
  if (io.dh0 && sg == 0) {  // the document's first chunks end its reverse chain
    if (n > 0) {
#pragma unroll
      for (int jj = 0; jj < 2; jj++)
#pragma unroll
        for (int hh = 0; hh < 2; hh++) {
          const int i = 16 * mI + gq + 8 * hh, c = 16 * jn + 8 * jj + 2 * tq;
          *reinterpret_cast<float2*>(io.dh0 + dh + i * DV + col0 + c) = make_float2(acc[jj][2 * hh], acc[jj][2 * hh + 1]);
        }
    } else {
      for (int idx = tid; idx < DK * NSC; idx += CTH) {
        const int i = idx / NSC, jc = idx % NSC;
        io.dh0[dh + i * DV + col0 + jc] = io.dh_final ? io.dh_final[dh + i * DV + col0 + jc] : 0.f;
      }
    }
  }
}

// bwd_seg: the composites of split backward chains (Dims::seg; the forward's
// segment table).  One CTA of four warps per (unit, head, 32 value columns)
// whose unit is a segment after its document's first: Y = [Psi | D] (32 x 64;
// Psi the product of the segment's M_c^T, D the gradient its reverse chain
// reaches from zero) by Y <- M_c^T Y + [0 | QW_c^T dO_c] over its chunks from
// the last, from [I | 0], with bwd_scan's products and four-stage ring (M | QW
// by bulk copy, dO rows by cp.async).  Psi is the same for both halves; half 0
// stores it (over the forward's composites, consumed by then).
struct BSegSm {
  BChainStage st[BSTG];
  bf16 Y[2][2 * DK * 2 * NSC];  // [Psi | D] (split), double-buffered
  uint64_t bar[BSTG];
};
static_assert(offsetof(BSegSm, Y) % 16 == 0, "operand tiles need 16-byte alignment");

__global__ void __launch_bounds__(CTH) bwd_seg_kernel(Dims d, BwdIO io, Ws w) {
  extern __shared__ __align__(128) unsigned char smraw[];
  BSegSm& sm = *reinterpret_cast<BSegSm*>(smraw);
  const int tid = threadIdx.x, warp = tid >> 5;
  const int lane = tid & 31, gq = lane >> 2, tq = lane & 3;
  if (!saved_ok(d, w.tag, w.err)) return;
  const ChainCta cc = chain_cta(d, w);
  const int u = cc.unit, h = cc.h, half = cc.half, col0 = half * NSC;
  if (u < 0) return;
  const int4 un = w.useg[u];  // (document, first chunk in it, chunks, segment)
  if (un.w == 0) return;      // a document's first segment is not composed
  const int H = d.H, n = un.z, cb = w.doc_chunk0[un.x] + un.y, ce = cb + n;
  const DocSpan sp = doc_span(w, cb, n);
  constexpr int YK = 2 * NSC;  // columns of Y
  const Op Y0{sm.Y[0], sm.Y[0] + DK * YK, YK}, Y1{sm.Y[1], sm.Y[1] + DK * YK, YK};
  for (int idx = tid; idx < DK * YK / 2; idx += CTH) {  // [I | 0]
    const int i = idx / (YK / 2), jc = 2 * (idx % (YK / 2));
    op_store2(Y0, i, jc, i == jc ? 1.f : 0.f, i == jc + 1 ? 1.f : 0.f);
  }
  const bf16* dOg = (const bf16*)io.dO;
  if (tid == 0) {
    for (int s2 = 0; s2 < BSTG; s2++) mbar_init(&sm.bar[s2], 1);
    mbar_init_fence();
  }
  __syncthreads();  // the barriers are initialised before any thread waits on them
  auto prefetch = [&](int step) {  // always commits a cp.async group (empty past the end)
    if (step < n) {
      const int slot = step % BSTG;
      BChainStage& s = sm.st[slot];
      const int ci = ce - 1 - step, L = sp.L(n - 1 - step), t0 = sp.t0(n - 1 - step);
      const int64_t ch = (int64_t)ci * H + h;
      if (tid == 0) {  // M | QW, adjacent in the chain block and in the stage
        mbar_expect_tx(&sm.bar[slot], CB_KU1 - CB_M);
        bulk_g2s(s.M, chblk(w, ch) + CB_M, CB_KU1 - CB_M, &sm.bar[slot]);
      }
      for (int idx = tid; idx < C * NSC / 8; idx += CTH) {
        const int r = idx / (NSC / 8), p = idx % (NSC / 8);
        bf16* dst = s.dO + opix(r, 8 * p, NSC);
        if (r < L) cp16(dst, dOg + ((size_t)(t0 + r) * H + h) * DV + col0 + 8 * p);
        else *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    cp_commit();
  };
  for (int s = 0; s < BSTG - 1; s++) prefetch(s);
  const int mI = warp & 1, jn = warp >> 1;  // this warp's tile of Y: rows 16 mI .., columns 32 jn ..
  float yn[4][4];
  zero(yn);
  for (int step = 0; step < n; step++) {
    const BChainStage& s = sm.st[step % BSTG];
    asm volatile("cp.async.wait_group %0;\n" ::"n"(BSTG - 2));
    if (__syncthreads_or(!mbar_wait(&sm.bar[step % BSTG], (step / BSTG) & 1))) {  // a stage did not arrive in bound
      for (int k2 = step; k2 < n && k2 < step + BSTG - 1; k2++) mbar_wait(&sm.bar[k2 % BSTG], (k2 / BSTG) & 1);
      cp_wait_all();
      if (tid == 0) atomicExch(w.err, -7);
      return;
    }  // this step's stage and Y are visible; the other Y buffer and the slot of step - 1 are free
    prefetch(step + BSTG - 1);
    const Op Mo{const_cast<bf16*>(s.M), const_cast<bf16*>(s.M) + DK * DK, DK};
    const Op QWo{const_cast<bf16*>(s.QW), const_cast<bf16*>(s.QW) + C * DK, DK};
    const Op dOo{const_cast<bf16*>(s.dO), nullptr, NSC};
    const Op& Yc = (step & 1) ? Y1 : Y0;
    const Op& Yn = (step & 1) ? Y0 : Y1;
    zero(yn);
    gemm3<2, true, true>(yn, Mo, 16 * mI, 0, Yc, 32 * jn, 0, DK / 16);        // M^T Y
    if (jn == 1) gemm3<2, true, true>(yn, QWo, 16 * mI, 0, dOo, 0, 0, C / 16);  // + QW^T dO
#pragma unroll
    for (int jt = 0; jt < 4; jt++)
#pragma unroll
      for (int hh = 0; hh < 2; hh++)
        op_store2(Yn, 16 * mI + gq + 8 * hh, 32 * jn + 8 * jt + 2 * tq, yn[jt][2 * hh], yn[jt][2 * hh + 1]);
  }
  cp_wait_all();
  float* out = w.segc + ((int64_t)u * H + h) * DK * (DK + DV);  // Psi [DK][DK], then D [DK][DV]
  if (jn == 0 && half != 0) return;
#pragma unroll
  for (int jt = 0; jt < 4; jt++)
#pragma unroll
    for (int hh = 0; hh < 2; hh++) {
      const int r = 16 * mI + gq + 8 * hh, c = 8 * jt + 2 * tq;
      float* dst = jn == 0 ? out + r * DK + c : out + DK * DK + r * DV + col0 + c;
      *reinterpret_cast<float2*>(dst) = make_float2(yn[jt][2 * hh], yn[jt][2 * hh + 1]);
    }
}

// bwd_scan_norm: the reverse chain with the gated RMSNorm's backward fused in
// front of its dO.  With y = o r w s (s = sigmoid(g), r = 1 / sqrt(mean_j o_j^2
// + eps)) and dy given, by the chain rule through the norm:
//   dO_j = r a_j - o_j r^3 (sum_k a_k o_k) / dv,   a_j = dy_j w_j s_j
//   dg_j = dy_j o_j r w_j s_j (1 - s_j),           dw_j = sum over rows of dy_j o_j r s_j
// The two row sums need all dv columns; the two column-half CTAs of a
// (document, head) run as a cluster and exchange their halves' partials
// through distributed shared memory.  Warp-specialised: warps 0-3 carry the
// chain exactly as bwd_scan does (their own named barrier between reading and
// writing the state tile); warps 4-7 form, during step s, the next stage's dO
// (its operand tile, dO in global memory for bwd_grad, dg, and the dw partials),
// so the norm's work and the exchange stay off the chain's critical path.  Each
// stage brings M | QW (one bulk copy) and this half's dy, g (bf16) and the
// forward's fp32 o (tensor-map copies) on one barrier, two steps ahead.  No
// early return after the first cluster barrier (errors skip the remaining
// steps) and a final cluster barrier: no CTA exits while its peer may still
// address its shared memory.
struct BChainStageN {
  bf16 M[2 * DK * DK];
  bf16 QW[2 * C * DK];
  bf16 dO[C * NSC];              // formed here by the norm warps
  bf16 dy[C * NSC], g[C * NSC];  // [C][NSC], rows past the chunk end masked when used
  float o[C * NSC];
};
struct BChainSmN {
  BChainStageN st[NSTG];
  bf16 dS[2 * DK * NSC];
  uint64_t bar[NSTG];
  Xchg x;
};
static_assert(sizeof(BChainStageN) % 128 == 0 && offsetof(BChainStageN, QW) == 4 * DK * DK &&
                  offsetof(BChainStageN, dy) % 128 == 0 &&
                  offsetof(BChainStageN, g) % 128 == 0 && offsetof(BChainStageN, o) % 128 == 0,
              "tensor-copy targets need 128-byte alignment");
constexpr uint32_t BSTAGE_N_TX = (CB_KU1 - CB_M) + 2 * 2 * C * NSC + 4 * C * NSC;

__global__ void __launch_bounds__(2 * CTH, 2) bwd_scan_norm_kernel(Dims d, BwdIO io, Ws w,
                                                                const __grid_constant__ NMaps nmap) {
  extern __shared__ __align__(128) unsigned char smraw[];
  BChainSmN& sm = *reinterpret_cast<BChainSmN*>(smraw);
  const int doc = blockIdx.x, h = blockIdx.y, col0 = blockIdx.z * NSC, tid = threadIdx.x, warp = tid >> 5;
  const int lane = tid & 31, gq = lane >> 2, tq = lane & 3;
  const bool chain = warp < 4;
  pdl_release();  // bwd_grad may launch: it waits for this grid before reading dS and dO
  const bool ok0 = saved_ok(d, w.tag, w.err);
  const int H = d.H;
  const int cb = w.doc_chunk0[doc], ce = w.doc_chunk0[doc + 1], n = ok0 ? ce - cb : 0;
  const DocSpan sp = doc_span(w, cb, n);
  const int64_t dh = ((int64_t)doc * H + h) * DK * DV;
  const Op dS{sm.dS, sm.dS + DK * NSC, NSC};
  for (int idx = tid; idx < DK * NSC / 2; idx += 2 * CTH) {
    const int i = idx / (NSC / 2), jc = 2 * (idx % (NSC / 2));
    float2 v = make_float2(0.f, 0.f);
    if (io.dh_final && ok0) v = *reinterpret_cast<const float2*>(io.dh_final + dh + i * DV + col0 + jc);
    op_store2(dS, i, jc, v.x, v.y);
  }
  if (tid == 0) {
    for (int s2 = 0; s2 < NSTG; s2++) mbar_init(&sm.bar[s2], 1);
    for (int x2 = 0; x2 < NX; x2++) mbar_init(&sm.x.bar[x2], 1);  // one local arming per phase + the peer's bytes
    mbar_init_fence();
    for (int x2 = 0; x2 < NX; x2++) mbar_expect_tx(&sm.x.bar[x2], XBYTES);  // stages 0 .. NX - 1
  }
  __syncthreads();
  cluster_sync();  // both CTAs' barriers are initialised before any remote arrival
  const uint32_t peer = cluster_rank() ^ 1u;
  const uint32_t xpart = cluster_map(&sm.x.part[0][0], peer), xbar = cluster_map(&sm.x.bar[0], peer);
  // (norm warps) thread nt owns row nt / 2, columns 16 (nt % 2) .. of the CTA's 32
  const int nt = tid - CTH, nr = nt >> 1, nh = nt & 1;
  float nwv[16], dwacc[16];
#pragma unroll
  for (int j = 0; j < 16; j++) {
    nwv[j] = chain ? 0.f : io.nw[col0 + 16 * nh + j];
    dwacc[j] = 0.f;
  }
  auto prefetch = [&](int step) {  // one thread: M | QW (bulk) and dy, g, o (tensor maps) on one barrier
    if (step < n && tid == 0) {
      const int slot = step % NSTG;
      BChainStageN& s = sm.st[slot];
      const int ci = ce - 1 - step, t0 = sp.t0(n - 1 - step);
      const int64_t ch = (int64_t)ci * H + h;
      mbar_expect_tx(&sm.bar[slot], BSTAGE_N_TX);
      bulk_g2s(s.M, chblk(w, ch) + CB_M, CB_KU1 - CB_M, &sm.bar[slot]);
      tma_load_2d(s.dy, &nmap.dy, h * DV + col0, t0, &sm.bar[slot]);
      tma_load_2d(s.g, &nmap.g, h * DV + col0, t0, &sm.bar[slot]);
      tma_load_2d(s.o, &nmap.o, h * DV + col0, t0, &sm.bar[slot]);
    }
  };
  // (norm warps) this thread's 16 values of stage k's row nr, rows past the chunk end as zero
  auto norm_vals = [&](const BChainStageN& s, int L, float* dyv, float* ov, float* sgv) {
#pragma unroll
    for (int hh = 0; hh < 2; hh++) {
      const int o8 = nr * NSC + 16 * nh + 8 * hh;
      unpack8(*reinterpret_cast<const uint4*>(s.dy + o8), dyv + 8 * hh);
      unpack8(*reinterpret_cast<const uint4*>(s.g + o8), sgv + 8 * hh);
      const float4 a = *reinterpret_cast<const float4*>(s.o + o8), b = *reinterpret_cast<const float4*>(s.o + o8 + 4);
      ov[8 * hh] = a.x; ov[8 * hh + 1] = a.y; ov[8 * hh + 2] = a.z; ov[8 * hh + 3] = a.w;
      ov[8 * hh + 4] = b.x; ov[8 * hh + 5] = b.y; ov[8 * hh + 6] = b.z; ov[8 * hh + 7] = b.w;
    }
    const bool live = nr < L;
#pragma unroll
    for (int j = 0; j < 16; j++) {
      sgv[j] = live ? sigmoid_fast(sgv[j]) : 0.f;  // s_j
      if (!live) dyv[j] = ov[j] = 0.f;
    }
  };
  bool xfail = false, bad = false;
  // (norm warps) stage k's dO: wait for the stage, send the row partials, receive the peer's,
  // write the dO operand tile, dO and dg to global memory, and accumulate dw
  auto norm_stage = [&](int k) {
    BChainStageN& s = sm.st[k % NSTG];
    if (!mbar_wait(&sm.bar[k % NSTG], (k / NSTG) & 1)) {
      xfail = true;
      return;
    }
    const int L = sp.L(n - 1 - k), t0 = sp.t0(n - 1 - k), slot = k % NX;
    float dyv[16], ov[16], sgv[16];
    norm_vals(s, L, dyv, ov, sgv);
    float po = 0.f, pa = 0.f;
#pragma unroll
    for (int j = 0; j < 16; j++) {
      po += ov[j] * ov[j];
      pa += dyv[j] * nwv[j] * sgv[j] * ov[j];  // a_j o_j
    }
    po += __shfl_xor_sync(0xffffffffu, po, 1);
    pa += __shfl_xor_sync(0xffffffffu, pa, 1);
    if (nh == 0) st_async_f32x2(xpart + (uint32_t)((slot * C + nr) * 8), po, pa, xbar + (uint32_t)(slot * 8));
    float dOv[16];
    if (!mbar_wait_cluster(&sm.x.bar[slot], (k / NX) & 1)) {
      xfail = true;
#pragma unroll
      for (int j = 0; j < 16; j++) dOv[j] = 0.f;
    } else {
      if (nt == 0) mbar_expect_tx(&sm.x.bar[slot], XBYTES);  // armed for stage k + NX
      const float2 pp = sm.x.part[slot][nr];
      const float To = po + pp.x, Ta = pa + pp.y;
      const float rr = 1.0f / sqrtf(To * (1.0f / DV) + io.neps);
      const float cc = rr * rr * rr * Ta * (1.0f / DV);
      float dgv[16];
#pragma unroll
      for (int j = 0; j < 16; j++) {
        const float sg = sgv[j], or_ = ov[j] * rr;
        dOv[j] = rr * dyv[j] * nwv[j] * sg - ov[j] * cc;
        dgv[j] = dyv[j] * or_ * nwv[j] * sg * (1.f - sg);
        dwacc[j] += dyv[j] * or_ * sg;
      }
      if (nr < L) {
        const size_t gi = ((size_t)(t0 + nr) * H + h) * DV + col0 + 16 * nh;
#pragma unroll
        for (int hh = 0; hh < 2; hh++) {
          uint4 ud, ug;
          __nv_bfloat162* d2 = reinterpret_cast<__nv_bfloat162*>(&ud);
          __nv_bfloat162* g2 = reinterpret_cast<__nv_bfloat162*>(&ug);
#pragma unroll
          for (int e = 0; e < 4; e++) {
            d2[e] = __floats2bfloat162_rn(dOv[8 * hh + 2 * e], dOv[8 * hh + 2 * e + 1]);
            g2[e] = __floats2bfloat162_rn(dgv[8 * hh + 2 * e], dgv[8 * hh + 2 * e + 1]);
          }
          *reinterpret_cast<uint4*>((bf16*)io.dOw + gi + 8 * hh) = ud;
          *reinterpret_cast<uint4*>((bf16*)io.dg + gi + 8 * hh) = ug;
        }
      }
    }
#pragma unroll
    for (int hh = 0; hh < 2; hh++) {  // the dO operand tile (bf16, as stored for the per-chunk kernels)
      uint4 u;
      __nv_bfloat162* u2 = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
      for (int e = 0; e < 4; e++) u2[e] = __floats2bfloat162_rn(dOv[8 * hh + 2 * e], dOv[8 * hh + 2 * e + 1]);
      *reinterpret_cast<uint4*>(s.dO + opix(nr, 16 * nh + 8 * hh, NSC)) = u;
    }
  };
  for (int s = 0; s < NSTG - 1; s++) prefetch(s);
  if (!chain && n > 0) norm_stage(0);  // stage 0's dO before the chain starts
  float acc[2][4];
  zero(acc);
  const int mI = warp & 1, jn = (warp >> 1) & 1;
  for (int step = 0; step < n; step++) {
    const BChainStageN& s = sm.st[step % NSTG];
    const int ci = ce - 1 - step;
    if (__syncthreads_or(!mbar_wait(&sm.bar[step % NSTG], (step / NSTG) & 1) || xfail)) {  // a wait ran out
      for (int k2 = step; k2 < n && k2 < step + NSTG - 1; k2++) mbar_wait(&sm.bar[k2 % NSTG], (k2 / NSTG) & 1);
      if (tid == 0) atomicExch(w.err, -7);
      bad = true;
      break;
    }  // this step's stage, its dO tile and the last state update are visible
    prefetch(step + NSTG - 1);
    if (chain) {
      const Op Mo{const_cast<bf16*>(s.M), const_cast<bf16*>(s.M) + DK * DK, DK};
      const Op QWo{const_cast<bf16*>(s.QW), const_cast<bf16*>(s.QW) + C * DK, DK};
      const Op dOo{const_cast<bf16*>(s.dO), nullptr, NSC};
      float ax[2][4];
      zero(acc);
      zero(ax);
      gemm3<1, true, true>(ax, QWo, 16 * mI, 0, dOo, 16 * jn, 0, C / 16);
      gemm3<1, true, true>(acc, Mo, 16 * mI, 0, dS, 16 * jn, 0, DK / 16);
      slice_to_global(w.sdS + ((int64_t)ci * H + h) * 2 * DK * DV, sm.dS, col0, tid);
#pragma unroll
      for (int jj = 0; jj < 2; jj++)
#pragma unroll
        for (int e = 0; e < 4; e++) acc[jj][e] += ax[jj][e];
      asm volatile("bar.sync 1, %0;\n" ::"n"(CTH) : "memory");  // the chain warps' reads of the state tile are done
#pragma unroll
      for (int jj = 0; jj < 2; jj++)
#pragma unroll
        for (int hh = 0; hh < 2; hh++)
          op_store2(dS, 16 * mI + gq + 8 * hh, 16 * jn + 8 * jj + 2 * tq, acc[jj][2 * hh], acc[jj][2 * hh + 1]);
    } else if (step + 1 < n) {
      norm_stage(step + 1);  // the next stage's dO, while the chain works on this one
    }
  }
  if (__syncthreads_or(xfail) && !bad) {  // the last exchange ran out
    if (tid == 0) atomicExch(w.err, -7);
    bad = true;
  }
  if (io.dh0 && !bad && ok0) {
    if (n > 0) {
      if (chain)
#pragma unroll
        for (int jj = 0; jj < 2; jj++)
#pragma unroll
          for (int hh = 0; hh < 2; hh++) {
            const int i = 16 * mI + gq + 8 * hh, c = 16 * jn + 8 * jj + 2 * tq;
            *reinterpret_cast<float2*>(io.dh0 + dh + i * DV + col0 + c) =
                make_float2(acc[jj][2 * hh], acc[jj][2 * hh + 1]);
          }
    } else {
      for (int idx = tid; idx < DK * NSC; idx += 2 * CTH) {
        const int i = idx / NSC, jc = idx % NSC;
        io.dh0[dh + i * DV + col0 + jc] = io.dh_final ? io.dh_final[dh + i * DV + col0 + jc] : 0.f;
      }
    }
  }
  // dw partial of this (document, head): column sums over the 64 rows (the norm
  // threads of each half), in a fixed order, through the idle stage 0
  float* red = reinterpret_cast<float*>(&sm.st[0]);  // [CTH][16]
  __syncthreads();
  if (!chain)
#pragma unroll
    for (int j = 0; j < 16; j++) red[nt * 16 + j] = dwacc[j];
  __syncthreads();
  if (tid < NSC && !bad && ok0) {
    const int hf = tid >> 4, j = tid & 15;
    float a = 0.f;
    for (int r = 0; r < C; r++) a += red[(2 * r + hf) * 16 + j];
    w.pdw[((int64_t)doc * H + h) * DV + col0 + tid] = a;
  }
  cluster_sync();  // the peer no longer touches this CTA's shared memory
}

// ------------------------------------------------------------ backward chunk kernels

// Tensor-core rounds with several issuing threads.  A small product is bound by
// the issue of its MMAs (about 60 cycles each), not by the tensor core, so the
// independent products of a round (each with its own accumulator) are issued in
// parallel: lane 0 of warp q < NISS runs share(q) and commits to the round's
// barrier, or arrives on it plainly when share(q) issued nothing; the barrier
// (NISS arrivals) completes once every share's MMAs have.
constexpr int NISS = 4;
template <class F>
__device__ __forceinline__ void issue_round(uint64_t* bar, F share) {
  const int q = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0 && q < NISS) {
    tc::fence_after();
    if (share(q)) tc::commit(bar);
    else mbar_arrive(bar);
  }
}

__device__ __forceinline__ void blk_ij(int b, int& I, int& J) {
  I = b < 1 ? 0 : b < 3 ? 1 : b < 6 ? 2 : 3;
  J = b - I * (I + 1) / 2;
}
__device__ __forceinline__ int blk_of(int I, int J) { return I * (I + 1) / 2 + J; }

// The 8 accumulator values a thread holds of a 16 x 16 tile, in fragment
// order: bwd_grad and bwd_gate use the same warp -> tile mapping, so the
// hand-over is two float4 per thread, the second NTH float4 after the first
// (each store / load instruction of a warp covers 512 contiguous bytes).
__device__ __forceinline__ void frag_store(float* g, const float (&v)[2][4]) {
  float4* p = reinterpret_cast<float4*>(g) + threadIdx.x;
  p[0] = make_float4(v[0][0], v[0][1], v[0][2], v[0][3]);
  p[NTH] = make_float4(v[1][0], v[1][1], v[1][2], v[1][3]);
}
__device__ __forceinline__ void frag_load(const float* g, float (&v)[2][4]) {
  const float4* p = reinterpret_cast<const float4*>(g) + threadIdx.x;
  const float4 a = p[0], b = p[NTH];
  v[0][0] = a.x; v[0][1] = a.y; v[0][2] = a.z; v[0][3] = a.w;
  v[1][0] = b.x; v[1][1] = b.y; v[1][2] = b.z; v[1][3] = b.w;
}

// bwd_grad: one CTA per chunk-head (two per SM).  From the forward's saved
// operand tiles (T, P = scale P', W, U; A' fp32) and the chunk's entry state
// S and exit-state gradient dS' it forms
//   dE = P^T dO + KD dS',  E = U - W S,
//   dP' = scale dO E^T,  dKD = E dS'^T,  dQG = scale dO S^T,  dW = -dE S^T,
//   dgamma = rowsum(dS' .* S),  YU = T^T dE,  YW = T^T dW,  dv = beta YU,
//   dA = -(YU U^T + YW W^T) (strict lower),  MA = beta dA,
//   dbeta = rowsum(YU .* V) + rowsum(YW .* K^ e^G) + rowsum(dA .* A'),
// writes dv and db, and hands dP', MA, dQG, dKD, beta YW and dgamma to bwd_gate.
struct GradSm {
  __align__(16) bf16 wk[45056];  // work area (88 KB), regions bound in the kernel
  __align__(16) float gg[C * SQ];
  __align__(16) bf16 rk[C * DK];  // 16-byte cp.async / vector access
  float bet[C], braw[C], dbet[C], part[4 * C];
  float tot[NW * DK];
  uint64_t bar[3];  // bulk-load completion (saved tiles, the dA operands); MMA rounds
  uint32_t tslot;   // TMEM base address
};
static_assert(offsetof(GradSm, rk) % 16 == 0 && offsetof(GradSm, gg) % 16 == 0, "vector-accessed arrays");

template <bool CONV>
__global__ void __launch_bounds__(NTH, 2) bwd_grad_kernel(Dims d, BwdIO io, Ws w) {
  extern __shared__ __align__(128) unsigned char smraw[];
  GradSm& sm = *reinterpret_cast<GradSm*>(smraw);
  const int j = (int)(blockIdx.x / (unsigned)d.H), h = (int)(blockIdx.x % (unsigned)d.H), tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, tq = lane & 3;
  const bool gdn = d.gate != 0;
  const float* dtb = io.dt_bias + h * (gdn ? 1 : DK);
  float dtv[8];  // dt_bias of this thread's key channels 8 (tid % 4) ..
#pragma unroll
  for (int e = 0; e < 8; e++) dtv[e] = dtb[gdn ? 0 : 8 * (tid & 3) + e];
  const float alog = io.A_log[h];
  pdl_release();  // bwd_gate may launch: it waits for this grid before its hand-over reads
  const int tag = *w.tag, err = *w.err, L = w.chunk_len[j], t0 = w.chunk_tok0[j];  // one round trip
  if (tag != d.tag) {
    *w.err = -5;
    return;
  }
  if (err != 0 || L <= 0) return;
  const int H = d.H;
  const int64_t ch = (int64_t)j * H + h;
  const float a = expf(alog), scale = d.scale;
  bf16* wk = sm.wk;
  // work-area regions (bf16 offsets): dO 0 | S 4096 | dS' 8192 | P -> E 12288 |
  // W -> dW -> YW 20480 | U -> dE -> YU 24576 | raw f -> KD 32768 | T 36864;
  // reloaded for the dA products over the first four: U 0 | W 8192 | A' 12288
  const Op dO{wk, nullptr, DV}, S{wk + 4096, wk + 6144, DV}, dS{wk + 8192, wk + 10240, DV};
  const Op P{wk + 12288, wk + 16384, C}, E{wk + 12288, wk + 16384, DV};
  const Op W{wk + 20480, wk + 22528, DK}, U{wk + 24576, wk + 28672, DV};
  const Op KD{wk + 32768, wk + 34816, DK}, T{wk + 36864, wk + 40960, C};
  const Op dW = W, YW = W, dE = U, YU = U;
  const Op U2{wk, wk + 4096, DV}, W2{wk + 8192, wk + 10240, DK};
  bf16* fst = wk + 32768;

  // ---- group 1: raw k, f;  group 2: dO, S, dS', P, W, U, T  (CONV: k comes from the convolution below)
  for (int idx = tid; idx < C * 4; idx += NTH) {
    const int r = idx >> 2, p = idx & 3;
    if (r < L) {
      const size_t g = ((size_t)(t0 + r) * H + h) * DK + 8 * p;
      if (!CONV) cp16(sm.rk + r * DK + 8 * p, (const bf16*)io.k + g);
      if (!gdn) cp16(fst + r * DK + 8 * p, (const bf16*)io.f + g);
    }
  }
  cp_commit();
  if (d.norm) pdl_wait();  // dO is then written by the fused-norm bwd_scan, the kernel before
  for (int idx = tid; idx < C * 8; idx += NTH) {
    const int r = idx >> 3, p = idx & 7;
    bf16* dst = wk + opix(r, 8 * p, DV);
    if (r < L) cp16(dst, (const bf16*)io.dO + ((size_t)(t0 + r) * H + h) * DV + 8 * p);
    else *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
  }
  cp_commit();
  if (tid == 0) {  // the saved tiles in one bulk transaction group
    mbar_init(&sm.bar[0], 1);
    mbar_init(&sm.bar[1], 1);
    mbar_init(&sm.bar[2], NISS);
    mbar_init_fence();
    mbar_expect_tx(&sm.bar[0], 2 * 4 * DK * DV + 2 * 4 * C * C + 4 * C * DK + 4 * C * DV);
    bulk_g2s(S.hi, w.sS + ch * 2 * DK * DV, 4 * DK * DV, &sm.bar[0]);
    bulk_g2s(P.hi, w.sP + ch * 2 * C * C, 4 * C * C, &sm.bar[0]);
    bulk_g2s(W.hi, w.sW + ch * 2 * C * DK, 4 * C * DK, &sm.bar[0]);
    bulk_g2s(U.hi, w.sU + ch * 2 * C * DV, 4 * C * DV, &sm.bar[0]);
    bulk_g2s(T.hi, w.sT + ch * 2 * C * C, 4 * C * C, &sm.bar[0]);
    pdl_wait();  // dS' is bwd_scan's (the kernel before): the forward's tiles above are not
    bulk_g2s(dS.hi, w.sdS + ch * 2 * DK * DV, 4 * DK * DV, &sm.bar[0]);
  }

  if (warp == 0) tc::tmem_alloc(&sm.tslot, TCOLS);  // published by the barrier below

  // ---- k^, G, beta (thread: row tid / 4, key channels 8 (tid % 4) .., value columns 16 (tid % 4) ..)
  const int r = tid >> 2, q4 = tid & 3;
  const bool in = r < L;
  uint4 vraw[2] = {make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u)};
  float vcv[CONV ? 16 : 1];  // CONV: this thread's v after the convolution
  float kcv[CONV ? 8 : 1];   // and its k
  float braw = 0.f, fs = 0.f;  // fs: the scalar gate input of this row
  if (in) {
    const size_t row = (size_t)(t0 + r) * H + h;
    if constexpr (CONV) {
      const int tmin = conv_tmin(w, j, t0);
      conv_load<16>(vcv, (const bf16*)io.v + h * DV + 16 * q4, io.ld, t0 + r, tmin, io.cwv + 4 * (h * DV + 16 * q4));
      conv_load<8>(kcv, (const bf16*)io.k + h * DK + 8 * q4, io.ld, t0 + r, tmin, io.cwk + 4 * (h * DK + 8 * q4));
    } else {
      const uint4* vp = reinterpret_cast<const uint4*>((const bf16*)io.v + row * DV + 16 * q4);
      vraw[0] = __ldg(vp);
      vraw[1] = __ldg(vp + 1);
    }
    braw = bfl(((const bf16*)io.b)[row]);
    if (gdn) fs = bfl(((const bf16*)io.f)[row]);
  } else if constexpr (CONV) {
#pragma unroll
    for (int e = 0; e < 16; e++) vcv[e] = 0.f;
#pragma unroll
    for (int e = 0; e < 8; e++) kcv[e] = 0.f;
  }
  asm volatile("cp.async.wait_group 1;\n" ::);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tb = sm.tslot;
  float kv[8], gv[8];
  if (in) {
    if constexpr (CONV) {
#pragma unroll
      for (int e = 0; e < 8; e++) kv[e] = kcv[e];
    } else {
      unpack8(*reinterpret_cast<const uint4*>(sm.rk + r * DK + 8 * q4), kv);
    }
    if (gdn) {
      const float g = -a * LOG2E * softplus_fast(fs + dtv[0]);
#pragma unroll
      for (int e = 0; e < 8; e++) gv[e] = g;
    } else {
      unpack8(*reinterpret_cast<const uint4*>(fst + r * DK + 8 * q4), gv);
#pragma unroll
      for (int e = 0; e < 8; e++) gv[e] = -a * LOG2E * softplus_fast(gv[e] + dtv[e]);
    }
  } else {
#pragma unroll
    for (int e = 0; e < 8; e++) kv[e] = gv[e] = 0.f;
  }
  {
    float sk = 0.f;
#pragma unroll
    for (int e = 0; e < 8; e++) sk += kv[e] * kv[e];
    sk += __shfl_xor_sync(0xffffffffu, sk, 1);
    sk += __shfl_xor_sync(0xffffffffu, sk, 2);
    const float ik = 1.0f / sqrtf(sk + L2_EPS);
#pragma unroll
    for (int e = 0; e < 8; e++) kv[e] *= ik;
  }
  if (q4 == 0) {
    sm.bet[r] = in ? sigmoid_fast(braw) : 0.f;
    sm.braw[r] = braw;
  }
#pragma unroll
  for (int e = 0; e < 8; e++) {
    float x = gv[e];
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      const float y2 = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y2;
    }
    gv[e] = x;
  }
  if (lane >= 28)
#pragma unroll
    for (int e = 0; e < 8; e++) sm.tot[warp * DK + 8 * q4 + e] = gv[e];
  __syncthreads();
  add_warp_prefix(gv, sm.tot, warp, lane, q4);
  store_row8(sm.gg, r, q4, gv);
  __syncthreads();
  float xkg[8];  // k^ e^G for the W term of dbeta
#pragma unroll
  for (int e = 0; e < 8; e += 2) {
    const int i = 8 * q4 + e;
    const float gl0 = sm.gg[(L - 1) * SQ + i], gl1 = sm.gg[(L - 1) * SQ + i + 1];
    op_store2(KD, r, i, kv[e] * ex2(gl0 - gv[e]), kv[e + 1] * ex2(gl1 - gv[e + 1]));
    xkg[e] = kv[e] * ex2(gv[e]);
    xkg[e + 1] = kv[e + 1] * ex2(gv[e + 1]);
  }
  cp_wait_all();
  fence_async_smem();  // KD and dO are read by the tensor core next
  tc::fence_before();
  if (__syncthreads_or(!mbar_wait(&sm.bar[0], 0))) {  // a bulk load did not complete in bound
    mbar_wait(&sm.bar[0], 0);
    if (warp == 0) tc::tmem_dealloc(tb, TCOLS);
    if (tid == 0) atomicExch(w.err, -7);
    return;
  }
  // MMA rounds: one thread issues, completion on bar[2] (phase mph), all warps
  // then read their fragments.  TMEM columns: dE 0 | E 64 | dKD 128 | dQG 160 |
  // dW' 192 | YW 224;  dP' reuses 0, YU 64, dA 128.
  uint32_t mph = 0;
  auto round_done = [&]() -> bool {  // uniform over the CTA
    const bool ok = mbar_wait(&sm.bar[2], mph);
    mph ^= 1;
    tc::fence_after();
    return !__syncthreads_or(!ok);
  };
  auto bail = [&]() {
    mbar_wait(&sm.bar[2], mph ^ 1);
    tc::fence_before();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tb, TCOLS);
    if (tid == 0) atomicExch(w.err, -7);
  };

  const int I = warp & 3, hk = warp >> 2;  // owner tile: rows 16 I .., columns 32 hk .. / 16 hk ..
  // ---- dE = P^T dO + KD dS' and E = U - W S
  issue_round(&sm.bar[2], [&](int q) {
    if (q == 0) {
      tc::gemm_split(tb + 0, tc::mnmaj(P), tc::mnmaj(dO), 64, C / 16, false);
      tc::gemm_split(tb + 0, tc::kmaj(KD), tc::mnmaj(dS), 64, DK / 16, true);
    } else if (q == 1) {
      tc::gemm_split(tb + 64, tc::kmaj(W), tc::mnmaj(S), 64, DK / 16, false);
    }
    return q < 2;
  });
  if (!round_done()) { bail(); return; }
  {
    float dEr[4][4], ws[4][4];
    tc::ld_frag<4>(tb + 0, 32 * hk, dEr);
    tc::ld_frag<4>(tb + 64, 32 * hk, ws);
    // each thread reads U at the positions it then overwrites with dE; E goes over P
#pragma unroll
    for (int jt = 0; jt < 4; jt++)
#pragma unroll
      for (int hh = 0; hh < 2; hh++) {
        const int rr = 16 * I + gq + 8 * hh, col = 32 * hk + 8 * jt + 2 * tq;
        const float e0 = op_get(U, rr, col) - ws[jt][2 * hh], e1 = op_get(U, rr, col + 1) - ws[jt][2 * hh + 1];
        op_store2(E, rr, col, e0, e1);
        op_store2(dE, rr, col, dEr[jt][2 * hh], dEr[jt][2 * hh + 1]);
      }
  }
  fence_async_smem();
  tc::fence_before();
  __syncthreads();
  // ---- dKD = E dS'^T, dQG = scale dO S^T (to bwd_gate), dW = -dE S^T (over W),
  //      dP' = scale dO E^T lower blocks (to bwd_gate), dgamma
  issue_round(&sm.bar[2], [&](int q) {
    if (q == 0) tc::gemm_split(tb + 128, tc::kmaj(E), tc::kmaj(dS), 32, DV / 16, false);
    else if (q == 1) tc::gemm_split(tb + 160, tc::kmaj(dO), tc::kmaj(S), 32, DV / 16, false);
    else if (q == 2) tc::gemm_split(tb + 192, tc::kmaj(dE), tc::kmaj(S), 32, DV / 16, false);
    else tc::gemm_split(tb + 0, tc::kmaj(dO), tc::kmaj(E), 64, DV / 16, false);
    return true;
  });
  if (warp < 4) {  // dgamma_i = sum_j dS'_ij S_ij: lane = row i % 8 x column chunks (lane / 8, + 4); a
                    // quarter-warp reads whole core matrices
    const int i = 8 * warp + (lane & 7);
    float acc1 = 0.f;
#pragma unroll
    for (int hc = 0; hc < 2; hc++) {
      const int o = opix(i, 8 * ((lane >> 3) + 4 * hc), DV);
      float x[8], y[8], xl[8], yl[8];
      unpack8(*reinterpret_cast<const uint4*>(dS.hi + o), x);
      unpack8(*reinterpret_cast<const uint4*>(dS.lo + o), xl);
      unpack8(*reinterpret_cast<const uint4*>(S.hi + o), y);
      unpack8(*reinterpret_cast<const uint4*>(S.lo + o), yl);
#pragma unroll
      for (int e = 0; e < 8; e++) acc1 += (x[e] + xl[e]) * (y[e] + yl[e]);
    }
    acc1 += __shfl_xor_sync(0xffffffffu, acc1, 8);
    acc1 += __shfl_xor_sync(0xffffffffu, acc1, 16);
    if (lane < 8) w.gdg[ch * DK + i] = acc1;
  }
  if (!round_done()) { bail(); return; }
  {
    float dKD[2][4], dQG[2][4], acc[2][4], pp[4][4];
    tc::ld_frag<2>(tb + 128, 16 * hk, dKD);
    tc::ld_frag<2>(tb + 160, 16 * hk, dQG);
    tc::ld_frag<2>(tb + 192, 16 * hk, acc);
    tc::ld_frag<4>(tb + 0, 32 * hk, pp);
    each(dQG, [&](int, int, float& v) { v *= scale; });
    frag_store(w.gKD + ch * NTH * 8, dKD);
    frag_store(w.gQG + ch * NTH * 8, dQG);
#pragma unroll
    for (int jt = 0; jt < 2; jt++)
#pragma unroll
      for (int hh = 0; hh < 2; hh++)
        op_store2(dW, 16 * I + gq + 8 * hh, 16 * hk + 8 * jt + 2 * tq, -acc[jt][2 * hh], -acc[jt][2 * hh + 1]);
#pragma unroll
    for (int jb = 0; jb < 2; jb++) {  // blocks (I, J) of this warp's 32 columns, J <= I
      const int J = 2 * hk + jb;
      if (J > I) continue;
      float* g = w.gDP + (ch * NBLK + blk_of(I, J)) * 16 * PB;
#pragma unroll
      for (int jt = 0; jt < 2; jt++)
#pragma unroll
        for (int hh = 0; hh < 2; hh++) {
          const int m = gq + 8 * hh, n = 8 * jt + 2 * tq;
          const int rr = 16 * I + m, s0 = 16 * J + n;
          const float* v = pp[2 * jb + jt];
          *reinterpret_cast<float2*>(g + m * PB + n) =
              make_float2(s0 <= rr ? scale * v[2 * hh] : 0.f, s0 + 1 <= rr ? scale * v[2 * hh + 1] : 0.f);
        }
    }
  }
  fence_async_smem();
  tc::fence_before();
  __syncthreads();
  // ---- U, W, A' for the dA products (bulk, over dO, S, dS', E: all read by now);
  //      YU = T^T dE, YW = T^T dW
  if (tid == 0) {
    mbar_expect_tx(&sm.bar[1], 4 * C * DV + 4 * C * DK + NBLK * 16 * PB * 4);
    bulk_g2s(U2.hi, w.sU + ch * 2 * C * DV, 4 * C * DV, &sm.bar[1]);
    bulk_g2s(W2.hi, w.sW + ch * 2 * C * DK, 4 * C * DK, &sm.bar[1]);
    bulk_g2s(wk + 12288, w.sA + ch * NBLK * 16 * PB, NBLK * 16 * PB * 4, &sm.bar[1]);
  }
  issue_round(&sm.bar[2], [&](int q) {
    if (q == 0) tc::gemm_split(tb + 64, tc::mnmaj(T), tc::mnmaj(dE), 64, C / 16, false);
    else if (q == 1) tc::gemm_split(tb + 224, tc::mnmaj(T), tc::mnmaj(dW), 32, C / 16, false);
    return q < 2;
  });
  if (!round_done()) { bail(); return; }
  {  // YU over dE, YW over dW (each thread overwrites only what it read... the MMA read them: done);
     // dv = beta YU; beta YW to bwd_gate
    float yu[4][4], yw[2][4];
    tc::ld_frag<4>(tb + 64, 32 * hk, yu);
    tc::ld_frag<2>(tb + 224, 16 * hk, yw);
    bf16* dvo = (bf16*)io.dv;
#pragma unroll
    for (int jt = 0; jt < 4; jt++)
#pragma unroll
      for (int hh = 0; hh < 2; hh++) {
        const int rr = 16 * I + gq + 8 * hh, col = 32 * hk + 8 * jt + 2 * tq;
        op_store2(YU, rr, col, yu[jt][2 * hh], yu[jt][2 * hh + 1]);
        if (rr < L) {
          if constexpr (CONV)  // fp32 gradient of the convolution's v output
            *reinterpret_cast<float2*>((float*)io.dv + (size_t)(t0 + rr) * io.ld + h * DV + col) =
                make_float2(sm.bet[rr] * yu[jt][2 * hh], sm.bet[rr] * yu[jt][2 * hh + 1]);
          else
            *reinterpret_cast<__nv_bfloat162*>(dvo + ((size_t)(t0 + rr) * H + h) * DV + col) =
                __floats2bfloat162_rn(sm.bet[rr] * yu[jt][2 * hh], sm.bet[rr] * yu[jt][2 * hh + 1]);
        }
      }
#pragma unroll
    for (int jt = 0; jt < 2; jt++)
#pragma unroll
      for (int hh = 0; hh < 2; hh++) {
        const int rr = 16 * I + gq + 8 * hh;
        op_store2(YW, rr, 16 * hk + 8 * jt + 2 * tq, yw[jt][2 * hh], yw[jt][2 * hh + 1]);
        yw[jt][2 * hh] *= sm.bet[rr];
        yw[jt][2 * hh + 1] *= sm.bet[rr];
      }
    frag_store(w.gKG + ch * NTH * 8, yw);
  }
  fence_async_smem();
  tc::fence_before();
  if (__syncthreads_or(!mbar_wait(&sm.bar[1], 0))) {
    mbar_wait(&sm.bar[1], 0);
    if (warp == 0) tc::tmem_dealloc(tb, TCOLS);
    if (tid == 0) atomicExch(w.err, -7);
    return;
  }
  // ---- dA = -(YU U^T + YW W^T) strict lower; dbeta (U and W terms, row layout); MA = beta dA
  //      (to bwd_gate) and the A' term of dbeta
  issue_round(&sm.bar[2], [&](int q) {
    if (q == 0) {
      tc::gemm_split(tb + 128, tc::kmaj(YU), tc::kmaj(U2), 64, DV / 16, false);
      tc::gemm_split(tb + 128, tc::kmaj(YW), tc::kmaj(W2), 64, DK / 16, true);
    }
    return q == 0;
  });
  {  // bf16 pairs read in the rotated order of store8_rot: the 32 lanes hit 32 banks
    float va[8], vb[8];
    if constexpr (CONV) {
#pragma unroll
      for (int e = 0; e < 8; e++) {
        va[e] = vcv[e];
        vb[e] = vcv[8 + e];
      }
    } else {
      unpack8(vraw[0], va);
      unpack8(vraw[1], vb);
    }
    rot_pairs(va, q4);
    rot_pairs(vb, q4);
    rot_pairs(xkg, q4);
    auto pair = [&](const Op& t, int c) {
      const int i = opix(r, c, t.K);
      const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(t.hi + i));
      const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(t.lo + i));
      return make_float2(hi.x + lo.x, hi.y + lo.y);
    };
    float acc = 0.f;
#pragma unroll
    for (int p = 0; p < 4; p++) {
      const int c2 = 2 * ((p + q4) & 3);
      const float2 u0 = pair(YU, 16 * q4 + c2), u1 = pair(YU, 16 * q4 + 8 + c2), y = pair(YW, 8 * q4 + c2);
      acc += u0.x * va[2 * p] + u0.y * va[2 * p + 1] + u1.x * vb[2 * p] + u1.y * vb[2 * p + 1];
      acc += y.x * xkg[2 * p] + y.y * xkg[2 * p + 1];
    }
    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
    acc += __shfl_xor_sync(0xffffffffu, acc, 2);
    if (q4 == 0) sm.dbet[r] = acc;
  }
  if (!round_done()) { bail(); return; }
  {
    float aa[4][4];
    tc::ld_frag<4>(tb + 128, 32 * hk, aa);
    const float* A2 = reinterpret_cast<const float*>(wk + 12288);
#pragma unroll
    for (int jb = 0; jb < 2; jb++) {
      const int J = 2 * hk + jb;
      float rs0 = 0.f, rs1 = 0.f;
      if (J <= I) {
        const int t = blk_of(I, J);
        float* g = w.gMA + (ch * NBLK + t) * 16 * PB;
        const float* ab = A2 + t * 16 * PB;
#pragma unroll
        for (int jt = 0; jt < 2; jt++)
#pragma unroll
          for (int hh = 0; hh < 2; hh++) {
            const int m = gq + 8 * hh, n = 8 * jt + 2 * tq;
            const int rr = 16 * I + m, s0 = 16 * J + n;
            const float* v = aa[2 * jb + jt];
            const float da0 = s0 < rr ? -v[2 * hh] : 0.f, da1 = s0 + 1 < rr ? -v[2 * hh + 1] : 0.f;
            const float2 a2 = *reinterpret_cast<const float2*>(ab + m * PB + n);
            const float pa = da0 * a2.x + da1 * a2.y;
            if (hh == 0) rs0 += pa; else rs1 += pa;
            *reinterpret_cast<float2*>(g + m * PB + n) = make_float2(sm.bet[rr] * da0, sm.bet[rr] * da1);
          }
      }
      rs0 += __shfl_xor_sync(0xffffffffu, rs0, 1);
      rs0 += __shfl_xor_sync(0xffffffffu, rs0, 2);
      rs1 += __shfl_xor_sync(0xffffffffu, rs1, 1);
      rs1 += __shfl_xor_sync(0xffffffffu, rs1, 2);
      if (J <= I && tq == 0) {
        sm.part[J * C + 16 * I + gq] = rs0;
        sm.part[J * C + 16 * I + gq + 8] = rs1;
      }
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tb, TCOLS);
  if (tid < L) {  // fixed-order sum over the column blocks: deterministic
    float acc = sm.dbet[tid];
    for (int J = 0; J <= (tid >> 4); J++) acc += sm.part[J * C + tid];
    ((bf16*)io.db)[(size_t)(t0 + tid) * H + h] = __float2bfloat16_rn(acc * sm.bet[tid] * sigmoid_fast(-sm.braw[tid]));
  }
}

// bwd_gate: one CTA per chunk-head.  The pairwise decay-ratio terms of dq^,
// dk^ and dG from dP' and MA (split tf32: their row and column sums enter dG
// with opposite signs and must cancel in the cumulative sum), the remaining
// dq^ / dk^ / dG terms, the reverse cumulative sum over the chunk into dg,
// the gate backward (df and the per-chunk partials of dA_log and dt_bias)
// and the L2-norm backward (dq, dk).
// CONV: q and k are the convolution's fp32 outputs (recomputed from x as the
// forward computed them), kept in fp32 so that the backward sees their bits.
template <bool CONV>
struct GateSm {
  typedef typename std::conditional<CONV, float, bf16>::type QK;
  float gg[C * SQ];           // G2 = G log2(e); then dq^
  float dp[NBLK * 16 * PB];   // dP' lower blocks; then dk^
  float ma[NBLK * 16 * PB];   // MA lower blocks; then dG - kdt and its suffix sums
  QK rq[C * DK], rk[C * DK];
  bf16 rf[C * DK];
  float inq[C], ink[C];
  float gam[DK], dgam[DK];
  float tot[NW * DK], ks[4 * DK], part[NW * DK], red[NW];
  // operand tiles of the pairwise terms, [C][DK] with columns swizzled by tix:
  // kl = k^ 2^(G_last(I) - G), qf / kf = q^ / k^ 2^(G - G_first(I)) over the
  // row's 16-row block I (each at most |q^|, |k^|)
  float kl[C * DK], qf[C * DK], kf[C * DK];
  // the pairwise terms' block-boundary factors, per key channel: 2^(G_last(J) - G_last(J - 1)) for
  // J = 1..3, then 2^(G_first(I2 + 1) - G_first(I2)) for I2 = 0..2
  float bfac[6][DK];
  int spanok[4];
  uint64_t bar;   // bulk-load completion of dP' and MA
  uint64_t tbar;  // (not CONV) the raw q, k, f tiles' tensor-map copies
};
// Element (r, c) of a swizzled [C][DK] tile: the four rows r = 0..3 (mod 4) of
// a fragment load put their eight columns in different bank groups.
__device__ __forceinline__ int tix(int r, int c) { return r * DK + (c ^ ((r & 3) << 3)); }

static_assert(offsetof(GateSm<false>, rq) % 16 == 0 && offsetof(GateSm<false>, rk) % 16 == 0 &&
                  offsetof(GateSm<false>, rf) % 16 == 0 && offsetof(GateSm<false>, dp) % 16 == 0 &&
                  offsetof(GateSm<false>, ma) % 16 == 0 && offsetof(GateSm<false>, kl) % 16 == 0 &&
                  offsetof(GateSm<false>, qf) % 16 == 0 && offsetof(GateSm<false>, kf) % 16 == 0 &&
                  offsetof(GateSm<true>, rk) % 16 == 0 && offsetof(GateSm<true>, rf) % 16 == 0 &&
                  offsetof(GateSm<true>, kl) % 16 == 0 && offsetof(GateSm<true>, qf) % 16 == 0 &&
                  offsetof(GateSm<true>, kf) % 16 == 0,
              "vector-accessed arrays");
__device__ __forceinline__ float fl(float x) { return x; }
__device__ __forceinline__ float fl(bf16 x) { return bfl(x); }
__device__ __forceinline__ void load8(const bf16* p, float* v) { unpack8(*reinterpret_cast<const uint4*>(p), v); }
__device__ __forceinline__ void load8(const float* p, float* v) {
  const float4 a = *reinterpret_cast<const float4*>(p), b = *reinterpret_cast<const float4*>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

template <bool CONV>
__global__ void __launch_bounds__(NTH, CONV ? 2 : 3) bwd_gate_kernel(Dims d, BwdIO io, Ws w,
                                                                    const __grid_constant__ TMaps tmap) {
  extern __shared__ __align__(128) unsigned char smraw[];
  GateSm<CONV>& sm = *reinterpret_cast<GateSm<CONV>*>(smraw);
  const int j = (int)(blockIdx.x / (unsigned)d.H), h = (int)(blockIdx.x % (unsigned)d.H), tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, tq = lane & 3;
  const bool gdn = d.gate != 0;
  const float* dtb = io.dt_bias + h * (gdn ? 1 : DK);
  float dtv[8];  // dt_bias of key channels 8 (tid % 4) .. (the prologue's rows)
#pragma unroll
  for (int e = 0; e < 8; e++) dtv[e] = dtb[gdn ? 0 : 8 * (tid & 3) + e];
  const float dtl = dtb[gdn ? 0 : lane];  // and of channel `lane` (the gate step)
  const float alog = io.A_log[h];
  pdl_release();  // bwd_reduce may launch (it waits for this grid)
  const int tag = *w.tag, err = *w.err, L = w.chunk_len[j], t0 = w.chunk_tok0[j];  // one round trip
  if (tag != d.tag) {
    *w.err = -5;
    return;
  }
  if (err != 0 || L <= 0) return;
  const int H = d.H;
  const int64_t ch = (int64_t)j * H + h;
  const float a = expf(alog);
  const bf16* fsc = (const bf16*)io.f + h;  // scalar gate: f of this head, stride H

  // ---- group 1: raw q, k, f (rows past the chunk end zeroed);  group 2: dP', MA
  //      (CONV: q and k from the convolution, each thread its own row r = tid / 4, channels 8 (tid % 4) ..)
  for (int idx = tid; idx < C * 4; idx += NTH) {
    const int r = idx >> 2, p = idx & 3, o = r * DK + 8 * p;
    if (r < L) {
      const size_t g = ((size_t)(t0 + r) * H + h) * DK + 8 * p;
      if constexpr (CONV) {
        const int tmin = conv_tmin(w, j, t0);
        float cq[8], ck[8];
        conv_load<8>(cq, (const bf16*)io.q + h * DK + 8 * p, io.ld, t0 + r, tmin, io.cwq + 4 * (h * DK + 8 * p));
        conv_load<8>(ck, (const bf16*)io.k + h * DK + 8 * p, io.ld, t0 + r, tmin, io.cwk + 4 * (h * DK + 8 * p));
        float4* q4p = reinterpret_cast<float4*>(reinterpret_cast<float*>(sm.rq) + o);
        float4* k4p = reinterpret_cast<float4*>(reinterpret_cast<float*>(sm.rk) + o);
        q4p[0] = make_float4(cq[0], cq[1], cq[2], cq[3]);
        q4p[1] = make_float4(cq[4], cq[5], cq[6], cq[7]);
        k4p[0] = make_float4(ck[0], ck[1], ck[2], ck[3]);
        k4p[1] = make_float4(ck[4], ck[5], ck[6], ck[7]);
        if (!gdn) cp16(sm.rf + o, (const bf16*)io.f + g);
      }  // (not CONV: tensor-map copies below)
    } else if (CONV) {
      const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int u = 0; u < (CONV ? 2 : 1); u++) {
        reinterpret_cast<uint4*>(sm.rq + o)[u] = z;
        reinterpret_cast<uint4*>(sm.rk + o)[u] = z;
      }
      *reinterpret_cast<uint4*>(sm.rf + o) = z;
    }
  }
  cp_commit();
  if (!CONV && tid == 0) {  // the raw q, k (and f) tiles [C][DK], rows past the chunk end zeroed below
    mbar_init(&sm.tbar, 1);
    mbar_init_fence();
    mbar_expect_tx(&sm.tbar, (uint32_t)(2 * (gdn ? 2 : 3) * C * DK));
    tma_load_2d(sm.rq, &tmap.q, h * DK, t0, &sm.tbar);
    tma_load_2d(sm.rk, &tmap.k, h * DK, t0, &sm.tbar);
    if (!gdn) tma_load_2d(sm.rf, &tmap.f, h * DK, t0, &sm.tbar);
  }
  pdl_wait();  // every read below of bwd_grad's hand-over (the kernel before) follows this
  if (tid == 0) {
    mbar_init(&sm.bar, 1);
    mbar_init_fence();
    mbar_expect_tx(&sm.bar, 2 * NBLK * 16 * PB * 4);
    bulk_g2s(sm.dp, w.gDP + ch * NBLK * 16 * PB, NBLK * 16 * PB * 4, &sm.bar);
    bulk_g2s(sm.ma, w.gMA + ch * NBLK * 16 * PB, NBLK * 16 * PB * 4, &sm.bar);
  }
  if (tid < DK) sm.dgam[tid] = w.gdg[ch * DK + tid];
  if (tid < 4) sm.spanok[tid] = 1;
  cp_wait_all();
  __syncthreads();
  if constexpr (!CONV) {
    if (__syncthreads_or(!mbar_wait(&sm.tbar, 0))) {  // a copy did not land in bound
      mbar_wait(&sm.tbar, 0);
      mbar_wait(&sm.bar, 0);
      if (tid == 0) atomicExch(w.err, -7);
      return;
    }
    const int r = tid >> 2, o = r * DK + 8 * (tid & 3);  // rows past the chunk end: another document's, or zero
    if (r >= L) {
      const uint4 z = make_uint4(0u, 0u, 0u, 0u);
      *reinterpret_cast<uint4*>(sm.rq + o) = z;
      *reinterpret_cast<uint4*>(sm.rk + o) = z;
      *reinterpret_cast<uint4*>(sm.rf + o) = z;
    }
    __syncthreads();
  }

  // ---- q^, k^ norms and G (thread: row tid / 4, key channels 8 (tid % 4) ..)
  {
    const int r = tid >> 2, q4 = tid & 3;
    float qv[8], kv[8], gv[8];
    load8(sm.rq + r * DK + 8 * q4, qv);
    load8(sm.rk + r * DK + 8 * q4, kv);
    unpack8(*reinterpret_cast<const uint4*>(sm.rf + r * DK + 8 * q4), gv);
    const bool in = r < L;
    float sq = 0.f, sk = 0.f;
    const float gs = in && gdn ? -a * LOG2E * softplus_fast(bfl(fsc[(size_t)(t0 + r) * H]) + dtv[0]) : 0.f;
#pragma unroll
    for (int e = 0; e < 8; e++) {
      gv[e] = !in ? 0.f : gdn ? gs : -a * LOG2E * softplus_fast(gv[e] + dtv[e]);
      sq += qv[e] * qv[e];
      sk += kv[e] * kv[e];
    }
    sq += __shfl_xor_sync(0xffffffffu, sq, 1);
    sq += __shfl_xor_sync(0xffffffffu, sq, 2);
    sk += __shfl_xor_sync(0xffffffffu, sk, 1);
    sk += __shfl_xor_sync(0xffffffffu, sk, 2);
    if (q4 == 0) {
      sm.inq[r] = 1.0f / sqrtf(sq + L2_EPS);
      sm.ink[r] = 1.0f / sqrtf(sk + L2_EPS);
    }
#pragma unroll
    for (int e = 0; e < 8; e++) {
      float x = gv[e];
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        const float y2 = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y2;
      }
      gv[e] = x;
    }
    if (lane >= 28)
#pragma unroll
      for (int e = 0; e < 8; e++) sm.tot[warp * DK + 8 * q4 + e] = gv[e];
    __syncthreads();
    bool wide = false;
    add_warp_prefix(gv, sm.tot, warp, lane, q4);
    store_row8(sm.gg, r, q4, gv);
    __syncthreads();
    if (tid < 6 * DK) {  // once per CTA instead of in every warp's block loop
      const int f = tid / DK, i = tid % DK;
      const float* ga = sm.gg + (f < 3 ? 16 * f + 31 : 16 * (f - 3) + 16) * SQ;
      const float* gb = sm.gg + (f < 3 ? 16 * f + 15 : 16 * (f - 3)) * SQ;
      sm.bfac[f][i] = ex2(ga[i] - gb[i]);
    }
    const int I0 = r >> 4;
#pragma unroll
    for (int e = 0; e < 8; e++) {
      const int i = 8 * q4 + e;
      wide |= (r & 15) == 15 && sm.gg[(16 * I0) * SQ + i] - gv[e] > SPAN2;
      if (r == 0) sm.gam[i] = ex2(sm.gg[(L - 1) * SQ + i]);
    }
    if (wide) sm.spanok[I0] = 0;
    {  // the pairwise operand tiles of this row
      const float iq = sm.inq[r], ik = sm.ink[r];
      const float* gbr = sm.gg + (16 * I0) * SQ + 8 * q4;
      const float* ger = sm.gg + (16 * I0 + 15) * SQ + 8 * q4;
      float kl[8], qf[8], kf[8];
#pragma unroll
      for (int e = 0; e < 8; e++) {
        const float eF = ex2(gv[e] - gbr[e]), eL = ex2(ger[e] - gv[e]);
        kl[e] = kv[e] * ik * eL;
        qf[e] = qv[e] * iq * eF;
        kf[e] = kv[e] * ik * eF;
      }
      const int c0 = tix(r, 8 * q4);  // eight consecutive columns
      *reinterpret_cast<float4*>(sm.kl + c0) = make_float4(kl[0], kl[1], kl[2], kl[3]);
      *reinterpret_cast<float4*>(sm.kl + c0 + 4) = make_float4(kl[4], kl[5], kl[6], kl[7]);
      *reinterpret_cast<float4*>(sm.qf + c0) = make_float4(qf[0], qf[1], qf[2], qf[3]);
      *reinterpret_cast<float4*>(sm.qf + c0 + 4) = make_float4(qf[4], qf[5], qf[6], qf[7]);
      *reinterpret_cast<float4*>(sm.kf + c0) = make_float4(kf[0], kf[1], kf[2], kf[3]);
      *reinterpret_cast<float4*>(sm.kf + c0 + 4) = make_float4(kf[4], kf[5], kf[6], kf[7]);
    }
  }
  if (__syncthreads_or(!mbar_wait(&sm.bar, 0))) {  // a bulk load did not complete in bound
    mbar_wait(&sm.bar, 0);
    if (tid == 0) atomicExch(w.err, -7);
    return;
  }

  const int I = warp & 3, hk = warp >> 2;  // owner tile: rows 16 I .., key columns 16 hk ..
  const bool ok = sm.spanok[I];
  const float* gbI = sm.gg + (16 * I) * SQ;       // G at the block's first row
  const float* geI = sm.gg + (16 * I + 15) * SQ;  // and at its last
  // ---- pairwise terms: prow / arow (columns s of blocks J <= I), col (rows r of blocks I2 >= I)
  float prow[2][4], arow[2][4], col[2][4];
  zero(prow);
  zero(arow);
  zero(col);
  //      over the block pairs, with per-channel factors in Horner form (every ratio <= 1):
  //      prow = sum_J 2^(G_first(I) - G_last(J)) dP'_IJ kl_J (J ascending), col = sum_I2
  //      2^(G_first(I2) - G_last(I)) (dP'^T qf + MA^T kf)_I2 (I2 descending); the diagonal
  //      factor 2^span(I) only when the block is in range
  auto scale = [&](float (&x)[2][4], const float* ga, const float* gb) {  // x *= 2^(ga - gb) per column
#pragma unroll
    for (int jj = 0; jj < 2; jj++)
#pragma unroll
      for (int c1 = 0; c1 < 2; c1++) {
        const int i = 16 * hk + 8 * jj + 2 * tq + c1;
        const float f = ex2(ga[i] - gb[i]);
        x[jj][c1] *= f;
        x[jj][2 + c1] *= f;
      }
  };
  auto scalef = [&](float (&x)[2][4], const float* fac) {  // x *= fac per column
#pragma unroll
    for (int jj = 0; jj < 2; jj++)
#pragma unroll
      for (int c1 = 0; c1 < 2; c1++) {
        const float f = fac[16 * hk + 8 * jj + 2 * tq + c1];
        x[jj][c1] *= f;
        x[jj][2 + c1] *= f;
      }
  };
  const int Jl = ok ? I : I - 1;  // the last block J of prow / arow
  for (int J = 0; J <= Jl; J++) {
    const float* DPb = sm.dp + blk_of(I, J) * 16 * PB;
    const float* MAb = sm.ma + blk_of(I, J) * 16 * PB;
    if (J > 0) {  // 2^(G_last(J) - G_last(J - 1))
      scalef(prow, sm.bfac[J - 1]);
      scalef(arow, sm.bfac[J - 1]);
    }
    rows16_2a<2>(prow, arow, 2, [&](int m, int k) { return DPb[m * PB + k]; },
                 [&](int m, int k) { return MAb[m * PB + k]; },
                 [&](int k, int jj, int n) { return sm.kl[tix(16 * J + k, 16 * hk + 8 * jj + n)]; });
  }
  if (Jl >= 0) {
    scale(prow, gbI, sm.gg + (16 * Jl + 15) * SQ);
    scale(arow, gbI, sm.gg + (16 * Jl + 15) * SQ);
  }
  const int Il = ok ? I : I + 1;  // the last block I2 of col
  for (int I2 = 3; I2 >= Il; I2--) {
    const float* DPb = sm.dp + blk_of(I2, I) * 16 * PB;
    const float* MAb = sm.ma + blk_of(I2, I) * 16 * PB;
    if (I2 < 3) scalef(col, sm.bfac[3 + I2]);  // 2^(G_first(I2 + 1) - G_first(I2))
    rows16_ab<2>(col, 2, [&](int m, int k) { return DPb[k * PB + m]; },
                 [&](int m, int k) { return MAb[k * PB + m]; },
                 [&](int k, int jj, int n) {
                   const int t = tix(16 * I2 + k, 16 * hk + 8 * jj + n);
                   return make_float2(sm.qf[t], sm.kf[t]);
                 });
  }
  if (Il <= 3) scale(col, sm.gg + (16 * Il) * SQ, geI);
  // ---- assemble dq^, dk^, dG - kdt per owned element; column totals of kdt
  float dQG[2][4], dKD[2][4], dkg[2][4];  // bwd_grad's hand-over (L2-resident: prefetched a wave ahead)
  frag_load(w.gQG + ch * NTH * 8, dQG);
  frag_load(w.gKD + ch * NTH * 8, dKD);
  frag_load(w.gKG + ch * NTH * 8, dkg);
  float dqh[2][4], dkh[2][4], dGk[2][4], kcol[2][2];
  {
    const float* DPd = sm.dp + blk_of(I, I) * 16 * PB;
    const float* MAd = sm.ma + blk_of(I, I) * 16 * PB;
#pragma unroll
    for (int jj = 0; jj < 2; jj++) {
      kcol[jj][0] = kcol[jj][1] = 0.f;
#pragma unroll
      for (int e = 0; e < 4; e++) {
        const int m = gq + 8 * (e >> 1), rr = 16 * I + m, i = 16 * hk + 8 * jj + 2 * tq + (e & 1);
        const float G = sm.gg[rr * SQ + i];
        const float eL = ex2(G - gbI[i]), eR = ex2(geI[i] - G);
        float pr = prow[jj][e] * eL, ar = arow[jj][e] * eL, cl = col[jj][e] * eR;
        if (!ok) {  // exact diagonal-block terms (rows past the chunk end are zero)
          for (int s = 16 * I; s < 16 * I + 16 && s < L; s++) {
            const int n = s - 16 * I;
            const float ks = fl(sm.rk[s * DK + i]) * sm.ink[s], qs = fl(sm.rq[s * DK + i]) * sm.inq[s];
            if (s <= rr) {
              const float ex = ex2(G - sm.gg[s * SQ + i]);
              pr += DPd[m * PB + n] * ks * ex;
              ar += MAd[m * PB + n] * ks * ex;
            }
            if (s >= rr) {
              const float ex = ex2(sm.gg[s * SQ + i] - G);
              cl += (DPd[n * PB + m] * qs + MAd[n * PB + m] * ks) * ex;
            }
          }
        }
        const float q = fl(sm.rq[rr * DK + i]) * sm.inq[rr], k = fl(sm.rk[rr * DK + i]) * sm.ink[rr];
        const float Gm = ex2(G), kdf = ex2(sm.gg[(L - 1) * SQ + i] - G);
        const float kdt = dKD[jj][e] * k * kdf;
        dqh[jj][e] = pr + dQG[jj][e] * Gm;
        dkh[jj][e] = ar + cl + dkg[jj][e] * Gm + dKD[jj][e] * kdf;
        dGk[jj][e] = q * pr + k * ar - k * cl + dQG[jj][e] * q * Gm + dkg[jj][e] * k * Gm - kdt;
        kcol[jj][e & 1] += kdt;
      }
    }
  }
#pragma unroll
  for (int jj = 0; jj < 2; jj++)
#pragma unroll
    for (int c2 = 0; c2 < 2; c2++) {
      float x = kcol[jj][c2];
      x += __shfl_xor_sync(0xffffffffu, x, 4);
      x += __shfl_xor_sync(0xffffffffu, x, 8);
      x += __shfl_xor_sync(0xffffffffu, x, 16);
      kcol[jj][c2] = x;
    }
  __syncthreads();  // every read of G, dP' and MA is done
  float* dqs = sm.gg;
  float* dks = sm.dp;
  float* dgs = sm.ma;
#pragma unroll
  for (int jj = 0; jj < 2; jj++) {
#pragma unroll
    for (int e = 0; e < 4; e++) {
      const int rr = 16 * I + gq + 8 * (e >> 1), i = 16 * hk + 8 * jj + 2 * tq + (e & 1);
      dqs[rr * SQ + i] = dqh[jj][e];
      dks[rr * SQ + i] = dkh[jj][e];
      dgs[rr * SQ + i] = dGk[jj][e];
    }
    if (gq == 0) {
      sm.ks[I * DK + 16 * hk + 8 * jj + 2 * tq] = kcol[jj][0];
      sm.ks[I * DK + 16 * hk + 8 * jj + 2 * tq + 1] = kcol[jj][1];
    }
  }
  __syncthreads();
  // ---- reverse cumulative sum over the chunk:
  //      dg_t = sum_{r >= t} (dG_r - kdt_r) + sum_r kdt_r + dgamma gamma
  {
    float run = 0.f;
#pragma unroll
    for (int m = 7; m >= 0; m--) {
      const int rr = 8 * warp + m;
      run += dgs[rr * SQ + lane];
      dgs[rr * SQ + lane] = run;
    }
    sm.tot[warp * DK + lane] = run;
  }
  __syncthreads();
  {
    float off = sm.dgam[lane] * sm.gam[lane];
    for (int i4 = 0; i4 < 4; i4++) off += sm.ks[i4 * DK + lane];
#pragma unroll
    for (int w2 = 1; w2 < NW; w2++)
      if (w2 > warp) off += sm.tot[w2 * DK + lane];
    bf16* dfo = (bf16*)io.df;
    float pdt = 0.f, pA = 0.f;
#pragma unroll
    for (int m = 0; m < 8; m++) {
      const int rr = 8 * warp + m;
      if (rr < L) {  // uniform over the warp
        const float dg = dgs[rr * SQ + lane] + off;
        const float x = (gdn ? bfl(fsc[(size_t)(t0 + rr) * H]) : bfl(sm.rf[rr * DK + lane])) + dtl;
        const float g = -a * softplus_fast(x);
        const float dx = dg * (-a) * sigmoid_fast(x);
        if (gdn) {  // the scalar gate feeds every channel: its gradient is the channel sum
          const float ds = warp_sum(dx);
          if (lane == 0) dfo[(size_t)(t0 + rr) * H + h] = __float2bfloat16_rn(ds);
        } else {
          dgs[rr * SQ + lane] = dx;  // over the value just read: this warp's rows, stored below
        }
        pdt += dx;
        pA += dg * g;
      }
    }
    if (!gdn) {  // df of the warp's 8 rows: lane = row lane / 4, channels 8 (lane % 4) .., one 16-byte store
      __syncwarp();
      const int m = lane >> 2, rr = 8 * warp + m, c0 = 8 * (lane & 3);
      if (rr < L) {
        const float4 x0 = *reinterpret_cast<const float4*>(dgs + rr * SQ + c0);
        const float4 x1 = *reinterpret_cast<const float4*>(dgs + rr * SQ + c0 + 4);
        uint4 u;
        __nv_bfloat162* u2 = reinterpret_cast<__nv_bfloat162*>(&u);
        u2[0] = __floats2bfloat162_rn(x0.x, x0.y);
        u2[1] = __floats2bfloat162_rn(x0.z, x0.w);
        u2[2] = __floats2bfloat162_rn(x1.x, x1.y);
        u2[3] = __floats2bfloat162_rn(x1.z, x1.w);
        *reinterpret_cast<uint4*>(dfo + ((size_t)(t0 + rr) * H + h) * DK + c0) = u;
      }
    }
    sm.part[warp * DK + lane] = pdt;
    pA = warp_sum(pA);
    if (lane == 0) sm.red[warp] = pA;
  }
  __syncthreads();
  if (tid < DK) {
    float s = 0.f;
    for (int w2 = 0; w2 < NW; w2++) s += sm.part[w2 * DK + tid];
    w.pdt[ch * DK + tid] = s;
  }
  if (tid == 0) {
    float s = 0.f;
    for (int w2 = 0; w2 < NW; w2++) s += sm.red[w2];
    w.pA[ch] = s;
  }
  // ---- L2-norm backward (thread: row tid / 4, key channels 8 (tid % 4) ..)
  {
    const int r = tid >> 2, q4 = tid & 3;
    float qv[8], kv[8], dqv[8], dkv[8], pq = 0.f, pk = 0.f;
    load8(sm.rq + r * DK + 8 * q4, qv);
    load8(sm.rk + r * DK + 8 * q4, kv);
    const float iq = sm.inq[r], ik = sm.ink[r];
#pragma unroll
    for (int e = 0; e < 8; e++) {
      qv[e] *= iq;
      kv[e] *= ik;
      dqv[e] = dqs[r * SQ + 8 * q4 + e];
      dkv[e] = dks[r * SQ + 8 * q4 + e];
      pq += qv[e] * dqv[e];
      pk += kv[e] * dkv[e];
    }
    pq += __shfl_xor_sync(0xffffffffu, pq, 1);
    pq += __shfl_xor_sync(0xffffffffu, pq, 2);
    pk += __shfl_xor_sync(0xffffffffu, pk, 1);
    pk += __shfl_xor_sync(0xffffffffu, pk, 2);
    if (r < L) {
      if constexpr (CONV) {  // fp32 gradients of the convolution's q and k outputs
        float oq[8], ok[8];
#pragma unroll
        for (int e = 0; e < 8; e++) {
          oq[e] = (dqv[e] - qv[e] * pq) * iq;
          ok[e] = (dkv[e] - kv[e] * pk) * ik;
        }
        const size_t off = (size_t)(t0 + r) * io.ld + h * DK + 8 * q4;
        float4* pq4 = reinterpret_cast<float4*>((float*)io.dq + off);
        float4* pk4 = reinterpret_cast<float4*>((float*)io.dk + off);
        pq4[0] = make_float4(oq[0], oq[1], oq[2], oq[3]);
        pq4[1] = make_float4(oq[4], oq[5], oq[6], oq[7]);
        pk4[0] = make_float4(ok[0], ok[1], ok[2], ok[3]);
        pk4[1] = make_float4(ok[4], ok[5], ok[6], ok[7]);
      } else {
        uint4 uq, uk;
        __nv_bfloat162* pq2 = reinterpret_cast<__nv_bfloat162*>(&uq);
        __nv_bfloat162* pk2 = reinterpret_cast<__nv_bfloat162*>(&uk);
#pragma unroll
        for (int e = 0; e < 4; e++) {
          pq2[e] =
              __floats2bfloat162_rn((dqv[2 * e] - qv[2 * e] * pq) * iq, (dqv[2 * e + 1] - qv[2 * e + 1] * pq) * iq);
          pk2[e] =
              __floats2bfloat162_rn((dkv[2 * e] - kv[2 * e] * pk) * ik, (dkv[2 * e + 1] - kv[2 * e + 1] * pk) * ik);
        }
        const size_t off = ((size_t)(t0 + r) * H + h) * DK + 8 * q4;
        *reinterpret_cast<uint4*>((bf16*)io.dq + off) = uq;
        *reinterpret_cast<uint4*>((bf16*)io.dk + off) = uk;
      }
    }
  }
}

}  // namespace fast

static_assert(sizeof(fast::FwdSm) <= 232448, "fused forward shared memory exceeds 227 KB");
static_assert(sizeof(fast::ChunkSm) <= 113 * 1024, "per-chunk forward must fit two CTAs per SM");

static_assert(sizeof(fast::GradSm) <= 112 * 1024, "chunk-gradient kernel must fit two CTAs per SM");
static_assert(sizeof(fast::BChainSmN) <= 113 * 1024, "fused-norm reverse chain must fit two CTAs per SM");
static_assert(sizeof(fast::FChainSm<true>) <= 113 * 1024, "fused-norm forward chain must fit two CTAs per SM");
static_assert(sizeof(fast::FChainSm<false>) <= 113 * 1024 && sizeof(fast::BChainSm) <= 113 * 1024,
              "the chains must fit two CTAs per SM");
static_assert(sizeof(fast::GateSm<false>) <= 75 * 1024, "gate kernel must fit three CTAs per SM");
static_assert(sizeof(fast::GateSm<true>) <= 113 * 1024, "gate kernel (fused convolution) must fit two CTAs per SM");

bool fast_path(int dtype, int dk, int dv) { return dtype == 0 && dk == fast::DK && dv == fast::DV; }

static PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 enc = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &qr) !=
            cudaSuccess ||
        qr != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }();
  return enc;
}

// One 2-D map over [Ntok][H dh] elements (esz bytes each) with a box of bx columns x C tokens.
static bool encode_rows(CUtensorMap* m, const void* base, int Ntok, int H, int dh, int bx, bool fp32) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tmap_encoder();
  if (!enc) return false;
  const int esz = fp32 ? 4 : 2;
  const cuuint64_t dims[2] = {(cuuint64_t)H * dh, (cuuint64_t)Ntok};
  const cuuint64_t strides[1] = {(cuuint64_t)H * dh * esz};
  const cuuint32_t box[2] = {(cuuint32_t)bx, (cuuint32_t)C};
  const cuuint32_t es[2] = {1, 1};
  return enc(m, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base),
             dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_nmaps(NMaps* nm, const void* g, const void* dy, const float* o, int Ntok, int H, int dv) {
  *nm = NMaps{};
  return encode_rows(&nm->g, g, Ntok, H, dv, fast::NSC, false) && (!dy || encode_rows(&nm->dy, dy, Ntok, H, dv, fast::NSC, false)) &&
         (!o || encode_rows(&nm->o, o, Ntok, H, dv, fast::NSC, true));
}

bool encode_tmaps(TMaps* tm, const void* q, const void* k, const void* v, const void* f, int Ntok, int H, int dk,
                  int dv, bool channel_gate) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tmap_encoder();
  if (!enc) return false;
  auto one = [&](CUtensorMap* m, const void* base, int dh) {  // [Ntok][H dh] bf16, box dh x C
    const cuuint64_t dims[2] = {(cuuint64_t)H * dh, (cuuint64_t)Ntok};
    const cuuint64_t strides[1] = {(cuuint64_t)H * dh * 2};
    const cuuint32_t box[2] = {(cuuint32_t)dh, (cuuint32_t)C};
    const cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  };
  *tm = TMaps{};
  return one(&tm->q, q, dk) && one(&tm->k, k, dk) && one(&tm->v, v, dv) && (!channel_gate || one(&tm->f, f, dk));
}

// CTAs of the per-chunk kernels in flight on the current device (two per SM).
static int wave_ctas() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cached[dev] = 2 * n;
  }
  return cached[dev];
}

int fast_chain_slots() { return wave_ctas(); }  // fwd_state: two CTAs per SM, like the per-chunk kernels

cudaError_t launch_fast_fwd(const Dims& d0, const FwdIO& io, const Ws& w, cudaStream_t st, bool fused) {
  Dims d = d0;
  d.ahead = wave_ctas() / 2;  // fwd_chunk's L2 prefetch: the CTA half a wave later
  cudaError_t e;
  if (fused) {
    const size_t smem = sizeof(fast::FwdSm);
    e = cudaFuncSetAttribute(fast::fwd_chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    prof_begin(K_FWD_CHAIN, st);
    fast::fwd_chain_kernel<<<dim3(d.n_docs, d.H), fast::NTH, smem, st>>>(d, io, w);
    prof_end(K_FWD_CHAIN, st);
    return cudaGetLastError();
  }
  const size_t s1 = sizeof(fast::ChunkSm), s2 = sizeof(fast::FChainSm<false>), s2n = sizeof(fast::FChainSm<true>);
  e = cudaFuncSetAttribute(fast::fwd_chunk_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s1);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(fast::fwd_chunk_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s1);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(fast::fwd_state_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s2);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(fast::fwd_state_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s2n);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(fast::fwd_seg_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sizeof(fast::SegSm));
  if (e != cudaSuccess) return e;
  prof_begin(K_FWD_CHUNK, st);
  if (d.conv)
    e = launch_pdl(fast::fwd_chunk_kernel<true>, dim3(d.nc_max * d.H), dim3(fast::NTH), s1, st, d, io, w);
  else
    e = launch_pdl(fast::fwd_chunk_kernel<false>, dim3(d.nc_max * d.H), dim3(fast::NTH), s1, st, d, io, w);
  prof_end(K_FWD_CHUNK, st);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // one CTA per (document, head, column half); with split chains one per (segment unit, head,
  // half) on a 1-D grid (chain_cta)
  static_assert(fast::DV / fast::NSC == 2, "two column halves");
  const dim3 grid = d.seg ? dim3((unsigned)d.nu * d.H * 2) : dim3(d.n_docs, d.H, 2);
  NMaps nm = {};
  if (d.seg) {  // the segments' composites first
    prof_begin(K_FWD_SEG, st);
    e = launch_pdl(fast::fwd_seg_kernel, grid, dim3(fast::CTH), sizeof(fast::SegSm), st, d, io, w);
    prof_end(K_FWD_SEG, st);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (d.norm) {  // the two column halves of a (document, head, or segment) as one cluster
    if (!encode_nmaps(&nm, io.ng, nullptr, nullptr, d.Ntok, d.H, fast::DV)) return cudaErrorInvalidValue;
    prof_begin(K_FWD_STATE_NORM, st);
    e = launch_cluster(fast::fwd_state_kernel<true>, grid, dim3(2 * fast::CTH), s2n, st, 2, true, d, io, w, nm);
    prof_end(K_FWD_STATE_NORM, st);
  } else {
    prof_begin(K_FWD_STATE, st);
    e = launch_pdl(fast::fwd_state_kernel<false>, grid, dim3(2 * fast::CTH), s2, st, d, io, w, nm);
    prof_end(K_FWD_STATE, st);
  }
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_fast_bwd(const Dims& d0, const BwdIO& io, const Ws& w, cudaStream_t st) {
  Dims d = d0;
  d.ahead = 0;  // the backward's chunk kernels prefetch nothing (measured: the L2 prefetch of the next wave slowed them)
  const size_t sc = sizeof(fast::BChainSm), scn = sizeof(fast::BChainSmN), s1 = sizeof(fast::GradSm),
               s2 = d.conv ? sizeof(fast::GateSm<true>) : sizeof(fast::GateSm<false>);
  cudaError_t e = cudaFuncSetAttribute(fast::bwd_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sc);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(fast::bwd_scan_norm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)scn);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(fast::bwd_grad_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s1);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(fast::bwd_grad_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s1);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(fast::bwd_gate_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sizeof(fast::GateSm<false>));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(fast::bwd_gate_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sizeof(fast::GateSm<true>));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(fast::bwd_seg_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sizeof(fast::BSegSm));
  if (e != cudaSuccess) return e;
  const dim3 grid = d.seg && !d.norm ? dim3((unsigned)d.nu * d.H * 2) : dim3(d.n_docs, d.H, 2);  // (chain_cta)
  if (d.norm) {  // the two column halves of a (document, head) as one cluster
    NMaps nm;
    if (!encode_nmaps(&nm, io.ng, io.dy, w.nO, d.Ntok, d.H, fast::DV)) return cudaErrorInvalidValue;
    prof_begin(K_BWD_SCAN_NORM, st);
    e = launch_cluster(fast::bwd_scan_norm_kernel, grid, dim3(2 * fast::CTH), scn, st, 2, false, d, io, w, nm);
    prof_end(K_BWD_SCAN_NORM, st);
  } else {
    if (d.seg) {  // the later segments' composites first
      prof_begin(K_BWD_SEG, st);
      fast::bwd_seg_kernel<<<grid, fast::CTH, sizeof(fast::BSegSm), st>>>(d, io, w);
      prof_end(K_BWD_SEG, st);
      e = cudaGetLastError();
      if (e != cudaSuccess) return e;
    }
    prof_begin(K_BWD_SCAN, st);
    fast::bwd_scan_kernel<<<grid, fast::CTH, sc, st>>>(d, io, w);
    prof_end(K_BWD_SCAN, st);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) return e;
  prof_begin(K_BWD_GRAD, st);
  e = d.conv ? launch_pdl(fast::bwd_grad_kernel<true>, dim3(d.nc_max * d.H), dim3(fast::NTH), s1, st, d, io, w)
             : launch_pdl(fast::bwd_grad_kernel<false>, dim3(d.nc_max * d.H), dim3(fast::NTH), s1, st, d, io, w);
  prof_end(K_BWD_GRAD, st);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  prof_begin(K_BWD_GATE, st);
  TMaps tm = {};
  if (!d.conv && !encode_tmaps(&tm, io.q, io.k, io.v, io.f, d.Ntok, d.H, fast::DK, fast::DV, d.gate == 0))
    return cudaErrorInvalidValue;
  e = d.conv ? launch_pdl(fast::bwd_gate_kernel<true>, dim3(d.nc_max * d.H), dim3(fast::NTH), s2, st, d, io, w, tm)
             : launch_pdl(fast::bwd_gate_kernel<false>, dim3(d.nc_max * d.H), dim3(fast::NTH), s2, st, d, io, w, tm);
  prof_end(K_BWD_GATE, st);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_bwd_reduce(d, io, w, st);  // (with the fused norm also dw, in one more block)
}

}  // namespace kda
