// C ABI of the KDA library: argument validation, workspace layout, the
// varlen chunk table, launch order and per-kernel timing.
#include "../../include/kda.h"
#include "kda_internal.cuh"

#include <stdio.h>
#include <string.h>

#include <mutex>

namespace kda {

// ------------------------------------------------------------ chunk table
// One CTA builds the chunk table from the document offsets: document i of
// length L_i owns ceil(L_i / C) chunks, the last one partial.  Chunks always
// start at a document start, so a state never crosses a document boundary
// (torchtitan PR "[kimi k3] Support sample packing in KDA", Verification).
// Equal-length rows use the same table with offsets b * T.
constexpr int ORD_BUCKETS = 2048;  // document chunk counts the dispatch order sorts
// Inclusive scan of x over the block (a multiple of 32 threads, at most
// 1024), with the block's sum in *total; every thread calls it.
__device__ int block_incl_scan(int x, int* s_wsum, int* total) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = (int)(blockDim.x >> 5);
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_wsum[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int y = lane < nw ? s_wsum[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int z = __shfl_up_sync(0xffffffffu, y, o);
      if (lane >= o) y += z;
    }
    s_wsum[lane] = y;
  }
  __syncthreads();
  const int incl = x + (warp > 0 ? s_wsum[warp - 1] : 0);
  *total = s_wsum[nw - 1];
  __syncthreads();  // s_wsum is free again
  return incl;
}

// order[0 .. n) <- 0 .. n - 1 by decreasing key(i) >= 0, keys at or past
// ORD_BUCKETS sharing the top bucket; equal keys in any order (a chain's result
// does not depend on when it runs).  A counting sort in shared memory: every
// thread of the 1024-thread block calls it.
template <class K>
__device__ void order_desc(int n, K key, int32_t* order, int* s_cnt, int* s_wsum) {
  const int tid = threadIdx.x;
  for (int b = tid; b < ORD_BUCKETS; b += blockDim.x) s_cnt[b] = 0;
  __syncthreads();
  for (int i = tid; i < n; i += blockDim.x) atomicAdd(&s_cnt[min(key(i), ORD_BUCKETS - 1)], 1);
  __syncthreads();
  {  // s_cnt[b] <- items of larger keys: thread t owns buckets 2 (N - 1 - t) + {1, 0}
    static_assert(ORD_BUCKETS == 2048, "two buckets per thread of a 1024-thread block");
    const int b0 = ORD_BUCKETS - 2 * (tid + 1);
    const int c1 = s_cnt[b0 + 1], c0 = s_cnt[b0];
    int total;
    const int ex = block_incl_scan(c1 + c0, s_wsum, &total) - (c1 + c0);
    s_cnt[b0 + 1] = ex;
    s_cnt[b0] = ex + c1;
  }
  __syncthreads();
  for (int i = tid; i < n; i += blockDim.x) order[atomicAdd(&s_cnt[min(key(i), ORD_BUCKETS - 1)], 1)] = i;
}

__global__ void __launch_bounds__(1024) chunk_table_kernel(const int32_t* cu, Dims d, Ws w) {
  __shared__ int s_bad;
  __shared__ int s_cnt[ORD_BUCKETS];
  __shared__ int s_carry;
  __shared__ int s_wsum[32];
  // With equal rows the tensor-core fwd_chunk reads no table and runs alongside this kernel (it
  // waits for this grid only before it ends): the error word is reset before it may launch.
  if (d.rows && threadIdx.x == 0) *w.err = KDA_OK;
  pdl_release();  // fwd_chunk may launch; it waits for this table before reading it
  const int tid = threadIdx.x, n = d.n_docs;
  auto off = [&](int i) -> int { return cu ? cu[i] : i * d.T; };
  if (tid == 0) {
    s_bad = (off(0) != 0 || off(n) != d.Ntok) ? 1 : 0;
    s_carry = 0;
  }
  __syncthreads();
  for (int i = tid; i < n; i += blockDim.x)
    if (off(i + 1) < off(i)) atomicOr(&s_bad, 1);
  __syncthreads();
  if (!s_bad) {
    for (int base = 0; base < n; base += blockDim.x) {
      const int i = base + tid;
      const int nc = i < n ? (off(i + 1) - off(i) + C - 1) / C : 0;
      int total;
      const int incl = block_incl_scan(nc, s_wsum, &total);
      if (i < n) w.doc_chunk0[i] = s_carry + incl - nc;
      __syncthreads();
      if (tid == 0) s_carry += total;
      __syncthreads();
    }
    if (tid == 0 && s_carry > d.nc_max) s_bad = 1;  // cannot happen for valid offsets
    __syncthreads();
  }
  if (s_bad) {
    if (tid == 0) { *w.err = KDA_ERR_BAD_SEQLENS; *w.n_chunks = 0; *w.tag = 0; }
    for (int j = tid; j < d.nc_max; j += blockDim.x) w.chunk_len[j] = 0;
    return;
  }
  if (tid == 0) {
    w.doc_chunk0[n] = s_carry;
    *w.n_chunks = s_carry;
    if (!d.rows) *w.err = KDA_OK;  // (equal rows: reset above)
    *w.tag = d.save ? d.tag : 0;
  }
  for (int i = tid; i < n; i += blockDim.x) {
    int a = off(i), L = off(i + 1) - a, c0 = w.doc_chunk0[i];
    for (int c = 0; c * C < L; c++) {
      w.chunk_tok0[c0 + c] = a + c * C;
      w.chunk_len[c0 + c] = min(C, L - c * C);
      w.chunk_doc[c0 + c] = i;
    }
  }
  for (int j = s_carry + tid; j < d.nc_max; j += blockDim.x) w.chunk_len[j] = 0;
  if (d.seg) {  // the segment table of the tensor-core forward chains (seg_split, seg_count)
    __shared__ int s_nmax, s_ucarry;
    if (tid == 0) { s_nmax = 0; s_ucarry = 0; }
    __syncthreads();  // doc_chunk0 (written above by other threads) is visible
    int mx = 0;
    for (int i = tid; i < n; i += blockDim.x) mx = max(mx, w.doc_chunk0[i + 1] - w.doc_chunk0[i]);
    atomicMax(&s_nmax, mx);
    __syncthreads();
    const bool split = seg_split(s_nmax, s_carry, d.H, d.slots);
    const int len = seg_len(s_nmax);
    for (int base = 0; base < n; base += blockDim.x) {
      const int i = base + tid;
      const int nc = i < n ? w.doc_chunk0[i + 1] - w.doc_chunk0[i] : 0;
      const int ns = i < n ? seg_count(nc, split, len) : 0;
      int total;
      const int u0 = s_ucarry + block_incl_scan(ns, s_wsum, &total) - ns;
      for (int sg = 0; sg < ns; sg++) {
        const int c0 = sg * len;
        if (u0 + sg < d.nu) w.useg[u0 + sg] = make_int4(i, c0, ns > 1 ? min(len, nc - c0) : nc, sg);
      }
      __syncthreads();
      if (tid == 0) s_ucarry += total;
      __syncthreads();
    }
    if (tid == 0) {  // d.nu bounds the count (the host's own count or seg_units_max); past it, refuse
      *w.n_units = min(s_ucarry, d.nu);
      if (s_ucarry > d.nu) *w.err = KDA_ERR_INVALID_ARG;
    }
    __syncthreads();  // the table (written by every thread) and the count are visible
    // the chain grids take the heaviest units first: a later segment folds one composite per
    // earlier segment before its chunks
    order_desc(min(s_ucarry, d.nu), [&](int u) { const int4 un = w.useg[u]; return un.z + un.w; }, w.uorder,
               s_cnt, s_wsum);
  }
  // The documents by decreasing chunk count: the general scans run one CTA per
  // (document, head, column slice) in this order, longest first, so that a grid
  // of more chains than resident CTAs ends about when its longest chain does
  // instead of when a long chain dispatched last does.
  if (d.fast) return;  // (the tensor-core chains order their units above, when split)
  __syncthreads();  // doc_chunk0 (written above by other threads) is visible
  order_desc(n, [&](int i) { return w.doc_chunk0[i + 1] - w.doc_chunk0[i]; }, w.doc_order, s_cnt, s_wsum);
}

cudaError_t launch_chunk_table(const int32_t* cu, const Dims& d, const Ws& w, cudaStream_t st) {
  prof_begin(K_TABLE, st);
  chunk_table_kernel<<<1, 1024, 0, st>>>(cu, d, w);
  prof_end(K_TABLE, st);
  return cudaGetLastError();
}

// ------------------------------------------------------------ timing
namespace {
constexpr int MAX_EV = 8192;
struct Prof {
  bool on = false;
  int n = 0;
  cudaEvent_t ev[MAX_EV][2];
  int kid[MAX_EV];
  bool created = false;
};
Prof g_prof;
int g_open = -1;
}  // namespace

void prof_begin(int kid, cudaStream_t st) {
  if (!g_prof.on || g_prof.n >= MAX_EV) { g_open = -1; return; }
  g_open = g_prof.n++;
  g_prof.kid[g_open] = kid;
  cudaEventRecord(g_prof.ev[g_open][0], st);
}
void prof_end(int kid, cudaStream_t st) {
  (void)kid;
  if (g_open < 0) return;
  cudaEventRecord(g_prof.ev[g_open][1], st);
  g_open = -1;
}

// ------------------------------------------------------------ layout
static size_t align_up(size_t x) { return (x + 255) & ~(size_t)255; }

struct Layout {
  size_t total;
  size_t off_err, off_nch, off_dc0, off_ct0, off_cl, off_cd, off_ord;
  size_t off_W, off_U, off_P, off_QG, off_KD, off_gam, off_Sent, off_CH;
  size_t off_sT, off_sP, off_sW, off_sU, off_sA, off_gDP, off_gMA, off_gQG, off_gKD, off_gKG, off_gdg;
  size_t off_dE, off_dSn, off_pA, off_pdt, off_scr, off_nO, off_pdw, off_nrm, off_cg, off_cpart;
  size_t off_useg, off_uord, off_nu, off_segc;
};

// Upper bound on the segment units of a split forward chain: a document of n
// chunks has at most n / SEG + 1 segments (segments have at least SEG chunks).
static int64_t seg_units_max(const Dims& d) { return (int64_t)d.n_docs + (d.nc_max + SEG - 1) / SEG; }

// Workspace layout.  Both paths start with the error word, the saved-problem
// tag and the chunk table.  The tensor-core path (d.fast) keeps per chunk and
// head one block of M, QW (read again by the backward scan), KU and PU, and for the
// backward the entry states, the state gradients and the parameter-gradient
// partials; its fused forward (fused = true) needs the table alone.  The
// general path keeps its fp32 intra-chunk factors and scratch.
static Layout layout(const Dims& d, int for_bwd, bool fused = false) {
  Layout L = {};
  size_t o = 0;
  const size_t nch = (size_t)d.nc_max * d.H;
  auto take = [&](size_t bytes) { size_t r = o; o = align_up(o + bytes); return r; };
  L.off_err = take(8);  // error word, then the saved-problem tag
  L.off_nch = take(4);
  L.off_dc0 = take(4 * (size_t)(d.n_docs + 1));
  L.off_ct0 = take(4 * (size_t)d.nc_max);
  L.off_cl = take(4 * (size_t)d.nc_max);
  L.off_cd = take(4 * (size_t)d.nc_max);
  L.off_ord = take(4 * (size_t)d.n_docs);
  if (d.fast) {
    if (!fused) {
      L.off_CH = take(4 * nch * (d.dk * d.dk + C * d.dk + d.dk * d.dv + C * d.dv));  // M, QW, KU, PU
      const size_t nu = (size_t)seg_units_max(d);
      L.off_useg = take(16 * nu);  // the segment table of split forward chains
      L.off_uord = take(4 * nu);
      L.off_nu = take(4);
      L.off_segc = take(4 * nu * d.H * d.dk * (d.dk + d.dv));  // and the segments' composites
    }
    if (for_bwd) {
      L.off_Sent = take(4 * nch * d.dk * d.dv);  // entry states for the backward (split-bf16 tiles)
      L.off_dSn = take(4 * nch * d.dk * d.dv);
      L.off_pA = take(4 * nch);
      L.off_pdt = take(4 * nch * d.dk);
      L.off_sT = take(4 * nch * C * C);
      L.off_sP = take(4 * nch * C * C);
      L.off_sW = take(4 * nch * C * d.dk);
      L.off_sU = take(4 * nch * C * d.dv);
      L.off_sA = take(4 * nch * 10 * 16 * 20);  // A' blocks, rows padded to 20
      L.off_gDP = take(4 * nch * 10 * 16 * 20);
      L.off_gMA = take(4 * nch * 10 * 16 * 20);
      L.off_gQG = take(4 * nch * C * d.dk);
      L.off_gKD = take(4 * nch * C * d.dk);
      L.off_gKG = take(4 * nch * C * d.dk);
      L.off_gdg = take(4 * nch * d.dk);
    }
    if (for_bwd >= 2) {  // kda_fwd_norm_gate / kda_fwd_conv saving for their backward
      L.off_nO = take(4 * (size_t)d.Ntok * d.H * d.dv);
      L.off_pdw = take(4 * (size_t)d.n_docs * d.H * d.dv);
    }
    if (for_bwd == 3) {  // the fused convolution's backward
      const int64_t Cc = (int64_t)d.H * (2 * d.dk + d.dv);
      L.off_cg = take(4 * (size_t)d.Ntok * Cc);
      L.off_cpart = take(kda_short_conv_workspace_size(d.Ntok, (int)Cc));
    }
    L.total = o;
    return L;
  }
  L.off_W = take(4 * nch * C * d.dk);
  L.off_U = take(4 * nch * C * d.dv);
  L.off_P = take(4 * nch * C * C);
  L.off_QG = take(4 * nch * C * d.dk);
  L.off_KD = take(4 * nch * C * d.dk);
  L.off_gam = take(4 * nch * d.dk);
  if (for_bwd) {
    L.off_Sent = take(4 * nch * d.dk * d.dv);
    L.off_dE = take(4 * nch * C * d.dv);
    L.off_dSn = take(4 * nch * d.dk * d.dv);
    L.off_pA = take(4 * nch);
    L.off_pdt = take(4 * nch * d.dk);
    L.off_scr = take(4 * nch * (size_t)bwd_scratch_floats(d.dk, d.dv));
  }
  if (for_bwd == 2) {  // kda_fwd_norm_gate saving for kda_bwd_norm_gate: o, the norm kernels' partials
    L.off_nO = take(4 * (size_t)d.Ntok * d.H * d.dv);
    L.off_nrm = take(kda_norm_gate_workspace_size((int64_t)d.Ntok * d.H, d.dv));
  }
  L.total = o;
  return L;
}

static Ws bind(void* ws, const Layout& L, const Dims& d, int for_bwd) {
  char* p = (char*)ws;
  auto at = [&](size_t off) { return off ? (float*)(p + off) : nullptr; };
  auto bat = [&](size_t off) { return off ? (__nv_bfloat16*)(p + off) : nullptr; };
  Ws w;
  w.err = (int32_t*)(p + L.off_err);
  w.tag = (int32_t*)(p + L.off_err + 4);
  w.n_chunks = (int32_t*)(p + L.off_nch);
  w.doc_chunk0 = (int32_t*)(p + L.off_dc0);
  w.chunk_tok0 = (int32_t*)(p + L.off_ct0);
  w.chunk_len = (int32_t*)(p + L.off_cl);
  w.chunk_doc = (int32_t*)(p + L.off_cd);
  w.doc_order = (int32_t*)(p + L.off_ord);
  w.useg = L.off_useg ? (int4*)(p + L.off_useg) : nullptr;
  w.uorder = L.off_uord ? (int32_t*)(p + L.off_uord) : nullptr;
  w.n_units = L.off_nu ? (int32_t*)(p + L.off_nu) : nullptr;
  w.segc = at(L.off_segc);
  w.W = at(L.off_W);
  w.U = at(L.off_U);
  w.P = at(L.off_P);
  w.QG = at(L.off_QG);
  w.KD = at(L.off_KD);
  w.gam = at(L.off_gam);
  w.Sent = for_bwd ? at(L.off_Sent) : nullptr;
  w.chb = L.off_CH ? (unsigned char*)(p + L.off_CH) : nullptr;
  w.dE = for_bwd ? at(L.off_dE) : nullptr;
  w.dSn = for_bwd ? at(L.off_dSn) : nullptr;
  w.pA = for_bwd ? at(L.off_pA) : nullptr;
  w.pdt = for_bwd ? at(L.off_pdt) : nullptr;
  w.scr = for_bwd ? at(L.off_scr) : nullptr;
  w.scr_per_ch = bwd_scratch_floats(d.dk, d.dv);
  w.sS = d.fast ? bat(L.off_Sent) : nullptr;
  w.sdS = d.fast && for_bwd ? bat(L.off_dSn) : nullptr;
  w.sT = bat(L.off_sT);
  w.sP = bat(L.off_sP);
  w.sW = bat(L.off_sW);
  w.sU = bat(L.off_sU);
  w.sA = at(L.off_sA);
  w.gDP = at(L.off_gDP);
  w.gMA = at(L.off_gMA);
  w.gQG = at(L.off_gQG);
  w.gKD = at(L.off_gKD);
  w.gKG = at(L.off_gKG);
  w.gdg = at(L.off_gdg);
  w.nO = at(L.off_nO);
  w.cg = at(L.off_cg);
  w.cpart = at(L.off_cpart);
  w.pdw = at(L.off_pdw);
  w.nrm = at(L.off_nrm);
  return w;
}

// Failure-detection test hook (kda_test_stage_timeout); 0 in normal use.
static int g_test_tx_extra = 0;

// The tensor-core state chains' grids: whether long chains may be split into
// segments (Dims::seg) and how many units the grids cover (Dims::nu).  (With
// the fused norm only the forward chain splits: the reverse chain forms dO
// itself, which the backward's composites would need beforehand.)  With the lengths known on the
// host (equal rows, or a host copy of cu_seqlens) the rule of seg_split is
// applied here and the grid is exact; with device-only offsets the chunk
// table applies it and the grid covers the most units any offsets can give.
static void chain_split_rule(const kda_problem* p, Dims& d) {
  d.seg = 0;
  d.nu = d.n_docs;
  if (!d.fast) return;
  d.slots = fast_chain_slots();
  if (d.slots <= 0) return;
  const long long grid_max = 2147483647LL / (2LL * d.H);  // the split grids are one-dimensional
  if (p->cu_seqlens && !p->cu_seqlens_host) {
    if (seg_units_max(d) > grid_max) return;
    d.seg = 1;
    d.nu = (int)seg_units_max(d);
    return;
  }
  const int32_t* c = p->cu_seqlens_host;
  auto chunks = [&](int i) { return c ? (c[i + 1] - c[i] + C - 1) / C : (d.T + C - 1) / C; };
  int n_max = 0;
  long long total = 0;
  for (int i = 0; i < d.n_docs; i++) {
    const int n = chunks(i);
    n_max = n > n_max ? n : n_max;
    total += n;
  }
  if (!seg_split(n_max, total, d.H, d.slots)) return;
  const int len = seg_len(n_max);
  long long units = 0;
  for (int i = 0; i < d.n_docs; i++) units += seg_count(chunks(i), true, len);
  if (units > grid_max) return;
  d.seg = 1;
  d.nu = (int)units;
}

// The plan of chain_split_rule, for the forward and again for its backward,
// which reads the forward's segment table: a plan that differs (another
// device's SM count) makes a different saved-problem tag, so that the
// backward refuses the workspace.
static void plan_chain_split(const kda_problem* p, Dims& d) {
  chain_split_rule(p, d);
  if (d.seg) d.tag ^= (int32_t)(((uint32_t)d.nu * 2654435761u) << 4 | 8u);
}

// The forward launch sequence shared by kda_fwd and kda_fwd_noalloc.
static cudaError_t run_forward(const kda_problem* p, Dims d, const FwdIO& io, const Ws& w, cudaStream_t stream,
                               bool fused = false) {
  d.tx_extra = g_test_tx_extra;
  if (!fused) plan_chain_split(p, d);
  cudaError_t e = launch_chunk_table(p->cu_seqlens, d, w, stream);
  if (e != cudaSuccess) return e;
  if (d.fast) return launch_fast_fwd(d, io, w, stream, fused);
  e = launch_fwd_intra(p->dtype, d, io, w, stream);
  if (e == cudaSuccess) e = launch_fwd_scan(p->dtype, d, io, w, stream);
  return e;
}

static bool supported(int dk, int dv) {
  return (dk == 32 && dv == 64) || (dk == 64 && dv == 64) || (dk == 64 && dv == 128) || (dk == 128 && dv == 128);
}

static bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

// Validates the problem and fills the dims.  Pure host code: no CUDA call.
static kda_status check_problem(const kda_problem* p, Dims* d) {
  if (!p) return KDA_ERR_INVALID_ARG;
  if (p->B <= 0 || p->T <= 0 || p->H <= 0 || p->dk <= 0 || p->dv <= 0) return KDA_ERR_INVALID_ARG;
  if (p->dtype != KDA_BF16 && p->dtype != KDA_F32) return KDA_ERR_INVALID_ARG;
  if (p->gate != KDA_GATE_CHANNEL && p->gate != KDA_GATE_SCALAR) return KDA_ERR_INVALID_ARG;
  if (!supported(p->dk, p->dv)) return KDA_ERR_UNSUPPORTED;
  const int64_t ntok = (int64_t)p->B * p->T;
  if (ntok > (int64_t)1 << 30 || p->H > 4096) return KDA_ERR_INVALID_ARG;
  int n_docs = p->B;
  if (p->cu_seqlens) {
    if (p->n_docs <= 0 || p->n_docs > (1 << 24)) return KDA_ERR_INVALID_ARG;
    if (!aligned(p->cu_seqlens, 4)) return KDA_ERR_ALIGNMENT;
    n_docs = p->n_docs;
    if (p->cu_seqlens_host) {
      const int32_t* c = p->cu_seqlens_host;
      if (c[0] != 0 || (int64_t)c[n_docs] != ntok) return KDA_ERR_BAD_SEQLENS;
      for (int i = 0; i < n_docs; i++)
        if (c[i + 1] < c[i]) return KDA_ERR_BAD_SEQLENS;
    }
  } else if (p->cu_seqlens_host) {
    return KDA_ERR_INVALID_ARG;
  }
  d->B = p->B;
  d->T = p->T;
  d->Ntok = (int)ntok;
  d->H = p->H;
  d->dk = p->dk;
  d->dv = p->dv;
  d->n_docs = n_docs;
  d->scale = p->scale > 0.f ? p->scale : 1.0f / sqrtf((float)p->dk);
  // upper bound on sum_i ceil(L_i / C) over any valid offsets
  int64_t ncm = p->cu_seqlens ? (ntok + (int64_t)(C - 1) * n_docs) / C
                              : (int64_t)p->B * ((p->T + C - 1) / C);
  if (ncm < 1) ncm = 1;
  if (ncm > (int64_t)1 << 30) return KDA_ERR_INVALID_ARG;
  if (ncm * p->H > (int64_t)2147483647) return KDA_ERR_INVALID_ARG;  // one CTA per chunk-head on a 1-D grid
  d->nc_max = (int)ncm;
  uint32_t hsh = 2166136261u;  // FNV-1a over the sizes that fix the layout
  const int32_t vals[9] = {p->B, p->T, p->H, p->dk, p->dv, p->dtype, n_docs, p->gate, 0x4b4441};
  for (int i = 0; i < 9; i++) { hsh ^= (uint32_t)vals[i]; hsh *= 16777619u; }
  d->tag = (int32_t)(hsh | 1u);
  d->save = 0;
  d->fast = fast_path(p->dtype, p->dk, p->dv) ? 1 : 0;
  d->ahead = 0;
  d->gate = p->gate;
  d->norm = 0;
  d->conv = 0;
  d->tx_extra = 0;
  d->rows = p->cu_seqlens ? 0 : 1;
  d->seg = 0;
  d->nu = n_docs;
  d->slots = 0;
  return KDA_OK;
}

}  // namespace kda

using namespace kda;

extern "C" {

size_t kda_workspace_size(const kda_problem* p, int for_backward) {
  Dims d;
  if (check_problem(p, &d) != KDA_OK) return 0;
  return layout(d, (for_backward == 2 || for_backward == 3) ? for_backward : for_backward ? 1 : 0).total;
}

static kda_status status_of(cudaError_t e) { return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA; }

}  // extern "C"

namespace {
// The gated RMSNorm epilogue's arguments of the fused entry points.
struct NormArgs {
  const void* g;
  const float* w;
  float eps;
};
// The short convolution's arguments: x [Ntok, H (2 dk + dv)] (the q | k | v
// blocks before the convolution) and its taps [H (2 dk + dv), 4].
struct ConvArgs {
  const void* x;
  const float* w;
};
// Points the q, k, v inputs (and the convolution taps) of io at the blocks of x.
template <class IO>
void bind_conv(IO& io, const Dims& d, const ConvArgs& cv) {
  const size_t qk = (size_t)d.H * d.dk;
  const __nv_bfloat16* x = (const __nv_bfloat16*)cv.x;
  io.q = x;
  io.k = x + qk;
  io.v = x + 2 * qk;
  io.ld = d.H * (2 * d.dk + d.dv);
  io.cwq = cv.w;
  io.cwk = cv.w + 4 * qk;
  io.cwv = cv.w + 8 * qk;
}

kda_status fwd_impl(const kda_problem* p, const void* q, const void* k, const void* v, const void* f, const void* b,
                    const float* A_log, const float* dt_bias, const float* h0, void* o, float* h_final,
                    int save_for_backward, void* workspace, size_t workspace_bytes, cudaStream_t stream,
                    const NormArgs* nm, void* y, const ConvArgs* cv = nullptr) {
  Dims d;
  kda_status s = check_problem(p, &d);
  if (s != KDA_OK) return s;
  if (nm && !d.fast && p->dtype != KDA_F32) return KDA_ERR_UNSUPPORTED;  // bf16 needs the fused kernels
  if (cv && !d.fast) return KDA_ERR_UNSUPPORTED;                         // the convolution is fused only there
  if (cv) {
    if (!cv->x || !cv->w) return KDA_ERR_INVALID_ARG;
    if (!aligned(cv->x, 16) || !aligned(cv->w, 16)) return KDA_ERR_ALIGNMENT;
    q = k = v = cv->x;  // checked below; bound to the blocks of x after the checks
  }
  const int fb = save_for_backward ? (cv ? 3 : nm ? 2 : 1) : 0;
  // o may be omitted with the norm, except as the composed path's intermediate when nothing is saved
  const bool need_o = !nm || (!d.fast && !fb);
  if (!q || !k || !v || !f || !b || !A_log || !dt_bias || (need_o && !o)) return KDA_ERR_INVALID_ARG;
  if (nm && (!nm->g || !nm->w || !y)) return KDA_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, f, b, A_log, dt_bias};
  for (const void* x : ptrs)
    if (!aligned(x, 16)) return KDA_ERR_ALIGNMENT;
  if ((o && !aligned(o, 16)) || (h0 && !aligned(h0, 16)) || (h_final && !aligned(h_final, 16))) return KDA_ERR_ALIGNMENT;
  if (nm && (!aligned(nm->g, 16) || !aligned(nm->w, 16) || !aligned(y, 16))) return KDA_ERR_ALIGNMENT;
  if (!workspace) return KDA_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return KDA_ERR_ALIGNMENT;
  Layout L = layout(d, fb);
  if (workspace_bytes < L.total) return KDA_ERR_WORKSPACE;
  Ws w = bind(workspace, L, d, fb ? 1 : 0);
  d.save = fb ? 1 : 0;
  if (nm) d.tag ^= 2;  // a workspace saved with the norm (or the convolution) serves that backward only
  if (cv) d.tag ^= 4;
  const float eps = nm && nm->eps > 0.f ? nm->eps : 1e-6f;
  FwdIO io{q, k, v, f, b, A_log, dt_bias, h0, o, h_final, d.save, nullptr, nullptr, 0.f, nullptr,
           d.H * d.dk, nullptr, nullptr, nullptr};
  if (cv) {
    d.conv = 1;
    bind_conv(io, d, *cv);
  }
  if (nm && d.fast) {  // fused into the forward chain's output warps
    d.norm = 1;
    io.ng = nm->g;
    io.nw = nm->w;
    io.neps = eps;
    io.y = y;
  }
  if (nm && !d.fast && fb) io.o = w.nO;  // fp32 io: the saved copy of o is the KDA output itself
  if (run_forward(p, d, io, w, stream) != cudaSuccess) return KDA_ERR_CUDA;
  if (nm && !d.fast) {  // other head shapes (fp32 io): the standalone epilogue kernel on o
    const int64_t rows = (int64_t)d.Ntok * d.H;
    s = kda_norm_gate_fwd(rows, d.dv, p->dtype, eps, io.o, nm->g, nm->w, y, stream);
    if (s != KDA_OK) return s;
    if (fb && o && cudaMemcpyAsync(o, w.nO, (size_t)rows * d.dv * 4, cudaMemcpyDeviceToDevice, stream) != cudaSuccess)
      return KDA_ERR_CUDA;
  }
  return KDA_OK;
}

kda_status bwd_impl(const kda_problem* p, const void* q, const void* k, const void* v, const void* f, const void* b,
                    const float* A_log, const float* dt_bias, const void* dO, const float* dh_final, void* dq,
                    void* dk, void* dv, void* df, void* db, float* dA_log, float* ddt_bias, float* dh0,
                    void* workspace, size_t workspace_bytes, cudaStream_t stream, const NormArgs* nm,
                    const void* dy, void* dg, float* dw, const ConvArgs* cv = nullptr, void* dx = nullptr,
                    float* dcw = nullptr) {
  Dims d;
  kda_status s = check_problem(p, &d);
  if (s != KDA_OK) return s;
  if (nm && !d.fast && p->dtype != KDA_F32) return KDA_ERR_UNSUPPORTED;
  if (cv && !d.fast) return KDA_ERR_UNSUPPORTED;
  if (cv) {
    if (!cv->x || !cv->w || !dx || !dcw) return KDA_ERR_INVALID_ARG;
    if (!aligned(cv->x, 16) || !aligned(cv->w, 16) || !aligned(dx, 16) || !aligned(dcw, 16)) return KDA_ERR_ALIGNMENT;
    q = k = v = cv->x;  // bound to the blocks of x below
  }
  if (cv) dq = dk = dv = dx;  // the gradients of the convolution's outputs go to the workspace (below)
  if (!q || !k || !v || !f || !b || !A_log || !dt_bias || !dO || !dq || !dk || !dv || !df || !db ||
      !dA_log || !ddt_bias)
    return KDA_ERR_INVALID_ARG;
  if (nm && (!nm->g || !nm->w || !dy || !dg || !dw)) return KDA_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, f, b, A_log, dt_bias, dO, dq, dk, dv, df, db, dA_log, ddt_bias};
  for (const void* x : ptrs)
    if (!aligned(x, 16)) return KDA_ERR_ALIGNMENT;
  if ((dh_final && !aligned(dh_final, 16)) || (dh0 && !aligned(dh0, 16))) return KDA_ERR_ALIGNMENT;
  if (nm) {
    const void* np[] = {nm->g, nm->w, dy, dg, dw};
    for (const void* x : np)
      if (!aligned(x, 16)) return KDA_ERR_ALIGNMENT;
  }
  if (!workspace) return KDA_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return KDA_ERR_ALIGNMENT;
  Layout L = layout(d, cv ? 3 : nm ? 2 : 1);
  if (workspace_bytes < L.total) return KDA_ERR_WORKSPACE;
  Ws w = bind(workspace, L, d, 1);
  if (nm) d.tag ^= 2;
  if (cv) d.tag ^= 4;
  const float eps = nm && nm->eps > 0.f ? nm->eps : 1e-6f;
  BwdIO io{q, k, v, f, b, A_log, dt_bias, dO, dh_final, dq, dk, dv, df, db, dA_log, ddt_bias, dh0,
           nullptr, nullptr, 0.f, nullptr, nullptr, nullptr, nullptr, d.H * d.dk, nullptr, nullptr, nullptr};
  if (cv) {  // q, k, v from x; dq, dk, dv the fp32 gradients of the convolution's outputs
    d.conv = 1;
    bind_conv(io, d, *cv);
    const size_t qk = (size_t)d.H * d.dk;
    io.dq = w.cg;
    io.dk = w.cg + qk;
    io.dv = w.cg + 2 * qk;
  }
  if (nm && d.fast) {  // fused into the reverse chain, which writes dO for the per-chunk kernels
    d.norm = 1;
    io.ng = nm->g;
    io.nw = nm->w;
    io.neps = eps;
    io.dy = dy;
    io.dOw = const_cast<void*>(dO);
    io.dg = dg;
    io.dw = dw;
  }
  if (nm && !d.fast) {  // other head shapes (fp32 io): the standalone epilogue backward writes dO first
    const int64_t rows = (int64_t)d.Ntok * d.H;
    s = kda_norm_gate_bwd(rows, d.dv, p->dtype, eps, w.nO, nm->g, nm->w, dy, const_cast<void*>(dO), dg, dw, w.nrm,
                          kda_norm_gate_workspace_size(rows, d.dv), stream);
    if (s != KDA_OK) return s;
  }
  if (d.fast) {
    plan_chain_split(p, d);  // the forward's plan (its segment table is in the workspace)
    cudaError_t e = launch_fast_bwd(d, io, w, stream);
    if (e == cudaSuccess && cv) {  // dx, dw of the convolution from its outputs' gradients
      const int Cc = d.H * (2 * d.dk + d.dv);
      e = launch_conv_bwd_fused(d.Ntok, Cc, p->cu_seqlens, d.n_docs, p->cu_seqlens ? (int64_t)d.Ntok : (int64_t)d.T,
                                (const __nv_bfloat16*)cv->x, cv->w, w.cg, (__nv_bfloat16*)dx, w.cpart, dcw, stream);
    }
    return status_of(e);
  }
  cudaError_t e = launch_bwd_scan(p->dtype, d, io, w, stream);
  if (e == cudaSuccess) e = launch_bwd_intra(p->dtype, d, io, w, stream);
  if (e == cudaSuccess) e = launch_bwd_reduce(d, io, w, stream);
  return status_of(e);
}
}  // namespace

extern "C" {

kda_status kda_fwd(const kda_problem* p, const void* q, const void* k, const void* v, const void* f,
                   const void* b, const float* A_log, const float* dt_bias, const float* h0, void* o,
                   float* h_final, int save_for_backward, void* workspace, size_t workspace_bytes,
                   cudaStream_t stream) {
  return fwd_impl(p, q, k, v, f, b, A_log, dt_bias, h0, o, h_final, save_for_backward, workspace, workspace_bytes,
                  stream, nullptr, nullptr);
}

kda_status kda_bwd(const kda_problem* p, const void* q, const void* k, const void* v, const void* f,
                   const void* b, const float* A_log, const float* dt_bias, const float* h0,
                   const void* dO, const float* dh_final, void* dq, void* dk, void* dv, void* df,
                   void* db, float* dA_log, float* ddt_bias, float* dh0, void* workspace,
                   size_t workspace_bytes, cudaStream_t stream) {
  (void)h0;  // the entry states were saved by kda_fwd
  return bwd_impl(p, q, k, v, f, b, A_log, dt_bias, dO, dh_final, dq, dk, dv, df, db, dA_log, ddt_bias, dh0,
                  workspace, workspace_bytes, stream, nullptr, nullptr, nullptr, nullptr);
}

kda_status kda_fwd_norm_gate(const kda_problem* p, const void* q, const void* k, const void* v, const void* f,
                             const void* b, const float* A_log, const float* dt_bias, const float* h0,
                             const void* g, const float* w, float eps, void* o, void* y, float* h_final,
                             int save_for_backward, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  const NormArgs nm{g, w, eps};
  return fwd_impl(p, q, k, v, f, b, A_log, dt_bias, h0, o, h_final, save_for_backward, workspace, workspace_bytes,
                  stream, &nm, y);
}

kda_status kda_fwd_conv(const kda_problem* p, const void* x, const float* conv_w, const void* f, const void* b,
                        const float* A_log, const float* dt_bias, const float* h0, const void* g, const float* w,
                        float eps, void* o, void* y, float* h_final, int save_for_backward, void* workspace,
                        size_t workspace_bytes, cudaStream_t stream) {
  const ConvArgs cv{x, conv_w};
  const NormArgs nm{g, w, eps};
  return fwd_impl(p, nullptr, nullptr, nullptr, f, b, A_log, dt_bias, h0, o, h_final, save_for_backward, workspace,
                  workspace_bytes, stream, g ? &nm : nullptr, y, &cv);
}

kda_status kda_bwd_conv(const kda_problem* p, const void* x, const float* conv_w, const void* f, const void* b,
                        const float* A_log, const float* dt_bias, const float* h0, const void* g, const float* w,
                        float eps, const void* dy, const float* dh_final, void* dO, void* dg, float* dw, void* dx,
                        float* dconv_w, void* df, void* db, float* dA_log, float* ddt_bias, float* dh0,
                        void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  (void)h0;
  const ConvArgs cv{x, conv_w};
  const NormArgs nm{g, w, eps};
  // without the norm, dy is the gradient of o itself
  return bwd_impl(p, nullptr, nullptr, nullptr, f, b, A_log, dt_bias, g ? dO : dy, dh_final, nullptr, nullptr,
                  nullptr, df, db, dA_log, ddt_bias, dh0, workspace, workspace_bytes, stream, g ? &nm : nullptr,
                  dy, dg, dw, &cv, dx, dconv_w);
}

kda_status kda_bwd_norm_gate(const kda_problem* p, const void* q, const void* k, const void* v, const void* f,
                             const void* b, const float* A_log, const float* dt_bias, const float* h0,
                             const void* g, const float* w, float eps, const void* dy, const float* dh_final,
                             void* dO, void* dg, float* dw, void* dq, void* dk, void* dv, void* df, void* db,
                             float* dA_log, float* ddt_bias, float* dh0, void* workspace, size_t workspace_bytes,
                             cudaStream_t stream) {
  (void)h0;
  const NormArgs nm{g, w, eps};
  return bwd_impl(p, q, k, v, f, b, A_log, dt_bias, dO, dh_final, dq, dk, dv, df, db, dA_log, ddt_bias, dh0,
                  workspace, workspace_bytes, stream, &nm, dy, dg, dw);
}

kda_status kda_test_stage_timeout(int enable) {
  g_test_tx_extra = enable ? 16 : 0;
  return KDA_OK;
}

kda_status kda_device_status(const void* workspace, cudaStream_t stream) {
  if (!workspace) return KDA_ERR_WORKSPACE;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return KDA_ERR_CUDA;
  int32_t v = 0;
  if (cudaMemcpy(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return KDA_ERR_CUDA;
  return (kda_status)v;
}

const char* kda_strerror(kda_status s) {
  switch (s) {
    case KDA_OK: return "ok";
    case KDA_ERR_INVALID_ARG: return "invalid argument (null pointer, size or dtype)";
    case KDA_ERR_UNSUPPORTED: return "unsupported (dk, dv): supported are (32,64), (64,64), (64,128), (128,128)";
    case KDA_ERR_ALIGNMENT: return "misaligned pointer (tensors need 16-byte, workspace 256-byte alignment)";
    case KDA_ERR_BAD_SEQLENS: return "cu_seqlens must start at 0, be non-decreasing and end at B*T";
    case KDA_ERR_WORKSPACE: return "workspace missing or smaller than kda_workspace_size()";
    case KDA_ERR_CUDA: return "a CUDA runtime call or kernel launch failed";
    case KDA_ERR_DEVICE: return "the device flagged an error";
  }
  return "unknown status";
}

static const char* const k_names[K_COUNT] = {"chunk_table", "fwd_intra", "fwd_scan", "bwd_scan",
                                             "bwd_intra", "bwd_reduce", "fwd_chain", "fwd_chunk",
                                             "fwd_state", "bwd_grad",  "bwd_gate",   "decode",
                                             "norm_gate_fwd", "norm_gate_bwd", "norm_gate_reduce",
                                             "conv_fwd",  "conv_bwd",  "conv_reduce",
                                             "fwd_state_norm", "bwd_scan_norm", "fwd_seg", "bwd_seg"};

const char* kda_prof_kernel_name(int i) { return (i >= 0 && i < K_COUNT) ? k_names[i] : nullptr; }

kda_status kda_prof_start(void) {
  if (!g_prof.created) {
    for (int i = 0; i < MAX_EV; i++)
      for (int j = 0; j < 2; j++)
        if (cudaEventCreate(&g_prof.ev[i][j]) != cudaSuccess) return KDA_ERR_CUDA;
    g_prof.created = true;
  }
  g_prof.n = 0;
  g_prof.on = true;
  return KDA_OK;
}

kda_status kda_prof_stop(double* total_ms, int64_t* launches, int n) {
  if (!g_prof.created) return KDA_ERR_INVALID_ARG;
  g_prof.on = false;
  for (int i = 0; i < n; i++) { if (total_ms) total_ms[i] = 0; if (launches) launches[i] = 0; }
  for (int e = 0; e < g_prof.n; e++) {
    if (cudaEventSynchronize(g_prof.ev[e][1]) != cudaSuccess) return KDA_ERR_CUDA;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, g_prof.ev[e][0], g_prof.ev[e][1]) != cudaSuccess) return KDA_ERR_CUDA;
    int kid = g_prof.kid[e];
    if (kid < n) {
      if (total_ms) total_ms[kid] += ms;
      if (launches) launches[kid] += 1;
    }
  }
  g_prof.n = 0;
  return KDA_OK;
}

}  // extern "C"

// ------------------------------------------------------------ allocation-free forward
// The forward's scratch for kda_fwd_noalloc lives in this fixed array (see
// include/kda.h).  Host code must not pass the symbol itself to a kernel:
// on the host it names a stand-in, not device memory.  Its device address
// is looked up once per device (with that device current) and cached.
static __device__ __align__(256) unsigned char g_noalloc_scratch[KDA_NOALLOC_SCRATCH_BYTES];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

kda_status noalloc_scratch(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KDA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return KDA_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return KDA_OK;
}
}  // namespace

extern "C" kda_status kda_fwd_noalloc(const kda_problem* p, const void* q, const void* k, const void* v,
                                      const void* f, const void* b, const float* A_log, const float* dt_bias,
                                      const float* h0, void* o, float* h_final, cudaStream_t stream) {
  Dims d;
  kda_status s = check_problem(p, &d);
  if (s != KDA_OK) return s;
  if (!q || !k || !v || !f || !b || !A_log || !dt_bias || !o) return KDA_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, f, b, A_log, dt_bias, o};
  for (const void* x : ptrs)
    if (!aligned(x, 16)) return KDA_ERR_ALIGNMENT;
  if ((h0 && !aligned(h0, 16)) || (h_final && !aligned(h_final, 16))) return KDA_ERR_ALIGNMENT;
  Layout L = layout(d, 0, true);
  if (L.total > KDA_NOALLOC_SCRATCH_BYTES) return KDA_ERR_WORKSPACE;  // beyond the fixed array
  void* scratch = nullptr;
  s = noalloc_scratch(&scratch);
  if (s != KDA_OK) return s;
  Ws w = bind(scratch, L, d, 0);
  d.save = 0;
  FwdIO io{q, k, v, f, b, A_log, dt_bias, h0, o, h_final, 0};
  return run_forward(p, d, io, w, stream, true) == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

// The error word of the fixed array sits at its byte 0, like a workspace's.
extern "C" kda_status kda_noalloc_status(cudaStream_t stream) {
  void* scratch = nullptr;
  const kda_status s = noalloc_scratch(&scratch);
  if (s != KDA_OK) return s;
  return kda_device_status(scratch, stream);
}
