// Internal declarations shared by the CUDA translation units of the KDA
// library (not part of the C ABI).
#pragma once
#include <cuda.h>  // CUtensorMap (the maps are encoded through the runtime's driver entry point)
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <stddef.h>

namespace kda {

constexpr int C = 64;          // chunk length (tokens)
constexpr float L2_EPS = 1e-6f; // q/k L2-norm epsilon

// Kernel ids for the per-kernel timing brackets.
enum KernelId {
  K_TABLE = 0,
  K_FWD_INTRA,
  K_FWD_SCAN,
  K_BWD_SCAN,
  K_BWD_INTRA,
  K_BWD_REDUCE,
  K_FWD_CHAIN,
  K_FWD_CHUNK,
  K_FWD_STATE,
  K_BWD_GRAD,
  K_BWD_GATE,
  K_DECODE,
  K_NORM_FWD,
  K_NORM_BWD,
  K_NORM_RED,
  K_CONV_FWD,
  K_CONV_BWD,
  K_CONV_RED,
  K_FWD_STATE_NORM,
  K_BWD_SCAN_NORM,
  K_FWD_SEG,
  K_BWD_SEG,
  K_COUNT
};

// Splitting long state chains (tensor-core path).  The forward state chain is
// affine, S_{c+1} = M_c S_c + KU_c, so a run of chunks composes into one map
// S -> Phi S + B; so is the backward's reverse chain (dS -> Psi dS + D).  When
// a workload's longest document has more than SPLIT_MIN chunks and more than
// twice the average chain length per resident chain CTA (a chain-bound
// workload: a few long chains finish long after the rest), every document of
// more than SPLIT_MIN chunks is cut into segments of seg_len(n_max) chunks.
// Per direction one kernel composes each segment but the one its chain starts
// in; the chain kernel starts every other segment from the composites on its
// way folded onto the document's initial state (final-state gradient): one
// small product per segment, so segments grow with the longest document, about
// sqrt(n_max) chunks and at least SEG.  The same rule runs on the host (to size
// the launch) and in the chunk-table kernel (to build the segment table).
constexpr int SEG = 16, SPLIT_MIN = 32;
__host__ __device__ inline bool seg_split(int n_max, long long total_chunks, int H, int slots) {
  if (n_max <= SPLIT_MIN || slots <= 0) return false;
  const long long avg = (total_chunks * H * 2 + slots - 1) / slots;  // chain steps per resident chain CTA
  return n_max > 2 * avg;
}
// Chunks per segment: the least multiple of SEG whose square covers n_max.
__host__ __device__ inline int seg_len(int n_max) {
  int s = SEG;
  while ((long long)s * s < n_max) s += SEG;
  return s;
}
// Segments of a document of n chunks.
__host__ __device__ inline int seg_count(int n, bool split, int len) {
  return split && n > SPLIT_MIN ? (n + len - 1) / len : 1;
}

// Device-side view of the caller's workspace.  Offsets are fixed by
// layout_workspace() from the problem sizes; the error word sits at byte 0.
struct Ws {
  int32_t* err;         // [1]  device error word (kda_status value)
  int32_t* tag;         // [1]  problem tag of the forward that saved this workspace
  int32_t* n_chunks;    // [1]
  int32_t* doc_chunk0;  // [n_docs + 1] first chunk of each document
  int32_t* chunk_tok0;  // [nc_max] first flattened token of each chunk
  int32_t* chunk_len;   // [nc_max] tokens in the chunk (1..C), 0 = unused
  int32_t* chunk_doc;   // [nc_max]
  int32_t* doc_order;   // [n_docs] documents by decreasing chunk count (the general scans' dispatch order)
  // tensor-core state chains split into segments (Dims::seg): per unit (document, first chunk
  // within it, chunks, segment index), a document's segments consecutive; the unit count; and
  // per unit and head a composite ([dk][dk] then [dk][dv], fp32): in the forward [Phi | B] of
  // every segment but a document's last, in the backward [Psi | D] of every segment but its first
  int4* useg;
  int32_t* uorder;  // units by decreasing work (chunks plus folded segments): the chain grids' dispatch order
  int32_t* n_units;
  float* segc;
  // forward intermediates, per chunk-head ch = chunk * H + h
  float* W;    // [ch][C][dk]  T diag(beta) (K^ * Gamma)
  float* U;    // [ch][C][dv]  T diag(beta) V
  float* P;    // [ch][C][C]   scale * inclusive-lower (Q^ K^T with decay ratios)
  float* QG;   // [ch][C][dk]  scale * Q^ * Gamma
  float* KD;   // [ch][C][dk]  K^ * exp(G_last - G)
  float* gam;  // [ch][dk]     exp(G_last)
  float* Sent; // [ch][dk][dv] state entering the chunk (saved for backward)
  // tensor-core path, split-bf16 operand tiles (hi tile, then lo tile): S
  // entering the chunk (forward chain); T, P = scale P', W, U saved by the
  // forward; the state gradient leaving the chunk (backward chain)
  __nv_bfloat16 *sS, *sT, *sP, *sW, *sU, *sdS;
  // M = Diag(gamma) - KD^T W [ch][dk][dk] and QW = QG - P W [ch][C][dk] (split
  // tiles from the per-chunk forward; both chains read them)
  // tensor-core forward: per chunk-head the chain operands M, QW (split bf16) and KU, PU (fp32,
  // per 32-column half in fragment order) in one block, [KU0 | PU0 | M | QW | KU1 | PU1]
  unsigned char* chb;
  float* sA;   // [ch][10][16][16] A' (unscaled) lower 16 x 16 blocks
  // tensor-core backward, bwd_grad -> bwd_gate
  float *gDP, *gMA;        // [ch][10][16][16] dP', beta dA lower blocks
  float *gQG, *gKD, *gKG;  // [ch][256 threads][8] dQG, dKD, beta YW in fragment order
  float* gdg;              // [ch][dk] dgamma
  // backward
  float* dE;   // [ch][C][dv]  gradient of E = U - W S
  float* dSn;  // [ch][dk][dv] gradient of the state leaving the chunk
  float* pA;   // [ch]         per chunk-head partial of dA_log
  float* pdt;  // [ch][dk]     per chunk-head partial of ddt_bias
  // saved by kda_fwd_norm_gate for kda_bwd_norm_gate (workspace for_backward = 2)
  float* nO;   // [Ntok][H][dv] the pre-norm KDA output o in fp32
  float* pdw;  // [n_docs * H][dv] per (document, head) partial of the gated norm's dw (fused backward)
  float* nrm;  // other head shapes: the standalone norm backward's per-CTA dw partials
  // the fused convolution's backward (workspace for_backward = 3)
  float* cg;     // [Ntok][C] fp32 gradients of the convolution's outputs (q | k | v blocks)
  float* cpart;  // its weight-gradient partials
  float* scr;  // [ch][scr_per_ch] backward scratch
  int64_t scr_per_ch;
};

struct Dims {
  int Ntok, H, dk, dv, n_docs, nc_max, B, T;
  float scale;
  int32_t tag;   // nonzero hash of the problem; the forward stores it when saving
  int32_t save;  // forward saves for the backward
  int32_t fast;  // bf16 io with dk = 32, dv = 64: tensor-core kernels
  int32_t ahead; // CTAs in flight (one wave) of the per-chunk tensor-core kernels: their L2 prefetch distance
  int32_t gate;  // 0: per key channel (KDA); 1: scalar per head (GDN), f [Ntok, H], dt_bias [H]
  int32_t norm;  // the gated RMSNorm epilogue is fused into the chains (tensor-core path)
  int32_t conv;  // the short convolution is fused into the per-chunk kernels' prologue (tensor-core path)
  int32_t tx_extra;  // failure-detection test hook (kda_test_stage_timeout): bytes the forward chain's stage
                     // barriers expect beyond what their copies deliver; 0 outside that test
  int32_t rows;   // no cu_seqlens: the documents are the B rows of T tokens (chunk j's tokens follow from j)
  int32_t seg;    // (tensor-core chains) the chunk table decides whether to split long chains (seg_split)
  int32_t nu;     // units of the forward chain grid: documents, or with seg an upper bound on the segments
  int32_t slots;  // resident forward chain CTAs on the device (the split rule's denominator)
};

// Backward kernels refuse a workspace that no saving forward of the same
// problem filled (flagging KDA_ERR_WORKSPACE instead of reading garbage).
__device__ __forceinline__ bool saved_ok(const Dims& d, const int32_t* tag, int32_t* err) {
  if (*tag != d.tag) {
    *err = -5;
    return false;
  }
  return *err == 0;
}

struct FwdIO {
  const void *q, *k, *v, *f, *b;
  const float *A_log, *dt_bias, *h0;
  void* o;
  float* h_final;
  int save;
  // fused gated RMSNorm epilogue (Dims::norm): y = o r w sigmoid(g) per row
  const void* ng;   // gate g [Ntok, H, dv]
  const float* nw;  // weight w [dv]
  float neps;
  void* y;          // [Ntok, H, dv]
  // fused short convolution (Dims::conv): q, k, v point at the q, k, v channel
  // blocks of the pre-convolution projection x [Ntok, C] (C = H (2 dk + dv)),
  // whose rows are ld elements apart, and cwq / cwk / cwv at the blocks' taps
  // ([channels][4] fp32); the kernels apply the convolution and silu on load
  int ld;
  const float *cwq, *cwk, *cwv;
};

struct BwdIO {
  const void *q, *k, *v, *f, *b;
  const float *A_log, *dt_bias;
  const void* dO;
  const float* dh_final;
  void *dq, *dk, *dv, *df, *db;
  float *dA_log, *ddt_bias, *dh0;
  // fused gated RMSNorm backward (Dims::norm): from dy, g, w and the fp32 o the
  // forward saved (Ws::nO) the reverse chain forms dO itself and writes it to
  // dOw (dO above then names the same buffer for the per-chunk kernels), dg and
  // the dw partials
  const void* ng;
  const float* nw;
  float neps;
  const void* dy;
  void* dOw;
  void* dg;
  float* dw;
  // fused short convolution (Dims::conv): inputs as in FwdIO; dq, dk, dv are
  // then the fp32 gradients of the convolution's outputs, rows ld apart (the
  // q, k, v blocks of a [Ntok, C] buffer the convolution's backward reads)
  int ld;
  const float *cwq, *cwk, *cwv;
};

// TMA tensor maps of the raw per-token inputs, each viewed as a 2-D [Ntok][H d]
// bf16 tensor with a box of one head's d channels x C tokens (encoded on the
// host per call; unused fields are zero).
struct TMaps {
  CUtensorMap q, k, v, f;
};
// Encodes the maps for bf16 q, k, f [Ntok, H, dk] and v [Ntok, H, dv]
// (f only for the per-channel gate); false if the driver refuses.
bool encode_tmaps(TMaps* tm, const void* q, const void* k, const void* v, const void* f, int Ntok, int H, int dk,
                  int dv, bool channel_gate);
// The fused gated norm's per-row tensors, [Ntok][H dv] with a box of 32 value
// columns x C tokens: the gate g and dy (bf16) and the saved fp32 o.
struct NMaps {
  CUtensorMap g, dy, o;
};
bool encode_nmaps(NMaps* nm, const void* g, const void* dy, const float* o, int Ntok, int H, int dv);

// Launch wrappers (return cudaGetLastError of their launches).
// Launches kernel k with the programmatic-stream-serialization attribute (see pdl_wait).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, args...);
}
// Launches kernel k in thread-block clusters of cz CTAs along z (the grid's z
// extent a multiple of cz), with the programmatic-stream-serialization
// attribute when pdl is set.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_cluster(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, int cz,
                                  bool pdl, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  at[1].id = cudaLaunchAttributeClusterDimension;  // cz CTAs along z, or along x for a 1-D grid
  const bool along_x = grid.y == 1 && grid.z == 1;
  at[1].val.clusterDim.x = along_x ? cz : 1;
  at[1].val.clusterDim.y = 1;
  at[1].val.clusterDim.z = along_x ? 1 : cz;
  cfg.attrs = pdl ? at : at + 1;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, k, args...);
}
cudaError_t launch_chunk_table(const int32_t* cu, const Dims& d, const Ws& w, cudaStream_t st);
cudaError_t launch_fwd_intra(int dtype, const Dims& d, const FwdIO& io, const Ws& w, cudaStream_t st);
cudaError_t launch_fwd_scan(int dtype, const Dims& d, const FwdIO& io, const Ws& w, cudaStream_t st);
cudaError_t launch_bwd_scan(int dtype, const Dims& d, const BwdIO& io, const Ws& w, cudaStream_t st);
cudaError_t launch_bwd_intra(int dtype, const Dims& d, const BwdIO& io, const Ws& w, cudaStream_t st);
cudaError_t launch_bwd_reduce(const Dims& d, const BwdIO& io, const Ws& w, cudaStream_t st);
bool fast_path(int dtype, int dk, int dv);
// fused: the single-kernel forward that needs only the chunk table (used by
// kda_fwd_noalloc); else the per-chunk kernel and the state chain.
cudaError_t launch_fast_fwd(const Dims& d, const FwdIO& io, const Ws& w, cudaStream_t st, bool fused);
// Resident forward-chain CTAs of the tensor-core path on the current device (two per SM).
int fast_chain_slots();
cudaError_t launch_fast_bwd(const Dims& d, const BwdIO& io, const Ws& w, cudaStream_t st);

// The fused convolution's backward: dx and dw from x and the fp32 gradients of
// the convolution's outputs (documents: cu, or rows of row_len tokens).
cudaError_t launch_conv_bwd_fused(int64_t n_tok, int C, const int32_t* cu, int n_docs, int64_t row_len,
                                  const __nv_bfloat16* x, const float* w, const float* dy, __nv_bfloat16* dx,
                                  float* part, float* dw, cudaStream_t st);

// out[c] = sum over the rows of a [nrows][ncols] fp32 array, in a fixed order.
cudaError_t launch_sum_rows(const float* part, int nrows, int ncols, float* out, cudaStream_t st);

// Timing brackets (no-ops unless kda_prof_start() armed them).
void prof_begin(int kid, cudaStream_t st);
void prof_end(int kid, cudaStream_t st);

// Bytes of backward scratch per chunk-head.
inline int64_t bwd_scratch_floats(int dk, int dv) {
  return (int64_t)C * dv * 2 + (int64_t)C * dk * 8;
}

// ------------------------------------------------------------ device helpers
__device__ __forceinline__ float ldf(const float* p) { return *p; }
__device__ __forceinline__ float ldf(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void stf(float* p, float x) { *p = x; }
__device__ __forceinline__ void stf(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

__device__ __forceinline__ float softplus_f(float x) {
  return fmaxf(x, 0.0f) + log1pf(expf(-fabsf(x)));
}
__device__ __forceinline__ float sigmoid_f(float x) { return 1.0f / (1.0f + expf(-x)); }
// Sigmoid from the fast exponential and the fast division intrinsic (relative
// error ~1e-6; 0 once exp(-x) overflows, the function's limit): for the
// streaming epilogue / prologue kernels whose outputs are stored in bf16 or
// fp32 and need no more.
__device__ __forceinline__ float sigmoid_fast(float x) { return __fdividef(1.0f, 1.0f + __expf(-x)); }
// Softplus from the same intrinsics (absolute error below 1e-6): for the
// tensor-core path, where it sets the log-decay g = -exp(A_log) softplus(.)
// that then enters bf16-split products.
// 2^x by the hardware approximation (PTX ex2.approx.ftz: relative error about
// 2^-22; results below 2^-126 flush to zero, far below anything a decay factor
// contributes next to O(1) values).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float softplus_fast(float x) { return fmaxf(x, 0.0f) + __logf(1.0f + __expf(-fabsf(x))); }

// Programmatic dependent launch.  A kernel launched by launch_pdl may start
// while the kernel before it in the stream is finishing: pdl_wait() returns
// once that grid has completed and its writes are visible (at once when the
// kernel was launched normally, or the previous grid never released), and
// must precede every read of what that grid wrote; pdl_release() lets the
// next grid launch once every CTA of this grid has called it or exited.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_release() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

}  // namespace kda
