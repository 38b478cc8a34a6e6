/*
 * kda.h -- C ABI of the GB300 (sm_103a) Kimi Delta Attention library.
 *
 * Operation (per document and per head, tokens in order):
 *   q^ = q / sqrt(sum q^2 + 1e-6)          k^ likewise   (over the key dim dk)
 *   g  = -exp(A_log[h]) * softplus(f + dt_bias[h, :])    per key channel
 *   beta = sigmoid(b)                                    per token and head
 *   S_t = (I - beta_t k^_t k^_t^T) Diag(exp g_t) S_{t-1} + beta_t k^_t v_t^T
 *   o_t = scale * S_t^T q^_t
 * with S (dk x dv, fp32) reset to the document's initial state at every
 * document start.  Sources: "Pure KDA 300M" guide (Primus, ROCm docs),
 * Overview (softplus decay gate with learnable A_log and dt_bias, delta-rule
 * recurrence) and "Configs and tools" (one beta per value head); openkimi
 * README, "What is implemented" (fused Q/K norm, decay gate and beta; fp32
 * recurrent state); torchtitan PR "[kimi k3] Support sample packing in KDA"
 * (state reset at cu_seqlens document boundaries).
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers owned by the caller.  The
 *    library never allocates device memory at run time; scratch lives in the
 *    caller's workspace.  The one exception is kda_fwd_noalloc(), whose
 *    scratch is a fixed static array (KDA_NOALLOC_SCRATCH_BYTES, 32 MiB)
 *    reserved on every GPU that loads the library.  Host pointers are named
 *    *_host.
 *  - Calls are asynchronous on the given stream; nothing synchronises the
 *    device except kda_device_status() and kda_prof_stop().
 *  - CUDA graphs: kda_fwd, kda_bwd, kda_decode and the norm and convolution
 *    calls issue only kernel launches on the given stream, so they can be
 *    captured (cudaStreamBeginCapture) and replayed; a replay reads the
 *    captured pointers' current contents and gives the bits of an eager call.
 *    kda_device_status() and kda_prof_stop() synchronise and cannot be
 *    captured; the first kda_fwd_noalloc() on a device must precede capture.
 *  - Arguments are validated on the host before any launch; a failed check
 *    returns its status and launches nothing.  An invalid cu_seqlens array
 *    that only exists on the device is caught by the device (no work is done,
 *    outputs are left unwritten) and reported by kda_device_status().
 *  - Layouts are contiguous, token-major, over Ntok = B*T flattened tokens:
 *      q, k, f, dq, dk, df : [B, T, H, dk]
 *      v, o, dO, dv        : [B, T, H, dv]
 *      b, db               : [B, T, H]
 *      A_log, dA_log       : [H] fp32       dt_bias, ddt_bias : [H, dk] fp32
 *    With gate = KDA_GATE_SCALAR (the scalar-gated Gated DeltaNet variant, one
 *    log-decay per token and head broadcast over the dk channels; the openkimi
 *    README, "Testing and verification", contrasts it with KDA's channel-wise
 *    decay): f, df : [B, T, H] and dt_bias, ddt_bias : [H].
 *      h0, h_final, dh_final, dh0 : [n_docs, H, dk, dv] fp32
 *  - Alignment: every tensor pointer 16-byte aligned; workspace 256-byte.
 *  - Gradient outputs are overwritten, never accumulated.
 */
#ifndef KDA_GB300_H
#define KDA_GB300_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime.h>

#if defined(__GNUC__)
#define KDA_API __attribute__((visibility("default")))
#else
#define KDA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kda_status {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = -1,  /* null pointer, non-positive size, bad dtype */
    KDA_ERR_UNSUPPORTED = -2,  /* (dk, dv) pair not compiled in */
    KDA_ERR_ALIGNMENT = -3,    /* a pointer violates the alignment rule */
    KDA_ERR_BAD_SEQLENS = -4,  /* cu_seqlens not 0 = c0 <= c1 <= ... = B*T */
    KDA_ERR_WORKSPACE = -5,    /* workspace missing or smaller than kda_workspace_size() */
    KDA_ERR_CUDA = -6,         /* a CUDA runtime call failed (launch error) */
    KDA_ERR_DEVICE = -7        /* the device flagged an error (see kda_device_status) */
} kda_status;

typedef enum kda_dtype { KDA_BF16 = 0, KDA_F32 = 1 } kda_dtype;

/* Problem description shared by every call.
 *  B, T      : rows and tokens per row; the token axis is flattened to B*T.
 *  H         : heads; dk / dv : key / value head dims.  Supported (dk, dv):
 *              (32, 64), (64, 64), (64, 128), (128, 128).
 *  dtype     : kda_dtype of q, k, v, f, b, o, dO and dq, dk, dv, df, db.
 *  scale     : output scale; <= 0 selects 1/sqrt(dk).
 *  n_docs    : number of documents when cu_seqlens is given (>= 1).
 *  cu_seqlens: DEVICE int32 [n_docs + 1] document offsets into the flattened
 *              token axis, or NULL for equal-length rows (n_docs = B,
 *              documents are the rows).  Zero-length documents are allowed:
 *              their final state is their initial state.
 *  cu_seqlens_host : optional HOST copy of cu_seqlens; when given it is
 *              validated on the host (KDA_ERR_BAD_SEQLENS before any launch).
 */
typedef enum kda_gate {
    KDA_GATE_CHANNEL = 0,  /* KDA: one log-decay per key channel, f [.., H, dk], dt_bias [H, dk] */
    KDA_GATE_SCALAR = 1    /* scalar-gated (GDN): one per head, f [.., H], dt_bias [H]; df [.., H], ddt_bias [H] */
} kda_gate;

typedef struct kda_problem {
    int32_t B, T, H, dk, dv;
    int32_t dtype;
    float scale;
    int32_t n_docs;
    const int32_t* cu_seqlens;
    const int32_t* cu_seqlens_host;
    int32_t gate;          /* kda_gate */
} kda_problem;

/* Bytes of device workspace kda_fwd / kda_bwd need for this problem
 * (for_backward = 0: forward only; 1: forward that saves for the backward,
 * and the backward; 2: kda_fwd_norm_gate saving for kda_bwd_norm_gate, and
 * that backward; 3: kda_fwd_conv saving for kda_bwd_conv, and that
 * backward).  Returns 0 for an invalid problem. */
KDA_API size_t kda_workspace_size(const kda_problem* p, int for_backward);

/* Forward.  Writes o and, when non-NULL, h_final.  h0 may be NULL (zero
 * initial state).  With save_for_backward = 1 the workspace (sized with
 * for_backward = 1) keeps what kda_bwd needs; it must then be passed to
 * kda_bwd unmodified, with the same inputs.  Streams: stream 0 is the legacy
 * default stream.
 * bf16 io at dk=32/dv=64: when the batch is chain-bound (its longest document
 * has more than 32 chunks of 64 tokens and more than twice the average chain
 * length per resident chain CTA of the device), documents of more than 32
 * chunks run their state chains as segments composed in parallel and folded
 * onto h0 (the same map, a different rounding order: such a document's last
 * bits can differ from its run in a batch that is not chain-bound).  The plan
 * depends on the device's SM count; kda_bwd on a device that plans
 * differently refuses the workspace (KDA_ERR_WORKSPACE from
 * kda_device_status). */
KDA_API kda_status kda_fwd(const kda_problem* p,
                   const void* q, const void* k, const void* v, const void* f, const void* b,
                   const float* A_log, const float* dt_bias, const float* h0,
                   void* o, float* h_final,
                   int save_for_backward, void* workspace, size_t workspace_bytes,
                   cudaStream_t stream);

/* Backward of the loss sum(o * dO) + sum(h_final * dh_final).  Requires the
 * workspace filled by kda_fwd(save_for_backward = 1) on the same inputs (and
 * a device of the same SM count, see kda_fwd).
 * dh_final may be NULL (zero); dh0 may be NULL (not returned).  Writes dq,
 * dk, dv, df, db (dtype), dA_log [H] and ddt_bias [H, dk] (fp32, summed over
 * all tokens in a fixed order: deterministic). */
KDA_API kda_status kda_bwd(const kda_problem* p,
                   const void* q, const void* k, const void* v, const void* f, const void* b,
                   const float* A_log, const float* dt_bias, const float* h0,
                   const void* dO, const float* dh_final,
                   void* dq, void* dk, void* dv, void* df, void* db,
                   float* dA_log, float* ddt_bias, float* dh0,
                   void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Forward with the gated RMSNorm output epilogue fused in ("Pure KDA 300M"
 * guide, Overview: per-head output gate and RMSNorm with eps 1e-6; openkimi
 * README, "What is implemented": fused RMSNorm plus sigmoid gate on the KDA
 * output).  Per token and head, over the value dim dv:
 *   y_j = o_j r w_j sigmoid(g_j),   r = 1 / sqrt(mean_k o_k^2 + eps)
 * where o is the KDA output of kda_fwd.  g, y : [B, T, H, dv] in dtype; w :
 * [dv] fp32, shared by the heads; eps <= 0 selects 1e-6.  o (the pre-norm
 * output, dtype) is written when non-NULL and may be NULL, except on the
 * composed path below without save_for_backward (there it is the
 * intermediate).  With save_for_backward the workspace must hold
 * kda_workspace_size(p, 2) bytes: it keeps o in fp32 for kda_bwd_norm_gate, so
 * that the backward does not depend on a rounding of o.  Other arguments and
 * statuses are those of kda_fwd.
 * bf16 io at dk=32/dv=64: the norm runs inside the state chain's output stage
 * (the two column halves of a row exchange their sums of squares between the
 * two CTAs of a thread-block cluster), so o need not round-trip through
 * memory.  fp32 io, any supported (dk, dv): kda_fwd then the
 * kda_norm_gate_fwd kernel inside the same call.  bf16 io at other head
 * shapes: KDA_ERR_UNSUPPORTED (compose kda_fwd and kda_norm_gate_fwd). */
KDA_API kda_status kda_fwd_norm_gate(const kda_problem* p,
                   const void* q, const void* k, const void* v, const void* f, const void* b,
                   const float* A_log, const float* dt_bias, const float* h0,
                   const void* g, const float* w, float eps,
                   void* o, void* y, float* h_final,
                   int save_for_backward, void* workspace, size_t workspace_bytes,
                   cudaStream_t stream);

/* Backward of the loss sum(y * dy) + sum(h_final * dh_final) through the
 * fused forward above: writes dO (the gradient of the pre-norm output o,
 * [B, T, H, dv] in dtype; an output, also read by the later kernels of this
 * call), dg ([B, T, H, dv] in dtype), dw ([dv] fp32, summed in a fixed order)
 * and every output of kda_bwd.  g, w, eps are the forward's; o comes from the
 * workspace, which must be the one kda_fwd_norm_gate(save_for_backward = 1)
 * filled on the same inputs (kda_workspace_size(p, 2) bytes; a workspace
 * saved by kda_fwd is refused by the device, see kda_device_status).
 * bf16 io at dk=32/dv=64: the norm's backward runs inside the reverse state
 * chain, which forms dO on chip for its own products.  fp32 io, other head
 * shapes: the kda_norm_gate_bwd kernel, then the kda_bwd kernels.  bf16 io at
 * other head shapes: KDA_ERR_UNSUPPORTED. */
KDA_API kda_status kda_bwd_norm_gate(const kda_problem* p,
                   const void* q, const void* k, const void* v, const void* f, const void* b,
                   const float* A_log, const float* dt_bias, const float* h0,
                   const void* g, const float* w, float eps,
                   const void* dy, const float* dh_final,
                   void* dO, void* dg, float* dw,
                   void* dq, void* dk, void* dv, void* df, void* db,
                   float* dA_log, float* ddt_bias, float* dh0,
                   void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* The layer around the KDA path in one call each way: the varlen short causal
 * convolution (width 4, silu) on the concatenated q | k | v projection, KDA,
 * and optionally the gated RMSNorm epilogue ("Pure KDA 300M" guide,
 * Overview: short-conv kernel size 4, depthwise on the concatenated QKV, then
 * the KDA recurrence, per-head output gate and RMSNorm; torchtitan PR "[kimi
 * k3] Support sample packing in KDA": the convolution window and the state
 * both reset at document starts):
 *   q | k | v = silu(conv4(x)),   o = KDA(q, k, v, f, b, ...),   y = o r w sigmoid(g)
 * x : [B, T, H (2 dk + dv)] in dtype, the q channels (h dk + i) first, then k,
 * then v (h dv + j); conv_w : [H (2 dk + dv), 4] fp32, tap j multiplying
 * x_{t-3+j}; tokens before the document start read as 0 (documents are the
 * rows, or cu_seqlens).  g == NULL: no norm (o is written, y unused); else as
 * kda_fwd_norm_gate (o optional).  bf16 io at dk=32/dv=64 only (other shapes:
 * KDA_ERR_UNSUPPORTED): the per-chunk kernels apply the convolution and silu
 * to the rows they load (with the three tokens before the chunk), so q, k, v
 * never exist in memory.  Saving for the backward needs
 * kda_workspace_size(p, 3) bytes. */
KDA_API kda_status kda_fwd_conv(const kda_problem* p, const void* x, const float* conv_w,
                   const void* f, const void* b, const float* A_log, const float* dt_bias, const float* h0,
                   const void* g, const float* w, float eps,
                   void* o, void* y, float* h_final,
                   int save_for_backward, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Backward of kda_fwd_conv: the loss sum(y * dy) (with the norm; dy then
 * [B, T, H, dv], and dO, dg, dw are written as in kda_bwd_norm_gate) or
 * sum(o * dy) (g == NULL; dO, dg, dw unused), plus sum(h_final * dh_final).
 * Writes dx [B, T, H (2 dk + dv)] (dtype), dconv_w [H (2 dk + dv), 4] (fp32,
 * summed in a fixed order), df, db, dA_log, ddt_bias and dh0 (NULL: not
 * returned).  The per-chunk kernels recompute q, k, v from x and write the
 * fp32 gradients of the convolution's outputs into the workspace; one
 * streaming kernel then forms dx and the tap gradients (its window crosses
 * chunk boundaries).  The workspace must come from kda_fwd_conv with
 * save_for_backward = 1 on the same inputs. */
KDA_API kda_status kda_bwd_conv(const kda_problem* p, const void* x, const float* conv_w,
                   const void* f, const void* b, const float* A_log, const float* dt_bias, const float* h0,
                   const void* g, const float* w, float eps,
                   const void* dy, const float* dh_final,
                   void* dO, void* dg, float* dw,
                   void* dx, float* dconv_w, void* df, void* db,
                   float* dA_log, float* ddt_bias, float* dh0,
                   void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Synchronises `stream` and reads the device-side error word kept in the
 * workspace (KDA_OK, or the status the device flagged, e.g.
 * KDA_ERR_BAD_SEQLENS for offsets that were only on the device). */
KDA_API kda_status kda_device_status(const void* workspace, cudaStream_t stream);

/* Failure-detection test hook.  Every wait of the library's kernels on an
 * mbarrier (bulk-copy completion, a cluster peer's data) gives up after about
 * a second; the kernel then flags KDA_ERR_DEVICE in the workspace's
 * error word, skips its remaining work and returns, leaving the context
 * usable.  While enable != 0, later tensor-core forwards (bf16, dk=32/dv=64)
 * make the forward state chain's stage barriers (and those of its composing
 * kernel, when the chain runs split) expect 16 bytes more than each copy
 * delivers, so those waits run out (every copy issued still completes):
 * kda_device_status() then reports KDA_ERR_DEVICE, and the outputs are not
 * valid.  Off by default; process-wide, not thread-safe; for tests only. */
KDA_API kda_status kda_test_stage_timeout(int enable);

/* Human-readable text for a status. */
KDA_API const char* kda_strerror(kda_status s);

/* Per-kernel timing.  kda_prof_start() arms CUDA-event brackets around every
 * kernel the library launches afterwards (on the launch stream); kda_prof_stop()
 * synchronises those events and returns, for each kernel id i < n, the summed
 * milliseconds and the launch count, then disarms.  Not thread-safe; for
 * benchmarks.  kda_prof_kernel_name(i) names kernel id i (NULL past the end). */
KDA_API kda_status kda_prof_start(void);
KDA_API kda_status kda_prof_stop(double* total_ms, int64_t* launches, int n);
KDA_API const char* kda_prof_kernel_name(int i);

/* Forward without any caller-provided workspace (no counterpart in the
 * paper; this is a convenience of this library).
 *
 * Who needs it: callers that cannot or must not call cudaMalloc -- for
 * example a host program that has given all device memory to its own pool
 * and exposes no allocator to plug-ins, or a latency-critical loop where the
 * device synchronisation that cudaMalloc/cudaFree can imply is not
 * acceptable.  Such callers still own q, k, v, f, b, A_log, dt_bias, h0, o and
 * h_final; only the forward's scratch moves into a fixed array inside the
 * library.
 *
 * The array is KDA_NOALLOC_SCRATCH_BYTES (32 MiB) of device memory, reserved
 * on every GPU that loads this library for as long as the process lives.  A
 * problem whose scratch does not fit is rejected with KDA_ERR_WORKSPACE
 * before anything is launched.  The scratch is:
 *  - bf16 io at dk=32/dv=64: the chunk table only (a single-kernel forward
 *    carries each document's state itself), about 12 bytes per 64-token
 *    chunk plus 4 per document -- up to about 2.8 million chunks, far more
 *    than kda_workspace_size(p, 0), which counts the two-kernel forward's
 *    per-chunk products, would suggest;
 *  - every other shape or fp32 io: exactly kda_workspace_size(p, 0) (fp32
 *    intra-chunk factors, about 56 KB per chunk and head at 32/64 fp32,
 *    roughly 600 chunk-heads).
 * Nothing is saved for kda_bwd.
 *
 * The first call on a device looks up the array's device address on that
 * device (the device must be current); make that first call before any
 * stream capture.  Every call on a device shares the same array and leaves
 * its contents behind (nothing in it needs to start zeroed: each call writes
 * everything it later reads).  Calls whose work overlaps on the GPU -- on
 * different streams, or from different host threads -- race on the array
 * and give wrong results: serialise them.  Arguments and host-side statuses
 * are those of kda_fwd with save_for_backward = 0.  Offsets that exist only
 * on the device (cu_seqlens without cu_seqlens_host) are checked by the
 * device; a rejection leaves o and h_final unwritten and is reported by
 * kda_noalloc_status(), not by the return value. */
#define KDA_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
KDA_API kda_status kda_fwd_noalloc(const kda_problem* p,
                   const void* q, const void* k, const void* v, const void* f, const void* b,
                   const float* A_log, const float* dt_bias, const float* h0,
                   void* o, float* h_final, cudaStream_t stream);

/* Synchronises `stream` and returns the device-side status of the last
 * kda_fwd_noalloc() on the current device (KDA_OK, or e.g.
 * KDA_ERR_BAD_SEQLENS for offsets that were only on the device); the error
 * word lives in the same fixed array, so the call must follow the forward it
 * checks before any other kda_fwd_noalloc() on that device.  Allocates
 * nothing. */
KDA_API kda_status kda_noalloc_status(cudaStream_t stream);

/* Single-token recurrent step (decode): one token for each of n_seq
 * independent sequences, applied to their states in place.  Per sequence and
 * head, the same recurrence as above for one token ("Pure KDA 300M" guide,
 * Overview; the inference-only forward backend discussed in the openkimi
 * README, "Testing and verification"):
 *   S <- (I - beta k^ k^T) Diag(exp g) S + beta k^ v^T,   o = scale S^T q^
 * Layouts (device pointers, 16-byte aligned, contiguous):
 *   q, k, f : [n_seq, H, dk]     v, o : [n_seq, H, dv]     b : [n_seq, H]
 *   A_log : [H] fp32    dt_bias : [H, dk] fp32
 *   state : [n_seq, H, dk, dv] fp32, read and overwritten with the new state
 * dtype is KDA_BF16 or KDA_F32 for q, k, v, f, b and o; (dk, dv) as kda_fwd;
 * gate as kda_problem.gate (KDA_GATE_SCALAR: f [n_seq, H], dt_bias [H]);
 * scale <= 0 selects 1/sqrt(dk).  Needs no workspace.  Returns
 * KDA_ERR_INVALID_ARG / _UNSUPPORTED / _ALIGNMENT before any launch, or
 * KDA_ERR_CUDA if the launch fails.  Steps on the same stream chain: each reads
 * the state the previous one wrote. */
KDA_API kda_status kda_decode(int n_seq, int H, int dk, int dv, int dtype, int gate, float scale,
                   const void* q, const void* k, const void* v, const void* f, const void* b,
                   const float* A_log, const float* dt_bias, float* state, void* o,
                   cudaStream_t stream);

/* Gated RMSNorm output epilogue, per row (token and head) over the value dim
 * dv ("Pure KDA 300M" guide, Overview: per-head output gate and RMSNorm with
 * eps 1e-6; openkimi README, "What is implemented": fused RMSNorm plus sigmoid
 * gate on the KDA output):
 *   r = 1 / sqrt(mean_j x_j^2 + eps),   y_j = x_j * r * w_j * sigmoid(g_j)
 * x (the KDA output o), g (the output gate), y, dy, dx, dg : [n_rows, dv] in
 * dtype (KDA_BF16 or KDA_F32); w, dw : [dv] fp32, one weight vector shared by
 * the heads; dv is 64 or 128; eps <= 0 selects 1e-6.  Device pointers,
 * 16-byte aligned.  The backward overwrites dx (the dO of kda_bwd), dg and dw;
 * its scratch (per-CTA partials of dw, summed in a fixed order) is
 * kda_norm_gate_workspace_size(n_rows, dv) bytes (0 for invalid sizes). */
KDA_API size_t kda_norm_gate_workspace_size(int64_t n_rows, int dv);
KDA_API kda_status kda_norm_gate_fwd(int64_t n_rows, int dv, int dtype, float eps,
                   const void* x, const void* g, const float* w, void* y, cudaStream_t stream);
KDA_API kda_status kda_norm_gate_bwd(int64_t n_rows, int dv, int dtype, float eps,
                   const void* x, const void* g, const float* w, const void* dy,
                   void* dx, void* dg, float* dw, void* workspace, size_t workspace_bytes,
                   cudaStream_t stream);

/* Varlen short causal depthwise convolution, kernel width 4, the step before
 * the KDA path on the concatenated q | k | v channels ("Pure KDA 300M" guide,
 * Overview: short-conv kernel size 4, depthwise on the concatenated QKV; its
 * troubleshooting section uses FLA's causal_conv1d on [B, T, D]; torchtitan PR
 * "[kimi k3] Support sample packing in KDA": per-document reset):
 *   z_t,c = sum_{j<4} w[c, j] x_{t-3+j, c}   (x before the document start is 0)
 *   y_t,c = silu(z_t,c) = z sigmoid(z) (activation 1), or z (activation 0)
 * x, y, dy, dx : [n_tok, C] token-major in dtype (C a multiple of 8 for bf16,
 * 4 for fp32; 16-byte aligned); w, dw : [C, 4] fp32 (w 16-byte aligned).  cu_seqlens (device
 * int32 [n_docs + 1], 0 = c0 <= ... = n_tok) delimits documents; NULL is one
 * document.  The backward overwrites dx and dw (per-tile partials of dw in the
 * workspace, summed in a fixed order): kda_short_conv_workspace_size(n_tok, C)
 * bytes. */
KDA_API size_t kda_short_conv_workspace_size(int64_t n_tok, int C);
KDA_API kda_status kda_short_conv_fwd(int64_t n_tok, int C, int dtype, int activation,
                   const int32_t* cu_seqlens, int n_docs, const void* x, const float* w, void* y,
                   cudaStream_t stream);
KDA_API kda_status kda_short_conv_bwd(int64_t n_tok, int C, int dtype, int activation,
                   const int32_t* cu_seqlens, int n_docs, const void* x, const float* w, const void* dy,
                   void* dx, float* dw, void* workspace, size_t workspace_bytes, cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* KDA_GB300_H */
