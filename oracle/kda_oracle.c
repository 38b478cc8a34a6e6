/*
 * Kimi Delta Attention (KDA) -- plain CPU oracle.  TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg use
 * this file.  The CUDA library never includes, links or calls it, and it
 * shares no header, helper or constant with the CUDA sources.
 *
 * What it computes (per document and per head, one token at a time):
 *
 *   q^ = q / sqrt(sum q^2 + eps),  k^ = k / sqrt(sum k^2 + eps)   (over dk)
 *   x  = f + dt_bias[h, :]
 *   g  = -exp(A_log[h]) * softplus(x)            per key channel, g <= 0
 *   beta = sigmoid(b)                            one scalar per token, head
 *   S' = Diag(exp g) S                           decay first
 *   e  = beta * (v - S'^T k^)                    delta-rule correction
 *   S  = S' + k^ e^T       == (I - beta k^ k^T) Diag(exp g) S + beta k^ v^T
 *   o  = scale * S^T q^                          post-update state
 *
 * Sources:
 *  - "Pure KDA 300M" guide (Primus, ROCm docs), Overview: per-head decay gate
 *    combining the f projection with learnable A_log and dt_bias through a
 *    softplus; delta-rule recurrence with no positional encoding.
 *  - "Pure KDA 300M" guide, "Configs and tools": the fused in_proj carries one
 *    beta row per value head, so beta is one scalar per token and head.
 *  - openkimi README, "What is implemented": an exact recurrent FP32-state
 *    KDA oracle, fused Q/K norm, decay gate and beta.
 *  - torchtitan PR "[kimi k3] Support sample packing in KDA", Verification:
 *    the recurrent state resets at each document boundary given by
 *    cu_seqlens; a packed row equals the separate per-document runs.
 *  The pages print no equations; the recurrence above is the method's
 *  defining update (decay, then the delta correction on the decayed state).
 *
 * Readings where the pages are silent:
 *  - L2-norm epsilon: eps is passed in (1e-6 by the callers).
 *  - softplus: exact form max(x,0) + log1p(exp(-|x|)), no linear cut-off.
 *  - scale multiplies the output; it is not folded into q before the norm.
 *  - a zero-length document is allowed: its final state is its initial state
 *    and its dS0 is its dS_final.
 *
 * Precision: REAL is double unless built with -DORACLE_REAL=float, which
 * gives the fp32-state variant.  Interfaces always take double arrays.
 *
 * Parity: every function here is pinned by the CPU tests (closed forms,
 * special cases, brute-force matrix products, finite differences and the
 * packed-vs-separate identity).  The epsilon and softplus readings above are
 * conventions the pages do not fix; they are "parity unpinned" as readings,
 * though the code that applies them is pinned.
 *
 * Layouts (token-major, flattened over batch rows):
 *   q, k, f : [Ntok, H, dk]    v, o, dO : [Ntok, H, dv]    b : [Ntok, H]
 *   A_log   : [H]              dt_bias  : [H, dk]
 *   states  : [n_seqs, H, dk, dv]
 *   cu_seqlens : n_seqs + 1 non-decreasing offsets into [0, Ntok]
 * A "unit" is one (document, head) pair; units are independent and the
 * caller may run disjoint unit lists in parallel threads.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifndef ORACLE_REAL
#define ORACLE_REAL double
#endif
typedef ORACLE_REAL real;

/* softplus(x) = log(1 + e^x), written so that it neither overflows nor
 * loses the small tail. */
static real sp_(real x) {
    real ax = x < 0 ? -x : x;
    return (x > 0 ? x : (real)0) + (real)log1p(exp((double)-ax));
}

static real sigm_(real x) { return (real)(1.0 / (1.0 + exp(-(double)x))); }

/* Per-token quantities of one head. */
typedef struct {
    real *qh, *kh;   /* normalised q, k  [dk] */
    real nq, nk;     /* their norms sqrt(sum x^2 + eps) */
    real *x, *g;     /* pre-softplus gate input and log-decay [dk] */
    real beta, braw;
} tok_t;

static void token_prologue(int dk, int H, int h, long t,
                           const double* q, const double* k, const double* f,
                           const double* b, real a, const double* dtb,
                           real eps, tok_t* T) {
    const double* qt = q + ((size_t)t * H + h) * dk;
    const double* kt = k + ((size_t)t * H + h) * dk;
    const double* ft = f + ((size_t)t * H + h) * dk;
    real sq = 0, sk = 0;
    for (int i = 0; i < dk; i++) { sq += (real)qt[i] * (real)qt[i]; sk += (real)kt[i] * (real)kt[i]; }
    T->nq = (real)sqrt((double)(sq + eps));
    T->nk = (real)sqrt((double)(sk + eps));
    for (int i = 0; i < dk; i++) {
        T->qh[i] = (real)qt[i] / T->nq;
        T->kh[i] = (real)kt[i] / T->nk;
        T->x[i] = (real)ft[i] + (real)dtb[i];
        T->g[i] = -a * sp_(T->x[i]);
    }
    T->braw = (real)b[(size_t)t * H + h];
    T->beta = sigm_(T->braw);
}

/* One forward token update S <- (I - beta k k^T) Diag(exp g) S + beta k v^T,
 * o = scale S^T q.  S is dk x dv row-major.  Optionally returns e. */
static void token_step(int dk, int dv, const tok_t* T, const double* vt, real scale,
                       real* S, real* u, real* e, double* ot) {
    for (int i = 0; i < dk; i++) {
        real al = (real)exp((double)T->g[i]);
        for (int j = 0; j < dv; j++) S[i * dv + j] *= al;          /* S' = Diag(a) S */
    }
    for (int j = 0; j < dv; j++) {                                  /* u = S'^T k */
        real s = 0;
        for (int i = 0; i < dk; i++) s += S[i * dv + j] * T->kh[i];
        u[j] = s;
        e[j] = T->beta * ((real)vt[j] - s);                         /* e = beta (v - u) */
    }
    for (int i = 0; i < dk; i++)                                    /* S = S' + k e^T */
        for (int j = 0; j < dv; j++) S[i * dv + j] += T->kh[i] * e[j];
    if (ot) {
        for (int j = 0; j < dv; j++) {                              /* o = scale S^T q */
            real s = 0;
            for (int i = 0; i < dk; i++) s += S[i * dv + j] * T->qh[i];
            ot[j] = (double)(scale * s);
        }
    }
}

static int tok_alloc(tok_t* T, int dk) {
    T->qh = (real*)calloc(4 * (size_t)dk, sizeof(real));
    if (!T->qh) return -1;
    T->kh = T->qh + dk; T->x = T->kh + dk; T->g = T->x + dk;
    return 0;
}

/*
 * Forward for a list of units.  o rows of the listed units and their final
 * states are written; nothing else is touched.  h0 / h_final may be NULL.
 * Returns 0, or -1 on allocation failure / bad arguments.
 */
int kda_oracle_forward(int Ntok, int H, int dk, int dv,
                       const double* q, const double* k, const double* v,
                       const double* f, const double* b,
                       const double* A_log, const double* dt_bias,
                       double scale, double eps,
                       int n_seqs, const int* cu_seqlens, const double* h0,
                       int n_units, const int* unit_seq, const int* unit_head,
                       double* o, double* h_final) {
    if (Ntok < 0 || H <= 0 || dk <= 0 || dv <= 0 || n_seqs < 0) return -1;
    real* S = (real*)malloc(sizeof(real) * ((size_t)dk * dv + 2 * (size_t)dv));
    tok_t T;
    if (!S || tok_alloc(&T, dk)) { free(S); return -1; }
    real* u = S + (size_t)dk * dv;
    real* e = u + dv;
    for (int n = 0; n < n_units; n++) {
        int sq = unit_seq[n], h = unit_head[n];
        if (sq < 0 || sq >= n_seqs || h < 0 || h >= H) { free(S); free(T.qh); return -1; }
        long t0 = cu_seqlens[sq], t1 = cu_seqlens[sq + 1];
        if (t0 < 0 || t1 < t0 || t1 > Ntok) { free(S); free(T.qh); return -1; }
        const double* h0u = h0 ? h0 + ((size_t)sq * H + h) * dk * dv : NULL;
        for (size_t i = 0; i < (size_t)dk * dv; i++) S[i] = h0u ? (real)h0u[i] : 0;
        real a = (real)exp(A_log[h]);
        for (long t = t0; t < t1; t++) {
            token_prologue(dk, H, h, t, q, k, f, b, a, dt_bias + (size_t)h * dk, (real)eps, &T);
            token_step(dk, dv, &T, v + ((size_t)t * H + h) * dv, (real)scale, S, u, e,
                       o + ((size_t)t * H + h) * dv);
        }
        if (h_final) {
            double* hf = h_final + ((size_t)sq * H + h) * dk * dv;
            for (size_t i = 0; i < (size_t)dk * dv; i++) hf[i] = (double)S[i];
        }
    }
    free(S); free(T.qh);
    return 0;
}

/*
 * Reverse-mode backward for a list of units, token by token in reverse.
 * The loss is  sum(o * dO) + sum(h_final * dh_final).  The states S_{t-1}
 * needed in reverse are recomputed forward from checkpoints taken every CK
 * tokens.  Gradients of the listed units' rows are written (overwritten);
 * the per-head parameter gradients are returned per unit
 * (dA_log_part[n], ddt_bias_part[n, dk]) so that the caller sums them.
 */
#define CK 64
int kda_oracle_backward(int Ntok, int H, int dk, int dv,
                        const double* q, const double* k, const double* v,
                        const double* f, const double* b,
                        const double* A_log, const double* dt_bias,
                        double scale, double eps,
                        int n_seqs, const int* cu_seqlens, const double* h0,
                        const double* dO, const double* dh_final,
                        int n_units, const int* unit_seq, const int* unit_head,
                        double* dq, double* dkk, double* dvv, double* df, double* db,
                        double* dA_log_part, double* ddt_bias_part, double* dh0) {
    if (Ntok < 0 || H <= 0 || dk <= 0 || dv <= 0 || n_seqs < 0) return -1;
    const size_t SS = (size_t)dk * dv;
    /* states before each token of the current segment, plus one scratch */
    real* seg = (real*)malloc(sizeof(real) * SS * (CK + 1));
    real* dS = (real*)malloc(sizeof(real) * (SS * 2 + 6 * (size_t)dv + 4 * (size_t)dk));
    tok_t T;
    if (!seg || !dS || tok_alloc(&T, dk)) { free(seg); free(dS); return -1; }
    real* Sp = dS + SS;             /* S' = Diag(alpha) S_{t-1} */
    real* u = Sp + SS;              /* S'^T k */
    real* e = u + dv;
    real* de = e + dv;
    real* du = de + dv;
    real* St = du + dv;             /* scratch dv */
    real* dqh = St + dv;
    real* dkh = dqh + dk;
    real* dal = dkh + dk;
    real* tmp = dal + dk;
    (void)tmp;
    real* ckp = NULL;
    size_t ck_cap = 0;
    for (int n = 0; n < n_units; n++) {
        int sq = unit_seq[n], h = unit_head[n];
        if (sq < 0 || sq >= n_seqs || h < 0 || h >= H) goto fail;
        long t0 = cu_seqlens[sq], t1 = cu_seqlens[sq + 1];
        if (t0 < 0 || t1 < t0 || t1 > Ntok) goto fail;
        long L = t1 - t0;
        long nseg = (L + CK - 1) / CK;
        if ((size_t)(nseg + 1) > ck_cap) {
            free(ckp);
            ck_cap = (size_t)nseg + 1;
            ckp = (real*)malloc(sizeof(real) * SS * ck_cap);
            if (!ckp) goto fail;
        }
        real a = (real)exp(A_log[h]);
        const double* dtb = dt_bias + (size_t)h * dk;
        const double* h0u = h0 ? h0 + ((size_t)sq * H + h) * SS : NULL;
        /* forward pass keeping the state at the start of every segment */
        real* S = seg;  /* use seg[0] as the running state */
        for (size_t i = 0; i < SS; i++) S[i] = h0u ? (real)h0u[i] : 0;
        for (long s = 0; s < nseg; s++) {
            memcpy(ckp + s * SS, S, sizeof(real) * SS);
            for (long t = t0 + s * CK; t < t0 + (s + 1) * CK && t < t1; t++) {
                token_prologue(dk, H, h, t, q, k, f, b, a, dtb, (real)eps, &T);
                token_step(dk, dv, &T, v + ((size_t)t * H + h) * dv, (real)scale, S, u, e, NULL);
            }
        }
        /* dS starts at dS_final */
        const double* dhf = dh_final ? dh_final + ((size_t)sq * H + h) * SS : NULL;
        for (size_t i = 0; i < SS; i++) dS[i] = dhf ? (real)dhf[i] : 0;
        real dAl = 0;
        real* ddtb = (real*)calloc((size_t)dk, sizeof(real));
        if (!ddtb) goto fail;
        for (long s = nseg - 1; s >= 0; s--) {
            long ta = t0 + s * CK, tb = ta + CK < t1 ? ta + CK : t1;
            /* seg[m] = state before token ta+m */
            memcpy(seg, ckp + s * SS, sizeof(real) * SS);
            for (long t = ta; t < tb - 1; t++) {
                real* nxt = seg + (size_t)(t - ta + 1) * SS;
                memcpy(nxt, seg + (size_t)(t - ta) * SS, sizeof(real) * SS);
                token_prologue(dk, H, h, t, q, k, f, b, a, dtb, (real)eps, &T);
                token_step(dk, dv, &T, v + ((size_t)t * H + h) * dv, (real)scale, nxt, u, e, NULL);
            }
            for (long t = tb - 1; t >= ta; t--) {
                const real* Sprev = seg + (size_t)(t - ta) * SS;
                token_prologue(dk, H, h, t, q, k, f, b, a, dtb, (real)eps, &T);
                const double* vt = v + ((size_t)t * H + h) * dv;
                const double* dot = dO + ((size_t)t * H + h) * dv;
                /* recompute S' = Diag(alpha) S_{t-1}, u, e and S_t */
                for (int i = 0; i < dk; i++) {
                    real al = (real)exp((double)T.g[i]);
                    for (int j = 0; j < dv; j++) Sp[i * dv + j] = al * Sprev[i * dv + j];
                }
                for (int j = 0; j < dv; j++) {
                    real s2 = 0;
                    for (int i = 0; i < dk; i++) s2 += Sp[i * dv + j] * T.kh[i];
                    u[j] = s2;
                    e[j] = T.beta * ((real)vt[j] - s2);
                }
                /* o = scale S_t^T q^ :  dq^ = scale S_t dO,  dS += scale q^ dO^T */
                for (int i = 0; i < dk; i++) {
                    real s2 = 0;
                    for (int j = 0; j < dv; j++) {
                        real Sij = Sp[i * dv + j] + T.kh[i] * e[j];
                        s2 += Sij * (real)dot[j];
                    }
                    dqh[i] = scale * s2;
                }
                for (int i = 0; i < dk; i++)
                    for (int j = 0; j < dv; j++) dS[i * dv + j] += (real)scale * T.qh[i] * (real)dot[j];
                /* S_t = S' + k^ e^T :  dk^ = dS e,  de = dS^T k^,  dS' = dS */
                for (int i = 0; i < dk; i++) {
                    real s2 = 0;
                    for (int j = 0; j < dv; j++) s2 += dS[i * dv + j] * e[j];
                    dkh[i] = s2;
                }
                for (int j = 0; j < dv; j++) {
                    real s2 = 0;
                    for (int i = 0; i < dk; i++) s2 += dS[i * dv + j] * T.kh[i];
                    de[j] = s2;
                }
                /* e = beta (v - u) */
                real dbeta = 0;
                for (int j = 0; j < dv; j++) {
                    dbeta += de[j] * ((real)vt[j] - u[j]);
                    dvv[((size_t)t * H + h) * dv + j] = (double)(T.beta * de[j]);
                    du[j] = -T.beta * de[j];
                }
                /* u = S'^T k^ :  dS' += k^ du^T,  dk^ += S' du */
                for (int i = 0; i < dk; i++) {
                    real s2 = 0;
                    for (int j = 0; j < dv; j++) {
                        dS[i * dv + j] += T.kh[i] * du[j];
                        s2 += Sp[i * dv + j] * du[j];
                    }
                    dkh[i] += s2;
                }
                /* S' = Diag(alpha) S_{t-1} :  dalpha_i = sum_j dS'_ij S_{t-1,ij},
                 * dS_{t-1} = Diag(alpha) dS' */
                for (int i = 0; i < dk; i++) {
                    real al = (real)exp((double)T.g[i]);
                    real s2 = 0;
                    for (int j = 0; j < dv; j++) {
                        s2 += dS[i * dv + j] * Sprev[i * dv + j];
                        dS[i * dv + j] *= al;
                    }
                    dal[i] = s2 * al;   /* dg = dalpha * alpha */
                }
                /* gate: g = -exp(A_log) softplus(x),  x = f + dt_bias */
                for (int i = 0; i < dk; i++) {
                    real dg = dal[i];
                    real dx = dg * (-a) * sigm_(T.x[i]);
                    df[((size_t)t * H + h) * dk + i] = (double)dx;
                    ddtb[i] += dx;
                    dAl += dg * T.g[i];
                }
                /* beta = sigmoid(b) */
                db[(size_t)t * H + h] = (double)(dbeta * T.beta * (1 - T.beta));
                /* L2 norm:  dx = (dx^ - x^ (x^ . dx^)) / n */
                real pq = 0, pk = 0;
                for (int i = 0; i < dk; i++) { pq += T.qh[i] * dqh[i]; pk += T.kh[i] * dkh[i]; }
                for (int i = 0; i < dk; i++) {
                    dq[((size_t)t * H + h) * dk + i] = (double)((dqh[i] - T.qh[i] * pq) / T.nq);
                    dkk[((size_t)t * H + h) * dk + i] = (double)((dkh[i] - T.kh[i] * pk) / T.nk);
                }
            }
        }
        if (dh0) {
            double* d0 = dh0 + ((size_t)sq * H + h) * SS;
            for (size_t i = 0; i < SS; i++) d0[i] = (double)dS[i];
        }
        dA_log_part[n] = (double)dAl;
        for (int i = 0; i < dk; i++) ddt_bias_part[(size_t)n * dk + i] = (double)ddtb[i];
        free(ddtb);
    }
    free(seg); free(dS); free(T.qh); free(ckp);
    return 0;
fail:
    free(seg); free(dS); free(T.qh); free(ckp);
    return -1;
}

/* Gate pieces exposed for the closed-form pins. */
double kda_oracle_gate(double A_log, double x) { return (double)(-(real)exp(A_log) * sp_((real)x)); }
double kda_oracle_sigmoid(double x) { return (double)sigm_((real)x); }
int kda_oracle_real_bytes(void) { return (int)sizeof(real); }
