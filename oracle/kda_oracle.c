/*
 * kda_oracle.c -- TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.
 *
 * A plain, slow, double-precision CPU statement of the delta-rule linear
 * attention forward with per-token decay.  Only the test-suite, the smoke
 * check and the CPU-baseline leg of the benchmark load this file's library;
 * the GPU library shares no code, header, table or helper with it.
 *
 * Source of the arithmetic (cited by page title and section):
 *
 *   [P1] ejkernel "kernels._xla.kernel_delta_attention._interface", function
 *        kda(): "The core recurrence"
 *            h_t = exp(decay_t) * h_{t-1} + k_t (x) (beta_t * (v_t - h_{t-1} @ k_t))
 *            o_t = h_t @ q_t
 *        with h_t the [head_dim, value_dim] memory of one head; "Parameters"
 *        (softmax_scale defaults to head_dim^-0.5 and scales the query;
 *        use_qk_l2norm normalises q and k; decay None means zeros;
 *        initial_state [B,H,dk,dv]); "Returns" (output [B,T,H,dv] and
 *        final_state [B,H,dk,dv]); "Algorithm Modes" (recurrent = pure
 *        sequential scan, chunked = parallel inside a chunk and sequential
 *        across chunks).
 *   [P2] TileOPs "Linear Attention Operators", DeltaNetFwdOp: packed
 *        variable-length mode with cu_seqlens, one state per sequence,
 *        key-major fp32 state.
 *   [P3] TileOPs "Linear Attention Operators", KDAFwdOp (Kimi Delta
 *        Attention): the gated delta rule with one log-space decay per key
 *        channel, g [B,T,H,K]; GLARecurrentFwdOp prints the per-channel
 *        retention as diag(exp(gk)) applied to the state.
 *   [P1'] the same page, kda_decay(): the per-token decay from a gate,
 *        A = -exp(A_log), decay = A * softplus(gate + dt_bias), never positive.
 *   [P3'] TileOPs "Linear Attention Operators", GDNFwdOp / KDAFwdOp:
 *        use_beta_sigmoid_in_kernel (beta = sigmoid(x)), allow_neg_eigval
 *        (beta = 2 sigmoid(x)), use_gate_in_kernel (the gate above, with A_log
 *        and dt_bias).
 *   [P4] kda-neuron-kernels README, "What this package provides" and
 *        "Functional warning": the exact chunked form uses the per-channel
 *        factor exp(gc_i - gc_j) inside the chunk; the recurrent form is exact.
 *
 * Readings taken where the page is silent:
 *   - h is [dk,dv], so "h @ k" is read as h^T k (a dv-vector) and the write
 *     "k (x) u" is the outer product k u^T.
 *   - The delta term reads the undecayed h_{t-1}, literally as printed.
 *   - softmax_scale multiplies the (normalised) query: o_t = h_t^T (scale*q_t).
 *   - L2 normalisation is x / max(||x||_2, 1e-12).
 *
 * Inputs arrive as float32 (every value the generators produce is exactly
 * representable in float32 -- bf16-rounded or plain fp32) and are widened
 * exactly to double; every operation is carried out in double.
 *
 * Layouts (row-major, contiguous):
 *   q, k  [B, T, H, dk]      v, o  [B, T, H, dv]      beta, decay [B, T, H]
 *   h0, hT [B, H, dk, dv]    (varlen: B == 1, T == total tokens, state [N,H,dk,dv])
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORACLE_NORM_EPS 1e-12

/* One independent problem: one head of one sequence. */
typedef struct {
    const float *q, *k, *v;       /* first token of the sequence, head h  */
    const float *beta, *decay;    /* idem; decay may be NULL (zeros)      */
    const float *gk;              /* per-channel decay [.., dk] or NULL   */
    long tok_stride_qk;           /* elements between tokens in q/k       */
    long tok_stride_v;            /* elements between tokens in v/o       */
    long tok_stride_g;            /* elements between tokens in beta/decay*/
    const double *h0;             /* [dk,dv] or NULL                      */
    double *o;                    /* first token of the sequence, head h  */
    double *hT;                   /* [dk,dv] or NULL                      */
    int T, dk, dv;
} oracle_problem;

typedef struct {
    int mode;                     /* 0 = recurrent scan, 1 = chunked form */
    int chunk;
    double scale;
    int use_l2;
    int per_channel;              /* 1: decay per key channel (gk)        */
    int decayed_read;             /* 1: the delta reads the decayed state */
} oracle_opts;

/* Read row x (length n, float32) into out (double), L2-normalised when asked,
 * then multiplied by mult. */
static void load_row(const float *x, int n, int use_l2, double mult, double *out)
{
    for (int i = 0; i < n; ++i) out[i] = (double)x[i];
    if (use_l2) {
        double ss = 0.0;
        for (int i = 0; i < n; ++i) ss += out[i] * out[i];
        double nrm = sqrt(ss);
        if (nrm < ORACLE_NORM_EPS) nrm = ORACLE_NORM_EPS;
        for (int i = 0; i < n; ++i) out[i] /= nrm;
    }
    for (int i = 0; i < n; ++i) out[i] *= mult;
}

/*
 * Recurrent mode [P1 "Algorithm Modes": the pure sequential scan], one token at
 * a time, exactly the printed recurrence:
 *   r   = h^T k_t                     (the "h_{t-1} @ k_t" readout)
 *   u   = beta_t (v_t - r)            (the delta term)
 *   h   = exp(decay_t) h + k_t u^T    (retention + rank-one write)
 *   o_t = h^T (scale q_t)             (readout from the updated memory)
 */
static void scan_problem(const oracle_problem *p, const oracle_opts *op)
{
    const int dk = p->dk, dv = p->dv;
    double *h = (double *)calloc((size_t)dk * dv, sizeof(double));
    double *kk = (double *)malloc(sizeof(double) * dk);
    double *qq = (double *)malloc(sizeof(double) * dk);
    double *r = (double *)malloc(sizeof(double) * dv);
    double *u = (double *)malloc(sizeof(double) * dv);
    if (p->h0) memcpy(h, p->h0, sizeof(double) * (size_t)dk * dv);

    for (int t = 0; t < p->T; ++t) {
        load_row(p->k + t * p->tok_stride_qk, dk, op->use_l2, 1.0, kk);
        load_row(p->q + t * p->tok_stride_qk, dk, op->use_l2, op->scale, qq);
        const float *vt = p->v + t * p->tok_stride_v;
        double b = (double)p->beta[t * p->tok_stride_g];
        double g = p->decay ? (double)p->decay[t * p->tok_stride_g] : 0.0;
        double a = exp(g);

        for (int j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (int i = 0; i < dk; ++i) acc += h[(size_t)i * dv + j] * kk[i];
            r[j] = acc;
        }
        for (int j = 0; j < dv; ++j) u[j] = b * ((double)vt[j] - r[j]);
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j)
                h[(size_t)i * dv + j] = a * h[(size_t)i * dv + j] + kk[i] * u[j];
        double *ot = p->o + t * p->tok_stride_v;
        for (int j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (int i = 0; i < dk; ++i) acc += h[(size_t)i * dv + j] * qq[i];
            ot[j] = acc;
        }
    }
    if (p->hT) memcpy(p->hT, h, sizeof(double) * (size_t)dk * dv);
    free(h); free(kk); free(qq); free(r); free(u);
}

/*
 * Chunked mode [P1 "Algorithm Modes": parallel inside a chunk, sequential
 * across chunks], in the WY / UT-transform form that the TileOPs DeltaNet
 * pipeline names (prepare_wy_repr -> (Aw, Au) -> w, u).  The form below is
 * derived from the recurrence above; for a chunk of n tokens starting from
 * state S, with G_t the inclusive in-chunk sum of decay, gamma_t = exp(G_t),
 * gamma_0 := 1 and "prev(t)" = t-1:
 *
 *   L[t][s] = beta_t (k_t . k_s) exp(G_{t-1} - G_s)             for s < t
 *   T       = (I + L)^{-1}                      (unit lower triangular)
 *   W       = T diag(beta_t exp(G_{t-1})) K      [n, dk]
 *   U0      = T diag(beta_t) V                   [n, dv]
 *   U       = U0 - W S                           (the chunk's delta terms u_t)
 *   Aqk[t][s] = (q_t . k_s) exp(G_t - G_s)                      for s <= t
 *   O       = diag(gamma_t) Q S + Aqk U
 *   S_next  = gamma_n S + sum_s exp(G_n - G_s) k_s u_s^T
 *
 * (k, q here are the normalised / scaled rows.)  Every exponent is a
 * difference G_a - G_b with a >= b.  T is formed explicitly by forward
 * substitution, one column at a time.
 */
static void chunked_problem(const oracle_problem *p, const oracle_opts *op)
{
    const int dk = p->dk, dv = p->dv, C = op->chunk;
    double *S = (double *)calloc((size_t)dk * dv, sizeof(double));
    double *K = (double *)malloc(sizeof(double) * (size_t)C * dk);
    double *Q = (double *)malloc(sizeof(double) * (size_t)C * dk);
    double *V = (double *)malloc(sizeof(double) * (size_t)C * dv);
    double *bt = (double *)malloc(sizeof(double) * C);
    double *G = (double *)malloc(sizeof(double) * C);
    double *Gp = (double *)malloc(sizeof(double) * C);
    double *L = (double *)calloc((size_t)C * C, sizeof(double));
    double *Tm = (double *)calloc((size_t)C * C, sizeof(double));
    double *Aqk = (double *)calloc((size_t)C * C, sizeof(double));
    double *W = (double *)malloc(sizeof(double) * (size_t)C * dk);
    double *U0 = (double *)malloc(sizeof(double) * (size_t)C * dv);
    double *U = (double *)malloc(sizeof(double) * (size_t)C * dv);
    double *Sn = (double *)malloc(sizeof(double) * (size_t)dk * dv);
    if (p->h0) memcpy(S, p->h0, sizeof(double) * (size_t)dk * dv);

    for (int c0 = 0; c0 < p->T; c0 += C) {
        const int n = (p->T - c0 < C) ? (p->T - c0) : C;
        /* rows of the chunk */
        double run = 0.0;
        for (int t = 0; t < n; ++t) {
            const int tt = c0 + t;
            load_row(p->k + tt * p->tok_stride_qk, dk, op->use_l2, 1.0, K + (size_t)t * dk);
            load_row(p->q + tt * p->tok_stride_qk, dk, op->use_l2, op->scale, Q + (size_t)t * dk);
            for (int j = 0; j < dv; ++j) V[(size_t)t * dv + j] = (double)p->v[tt * p->tok_stride_v + j];
            bt[t] = (double)p->beta[tt * p->tok_stride_g];
            Gp[t] = run;
            run += p->decay ? (double)p->decay[tt * p->tok_stride_g] : 0.0;
            G[t] = run;
        }
        /* L (strictly lower) and Aqk (lower, diagonal included) */
        for (int t = 0; t < n; ++t)
            for (int s = 0; s < n; ++s) {
                double kk = 0.0, qk = 0.0;
                for (int i = 0; i < dk; ++i) {
                    kk += K[(size_t)t * dk + i] * K[(size_t)s * dk + i];
                    qk += Q[(size_t)t * dk + i] * K[(size_t)s * dk + i];
                }
                L[(size_t)t * C + s] = (s < t) ? bt[t] * kk * exp(Gp[t] - G[s]) : 0.0;
                Aqk[(size_t)t * C + s] = (s <= t) ? qk * exp(G[t] - G[s]) : 0.0;
            }
        /* T = (I + L)^{-1}: column j solves (I + L) x = e_j by forward substitution */
        for (int j = 0; j < n; ++j)
            for (int t = 0; t < n; ++t) {
                double x = (t == j) ? 1.0 : 0.0;
                for (int s = 0; s < t; ++s) x -= L[(size_t)t * C + s] * Tm[(size_t)s * C + j];
                Tm[(size_t)t * C + j] = x;
            }
        /* W and U0 */
        for (int t = 0; t < n; ++t) {
            for (int i = 0; i < dk; ++i) {
                double acc = 0.0;
                for (int s = 0; s < n; ++s)
                    acc += Tm[(size_t)t * C + s] * bt[s] * exp(Gp[s]) * K[(size_t)s * dk + i];
                W[(size_t)t * dk + i] = acc;
            }
            for (int j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (int s = 0; s < n; ++s) acc += Tm[(size_t)t * C + s] * bt[s] * V[(size_t)s * dv + j];
                U0[(size_t)t * dv + j] = acc;
            }
        }
        /* U = U0 - W S */
        for (int t = 0; t < n; ++t)
            for (int j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (int i = 0; i < dk; ++i) acc += W[(size_t)t * dk + i] * S[(size_t)i * dv + j];
                U[(size_t)t * dv + j] = U0[(size_t)t * dv + j] - acc;
            }
        /* O = diag(gamma) Q S + Aqk U */
        for (int t = 0; t < n; ++t) {
            double *ot = p->o + (c0 + t) * p->tok_stride_v;
            for (int j = 0; j < dv; ++j) {
                double qs = 0.0, au = 0.0;
                for (int i = 0; i < dk; ++i) qs += Q[(size_t)t * dk + i] * S[(size_t)i * dv + j];
                for (int s = 0; s <= t; ++s) au += Aqk[(size_t)t * C + s] * U[(size_t)s * dv + j];
                ot[j] = exp(G[t]) * qs + au;
            }
        }
        /* S_next = gamma_n S + sum_s exp(G_n - G_s) k_s u_s^T */
        const double Gn = G[n - 1];
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j) {
                double acc = exp(Gn) * S[(size_t)i * dv + j];
                for (int s = 0; s < n; ++s)
                    acc += exp(Gn - G[s]) * K[(size_t)s * dk + i] * U[(size_t)s * dv + j];
                Sn[(size_t)i * dv + j] = acc;
            }
        memcpy(S, Sn, sizeof(double) * (size_t)dk * dv);
    }
    if (p->hT) memcpy(p->hT, S, sizeof(double) * (size_t)dk * dv);
    free(S); free(K); free(Q); free(V); free(bt); free(G); free(Gp); free(L);
    free(Tm); free(Aqk); free(W); free(U0); free(U); free(Sn);
}

/* ---------------------------------------------------------------------- */
/*
 * Per-key-channel decay [P3 KDAFwdOp, GLARecurrentFwdOp; P4].  The scalar
 * retention exp(decay_t) of [P1] becomes the diagonal D_t = diag(exp(g_t)),
 * g_t the dk-vector of log decays of token t: row i of the [dk,dv] memory
 * (key channel i) is scaled by exp(g_t[i]).  Where the delta term reads the
 * memory is taken from a flag:
 *   decayed_read = 0 (the order printed in [P1]):
 *       u_t = beta_t (v_t - h_{t-1}^T k_t),          h_t = D_t h_{t-1} + k_t u_t^T
 *   decayed_read = 1 (the gated delta rule that [P3] names):
 *       u_t = beta_t (v_t - (D_t h_{t-1})^T k_t),    h_t = D_t h_{t-1} + k_t u_t^T
 * and o_t = h_t^T (scale q_t) in both.  With every channel sharing one value,
 * decayed_read = 0 is the scalar recurrence above.  g NULL means zeros.
 */
static void scan_problem_gk(const oracle_problem *p, const oracle_opts *op)
{
    const int dk = p->dk, dv = p->dv;
    double *h = (double *)calloc((size_t)dk * dv, sizeof(double));
    double *kk = (double *)malloc(sizeof(double) * dk);
    double *qq = (double *)malloc(sizeof(double) * dk);
    double *a = (double *)malloc(sizeof(double) * dk);
    double *r = (double *)malloc(sizeof(double) * dv);
    double *u = (double *)malloc(sizeof(double) * dv);
    if (p->h0) memcpy(h, p->h0, sizeof(double) * (size_t)dk * dv);

    for (int t = 0; t < p->T; ++t) {
        load_row(p->k + t * p->tok_stride_qk, dk, op->use_l2, 1.0, kk);
        load_row(p->q + t * p->tok_stride_qk, dk, op->use_l2, op->scale, qq);
        const float *vt = p->v + t * p->tok_stride_v;
        const double b = (double)p->beta[t * p->tok_stride_g];
        for (int i = 0; i < dk; ++i)
            a[i] = p->gk ? exp((double)p->gk[t * p->tok_stride_qk + i]) : 1.0;

        /* readout of the memory the delta term sees */
        for (int j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (int i = 0; i < dk; ++i)
                acc += (op->decayed_read ? a[i] : 1.0) * h[(size_t)i * dv + j] * kk[i];
            r[j] = acc;
        }
        for (int j = 0; j < dv; ++j) u[j] = b * ((double)vt[j] - r[j]);
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j)
                h[(size_t)i * dv + j] = a[i] * h[(size_t)i * dv + j] + kk[i] * u[j];
        double *ot = p->o + t * p->tok_stride_v;
        for (int j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (int i = 0; i < dk; ++i) acc += h[(size_t)i * dv + j] * qq[i];
            ot[j] = acc;
        }
    }
    if (p->hT) memcpy(p->hT, h, sizeof(double) * (size_t)dk * dv);
    free(h); free(kk); free(qq); free(a); free(r); free(u);
}

/*
 * Chunked form of the per-channel recurrence, derived from it the same way as
 * the scalar chunked form above, with the cumulative decays now dk-vectors:
 * G_t[c] = sum of g_s[c] over the chunk's tokens s <= t, P_t[c] = G_{t-1}[c]
 * (0 for the first token), and R_t = G_t when the delta reads the decayed
 * memory, R_t = P_t otherwise.  For a chunk of n tokens starting from S:
 *
 *   L[t][s]   = beta_t sum_c k_t[c] k_s[c] exp(R_t[c] - G_s[c])       s < t
 *   T         = (I + L)^{-1}
 *   W         = T diag(beta) [k_t * exp(R_t)]_t                         [n, dk]
 *   U         = T diag(beta) V - W S
 *   Aqk[t][s] = sum_c q_t[c] k_s[c] exp(G_t[c] - G_s[c])               s <= t
 *   O         = [q_t * exp(G_t)]_t S + Aqk U
 *   S_next    = diag(exp(G_n)) S + sum_s [k_s * exp(G_n - G_s)] u_s^T
 *
 * ("*" is the elementwise product.)  Every exponent is a difference G_a - G_b
 * (or R_a - G_b) with a later index first, so it is <= 0 when g <= 0.  The
 * per-channel factors are kept inside the sums over c exactly as written: no
 * factorisation, no sub-chunk split.
 */
static void chunked_problem_gk(const oracle_problem *p, const oracle_opts *op)
{
    const int dk = p->dk, dv = p->dv, C = op->chunk;
    double *S = (double *)calloc((size_t)dk * dv, sizeof(double));
    double *K = (double *)malloc(sizeof(double) * (size_t)C * dk);
    double *Q = (double *)malloc(sizeof(double) * (size_t)C * dk);
    double *V = (double *)malloc(sizeof(double) * (size_t)C * dv);
    double *bt = (double *)malloc(sizeof(double) * C);
    double *G = (double *)malloc(sizeof(double) * (size_t)C * dk);
    double *R = (double *)malloc(sizeof(double) * (size_t)C * dk);
    double *L = (double *)calloc((size_t)C * C, sizeof(double));
    double *Tm = (double *)calloc((size_t)C * C, sizeof(double));
    double *Aqk = (double *)calloc((size_t)C * C, sizeof(double));
    double *W = (double *)malloc(sizeof(double) * (size_t)C * dk);
    double *U = (double *)malloc(sizeof(double) * (size_t)C * dv);
    double *Sn = (double *)malloc(sizeof(double) * (size_t)dk * dv);
    double *run = (double *)malloc(sizeof(double) * dk);
    if (p->h0) memcpy(S, p->h0, sizeof(double) * (size_t)dk * dv);

    for (int c0 = 0; c0 < p->T; c0 += C) {
        const int n = (p->T - c0 < C) ? (p->T - c0) : C;
        for (int c = 0; c < dk; ++c) run[c] = 0.0;
        for (int t = 0; t < n; ++t) {
            const int tt = c0 + t;
            load_row(p->k + tt * p->tok_stride_qk, dk, op->use_l2, 1.0, K + (size_t)t * dk);
            load_row(p->q + tt * p->tok_stride_qk, dk, op->use_l2, op->scale, Q + (size_t)t * dk);
            for (int j = 0; j < dv; ++j) V[(size_t)t * dv + j] = (double)p->v[tt * p->tok_stride_v + j];
            bt[t] = (double)p->beta[tt * p->tok_stride_g];
            for (int c = 0; c < dk; ++c) {
                const double prev = run[c];
                run[c] += p->gk ? (double)p->gk[tt * p->tok_stride_qk + c] : 0.0;
                G[(size_t)t * dk + c] = run[c];
                R[(size_t)t * dk + c] = op->decayed_read ? run[c] : prev;
            }
        }
        for (int t = 0; t < n; ++t)
            for (int s = 0; s < n; ++s) {
                double kk = 0.0, qk = 0.0;
                for (int c = 0; c < dk; ++c) {
                    const double ks = K[(size_t)s * dk + c], Gs = G[(size_t)s * dk + c];
                    if (s < t) kk += K[(size_t)t * dk + c] * ks * exp(R[(size_t)t * dk + c] - Gs);
                    if (s <= t) qk += Q[(size_t)t * dk + c] * ks * exp(G[(size_t)t * dk + c] - Gs);
                }
                L[(size_t)t * C + s] = (s < t) ? bt[t] * kk : 0.0;
                Aqk[(size_t)t * C + s] = (s <= t) ? qk : 0.0;
            }
        /* T = (I + L)^{-1}, column by column (forward substitution) */
        for (int j = 0; j < n; ++j)
            for (int t = 0; t < n; ++t) {
                double x = (t == j) ? 1.0 : 0.0;
                for (int s = 0; s < t; ++s) x -= L[(size_t)t * C + s] * Tm[(size_t)s * C + j];
                Tm[(size_t)t * C + j] = x;
            }
        /* W, then U = T diag(beta) V - W S */
        for (int t = 0; t < n; ++t)
            for (int c = 0; c < dk; ++c) {
                double acc = 0.0;
                for (int s = 0; s < n; ++s)
                    acc += Tm[(size_t)t * C + s] * bt[s] * K[(size_t)s * dk + c] *
                           exp(R[(size_t)s * dk + c]);
                W[(size_t)t * dk + c] = acc;
            }
        for (int t = 0; t < n; ++t)
            for (int j = 0; j < dv; ++j) {
                double tv = 0.0, ws = 0.0;
                for (int s = 0; s < n; ++s) tv += Tm[(size_t)t * C + s] * bt[s] * V[(size_t)s * dv + j];
                for (int c = 0; c < dk; ++c) ws += W[(size_t)t * dk + c] * S[(size_t)c * dv + j];
                U[(size_t)t * dv + j] = tv - ws;
            }
        /* O = [q_t * exp(G_t)] S + Aqk U */
        for (int t = 0; t < n; ++t) {
            double *ot = p->o + (c0 + t) * p->tok_stride_v;
            for (int j = 0; j < dv; ++j) {
                double qs = 0.0, au = 0.0;
                for (int c = 0; c < dk; ++c)
                    qs += Q[(size_t)t * dk + c] * exp(G[(size_t)t * dk + c]) * S[(size_t)c * dv + j];
                for (int s = 0; s <= t; ++s) au += Aqk[(size_t)t * C + s] * U[(size_t)s * dv + j];
                ot[j] = qs + au;
            }
        }
        /* S_next = diag(exp(G_n)) S + sum_s [k_s * exp(G_n - G_s)] u_s^T */
        const double *Gn = G + (size_t)(n - 1) * dk;
        for (int c = 0; c < dk; ++c)
            for (int j = 0; j < dv; ++j) {
                double acc = exp(Gn[c]) * S[(size_t)c * dv + j];
                for (int s = 0; s < n; ++s)
                    acc += exp(Gn[c] - G[(size_t)s * dk + c]) * K[(size_t)s * dk + c] *
                           U[(size_t)s * dv + j];
                Sn[(size_t)c * dv + j] = acc;
            }
        memcpy(S, Sn, sizeof(double) * (size_t)dk * dv);
    }
    if (p->hT) memcpy(p->hT, S, sizeof(double) * (size_t)dk * dv);
    free(S); free(K); free(Q); free(V); free(bt); free(G); free(R); free(L);
    free(Tm); free(Aqk); free(W); free(U); free(Sn); free(run);
}

/* ---------------------------------------------------------------------- */
/* Thread pool over independent problems (plain pthreads, static striding). */

typedef struct {
    const oracle_problem *probs;
    int nprob;
    const oracle_opts *opts;
    int tid, nthreads;
} worker_arg;

static void *worker(void *arg)
{
    worker_arg *w = (worker_arg *)arg;
    for (int i = w->tid; i < w->nprob; i += w->nthreads) {
        if (w->opts->per_channel) {
            if (w->opts->mode == 0) scan_problem_gk(&w->probs[i], w->opts);
            else chunked_problem_gk(&w->probs[i], w->opts);
        } else if (w->opts->mode == 0) {
            scan_problem(&w->probs[i], w->opts);
        } else {
            chunked_problem(&w->probs[i], w->opts);
        }
    }
    return NULL;
}

static int run_all(const oracle_problem *probs, int nprob, const oracle_opts *opts, int nthreads)
{
    if (nthreads <= 0) {
        long n = sysconf(_SC_NPROCESSORS_ONLN);
        nthreads = n > 0 ? (int)n : 1;
    }
    if (nthreads > nprob) nthreads = nprob > 0 ? nprob : 1;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * nthreads);
    worker_arg *args = (worker_arg *)malloc(sizeof(worker_arg) * nthreads);
    for (int i = 0; i < nthreads; ++i) {
        args[i].probs = probs; args[i].nprob = nprob; args[i].opts = opts;
        args[i].tid = i; args[i].nthreads = nthreads;
        if (i > 0) pthread_create(&th[i], NULL, worker, &args[i]);
    }
    worker(&args[0]);
    for (int i = 1; i < nthreads; ++i) pthread_join(th[i], NULL);
    free(th); free(args);
    return nthreads;
}

int kda_oracle_threads(void)
{
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

/*
 * Equal-length batch [P1 kda()].  mode 0 = recurrent scan, 1 = chunked form
 * with chunk size `chunk`.  scale <= 0 selects dk^-0.5 [P1 "Parameters"].
 * bh_list (pairs b*H+h) restricts the work to those heads when not NULL;
 * outputs of other heads are left untouched.  Returns the thread count used,
 * or a negative value on bad arguments.
 */
int kda_oracle_forward(const float *q, const float *k, const float *v,
                       const float *beta, const float *decay, const double *h0,
                       double *o, double *hT,
                       int B, int T, int H, int dk, int dv,
                       double scale, int use_l2, int mode, int chunk,
                       const int *bh_list, int n_bh, int nthreads)
{
    if (B < 0 || T < 0 || H <= 0 || dk <= 0 || dv <= 0) return -1;
    if (mode == 1 && chunk <= 0) return -2;
    oracle_opts op = { mode, chunk, scale > 0.0 ? scale : 1.0 / sqrt((double)dk), use_l2, 0, 0 };
    int nprob = bh_list ? n_bh : B * H;
    oracle_problem *pr = (oracle_problem *)malloc(sizeof(oracle_problem) * (nprob > 0 ? nprob : 1));
    for (int i = 0; i < nprob; ++i) {
        int bh = bh_list ? bh_list[i] : i;
        if (bh < 0 || bh >= B * H) { free(pr); return -3; }
        int b = bh / H, h = bh % H;
        oracle_problem *p = &pr[i];
        p->q = q + ((size_t)b * T * H + h) * dk;
        p->k = k + ((size_t)b * T * H + h) * dk;
        p->v = v + ((size_t)b * T * H + h) * dv;
        p->beta = beta + (size_t)b * T * H + h;
        p->decay = decay ? decay + (size_t)b * T * H + h : NULL;
        p->gk = NULL;
        p->tok_stride_qk = (long)H * dk;
        p->tok_stride_v = (long)H * dv;
        p->tok_stride_g = H;
        p->h0 = h0 ? h0 + (size_t)bh * dk * dv : NULL;
        p->o = o + ((size_t)b * T * H + h) * dv;
        p->hT = hT ? hT + (size_t)bh * dk * dv : NULL;
        p->T = T; p->dk = dk; p->dv = dv;
    }
    int used = run_all(pr, nprob, &op, nthreads);
    free(pr);
    return used;
}

/*
 * Packed variable-length batch [P2 DeltaNetFwdOp: cu_seqlens, B == 1, one
 * state per sequence].  Tokens of sequence n are rows cu_seqlens[n] ..
 * cu_seqlens[n+1]-1 of the [total, H, D] token arrays; state n is
 * h0/hT[n, h].  Each sequence runs the same scan (or chunked form) from its
 * own initial state.  n_h_list restricts to pairs n*H+h when not NULL.
 */
int kda_oracle_varlen(const float *q, const float *k, const float *v,
                      const float *beta, const float *decay, const double *h0,
                      double *o, double *hT,
                      const int *cu_seqlens, int N, int H, int dk, int dv,
                      double scale, int use_l2, int mode, int chunk,
                      const int *nh_list, int n_nh, int nthreads)
{
    if (N < 0 || H <= 0 || dk <= 0 || dv <= 0) return -1;
    if (mode == 1 && chunk <= 0) return -2;
    for (int n = 0; n < N; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n]) return -4;
    oracle_opts op = { mode, chunk, scale > 0.0 ? scale : 1.0 / sqrt((double)dk), use_l2, 0, 0 };
    int nprob = nh_list ? n_nh : N * H;
    oracle_problem *pr = (oracle_problem *)malloc(sizeof(oracle_problem) * (nprob > 0 ? nprob : 1));
    for (int i = 0; i < nprob; ++i) {
        int nh = nh_list ? nh_list[i] : i;
        if (nh < 0 || nh >= N * H) { free(pr); return -3; }
        int n = nh / H, h = nh % H;
        size_t t0 = (size_t)cu_seqlens[n];
        oracle_problem *p = &pr[i];
        p->q = q + (t0 * H + h) * dk;
        p->k = k + (t0 * H + h) * dk;
        p->v = v + (t0 * H + h) * dv;
        p->beta = beta + t0 * H + h;
        p->decay = decay ? decay + t0 * H + h : NULL;
        p->gk = NULL;
        p->tok_stride_qk = (long)H * dk;
        p->tok_stride_v = (long)H * dv;
        p->tok_stride_g = H;
        p->h0 = h0 ? h0 + (size_t)nh * dk * dv : NULL;
        p->o = o + (t0 * H + h) * dv;
        p->hT = hT ? hT + (size_t)nh * dk * dv : NULL;
        p->T = cu_seqlens[n + 1] - cu_seqlens[n]; p->dk = dk; p->dv = dv;
    }
    int used = run_all(pr, nprob, &op, nthreads);
    free(pr);
    return used;
}

/*
 * Per-key-channel decay [P3 KDAFwdOp], equal-length (cu_seqlens NULL: N
 * sequences of T tokens, token arrays [N,T,H,.]) or packed (cu_seqlens [N+1]:
 * token arrays [1,total,H,.], one state per sequence).  g is [rows,H,dk]
 * float32 or NULL (no decay).  decayed_read selects where the delta term reads
 * the memory (see scan_problem_gk).  mode 0 = recurrent scan, 1 = chunked
 * form.  list (flat n*H+h) restricts the work when not NULL.
 */
int kda_oracle_gk(const float *q, const float *k, const float *v,
                  const float *beta, const float *g, const double *h0,
                  double *o, double *hT, const int *cu_seqlens,
                  int N, int T, int H, int dk, int dv,
                  double scale, int use_l2, int decayed_read, int mode, int chunk,
                  const int *list, int n_list, int nthreads)
{
    if (N < 0 || T < 0 || H <= 0 || dk <= 0 || dv <= 0) return -1;
    if (mode == 1 && chunk <= 0) return -2;
    if (cu_seqlens)
        for (int n = 0; n < N; ++n)
            if (cu_seqlens[n + 1] < cu_seqlens[n]) return -4;
    oracle_opts op = { mode, chunk, scale > 0.0 ? scale : 1.0 / sqrt((double)dk), use_l2,
                       1, decayed_read ? 1 : 0 };
    int nprob = list ? n_list : N * H;
    oracle_problem *pr = (oracle_problem *)malloc(sizeof(oracle_problem) * (nprob > 0 ? nprob : 1));
    for (int i = 0; i < nprob; ++i) {
        int nh = list ? list[i] : i;
        if (nh < 0 || nh >= N * H) { free(pr); return -3; }
        int n = nh / H, h = nh % H;
        size_t t0 = cu_seqlens ? (size_t)cu_seqlens[n] : (size_t)n * T;
        oracle_problem *p = &pr[i];
        p->q = q + (t0 * H + h) * dk;
        p->k = k + (t0 * H + h) * dk;
        p->v = v + (t0 * H + h) * dv;
        p->beta = beta + t0 * H + h;
        p->decay = NULL;
        p->gk = g ? g + (t0 * H + h) * dk : NULL;
        p->tok_stride_qk = (long)H * dk;
        p->tok_stride_v = (long)H * dv;
        p->tok_stride_g = H;
        p->h0 = h0 ? h0 + (size_t)nh * dk * dv : NULL;
        p->o = o + (t0 * H + h) * dv;
        p->hT = hT ? hT + (size_t)nh * dk * dv : NULL;
        p->T = cu_seqlens ? cu_seqlens[n + 1] - cu_seqlens[n] : T;
        p->dk = dk; p->dv = dv;
    }
    int used = run_all(pr, nprob, &op, nthreads);
    free(pr);
    return used;
}

/*
 * [P1'] kda_decay(): decay = -exp(A_log[h]) * softplus(gate + dt_bias), with
 * softplus(x) = log(1 + exp(x)).  gate is [rows, H, K] (K = 1 for one decay per
 * head, K = dk for one per key channel), A_log [H], dt_bias [H, K] or NULL (zeros).
 * Written in double; out has gate's layout.
 */
void kda_oracle_gate_decay(const float *gate, const float *A_log, const float *dt_bias,
                           double *out, long rows, int H, int K)
{
    for (long r = 0; r < rows; ++r)
        for (int h = 0; h < H; ++h)
            for (int c = 0; c < K; ++c) {
                const size_t i = ((size_t)r * H + h) * K + c;
                const double x = (double)gate[i] + (dt_bias ? (double)dt_bias[(size_t)h * K + c] : 0.0);
                const double sp = x > 700.0 ? x : log1p(exp(x));
                out[i] = -exp((double)A_log[h]) * sp;
            }
}

/* [P3'] beta = sigmoid(x) = 1 / (1 + exp(-x)), or twice that with allow_neg_eigval. */
void kda_oracle_beta(const float *x, double *out, long n, int allow_neg_eigval)
{
    for (long i = 0; i < n; ++i) {
        const double s = 1.0 / (1.0 + exp(-(double)x[i]));
        out[i] = allow_neg_eigval ? 2.0 * s : s;
    }
}
