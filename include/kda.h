/*
 * kda.h -- C ABI of the GB300 (sm_103a) delta-rule linear-attention forward.
 *
 * What is computed (ejkernel "kernels._xla.kernel_delta_attention._interface",
 * kda(), "The core recurrence"), per batch entry b and head h, with the memory
 * h_t a [dk, dv] matrix:
 *
 *     k^_t = l2(k_t),  q~_t = scale * l2(q_t)          (l2 only if use_qk_l2norm)
 *     u_t  = beta_t * (v_t - h_{t-1}^T k^_t)
 *     h_t  = exp(decay_t) * h_{t-1} + k^_t u_t^T
 *     o_t  = h_t^T q~_t
 *
 * h_0 = initial_state (zeros when NULL); final_state = h_T.  scale <= 0 selects
 * dk^-0.5 (kda() "Parameters": softmax_scale).  decay NULL means zeros, i.e. no
 * decay (kda() "Parameters": decay).  l2(x) = x / max(||x||, 1e-12).
 *
 * Layouts (all row-major and contiguous, element counts not bytes):
 *   q, k          [B, T, H, dk]    dtype given by `dtype`
 *   v, o          [B, T, H, dv]    dtype given by `dtype` (o has the dtype of q/v)
 *   beta, decay   [B, T, H]        float32
 *   state         [B, H, dk, dv]   float32, key-major (TileOPs "Linear Attention
 *                                   Operators", GDNFwdOp: key-major fp32 state)
 * Packed variable-length calls use B == 1, T == total tokens, and one state per
 * sequence, [N, H, dk, dv] (TileOPs DeltaNetFwdOp: cu_seqlens).
 *
 * Ownership: the caller owns every buffer, including the workspace; the library
 * allocates no device memory and keeps no state between calls.  All pointers
 * passed to the compute entry points are DEVICE pointers (cudaMalloc'd or
 * equivalent) unless named *_host.
 *
 * Asynchrony and errors: every compute call only enqueues work on `stream`
 * (a cudaStream_t; NULL = the legacy default stream) and returns.  Argument
 * errors are detected on the host and returned before anything is enqueued.
 * A launch failure returns KDA_ERR_CUDA.  No call aborts, throws or traps.
 * A kernel whose bounded wait runs out records KDA_ERR_DEVICE_TIMEOUT in the
 * workspace header, read back by kda_query_device_error().
 *
 * Supported shapes: dk, dv in {32, 64, 128}; chunk_size in {16, 32, 64}.
 * The bf16 chunked prefill runs on the tcgen05 tensor-core path when
 * dk == dv in {64, 128} and chunk_size == 64; every other supported shape runs
 * on the fp32 CUDA-core chunk path.  Anything else returns KDA_ERR_UNSUPPORTED.
 * The tensor-core path is one cooperative kernel launch (it occupies every SM until it
 * ends); its workspace holds a fixed ring of chunk maps per chain (at most 40 chains), so
 * it does not grow with the sequence length.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, declared here so that this header needs no CUDA header. */
struct CUstream_st;
typedef struct CUstream_st *kda_stream_t;

typedef enum kda_status {
    KDA_OK = 0,
    KDA_ERR_NULL = 1,           /* a required pointer is NULL                         */
    KDA_ERR_SHAPE = 2,          /* a size is negative/zero where it must be positive   */
    KDA_ERR_DTYPE = 3,          /* unknown kda_dtype                                  */
    KDA_ERR_UNSUPPORTED = 4,    /* valid but not served (head dims, chunk size)        */
    KDA_ERR_ALIGN = 5,          /* a pointer is not 16-byte aligned                    */
    KDA_ERR_WORKSPACE = 6,      /* workspace NULL or smaller than the query returned   */
    KDA_ERR_CUDA = 7,           /* a CUDA launch or runtime call failed                */
    KDA_ERR_DEVICE_TIMEOUT = 8, /* a kernel's bounded wait ran out (see above)         */
    KDA_ERR_INDEX = 9           /* cu_seqlens not monotone / not ending at total_T     */
} kda_status;

/* Element type of q, k, v and o.  beta, decay and the state are always float32
 * (TileOPs DeltaNetFwdOp: the recurrent state is FP32). */
typedef enum kda_dtype { KDA_F32 = 0, KDA_BF16 = 1 } kda_dtype;

/*
 * Options of the *_ex and kda_gk_* entry points: the decay placement, and the gate and
 * beta prologues done inside the kernels (TileOPs "Linear Attention Operators", GDNFwdOp /
 * KDAFwdOp: use_gate_in_kernel, use_beta_sigmoid_in_kernel, allow_neg_eigval; ejkernel
 * kda_decay()).  A NULL pointer or a zeroed struct is the plain recurrence above.
 */
typedef struct kda_options {
    int decayed_read;       /* 0: the delta term reads h_{t-1} (the order printed above);
                               1: it reads the decayed memory, exp(decay_t) h_{t-1} (per key
                               channel: diag(exp g_t) h_{t-1}) -- the gated delta rule          */
    const float *A_log;     /* [H], device.  Non-NULL: decay (or g) holds the raw gate and the
                               kernels use  -exp(A_log[h]) * softplus(gate + dt_bias)  (kda_decay) */
    const float *dt_bias;   /* [H] for a per-head decay, [H, dk] for g; device; NULL = zeros     */
    int beta_sigmoid;       /* nonzero: beta holds logits and the kernels use sigmoid(beta) ...  */
    int allow_neg_eigval;   /* ... or 2 sigmoid(beta) when this is nonzero as well               */
    int v_heads_per_qk_head;/* m >= 2: grouped value heads (GDNFwdOp / KDAFwdOp: v, beta, g and
                               the output use HV = m * H heads).  The H argument counts the q/k
                               heads; v, o, beta, decay, g, A_log, dt_bias and the state have
                               HV heads, and value head hv reads q/k head hv / m.  0 or 1: none.
                               Workspace queries take the value-head count HV.                 */
    int state_v_first;      /* nonzero: initial_state / final_state / the decode state are
                               value-major [.., HV, dv, dk] (GDNFwdOp / KDAFwdOp state_v_first)
                               instead of key-major [.., HV, dk, dv]                           */
} kda_options;

/* Human-readable name of a status code (static storage, never NULL). */
const char *kda_status_string(kda_status s);

/* Library version, (major << 16) | minor. */
int kda_version(void);

/*
 * Workspace bytes that kda_chunk_fwd needs for these sizes (host-only query, no
 * CUDA call).  Always at least 256 bytes (the header that holds the device error
 * word).  Returns 0 if the sizes are invalid or unsupported.
 */
size_t kda_chunk_fwd_workspace(int B, int T, int H, int dk, int dv, int chunk_size,
                               kda_dtype dtype);

/*
 * Chunked prefill (kda() "Algorithm Modes": chunked -- parallel inside a chunk,
 * sequential across chunks; the chunk-local form is the WY / UT-transform
 * representation that TileOPs DeltaNetChunkFwdOp names prepare_wy_repr -> w, u).
 *
 *   q, k, v, beta        inputs, layouts above; must not be NULL when B*T > 0.
 *   decay                [B,T,H] float32, or NULL for no decay.
 *   initial_state        [B,H,dk,dv] float32, or NULL for zeros.
 *   o                    [B,T,H,dv] output, dtype of q.
 *   final_state          [B,H,dk,dv] float32 output; may alias initial_state
 *                        (the state is read before it is overwritten), or NULL
 *                        when the caller does not want it.
 *   scale                query scale; <= 0 selects dk^-0.5.
 *   chunk_size           16, 32 or 64 (result does not depend on it beyond rounding).
 *   use_qk_l2norm        nonzero: L2-normalise q and k rows (kda() default: True).
 *   ws, ws_bytes         device workspace, at least kda_chunk_fwd_workspace() bytes,
 *                        16-byte aligned; contents need not be initialised.
 * T == 0 is allowed: o is untouched and final_state = initial_state (or zeros).
 */
kda_status kda_chunk_fwd(const void *q, const void *k, const void *v,
                         const float *beta, const float *decay,
                         const float *initial_state, void *o, float *final_state,
                         int B, int T, int H, int dk, int dv, kda_dtype dtype,
                         float scale, int chunk_size, int use_qk_l2norm,
                         void *ws, size_t ws_bytes, kda_stream_t stream);

/*
 * Chunked prefill that allocates nothing and takes no workspace.  The pages have no
 * counterpart: this entry point exists for callers that cannot allocate device memory
 * where they call us -- a plugin inside a framework that owns the memory pool, code on a
 * latency-critical path where cudaMalloc/cudaFree would synchronise the device, or a
 * caller with no spare memory to hand over.
 *
 * Same arguments and results as kda_chunk_fwd without ws/ws_bytes, for the tensor-core
 * shapes only: dtype KDA_BF16, dk == dv in {64, 128}, chunk_size 64 (anything else
 * returns KDA_ERR_UNSUPPORTED).  Its scratch is one 48 MiB array that the library keeps
 * on every GPU that loads it, until the process exits.  The scratch needed is
 * 256 + 256 * ceil(64 C / 256) + 256 * ceil(128 (C + 1) / 256) + 32 C (D+64)^2 bytes for
 * C = min(B*H, 40) chains, at most about 45 MiB (D = 128), whatever B, T and H; a
 * problem whose scratch would not fit would return KDA_ERR_WORKSPACE before anything is
 * enqueued, which no supported problem does.
 *
 * The first call on a device looks the array's device address up (with that device
 * current) and keeps it for the life of the process; make that first call before any
 * stream capture, and do not reset the device (cudaDeviceReset) after it.  Every call
 * shares the one array, so calls that overlap on the GPU (on different streams, or from
 * different threads without ordering) race and corrupt each other's results; order them.
 * A kernel time-out of this entry point is recorded in the array's own header:
 * kda_query_device_error(NULL, stream) reads it (and clears it) on the current device.
 */
kda_status kda_chunk_fwd_noalloc(const void *q, const void *k, const void *v,
                                 const float *beta, const float *decay,
                                 const float *initial_state, void *o, float *final_state,
                                 int B, int T, int H, int dk, int dv, kda_dtype dtype,
                                 float scale, int chunk_size, int use_qk_l2norm,
                                 kda_stream_t stream);

/*
 * Recurrent prefill (kda() "Algorithm Modes": recurrent -- the pure sequential
 * scan; kda(use_chunked=False)).  Same arguments as kda_chunk_fwd without the
 * chunk size; needs no workspace.  One CUDA-core kernel, one token at a time.
 */
kda_status kda_recurrent_fwd(const void *q, const void *k, const void *v,
                             const float *beta, const float *decay,
                             const float *initial_state, void *o, float *final_state,
                             int B, int T, int H, int dk, int dv, kda_dtype dtype,
                             float scale, int use_qk_l2norm, kda_stream_t stream);

/*
 * Single-token decode (kda() "Algorithm Modes": single-step, seq_len == 1 with
 * an initial state; TileOPs DeltaNetRecurrentFwdOp gives the decay-free step
 *   v_new = beta (v - S^T k), o = S^T q + (q.k) v_new, S_new = S + k v_new^T).
 * With alpha = exp(decay) this kernel computes, per (b, h):
 *   r = S^T k^, p = S^T q~, u = beta (v - r), o = alpha p + (k^ . q~) u,
 *   S <- alpha S + k^ u^T           (in place).
 *   q, k  [B,1,H,dk];  v, o [B,1,H,dv];  beta, decay [B,1,H] (decay may be NULL);
 *   state [B,H,dk,dv] float32, read and overwritten in place; must not be NULL.
 * Needs no workspace.  o must not alias any input.
 */
kda_status kda_decode_step(const void *q, const void *k, const void *v,
                           const float *beta, const float *decay, float *state, void *o,
                           int B, int H, int dk, int dv, kda_dtype dtype, float scale,
                           int use_qk_l2norm, kda_stream_t stream);

/* Workspace bytes for kda_varlen_fwd (host-only query).  0 if invalid/unsupported. */
size_t kda_varlen_fwd_workspace(int N, int total_T, int H, int dk, int dv, int chunk_size,
                                kda_dtype dtype);

/*
 * Packed variable-length chunked prefill (TileOPs DeltaNetFwdOp / GDNFwdOp:
 * token tensors with B == 1, cu_seqlens [N+1] marks the sequences, one state per
 * sequence; lengths need not be multiples of the chunk size).
 *   q, k  [1,total_T,H,dk];  v, o [1,total_T,H,dv];  beta, decay [1,total_T,H].
 *   cu_seqlens        device int32 [N+1], cu_seqlens[0] == 0, non-decreasing,
 *                     cu_seqlens[N] == total_T.
 *   cu_seqlens_host   optional host copy of the same array; when given, it is
 *                     validated (KDA_ERR_INDEX) and used to size the launch;
 *                     when NULL the device array is trusted as documented.
 *   initial_state     [N,H,dk,dv] float32 or NULL (zeros);
 *   final_state       [N,H,dk,dv] float32 or NULL; may alias initial_state.
 * No chunk crosses a sequence boundary; a sequence of length 0 gets
 * final_state = initial_state.
 */
kda_status kda_varlen_fwd(const void *q, const void *k, const void *v,
                          const float *beta, const float *decay,
                          const int *cu_seqlens, const int *cu_seqlens_host,
                          int N, int total_T, int H, int dk, int dv,
                          const float *initial_state, void *o, float *final_state,
                          kda_dtype dtype, float scale, int chunk_size, int use_qk_l2norm,
                          void *ws, size_t ws_bytes, kda_stream_t stream);

/*
 * Per-key-channel decay: Kimi Delta Attention (TileOPs "Linear Attention Operators",
 * KDAFwdOp: the gated delta rule with one log-space decay per key channel, g [B,T,H,K];
 * GLARecurrentFwdOp writes that retention as diag(exp(gk)) applied to the state).
 * Per (b, h), with D_t = diag(exp(g_t)) scaling row i (key channel i) of the memory:
 *
 *     opt->decayed_read == 0:   u_t = beta_t * (v_t - h_{t-1}^T k^_t)
 *     opt->decayed_read != 0:   u_t = beta_t * (v_t - (D_t h_{t-1})^T k^_t)   (gated delta rule)
 *     h_t = D_t h_{t-1} + k^_t u_t^T,      o_t = h_t^T q~_t
 *
 * k^, q~, scale and use_qk_l2norm as above.  With every channel of g_t equal to decay_t
 * and decayed_read == 0 this is the recurrence at the top of this header; without decay
 * the two placements coincide.  opt (may be NULL) also selects the in-kernel gate
 * (g holds the raw gate; dt_bias is [H, dk]) and beta transforms.
 *   g   [B,T,H,dk] float32, the layout of q and k; NULL means no decay.  16-byte aligned.
 * Every other argument, layout and rule as kda_recurrent_fwd / kda_varlen_fwd /
 * kda_decode_step.  The three *_recurrent_fwd / decode entry points run on CUDA cores,
 * token by token (exact for any decay strength), and need no workspace.
 */
kda_status kda_gk_recurrent_fwd(const void *q, const void *k, const void *v,
                                const float *beta, const float *g,
                                const float *initial_state, void *o, float *final_state,
                                int B, int T, int H, int dk, int dv, kda_dtype dtype,
                                float scale, int use_qk_l2norm, const kda_options *opt,
                                kda_stream_t stream);

/*
 * Chunked prefill with per-key-channel decay: the same results as kda_gk_recurrent_fwd.
 * Arguments, workspace (its size is kda_chunk_fwd_workspace()), errors and device error
 * word as kda_chunk_fwd, plus g and opt as above.  bf16 with dk == dv in {64, 128}
 * and chunk_size 64 runs on the tensor cores: the chunk's per-channel factors
 * exp(G_t[c] - G_s[c]) are split at 16-token sub-blocks (kda-neuron-kernels README: the
 * exact sub-chunk form), and a sub-block whose decay spans more than e^60 in some channel
 * takes its diagonal entries from an exact CUDA-core evaluation, so no decay strength
 * overflows.  Every other supported shape runs the per-channel token-by-token kernel.
 */
kda_status kda_gk_chunk_fwd(const void *q, const void *k, const void *v,
                            const float *beta, const float *g,
                            const float *initial_state, void *o, float *final_state,
                            int B, int T, int H, int dk, int dv, kda_dtype dtype,
                            float scale, int chunk_size, int use_qk_l2norm, const kda_options *opt,
                            void *ws, size_t ws_bytes, kda_stream_t stream);

/* Packed chunked prefill with per-key-channel decay: kda_varlen_fwd's arguments and
 * workspace (kda_varlen_fwd_workspace()) plus g [1,total_T,H,dk] and opt. */
kda_status kda_gk_varlen_fwd(const void *q, const void *k, const void *v,
                             const float *beta, const float *g,
                             const int *cu_seqlens, const int *cu_seqlens_host,
                             int N, int total_T, int H, int dk, int dv,
                             const float *initial_state, void *o, float *final_state,
                             kda_dtype dtype, float scale, int chunk_size, int use_qk_l2norm,
                             const kda_options *opt, void *ws, size_t ws_bytes, kda_stream_t stream);

/* Packed form: q, k, g [1,total_T,H,dk]; v, o [1,total_T,H,dv]; beta [1,total_T,H];
 * cu_seqlens / cu_seqlens_host and the [N,H,dk,dv] states as kda_varlen_fwd. */
kda_status kda_gk_varlen_recurrent_fwd(const void *q, const void *k, const void *v,
                                       const float *beta, const float *g,
                                       const int *cu_seqlens, const int *cu_seqlens_host,
                                       int N, int total_T, int H, int dk, int dv,
                                       const float *initial_state, void *o, float *final_state,
                                       kda_dtype dtype, float scale, int use_qk_l2norm,
                                       const kda_options *opt, kda_stream_t stream);

/* One token per sequence: q, k, g [B,1,H,dk]; the state is updated in place. */
kda_status kda_gk_decode_step(const void *q, const void *k, const void *v,
                              const float *beta, const float *g, float *state, void *o,
                              int B, int H, int dk, int dv, kda_dtype dtype, float scale,
                              int use_qk_l2norm, const kda_options *opt, kda_stream_t stream);

/*
 * Gradients of the per-key-channel recurrence above (the backward of the training mode; the
 * kda-neuron-kernels README's kda_chunk_step_exact_bwd returns the same set): given
 * d_o = dL/do [B,T,H,dv] (dtype of q) and dfinal_state = dL/dfinal_state [B,H,dk,dv] fp32
 * (NULL = zero), writes the fp32 gradients
 *     dq, dk [B,T,H,dk];  dv [B,T,H,dv];  dbeta [B,T,H];  dg [B,T,H,dk] (NULL allowed;
 *     zeros when g is NULL);  dinitial_state [B,H,dk,dv] (NULL allowed)
 * with respect to the raw q and k (through the L2 normalisation and the scale), v, beta,
 * g and initial_state.  q, k, v, beta, g, initial_state, scale, use_qk_l2norm, decayed_read
 * as in the forward (equal-length batches, key-major states).  Token by token on CUDA
 * cores: a forward pass stores the state every 32 tokens, the backward pass recomputes each
 * 32-token stretch and walks it in reverse.  ws: at least
 * kda_gk_recurrent_bwd_workspace() bytes, 16-byte aligned.
 */
size_t kda_gk_recurrent_bwd_workspace(int B, int T, int H, int dk, int dv);
kda_status kda_gk_recurrent_bwd(const void *q, const void *k, const void *v,
                                const float *beta, const float *g,
                                const float *initial_state, const void *d_o,
                                const float *dfinal_state, float *dq, float *dk_out,
                                float *dv_out, float *dbeta, float *dg, float *dinitial_state,
                                int B, int T, int H, int dk, int dv, kda_dtype dtype,
                                float scale, int use_qk_l2norm, int decayed_read,
                                void *ws, size_t ws_bytes, kda_stream_t stream);

/*
 * Gradients of the path's own recurrence (one decay per head, decay [B,T,H] as in
 * kda_chunk_fwd; the delta reads h_{t-1}, or exp(decay_t) h_{t-1} with decayed_read): the
 * same as kda_gk_recurrent_bwd with every key channel's decay equal, so that
 *     ddecay [B,T,H] (NULL allowed; zeros when decay is NULL) = the sum over the key
 *     channels of the per-channel dg,
 * and dq, dk, dv, dbeta, dinitial_state as there.  decay may be NULL (no decay).  ws: at
 * least kda_recurrent_bwd_workspace() bytes (the same size as the per-channel backward's),
 * 16-byte aligned.  Errors: as kda_gk_recurrent_bwd; ddecay must be 4-byte aligned.
 */
size_t kda_recurrent_bwd_workspace(int B, int T, int H, int dk, int dv);
kda_status kda_recurrent_bwd(const void *q, const void *k, const void *v,
                             const float *beta, const float *decay,
                             const float *initial_state, const void *d_o,
                             const float *dfinal_state, float *dq, float *dk_out,
                             float *dv_out, float *dbeta, float *ddecay, float *dinitial_state,
                             int B, int T, int H, int dk, int dv, kda_dtype dtype,
                             float scale, int use_qk_l2norm, int decayed_read,
                             void *ws, size_t ws_bytes, kda_stream_t stream);

/*
 * The scalar-decay entry points with options (see kda_options): the same arguments, layouts,
 * workspace and errors as kda_chunk_fwd / kda_varlen_fwd / kda_recurrent_fwd /
 * kda_decode_step, plus `opt` (may be NULL).  A_log and dt_bias must be 4-byte aligned
 * (KDA_ERR_ALIGN); dt_bias without A_log is KDA_ERR_NULL.  With A_log given, decay must
 * not be NULL (it is the gate).
 */
kda_status kda_chunk_fwd_ex(const void *q, const void *k, const void *v,
                            const float *beta, const float *decay,
                            const float *initial_state, void *o, float *final_state,
                            int B, int T, int H, int dk, int dv, kda_dtype dtype,
                            float scale, int chunk_size, int use_qk_l2norm,
                            const kda_options *opt, void *ws, size_t ws_bytes,
                            kda_stream_t stream);
kda_status kda_varlen_fwd_ex(const void *q, const void *k, const void *v,
                             const float *beta, const float *decay,
                             const int *cu_seqlens, const int *cu_seqlens_host,
                             int N, int total_T, int H, int dk, int dv,
                             const float *initial_state, void *o, float *final_state,
                             kda_dtype dtype, float scale, int chunk_size, int use_qk_l2norm,
                             const kda_options *opt, void *ws, size_t ws_bytes,
                             kda_stream_t stream);
kda_status kda_recurrent_fwd_ex(const void *q, const void *k, const void *v,
                                const float *beta, const float *decay,
                                const float *initial_state, void *o, float *final_state,
                                int B, int T, int H, int dk, int dv, kda_dtype dtype,
                                float scale, int use_qk_l2norm, const kda_options *opt,
                                kda_stream_t stream);
kda_status kda_decode_step_ex(const void *q, const void *k, const void *v,
                              const float *beta, const float *decay, float *state, void *o,
                              int B, int H, int dk, int dv, kda_dtype dtype, float scale,
                              int use_qk_l2norm, const kda_options *opt, kda_stream_t stream);

/*
 * The decay from a gate on its own (ejkernel kda_decay()):
 *     decay[r, h, c] = -exp(A_log[h]) * softplus(gate[r, h, c] + dt_bias[h, c])
 * gate, decay [rows, H, K] float32 (K = 1: one decay per head; K = dk: per key channel);
 * A_log [H]; dt_bias [H, K] or NULL (zeros).  Device pointers; decay may alias gate.
 */
kda_status kda_gate_decay(const float *gate, const float *A_log, const float *dt_bias,
                          float *decay, long rows, int H, int K, kda_stream_t stream);

/*
 * Chunked backward on the tensor cores: the same gradients as kda_recurrent_bwd (dq, dk,
 * dv, dbeta, ddecay, dinitial_state of sum(o . d_o) + sum(final_state . dfinal_state)) for
 * the bf16 tensor-core shapes (dtype KDA_BF16, dk == dv in {64, 128}; anything else returns
 * KDA_ERR_UNSUPPORTED), computed by chunks of 64 tokens (kda-neuron-kernels README,
 * kda_chunk_step_exact_bwd; TileOPs DeltaNetChunkBwdOp): a forward launch that keeps every
 * chunk's map and state, a reverse walk dS_c = [E_c^T [dS_{c+1}; dO_c]] over the maps
 * (the transposed chunk map) that keeps every chunk's state gradient, and one kernel for
 * the chunk-local gradients of q, k, v, beta and the decay.  Arguments, layouts and errors
 * as kda_recurrent_bwd (equal-length batches, key-major states).  Arithmetic: bf16 maps and
 * state operands on the tensor cores as in the forward (the kept states and state gradients
 * are those bf16 operands), tf32 products with fp32 accumulation for the chunk gradients.
 * ws: at least kda_chunk_bwd_workspace() bytes, 16-byte aligned (it holds every chunk's
 * map and two bf16 states per chunk, ~136 KB per chunk and head at head dim 128, plus a
 * fixed scratch of at most 304 x 368 KB for the gradient kernel).
 */
size_t kda_chunk_bwd_workspace(int B, int T, int H, int dk, int dv);
kda_status kda_chunk_bwd(const void *q, const void *k, const void *v,
                         const float *beta, const float *decay,
                         const float *initial_state, const void *d_o,
                         const float *dfinal_state, float *dq, float *dk_out, float *dv_out,
                         float *dbeta, float *ddecay, float *dinitial_state,
                         int B, int T, int H, int dk, int dv, kda_dtype dtype,
                         float scale, int use_qk_l2norm, int decayed_read,
                         void *ws, size_t ws_bytes, kda_stream_t stream);

/*
 * Chunked backward with per-key-channel decay: the same gradients as kda_gk_recurrent_bwd
 * (dq, dk, dv, dbeta, dg, dinitial_state; TileOPs KDAFwdOp's recurrence, kda-neuron-kernels
 * README kda_chunk_step_exact_bwd) for the bf16 tensor-core shapes (dtype KDA_BF16, dk == dv
 * in {64, 128}; anything else returns KDA_ERR_UNSUPPORTED).  The two walks are those of
 * kda_chunk_bwd: a forward launch that keeps every chunk's map (built with the per-channel
 * factors, as kda_gk_chunk_fwd builds it) and the state entering every chunk, and the
 * reverse walk over the maps, which gives the gradient of the state leaving every chunk and
 * dinitial_state.  With both in hand every 64-token chunk is independent: the gradient
 * kernel walks each (chunk, head, 32 value columns) token by token, recomputing the chunk's
 * states from the kept one, all chunks at once.  Arguments, layouts and errors as
 * kda_gk_recurrent_bwd; g NULL means no decay (dg, if given, is zero-filled).  Arithmetic:
 * the maps, the kept states and state gradients and the recomputed states are bf16 (the
 * precision of the forward's tensor-core operands); every sum is fp32.  ws: at least
 * kda_gk_chunk_bwd_workspace() bytes, 16-byte aligned (every chunk's map and two bf16
 * states per chunk, ~136 KB per chunk and head at head dim 128, plus a fixed scratch of
 * 304 x 512 KB at head dim 128).
 */
size_t kda_gk_chunk_bwd_workspace(int B, int T, int H, int dk, int dv);
kda_status kda_gk_chunk_bwd(const void *q, const void *k, const void *v,
                            const float *beta, const float *g,
                            const float *initial_state, const void *d_o,
                            const float *dfinal_state, float *dq, float *dk_out, float *dv_out,
                            float *dbeta, float *dg, float *dinitial_state,
                            int B, int T, int H, int dk, int dv, kda_dtype dtype,
                            float scale, int use_qk_l2norm, int decayed_read,
                            void *ws, size_t ws_bytes, kda_stream_t stream);

/*
 * Read the device error word that the kernels of the most recent kda_chunk_fwd /
 * kda_varlen_fwd call on `ws` recorded (KDA_OK if none), then clear it.  Each of
 * those calls clears the word on its stream before its kernels run.  ws == NULL reads
 * the built-in array of kda_chunk_fwd_noalloc on the current device instead.
 * Synchronises `stream`; use the stream of that call.
 */
kda_status kda_query_device_error(const void *ws, kda_stream_t stream);

/*
 * Failure-detection probe (diagnostic; the pages have no counterpart).  Enqueues one small
 * kernel that runs the two bounded waits of the tensor-core prefill -- on an mbarrier phase
 * and on a publication flag -- against events that never happen, with a limit of
 * `limit_us` microseconds each (1 .. 2,000,000) instead of the kernels' 2 s.  Each wait
 * gives up, records KDA_ERR_DEVICE_TIMEOUT in the header of `ws` and returns; nothing
 * traps, and the context stays usable.  kda_query_device_error(ws) then returns
 * KDA_ERR_DEVICE_TIMEOUT once.  ws: device workspace of at least 256 bytes, 16-byte
 * aligned (its header only is used).  Returns KDA_ERR_NULL, KDA_ERR_WORKSPACE,
 * KDA_ERR_ALIGN, KDA_ERR_SHAPE (limit out of range) or KDA_ERR_CUDA on a launch failure.
 */
kda_status kda_diag_wait_timeout(void *ws, size_t ws_bytes, unsigned limit_us,
                                 kda_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
