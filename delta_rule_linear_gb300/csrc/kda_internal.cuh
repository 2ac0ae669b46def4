// kda_internal.cuh -- declarations shared by the translation units of libkda.so.
//
// The C ABI (include/kda.h) validates arguments on the host and then calls one of
// the launchers declared here.  Each launcher enqueues its kernels on the given
// stream and returns the launch status.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace kda {

// Element type of q, k, v, o.
enum class DType : int { F32 = 0, BF16 = 1 };

// Workspace header: the first 256 bytes of every workspace.  Kernels with a
// bounded wait record the first failure code in `error` (atomicCAS from 0).
struct WsHeader {
    int error;          // 0 = none; otherwise a kda_status value
    int where;          // kernel-defined location of the failure (diagnostic)
    unsigned probe;     // flag that the failure-detection probe waits on and nobody releases
    int pad[61];
};
static_assert(sizeof(WsHeader) == 256, "workspace header is 256 bytes");

// A batch of independent sequences that share H, dk, dv.  Sequence n covers
// token rows [seq_start(n), seq_start(n) + seq_len(n)) of the flattened
// [rows, H, D] token arrays.  Equal-length batches use cu_seqlens == nullptr and
// sequence n = batch entry b starts at b * T; packed varlen batches read the
// device prefix array cu_seqlens [nseq + 1].
struct SeqBatch {
    const void *q;            // [rows, H, dk]   (Tin)
    const void *k;            // [rows, H, dk]   (Tin)
    const void *v;            // [rows, H, dv]   (Tin)
    const float *beta;        // [rows, H]
    const float *decay;       // [rows, H] or nullptr (zeros)
    const float *gk;          // per-channel decay [rows, H, dk] or nullptr (per_channel only)
    int per_channel;          // 1: the decay is gk, one value per key channel
    int decayed_read;         // the delta term reads the decayed state
    const float *A_log;       // [H] or nullptr: decay / gk hold the raw gate (gate_decay below)
    const float *dt_bias;     // [H] (scalar) or [H, dk] (per channel) or nullptr
    int beta_sig, neg_eig;    // beta holds logits: sigmoid, or 2 sigmoid with neg_eig
    int G;                    // value heads per q/k head (H counts value heads; q/k have H / G)
    int v_first;              // states are value-major [.., dv, dk]
    const float *h0;          // [nseq, H, dk, dv] or nullptr (zeros)
    void *o;                  // [rows, H, dv]   (Tin)
    float *hT;                // [nseq, H, dk, dv] or nullptr
    const int *cu_seqlens;    // device [nseq + 1] or nullptr (equal length)
    int nseq;                 // B (equal length) or N (varlen)
    int T;                    // equal-length T; varlen: max sequence length (launch sizing)
    int H, dk, dv;
    int chunk;
    DType dtype;
    float scale;              // already resolved (> 0)
    int use_l2;
    WsHeader *ws;             // workspace header (device)
    void *ws_body;            // workspace after the header
    size_t ws_body_bytes;
};

struct DecodeArgs {
    const void *q, *k, *v;
    const float *beta, *decay;
    const float *gk;          // per-channel decay [B, H, dk] or nullptr (per_channel only)
    int per_channel, decayed_read;
    const float *A_log, *dt_bias;   // as in SeqBatch
    int beta_sig, neg_eig;
    int G;                          // value heads per q/k head (H counts value heads)
    int v_first;                    // the state is value-major [B, H, dv, dk]
    float *state;
    void *o;
    int B, H, dk, dv;
    DType dtype;
    float scale;
    int use_l2;
};

// Launchers (each returns the cudaGetLastError() status of its launches).
cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t s);
cudaError_t launch_recurrent(const SeqBatch &a, cudaStream_t s);
cudaError_t launch_chunk_simt(const SeqBatch &a, cudaStream_t s);
size_t chunk_simt_smem_bytes(int dk, int dv, int chunk);
// Copies (or zero-fills) final_state from initial_state for empty sequences.
cudaError_t launch_state_passthrough(const SeqBatch &a, cudaStream_t s);

// Tensor-core chunked prefill (bf16, dk == dv in {64, 128}, chunk 64).
bool chunk_tc_supported(int dk, int dv, int chunk, DType dt);
// Workspace bytes after the header: bounded by the chains' E_c rings (independent of the
// sequence length) plus, for packed sequences, the schedule tables.
size_t chunk_tc_scratch_bytes(int nseq, int H, int d, bool varlen);
// varlen: a.T bounds the longest sequence.
cudaError_t launch_chunk_tc(const SeqBatch &a, long total_rows, cudaStream_t s);
// The two walks of the chunked backward (equal-length bf16 batches; one decay per head, or
// per key channel with a.per_channel): a forward launch that keeps every chunk's map and
// writes the bf16 state at every chunk start (fstates [B, H, nc, D, D]; a.o, a.hT may be
// nullptr), then the reverse walk [dS_c; dV_c] = E_c^T [dS_{c+1}; dO_c] writing dv (fp32
// [B, T, H, D], or nullptr: not written), dh0 (or nullptr) and the gradient of the state
// leaving every chunk (bstates, same layout).  a.ws_body: at least chunk_tc_keep_bytes().
size_t chunk_tc_keep_bytes(int B, int H, int T, int d);
cudaError_t launch_chunk_tc_walks(const SeqBatch &a, const void *d_o, const float *dhT, float *dh0, float *dv,
                                  __nv_bfloat16 *fstates, __nv_bfloat16 *bstates, cudaStream_t s);
// Gradients of q, k, beta and the decay per chunk from the two walks' states (chunk_bwd.cu).
struct ChunkBwdArgs {
    const void *q, *k, *v, *d_o;       // bf16 [B, T, H, D]
    const float *beta, *decay;          // [B, T, H]; decay may be nullptr
    const __nv_bfloat16 *fstates, *bstates;   // [B, H, nc, D, D], bf16
    float *dq, *dk, *dv, *dbeta, *ddecay;   // outputs (ddecay may be nullptr)
    int B, T, H, D;
    float scale;
    int use_l2, decayed_read;
    float *scratch;                     // chunk_bwd_scratch_floats(D) per CTA
    int ctas;
};
size_t chunk_bwd_scratch_floats(int D);
int chunk_bwd_ctas(long nchunks);   // persistent CTAs of the gradient kernel
cudaError_t launch_chunk_bwd_grads(const ChunkBwdArgs &a, cudaStream_t s);
// Device address of kda_chunk_fwd_noalloc's built-in scratch array on the current device
// (its first bytes are a workspace header).
cudaError_t noalloc_header(void **out);
// One CTA runs the tensor-core kernels' bounded waits against events that never happen,
// each giving up after limit_ns and recording KDA_ERR_DEVICE_TIMEOUT in the header.
cudaError_t launch_timeout_probe(WsHeader *ws, uint64_t limit_ns, cudaStream_t s);

// Gradients of the per-channel recurrence (token by token; scan_bwd.cu).
struct BwdArgs {
    const void *q, *k, *v, *dout;      // [rows, H, dk | dv] (Tin)
    const float *beta, *g;             // [rows, H], [rows, H, dk] (g may be null)
    const float *decay;                // [rows, H]: one decay per head (used when g is null)
    float *ddecay;                     // its gradient [rows, H] (may be null)
    const float *h0, *dhT;             // [B, H, dk, dv] or null
    float *dq, *dk, *dv, *dbeta, *dg;  // fp32 gradients (dg may be null)
    float *dh0;                        // [B, H, dk, dv] or null
    int B, T, H, dkdim, dvdim;
    DType dtype;
    float scale;
    int use_l2, decayed_read;
    void *ws;                          // gk_bwd_scratch_bytes()
};
size_t gk_bwd_scratch_bytes(int nseq, int T, int H, int dk, int dv);
cudaError_t launch_gk_bwd(const BwdArgs &a, cudaStream_t s);
// The gradient kernels of the per-channel chunked backward (bf16, dk == dv in {64, 128}):
// every 64-token chunk walked token by token on its own, from the state entering it and the
// gradient of the state leaving it (fstates, bstates as launch_chunk_tc_walks writes them),
// then the gradients of the raw q, k.  scratch: gk_chunk_bwd_scratch_bytes(dk) (a.ws unused).
size_t gk_chunk_bwd_scratch_bytes(int dk);
cudaError_t launch_gk_chunk_bwd_grads(const BwdArgs &a, const __nv_bfloat16 *fstates,
                                      const __nv_bfloat16 *bstates, void *scratch, cudaStream_t s);

// L2 normalisation floor: x / max(||x||, kNormEps).
constexpr float kNormEps = 1e-12f;

template <typename T> __device__ __forceinline__ float to_f32(T x);
template <> __device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
    return __bfloat162float(x);
}
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// kda_decay (ejkernel kernel_delta_attention): the log decay from a gate,
// -exp(A_log) * softplus(gate + dt_bias), softplus(x) = log(1 + exp(x)).
// softplus(x) = max(x, 0) + log1p(e^-|x|): no overflow, and the relative accuracy of
// log1p where e^-|x| is small.
__device__ __forceinline__ float gate_decay_a(float gate, float a, float bias) {   // a = exp(A_log)
    const float x = gate + bias;
    return -a * (fmaxf(x, 0.f) + log1pf(__expf(-fabsf(x))));
}
__device__ __forceinline__ float gate_decay(float gate, float a_log, float bias) {
    return gate_decay_a(gate, expf(a_log), bias);
}
// beta from logits (TileOPs GDNFwdOp / KDAFwdOp): sigmoid(x), or 2 sigmoid(x)
__device__ __forceinline__ float beta_of(float x, int sig, int neg) {
    if (!sig) return x;
    const float s = __frcp_rn(1.f + __expf(-x));
    return neg ? 2.f * s : s;
}

// Token row range of sequence n.
__device__ __forceinline__ void seq_range(const SeqBatch &p, int n, long &start, int &len) {
    if (p.cu_seqlens) {
        int a = p.cu_seqlens[n], b = p.cu_seqlens[n + 1];
        start = a;
        len = b - a;
    } else {
        start = (long)n * p.T;
        len = p.T;
    }
}

}  // namespace kda
