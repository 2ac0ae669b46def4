// kda_api.cu -- the C ABI of include/kda.h: argument checks, workspace carving,
// dispatch to the kernels.  Nothing here allocates device memory.
#include <algorithm>
#include <math.h>
#include <string.h>

#include "../../include/kda.h"
#include "kda_internal.cuh"

using namespace kda;

namespace {

constexpr size_t kWsHeader = sizeof(WsHeader);

bool supported_head(int d) { return d == 32 || d == 64 || d == 128; }
bool supported_chunk(int c) { return c == 16 || c == 32 || c == 64; }
bool aligned16(const void *p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void *p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

float resolve_scale(float scale, int dk) { return scale > 0.f ? scale : 1.0f / sqrtf((float)dk); }

// Copies initial_state into final_state (or zero-fills it) for every sequence;
// used when a call has no tokens to process.
__global__ void state_passthrough_kernel(const float *h0, float *hT, size_t count) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < count;
         i += (size_t)gridDim.x * blockDim.x)
        hT[i] = h0 ? h0[i] : 0.f;
}

kda_status check_common(const void *q, const void *k, const void *v, const float *beta,
                        const float *decay, const float *h0, const void *o, const float *hT,
                        long rows, int H, int dk, int dv, kda_dtype dtype) {
    if (dtype != KDA_F32 && dtype != KDA_BF16) return KDA_ERR_DTYPE;
    if (H <= 0 || dk <= 0 || dv <= 0 || rows < 0) return KDA_ERR_SHAPE;
    if (!supported_head(dk) || !supported_head(dv)) return KDA_ERR_UNSUPPORTED;
    if (rows > 0 && (!q || !k || !v || !beta || !o)) return KDA_ERR_NULL;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(h0) ||
        !aligned16(hT) || !aligned4(beta) || !aligned4(decay))
        return KDA_ERR_ALIGN;
    return KDA_OK;
}

kda_status launch_status(cudaError_t e) { return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA; }

// heads of v, o, beta, the decay and the state: H (q/k heads) times the value-head group
int value_heads(int H, const kda_options *opt) {
    const long m = (opt && opt->v_heads_per_qk_head > 1) ? opt->v_heads_per_qk_head : 1;
    return (long)H * m > 0x7fffffffL ? H : (int)((long)H * m);
}

// kda_options -> the batch fields; `gate` is the decay (or g) pointer the gate would replace
kda_status apply_options(const kda_options *opt, const float *gate, SeqBatch &a) {
    if (!opt) return KDA_OK;
    if (!aligned4(opt->A_log) || !aligned4(opt->dt_bias)) return KDA_ERR_ALIGN;
    if (opt->dt_bias && !opt->A_log) return KDA_ERR_NULL;
    if (opt->A_log && !gate) return KDA_ERR_NULL;
    a.decayed_read = opt->decayed_read ? 1 : 0;
    a.A_log = opt->A_log;
    a.dt_bias = opt->dt_bias;
    a.beta_sig = opt->beta_sigmoid ? 1 : 0;
    a.neg_eig = (opt->beta_sigmoid && opt->allow_neg_eigval) ? 1 : 0;
    a.v_first = opt->state_v_first ? 1 : 0;
    if (opt->v_heads_per_qk_head < 0) return KDA_ERR_SHAPE;
    if (opt->v_heads_per_qk_head > 1) {   // a.H (q/k heads on entry) becomes the value-head count
        if ((long)a.H * opt->v_heads_per_qk_head > 0x7fffffffL) return KDA_ERR_SHAPE;
        a.G = opt->v_heads_per_qk_head;
        a.H *= a.G;
    }
    return KDA_OK;
}

__global__ void gate_decay_kernel(const float *gate, const float *A_log, const float *dt_bias,
                                  float *decay, long n, int H, int K) {
    for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x) {
        const int c = (int)(i % K), h = (int)((i / K) % H);
        decay[i] = gate_decay(gate[i], A_log[h], dt_bias ? dt_bias[(size_t)h * K + c] : 0.f);
    }
}

}  // namespace

namespace kda {
cudaError_t launch_state_passthrough(const SeqBatch &a, cudaStream_t s) {
    if (!a.hT) return cudaSuccess;
    const size_t count = (size_t)a.nseq * a.H * a.dk * a.dv;
    if (count == 0) return cudaSuccess;
    if (a.h0 == a.hT) return cudaSuccess;  // aliasing: already in place
    const int grid = (int)((count + 255) / 256 < 4096 ? (count + 255) / 256 : 4096);
    state_passthrough_kernel<<<grid, 256, 0, s>>>(a.h0, a.hT, count);
    return cudaGetLastError();
}
}  // namespace kda

extern "C" {

const char *kda_status_string(kda_status s) {
    switch (s) {
        case KDA_OK: return "ok";
        case KDA_ERR_NULL: return "a required pointer is NULL";
        case KDA_ERR_SHAPE: return "invalid size";
        case KDA_ERR_DTYPE: return "unknown dtype";
        case KDA_ERR_UNSUPPORTED: return "unsupported head dimension or chunk size";
        case KDA_ERR_ALIGN: return "pointer not aligned (16 bytes for tensors, 4 for beta/decay)";
        case KDA_ERR_WORKSPACE: return "workspace missing or too small";
        case KDA_ERR_CUDA: return "CUDA launch or runtime error";
        case KDA_ERR_DEVICE_TIMEOUT: return "a kernel's bounded wait ran out";
        case KDA_ERR_INDEX: return "cu_seqlens invalid (not monotone, or not 0..total_T)";
    }
    return "unknown status";
}

int kda_version(void) { return (0 << 16) | 1; }

static DType to_dtype(kda_dtype d) { return d == KDA_BF16 ? DType::BF16 : DType::F32; }

size_t kda_chunk_fwd_workspace(int B, int T, int H, int dk, int dv, int chunk_size,
                               kda_dtype dtype) {
    if (B < 0 || T < 0 || H <= 0) return 0;
    if (dtype != KDA_F32 && dtype != KDA_BF16) return 0;
    if (!supported_head(dk) || !supported_head(dv) || !supported_chunk(chunk_size)) return 0;
    if (chunk_tc_supported(dk, dv, chunk_size, to_dtype(dtype)) && B > 0 && T > 0)
        return kWsHeader + chunk_tc_scratch_bytes(B, H, dk, false);
    return kWsHeader;
}

size_t kda_varlen_fwd_workspace(int N, int total_T, int H, int dk, int dv, int chunk_size,
                                kda_dtype dtype) {
    if (N < 0 || total_T < 0 || H <= 0) return 0;
    if (dtype != KDA_F32 && dtype != KDA_BF16) return 0;
    if (!supported_head(dk) || !supported_head(dv) || !supported_chunk(chunk_size)) return 0;
    if (chunk_tc_supported(dk, dv, chunk_size, to_dtype(dtype)) && N > 0)
        return kWsHeader + chunk_tc_scratch_bytes(N, H, dk, true);
    return kWsHeader;
}

// total_rows: rows of the token arrays (B*T, or total_T for varlen).
static kda_status run_prefill(SeqBatch &a, bool chunked, long total_rows, cudaStream_t st) {
    if (a.nseq == 0) return KDA_OK;
    if (!a.cu_seqlens && a.T == 0) return launch_status(launch_state_passthrough(a, st));
    cudaError_t e;
    if (!chunked) {
        e = launch_recurrent(a, st);
    } else if (chunk_tc_supported(a.dk, a.dv, a.chunk, a.dtype)) {
        e = launch_chunk_tc(a, total_rows, st);
    } else if (a.per_channel) {
        e = launch_recurrent(a, st);   // the per-channel decay has no CUDA-core chunk kernel
    } else {
        e = launch_chunk_simt(a, st);
    }
    return launch_status(e);
}

kda_status kda_chunk_fwd(const void *q, const void *k, const void *v, const float *beta,
                         const float *decay, const float *initial_state, void *o,
                         float *final_state, int B, int T, int H, int dk, int dv,
                         kda_dtype dtype, float scale, int chunk_size, int use_qk_l2norm,
                         void *ws, size_t ws_bytes, kda_stream_t stream) {
    return kda_chunk_fwd_ex(q, k, v, beta, decay, initial_state, o, final_state, B, T, H, dk, dv,
                            dtype, scale, chunk_size, use_qk_l2norm, nullptr, ws, ws_bytes, stream);
}

kda_status kda_chunk_fwd_ex(const void *q, const void *k, const void *v, const float *beta,
                            const float *decay, const float *initial_state, void *o,
                            float *final_state, int B, int T, int H, int dk, int dv,
                            kda_dtype dtype, float scale, int chunk_size, int use_qk_l2norm,
                            const kda_options *opt, void *ws, size_t ws_bytes, kda_stream_t stream) {
    if (B < 0 || T < 0) return KDA_ERR_SHAPE;
    kda_status c = check_common(q, k, v, beta, decay, initial_state, o, final_state,
                                (long)B * T, H, dk, dv, dtype);
    if (c != KDA_OK) return c;
    if (!supported_chunk(chunk_size)) return KDA_ERR_UNSUPPORTED;
    const size_t need = kda_chunk_fwd_workspace(B, T, value_heads(H, opt), dk, dv, chunk_size, dtype);
    if (!ws || ws_bytes < need) return KDA_ERR_WORKSPACE;
    if (!aligned16(ws)) return KDA_ERR_ALIGN;
    SeqBatch a{};
    a.q = q; a.k = k; a.v = v; a.beta = beta; a.decay = decay; a.h0 = initial_state;
    a.o = o; a.hT = final_state; a.cu_seqlens = nullptr; a.nseq = B; a.T = T; a.H = H;
    a.dk = dk; a.dv = dv; a.chunk = chunk_size;
    a.dtype = dtype == KDA_BF16 ? DType::BF16 : DType::F32;
    a.scale = resolve_scale(scale, dk); a.use_l2 = use_qk_l2norm ? 1 : 0;
    if ((c = apply_options(opt, decay, a)) != KDA_OK) return c;
    a.ws = static_cast<WsHeader *>(ws);
    a.ws_body = static_cast<char *>(ws) + kWsHeader;
    a.ws_body_bytes = ws_bytes - kWsHeader;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(ws, 0, sizeof(int) * 2, st) != cudaSuccess) return KDA_ERR_CUDA;
    return run_prefill(a, true, (long)B * T, st);
}

kda_status kda_recurrent_fwd(const void *q, const void *k, const void *v, const float *beta,
                             const float *decay, const float *initial_state, void *o,
                             float *final_state, int B, int T, int H, int dk, int dv,
                             kda_dtype dtype, float scale, int use_qk_l2norm,
                             kda_stream_t stream) {
    return kda_recurrent_fwd_ex(q, k, v, beta, decay, initial_state, o, final_state, B, T, H, dk,
                                dv, dtype, scale, use_qk_l2norm, nullptr, stream);
}

kda_status kda_recurrent_fwd_ex(const void *q, const void *k, const void *v, const float *beta,
                                const float *decay, const float *initial_state, void *o,
                                float *final_state, int B, int T, int H, int dk, int dv,
                                kda_dtype dtype, float scale, int use_qk_l2norm,
                                const kda_options *opt, kda_stream_t stream) {
    if (B < 0 || T < 0) return KDA_ERR_SHAPE;
    kda_status c = check_common(q, k, v, beta, decay, initial_state, o, final_state,
                                (long)B * T, H, dk, dv, dtype);
    if (c != KDA_OK) return c;
    SeqBatch a{};
    a.q = q; a.k = k; a.v = v; a.beta = beta; a.decay = decay; a.h0 = initial_state;
    a.o = o; a.hT = final_state; a.cu_seqlens = nullptr; a.nseq = B; a.T = T; a.H = H;
    a.dk = dk; a.dv = dv; a.chunk = 0;
    a.dtype = dtype == KDA_BF16 ? DType::BF16 : DType::F32;
    a.scale = resolve_scale(scale, dk); a.use_l2 = use_qk_l2norm ? 1 : 0;
    if ((c = apply_options(opt, decay, a)) != KDA_OK) return c;
    return run_prefill(a, false, (long)B * T, reinterpret_cast<cudaStream_t>(stream));
}

kda_status kda_decode_step(const void *q, const void *k, const void *v, const float *beta,
                           const float *decay, float *state, void *o, int B, int H, int dk,
                           int dv, kda_dtype dtype, float scale, int use_qk_l2norm,
                           kda_stream_t stream) {
    return kda_decode_step_ex(q, k, v, beta, decay, state, o, B, H, dk, dv, dtype, scale,
                              use_qk_l2norm, nullptr, stream);
}

// the decode arguments' option fields, by way of a batch
// (d.H: the q/k heads on entry, the value heads on return)
static kda_status decode_options(const kda_options *opt, const float *gate, DecodeArgs &d) {
    SeqBatch a{};
    a.H = d.H;
    const kda_status c = apply_options(opt, gate, a);
    d.decayed_read = a.decayed_read; d.A_log = a.A_log; d.dt_bias = a.dt_bias;
    d.beta_sig = a.beta_sig; d.neg_eig = a.neg_eig; d.G = a.G; d.H = a.H; d.v_first = a.v_first;
    return c;
}

kda_status kda_decode_step_ex(const void *q, const void *k, const void *v, const float *beta,
                              const float *decay, float *state, void *o, int B, int H, int dk,
                              int dv, kda_dtype dtype, float scale, int use_qk_l2norm,
                              const kda_options *opt, kda_stream_t stream) {
    if (B < 0) return KDA_ERR_SHAPE;
    kda_status c = check_common(q, k, v, beta, decay, state, o, state, B, H, dk, dv, dtype);
    if (c != KDA_OK) return c;
    if (B > 0 && !state) return KDA_ERR_NULL;
    DecodeArgs a{};
    a.H = H;
    if ((c = decode_options(opt, decay, a)) != KDA_OK) return c;
    if (B == 0) return KDA_OK;
    a.q = q; a.k = k; a.v = v; a.beta = beta; a.decay = decay; a.state = state; a.o = o;
    a.B = B; a.dk = dk; a.dv = dv;
    a.dtype = dtype == KDA_BF16 ? DType::BF16 : DType::F32;
    a.scale = resolve_scale(scale, dk); a.use_l2 = use_qk_l2norm ? 1 : 0;
    return launch_status(launch_decode(a, reinterpret_cast<cudaStream_t>(stream)));
}

kda_status kda_varlen_fwd(const void *q, const void *k, const void *v, const float *beta,
                          const float *decay, const int *cu_seqlens, const int *cu_seqlens_host,
                          int N, int total_T, int H, int dk, int dv, const float *initial_state,
                          void *o, float *final_state, kda_dtype dtype, float scale,
                          int chunk_size, int use_qk_l2norm, void *ws, size_t ws_bytes,
                          kda_stream_t stream) {
    return kda_varlen_fwd_ex(q, k, v, beta, decay, cu_seqlens, cu_seqlens_host, N, total_T, H, dk,
                             dv, initial_state, o, final_state, dtype, scale, chunk_size,
                             use_qk_l2norm, nullptr, ws, ws_bytes, stream);
}

kda_status kda_varlen_fwd_ex(const void *q, const void *k, const void *v, const float *beta,
                             const float *decay, const int *cu_seqlens, const int *cu_seqlens_host,
                             int N, int total_T, int H, int dk, int dv, const float *initial_state,
                             void *o, float *final_state, kda_dtype dtype, float scale,
                             int chunk_size, int use_qk_l2norm, const kda_options *opt, void *ws,
                             size_t ws_bytes, kda_stream_t stream) {
    if (N < 0 || total_T < 0) return KDA_ERR_SHAPE;
    kda_status c = check_common(q, k, v, beta, decay, initial_state, o, final_state,
                                total_T, H, dk, dv, dtype);
    if (c != KDA_OK) return c;
    if (!supported_chunk(chunk_size)) return KDA_ERR_UNSUPPORTED;
    if (N > 0 && !cu_seqlens) return KDA_ERR_NULL;
    if (!aligned4(cu_seqlens)) return KDA_ERR_ALIGN;
    int max_len = total_T;
    if (cu_seqlens_host) {
        if (cu_seqlens_host[0] != 0 || cu_seqlens_host[N] != total_T) return KDA_ERR_INDEX;
        max_len = 0;
        for (int n = 0; n < N; ++n) {
            const int L = cu_seqlens_host[n + 1] - cu_seqlens_host[n];
            if (L < 0) return KDA_ERR_INDEX;
            if (L > max_len) max_len = L;
        }
    }
    const size_t need = kda_varlen_fwd_workspace(N, total_T, value_heads(H, opt), dk, dv, chunk_size, dtype);
    if (!ws || ws_bytes < need) return KDA_ERR_WORKSPACE;
    if (!aligned16(ws)) return KDA_ERR_ALIGN;
    if (N == 0) return KDA_OK;
    SeqBatch a{};
    a.q = q; a.k = k; a.v = v; a.beta = beta; a.decay = decay; a.h0 = initial_state;
    a.o = o; a.hT = final_state; a.cu_seqlens = cu_seqlens; a.nseq = N; a.T = max_len; a.H = H;
    a.dk = dk; a.dv = dv; a.chunk = chunk_size;
    a.dtype = dtype == KDA_BF16 ? DType::BF16 : DType::F32;
    a.scale = resolve_scale(scale, dk); a.use_l2 = use_qk_l2norm ? 1 : 0;
    if ((c = apply_options(opt, decay, a)) != KDA_OK) return c;
    a.ws = static_cast<WsHeader *>(ws);
    a.ws_body = static_cast<char *>(ws) + kWsHeader;
    a.ws_body_bytes = ws_bytes - kWsHeader;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(ws, 0, sizeof(int) * 2, st) != cudaSuccess) return KDA_ERR_CUDA;
    // Every sequence runs the chunk loop from its own cu_seqlens range; a sequence
    // of length 0 falls through the loop and stores its initial state.
    return run_prefill(a, true, total_T, st);
}

kda_status kda_gk_chunk_fwd(const void *q, const void *k, const void *v, const float *beta,
                            const float *g, const float *initial_state, void *o, float *final_state,
                            int B, int T, int H, int dk, int dv, kda_dtype dtype, float scale,
                            int chunk_size, int use_qk_l2norm, const kda_options *opt, void *ws,
                            size_t ws_bytes, kda_stream_t stream) {
    if (B < 0 || T < 0) return KDA_ERR_SHAPE;
    kda_status c = check_common(q, k, v, beta, nullptr, initial_state, o, final_state,
                                (long)B * T, H, dk, dv, dtype);
    if (c != KDA_OK) return c;
    if (!aligned16(g)) return KDA_ERR_ALIGN;
    if (!supported_chunk(chunk_size)) return KDA_ERR_UNSUPPORTED;
    const size_t need = kda_chunk_fwd_workspace(B, T, value_heads(H, opt), dk, dv, chunk_size, dtype);
    if (!ws || ws_bytes < need) return KDA_ERR_WORKSPACE;
    if (!aligned16(ws)) return KDA_ERR_ALIGN;
    SeqBatch a{};
    a.q = q; a.k = k; a.v = v; a.beta = beta; a.decay = nullptr; a.h0 = initial_state;
    a.gk = g; a.per_channel = 1;
    a.o = o; a.hT = final_state; a.cu_seqlens = nullptr; a.nseq = B; a.T = T; a.H = H;
    a.dk = dk; a.dv = dv; a.chunk = chunk_size;
    a.dtype = dtype == KDA_BF16 ? DType::BF16 : DType::F32;
    a.scale = resolve_scale(scale, dk); a.use_l2 = use_qk_l2norm ? 1 : 0;
    // without g there is no decay, and the scalar tensor-core path computes the same
    // recurrence (the per-channel prep reads g)
    if (!g && chunk_tc_supported(dk, dv, chunk_size, a.dtype)) a.per_channel = 0;
    if ((c = apply_options(opt, g, a)) != KDA_OK) return c;
    a.ws = static_cast<WsHeader *>(ws);
    a.ws_body = static_cast<char *>(ws) + kWsHeader;
    a.ws_body_bytes = ws_bytes - kWsHeader;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(ws, 0, sizeof(int) * 2, st) != cudaSuccess) return KDA_ERR_CUDA;
    return run_prefill(a, true, (long)B * T, st);
}

kda_status kda_gk_varlen_fwd(const void *q, const void *k, const void *v, const float *beta,
                             const float *g, const int *cu_seqlens, const int *cu_seqlens_host,
                             int N, int total_T, int H, int dk, int dv, const float *initial_state,
                             void *o, float *final_state, kda_dtype dtype, float scale,
                             int chunk_size, int use_qk_l2norm, const kda_options *opt, void *ws,
                             size_t ws_bytes, kda_stream_t stream) {
    if (N < 0 || total_T < 0) return KDA_ERR_SHAPE;
    kda_status c = check_common(q, k, v, beta, nullptr, initial_state, o, final_state,
                                total_T, H, dk, dv, dtype);
    if (c != KDA_OK) return c;
    if (!aligned16(g)) return KDA_ERR_ALIGN;
    if (!supported_chunk(chunk_size)) return KDA_ERR_UNSUPPORTED;
    if (N > 0 && !cu_seqlens) return KDA_ERR_NULL;
    if (!aligned4(cu_seqlens)) return KDA_ERR_ALIGN;
    int max_len = total_T;
    if (cu_seqlens_host) {
        if (cu_seqlens_host[0] != 0 || cu_seqlens_host[N] != total_T) return KDA_ERR_INDEX;
        max_len = 0;
        for (int n = 0; n < N; ++n) {
            const int L = cu_seqlens_host[n + 1] - cu_seqlens_host[n];
            if (L < 0) return KDA_ERR_INDEX;
            if (L > max_len) max_len = L;
        }
    }
    const size_t need = kda_varlen_fwd_workspace(N, total_T, value_heads(H, opt), dk, dv, chunk_size, dtype);
    if (!ws || ws_bytes < need) return KDA_ERR_WORKSPACE;
    if (!aligned16(ws)) return KDA_ERR_ALIGN;
    if (N == 0) return KDA_OK;
    SeqBatch a{};
    a.q = q; a.k = k; a.v = v; a.beta = beta; a.decay = nullptr; a.h0 = initial_state;
    a.gk = g; a.per_channel = 1;
    a.o = o; a.hT = final_state; a.cu_seqlens = cu_seqlens; a.nseq = N; a.T = max_len; a.H = H;
    a.dk = dk; a.dv = dv; a.chunk = chunk_size;
    a.dtype = dtype == KDA_BF16 ? DType::BF16 : DType::F32;
    a.scale = resolve_scale(scale, dk); a.use_l2 = use_qk_l2norm ? 1 : 0;
    // without g there is no decay, and the scalar tensor-core path computes the same
    // recurrence (the per-channel prep reads g)
    if (!g && chunk_tc_supported(dk, dv, chunk_size, a.dtype)) a.per_channel = 0;
    if ((c = apply_options(opt, g, a)) != KDA_OK) return c;
    a.ws = static_cast<WsHeader *>(ws);
    a.ws_body = static_cast<char *>(ws) + kWsHeader;
    a.ws_body_bytes = ws_bytes - kWsHeader;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(ws, 0, sizeof(int) * 2, st) != cudaSuccess) return KDA_ERR_CUDA;
    return run_prefill(a, true, total_T, st);
}

kda_status kda_gk_recurrent_fwd(const void *q, const void *k, const void *v, const float *beta,
                                const float *g, const float *initial_state, void *o,
                                float *final_state, int B, int T, int H, int dk, int dv,
                                kda_dtype dtype, float scale, int use_qk_l2norm,
                                const kda_options *opt, kda_stream_t stream) {
    if (B < 0 || T < 0) return KDA_ERR_SHAPE;
    kda_status c = check_common(q, k, v, beta, nullptr, initial_state, o, final_state,
                                (long)B * T, H, dk, dv, dtype);
    if (c != KDA_OK) return c;
    if (!aligned16(g)) return KDA_ERR_ALIGN;
    SeqBatch a{};
    a.q = q; a.k = k; a.v = v; a.beta = beta; a.decay = nullptr; a.h0 = initial_state;
    a.gk = g; a.per_channel = 1;
    a.o = o; a.hT = final_state; a.cu_seqlens = nullptr; a.nseq = B; a.T = T; a.H = H;
    a.dk = dk; a.dv = dv; a.chunk = 0;
    a.dtype = dtype == KDA_BF16 ? DType::BF16 : DType::F32;
    a.scale = resolve_scale(scale, dk); a.use_l2 = use_qk_l2norm ? 1 : 0;
    if ((c = apply_options(opt, g, a)) != KDA_OK) return c;
    return run_prefill(a, false, (long)B * T, reinterpret_cast<cudaStream_t>(stream));
}

kda_status kda_gk_varlen_recurrent_fwd(const void *q, const void *k, const void *v,
                                       const float *beta, const float *g,
                                       const int *cu_seqlens, const int *cu_seqlens_host,
                                       int N, int total_T, int H, int dk, int dv,
                                       const float *initial_state, void *o, float *final_state,
                                       kda_dtype dtype, float scale, int use_qk_l2norm,
                                       const kda_options *opt, kda_stream_t stream) {
    if (N < 0 || total_T < 0) return KDA_ERR_SHAPE;
    kda_status c = check_common(q, k, v, beta, nullptr, initial_state, o, final_state,
                                total_T, H, dk, dv, dtype);
    if (c != KDA_OK) return c;
    if (!aligned16(g)) return KDA_ERR_ALIGN;
    if (N > 0 && !cu_seqlens) return KDA_ERR_NULL;
    if (!aligned4(cu_seqlens)) return KDA_ERR_ALIGN;
    if (cu_seqlens_host) {
        if (cu_seqlens_host[0] != 0 || cu_seqlens_host[N] != total_T) return KDA_ERR_INDEX;
        for (int n = 0; n < N; ++n)
            if (cu_seqlens_host[n + 1] < cu_seqlens_host[n]) return KDA_ERR_INDEX;
    }
    if (N == 0) return KDA_OK;
    SeqBatch a{};
    a.q = q; a.k = k; a.v = v; a.beta = beta; a.decay = nullptr; a.h0 = initial_state;
    a.gk = g; a.per_channel = 1;
    a.o = o; a.hT = final_state; a.cu_seqlens = cu_seqlens; a.nseq = N; a.T = total_T; a.H = H;
    a.dk = dk; a.dv = dv; a.chunk = 0;
    a.dtype = dtype == KDA_BF16 ? DType::BF16 : DType::F32;
    a.scale = resolve_scale(scale, dk); a.use_l2 = use_qk_l2norm ? 1 : 0;
    if ((c = apply_options(opt, g, a)) != KDA_OK) return c;
    // every sequence scans its own cu_seqlens range; one of length 0 stores its
    // initial state (or zeros)
    return launch_status(launch_recurrent(a, reinterpret_cast<cudaStream_t>(stream)));
}

kda_status kda_gk_decode_step(const void *q, const void *k, const void *v, const float *beta,
                              const float *g, float *state, void *o, int B, int H, int dk,
                              int dv, kda_dtype dtype, float scale, int use_qk_l2norm,
                              const kda_options *opt, kda_stream_t stream) {
    if (B < 0) return KDA_ERR_SHAPE;
    kda_status c = check_common(q, k, v, beta, nullptr, state, o, state, B, H, dk, dv, dtype);
    if (c != KDA_OK) return c;
    if (!aligned16(g)) return KDA_ERR_ALIGN;
    if (B > 0 && !state) return KDA_ERR_NULL;
    DecodeArgs a{};
    a.H = H;
    if ((c = decode_options(opt, g, a)) != KDA_OK) return c;
    if (B == 0) return KDA_OK;
    a.q = q; a.k = k; a.v = v; a.beta = beta; a.decay = nullptr; a.state = state; a.o = o;
    a.gk = g; a.per_channel = 1;
    a.B = B; a.dk = dk; a.dv = dv;
    a.dtype = dtype == KDA_BF16 ? DType::BF16 : DType::F32;
    a.scale = resolve_scale(scale, dk); a.use_l2 = use_qk_l2norm ? 1 : 0;
    return launch_status(launch_decode(a, reinterpret_cast<cudaStream_t>(stream)));
}

kda_status kda_gate_decay(const float *gate, const float *A_log, const float *dt_bias,
                          float *decay, long rows, int H, int K, kda_stream_t stream) {
    if (rows < 0 || H <= 0 || K <= 0) return KDA_ERR_SHAPE;
    if (rows == 0) return KDA_OK;
    if (!gate || !A_log || !decay) return KDA_ERR_NULL;
    if (!aligned4(gate) || !aligned4(A_log) || !aligned4(dt_bias) || !aligned4(decay)) return KDA_ERR_ALIGN;
    const long n = rows * (long)H * K;
    const long blocks = std::min<long>((n + 255) / 256, 4096);
    gate_decay_kernel<<<(unsigned)blocks, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        gate, A_log, dt_bias, decay, n, H, K);
    return launch_status(cudaGetLastError());
}

size_t kda_gk_recurrent_bwd_workspace(int B, int T, int H, int dk, int dv) {
    if (B < 0 || T < 0 || H <= 0 || !supported_head(dk) || !supported_head(dv)) return 0;
    return kWsHeader + gk_bwd_scratch_bytes(B, T, H, dk, dv);
}

kda_status kda_gk_recurrent_bwd(const void *q, const void *k, const void *v, const float *beta,
                                const float *g, const float *initial_state, const void *d_o,
                                const float *dfinal_state, float *dq, float *dk_out, float *dv_out,
                                float *dbeta, float *dg, float *dinitial_state, int B, int T, int H,
                                int dk, int dv, kda_dtype dtype, float scale, int use_qk_l2norm,
                                int decayed_read, void *ws, size_t ws_bytes, kda_stream_t stream) {
    if (B < 0 || T < 0) return KDA_ERR_SHAPE;
    kda_status c = check_common(q, k, v, beta, nullptr, initial_state, d_o, dfinal_state,
                                (long)B * T, H, dk, dv, dtype);
    if (c != KDA_OK) return c;
    const long rows = (long)B * T;
    if (rows > 0 && (!dq || !dk_out || !dv_out || !dbeta)) return KDA_ERR_NULL;
    if (!aligned16(g) || !aligned16(dinitial_state) || !aligned4(dq) || !aligned4(dk_out) ||
        !aligned4(dv_out) || !aligned4(dbeta) || !aligned4(dg))
        return KDA_ERR_ALIGN;
    const size_t need = kda_gk_recurrent_bwd_workspace(B, T, H, dk, dv);
    if (!ws || ws_bytes < need) return KDA_ERR_WORKSPACE;
    if (!aligned16(ws)) return KDA_ERR_ALIGN;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (rows == 0) {   // nothing but the state: dh0 = dhT
        if (!dinitial_state || B == 0) return KDA_OK;
        const size_t n = (size_t)B * H * dk * dv * sizeof(float);
        if (dfinal_state) return launch_status(cudaMemcpyAsync(dinitial_state, dfinal_state, n, cudaMemcpyDeviceToDevice, st));
        return launch_status(cudaMemsetAsync(dinitial_state, 0, n, st));
    }
    BwdArgs a{};
    a.q = q; a.k = k; a.v = v; a.dout = d_o; a.beta = beta; a.g = g; a.h0 = initial_state;
    a.dhT = dfinal_state; a.dq = dq; a.dk = dk_out; a.dv = dv_out; a.dbeta = dbeta;
    a.dg = g ? dg : nullptr; a.dh0 = dinitial_state;
    a.B = B; a.T = T; a.H = H; a.dkdim = dk; a.dvdim = dv;
    a.dtype = dtype == KDA_BF16 ? DType::BF16 : DType::F32;
    a.scale = resolve_scale(scale, dk); a.use_l2 = use_qk_l2norm ? 1 : 0;
    a.decayed_read = decayed_read ? 1 : 0;
    a.ws = static_cast<char *>(ws) + kWsHeader;
    if (!g && dg &&   // dg without g: no decay, a zero gradient
        cudaMemsetAsync(dg, 0, (size_t)rows * H * dk * sizeof(float), st) != cudaSuccess)
        return KDA_ERR_CUDA;
    return launch_status(launch_gk_bwd(a, st));
}

size_t kda_recurrent_bwd_workspace(int B, int T, int H, int dk, int dv) {
    return kda_gk_recurrent_bwd_workspace(B, T, H, dk, dv);
}

kda_status kda_recurrent_bwd(const void *q, const void *k, const void *v, const float *beta,
                             const float *decay, const float *initial_state, const void *d_o,
                             const float *dfinal_state, float *dq, float *dk_out, float *dv_out,
                             float *dbeta, float *ddecay, float *dinitial_state, int B, int T, int H,
                             int dk, int dv, kda_dtype dtype, float scale, int use_qk_l2norm,
                             int decayed_read, void *ws, size_t ws_bytes, kda_stream_t stream) {
    if (B < 0 || T < 0) return KDA_ERR_SHAPE;
    kda_status c = check_common(q, k, v, beta, decay, initial_state, d_o, dfinal_state,
                                (long)B * T, H, dk, dv, dtype);
    if (c != KDA_OK) return c;
    const long rows = (long)B * T;
    if (rows > 0 && (!dq || !dk_out || !dv_out || !dbeta)) return KDA_ERR_NULL;
    if (!aligned16(dinitial_state) || !aligned4(dq) || !aligned4(dk_out) || !aligned4(dv_out) ||
        !aligned4(dbeta) || !aligned4(ddecay))
        return KDA_ERR_ALIGN;
    const size_t need = kda_recurrent_bwd_workspace(B, T, H, dk, dv);
    if (!ws || ws_bytes < need) return KDA_ERR_WORKSPACE;
    if (!aligned16(ws)) return KDA_ERR_ALIGN;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (rows == 0) {   // nothing but the state: dh0 = dhT
        if (!dinitial_state || B == 0) return KDA_OK;
        const size_t n = (size_t)B * H * dk * dv * sizeof(float);
        if (dfinal_state) return launch_status(cudaMemcpyAsync(dinitial_state, dfinal_state, n, cudaMemcpyDeviceToDevice, st));
        return launch_status(cudaMemsetAsync(dinitial_state, 0, n, st));
    }
    BwdArgs a{};
    a.q = q; a.k = k; a.v = v; a.dout = d_o; a.beta = beta; a.g = nullptr; a.h0 = initial_state;
    a.decay = decay; a.ddecay = decay ? ddecay : nullptr;
    a.dhT = dfinal_state; a.dq = dq; a.dk = dk_out; a.dv = dv_out; a.dbeta = dbeta;
    a.dg = nullptr; a.dh0 = dinitial_state;
    a.B = B; a.T = T; a.H = H; a.dkdim = dk; a.dvdim = dv;
    a.dtype = dtype == KDA_BF16 ? DType::BF16 : DType::F32;
    a.scale = resolve_scale(scale, dk); a.use_l2 = use_qk_l2norm ? 1 : 0;
    a.decayed_read = decayed_read ? 1 : 0;
    a.ws = static_cast<char *>(ws) + kWsHeader;
    if (!decay && ddecay &&   // ddecay without a decay: a zero gradient
        cudaMemsetAsync(ddecay, 0, (size_t)rows * H * sizeof(float), st) != cudaSuccess)
        return KDA_ERR_CUDA;
    return launch_status(launch_gk_bwd(a, st));
}

kda_status kda_query_device_error(const void *ws, kda_stream_t stream) {
    if (!ws) {   // the built-in scratch of kda_chunk_fwd_noalloc on the current device
        void *h = nullptr;
        if (noalloc_header(&h) != cudaSuccess) return KDA_ERR_CUDA;
        ws = h;
    }
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    WsHeader h;
    if (cudaMemcpyAsync(&h, ws, sizeof(int) * 2, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return KDA_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return KDA_ERR_CUDA;
    if (h.error != 0) {
        if (cudaMemsetAsync(const_cast<void *>(ws), 0, sizeof(int) * 2, st) != cudaSuccess)
            return KDA_ERR_CUDA;
        if (cudaStreamSynchronize(st) != cudaSuccess) return KDA_ERR_CUDA;
        return static_cast<kda_status>(h.error);
    }
    return KDA_OK;
}

kda_status kda_diag_wait_timeout(void *ws, size_t ws_bytes, unsigned limit_us,
                                 kda_stream_t stream) {
    if (!ws) return KDA_ERR_NULL;
    if (ws_bytes < kWsHeader) return KDA_ERR_WORKSPACE;
    if (!aligned16(ws)) return KDA_ERR_ALIGN;
    if (limit_us == 0 || limit_us > 2000000u) return KDA_ERR_SHAPE;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(ws, 0, sizeof(int) * 2, st) != cudaSuccess) return KDA_ERR_CUDA;
    return launch_timeout_probe(static_cast<WsHeader *>(ws), (uint64_t)limit_us * 1000u, st) ==
                   cudaSuccess
               ? KDA_OK
               : KDA_ERR_CUDA;
}

}  // extern "C"

// ---------------------------------------------------------------------------------
// Chunked backward (tensor cores): the forward walk keeping every chunk's map and state,
// the reverse walk over the maps, then the chunk-local gradients.
// Workspace after the header: the forward's kept scratch | states at every chunk start |
// incoming state gradients of every chunk | the gradient kernel's per-CTA scratch.
static size_t chunk_bwd_layout(int B, int T, int H, int d, size_t *off_states, size_t *off_dstates,
                               size_t *off_scratch) {
    const size_t keep = (chunk_tc_keep_bytes(B, H, T, d) + 255) / 256 * 256;
    const size_t st = (size_t)B * H * ((T + 63) / 64) * d * d * 2;   // bf16 states
    if (off_states) *off_states = kWsHeader + keep;
    if (off_dstates) *off_dstates = kWsHeader + keep + st;
    if (off_scratch) *off_scratch = kWsHeader + keep + 2 * st;
    const long nchunks = (long)B * H * ((T + 63) / 64);
    return kWsHeader + keep + 2 * st + (size_t)chunk_bwd_ctas(nchunks) * chunk_bwd_scratch_floats(d) * sizeof(float);
}

size_t kda_chunk_bwd_workspace(int B, int T, int H, int dk, int dv) {
    if (B < 0 || T < 0 || H <= 0 || dk != dv || (dk != 64 && dk != 128)) return 0;
    if (B == 0 || T == 0) return kWsHeader;
    return chunk_bwd_layout(B, T, H, dk, nullptr, nullptr, nullptr);
}

kda_status kda_chunk_bwd(const void *q, const void *k, const void *v, const float *beta,
                         const float *decay, const float *initial_state, const void *d_o,
                         const float *dfinal_state, float *dq, float *dk_out, float *dv_out,
                         float *dbeta, float *ddecay, float *dinitial_state, int B, int T, int H,
                         int dk, int dv, kda_dtype dtype, float scale, int use_qk_l2norm,
                         int decayed_read, void *ws, size_t ws_bytes, kda_stream_t stream) {
    if (B < 0 || T < 0) return KDA_ERR_SHAPE;
    kda_status c = check_common(q, k, v, beta, decay, initial_state, d_o, dfinal_state,
                                (long)B * T, H, dk, dv, dtype);
    if (c != KDA_OK) return c;
    if (dtype != KDA_BF16 || dk != dv || (dk != 64 && dk != 128)) return KDA_ERR_UNSUPPORTED;
    const long rows = (long)B * T;
    if (rows >= (1L << 31)) return KDA_ERR_UNSUPPORTED;
    if (rows > 0 && (!dq || !dk_out || !dv_out || !dbeta)) return KDA_ERR_NULL;
    if (!aligned16(dinitial_state) || !aligned4(dq) || !aligned4(dk_out) || !aligned4(dv_out) ||
        !aligned4(dbeta) || !aligned4(ddecay))
        return KDA_ERR_ALIGN;
    const size_t need = kda_chunk_bwd_workspace(B, T, H, dk, dv);
    if (!ws || ws_bytes < need) return KDA_ERR_WORKSPACE;
    if (!aligned16(ws)) return KDA_ERR_ALIGN;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (rows == 0) {   // nothing but the state: dh0 = dhT
        if (!dinitial_state || B == 0) return KDA_OK;
        const size_t n = (size_t)B * H * dk * dv * sizeof(float);
        if (dfinal_state) return launch_status(cudaMemcpyAsync(dinitial_state, dfinal_state, n, cudaMemcpyDeviceToDevice, st));
        return launch_status(cudaMemsetAsync(dinitial_state, 0, n, st));
    }
    size_t o_st = 0, o_dst = 0, o_scr = 0;
    chunk_bwd_layout(B, T, H, dk, &o_st, &o_dst, &o_scr);
    char *w = static_cast<char *>(ws);
    __nv_bfloat16 *fstates = reinterpret_cast<__nv_bfloat16 *>(w + o_st);
    __nv_bfloat16 *bstates = reinterpret_cast<__nv_bfloat16 *>(w + o_dst);
    if (cudaMemsetAsync(ws, 0, sizeof(int) * 2, st) != cudaSuccess) return KDA_ERR_CUDA;
    SeqBatch a{};
    a.q = q; a.k = k; a.v = v; a.beta = beta; a.decay = decay; a.h0 = initial_state;
    a.o = nullptr; a.hT = nullptr; a.cu_seqlens = nullptr; a.nseq = B; a.T = T; a.H = H;
    a.dk = dk; a.dv = dv; a.chunk = 64; a.dtype = DType::BF16;
    a.scale = resolve_scale(scale, dk); a.use_l2 = use_qk_l2norm ? 1 : 0;
    a.decayed_read = decayed_read ? 1 : 0;
    a.ws = static_cast<WsHeader *>(ws);
    a.ws_body = w + kWsHeader;
    a.ws_body_bytes = o_st - kWsHeader;
    // the reverse walk writes the state gradients and dh0; the value gradients come from the
    // gradient kernel (dV = diag(beta) T^T dU), which spares the walk their stores
    cudaError_t e = launch_chunk_tc_walks(a, d_o, dfinal_state, dinitial_state, nullptr, fstates, bstates, st);
    if (e != cudaSuccess) return launch_status(e);
    ChunkBwdArgs g{};
    g.q = q; g.k = k; g.v = v; g.d_o = d_o; g.beta = beta; g.decay = decay;
    g.fstates = fstates; g.bstates = bstates;
    g.dq = dq; g.dk = dk_out; g.dv = dv_out; g.dbeta = dbeta; g.ddecay = decay ? ddecay : nullptr;
    g.B = B; g.T = T; g.H = H; g.D = dk;
    g.scale = a.scale; g.use_l2 = a.use_l2; g.decayed_read = a.decayed_read;
    g.scratch = reinterpret_cast<float *>(w + o_scr);
    g.ctas = chunk_bwd_ctas((long)B * H * ((T + 63) / 64));
    if (!decay && ddecay &&   // ddecay without a decay: a zero gradient
        cudaMemsetAsync(ddecay, 0, (size_t)rows * H * sizeof(float), st) != cudaSuccess)
        return KDA_ERR_CUDA;
    return launch_status(launch_chunk_bwd_grads(g, st));
}

// header | kept maps | kept states | state gradients | the gradient kernel's scratch
static size_t gk_chunk_bwd_layout(int B, int T, int H, int d, size_t *off_states, size_t *off_dstates,
                                  size_t *off_scratch) {
    const size_t keep = (chunk_tc_keep_bytes(B, H, T, d) + 255) / 256 * 256;
    const size_t st = (size_t)B * H * ((T + 63) / 64) * d * d * 2;   // bf16 states
    if (off_states) *off_states = kWsHeader + keep;
    if (off_dstates) *off_dstates = kWsHeader + keep + st;
    if (off_scratch) *off_scratch = kWsHeader + keep + 2 * st;
    return kWsHeader + keep + 2 * st + gk_chunk_bwd_scratch_bytes(d);
}

size_t kda_gk_chunk_bwd_workspace(int B, int T, int H, int dk, int dv) {
    if (B < 0 || T < 0 || H <= 0 || dk != dv || (dk != 64 && dk != 128)) return 0;
    if (B == 0 || T == 0) return kWsHeader;
    return gk_chunk_bwd_layout(B, T, H, dk, nullptr, nullptr, nullptr);
}

kda_status kda_gk_chunk_bwd(const void *q, const void *k, const void *v, const float *beta,
                            const float *g, const float *initial_state, const void *d_o,
                            const float *dfinal_state, float *dq, float *dk_out, float *dv_out,
                            float *dbeta, float *dg, float *dinitial_state, int B, int T, int H,
                            int dk, int dv, kda_dtype dtype, float scale, int use_qk_l2norm,
                            int decayed_read, void *ws, size_t ws_bytes, kda_stream_t stream) {
    if (B < 0 || T < 0) return KDA_ERR_SHAPE;
    kda_status c = check_common(q, k, v, beta, nullptr, initial_state, d_o, dfinal_state,
                                (long)B * T, H, dk, dv, dtype);
    if (c != KDA_OK) return c;
    if (dtype != KDA_BF16 || dk != dv || (dk != 64 && dk != 128)) return KDA_ERR_UNSUPPORTED;
    const long rows = (long)B * T;
    if (rows >= (1L << 31)) return KDA_ERR_UNSUPPORTED;
    if (rows > 0 && (!dq || !dk_out || !dv_out || !dbeta)) return KDA_ERR_NULL;
    if (!aligned16(g) || !aligned16(dinitial_state) || !aligned4(dq) || !aligned4(dk_out) ||
        !aligned4(dv_out) || !aligned4(dbeta) || !aligned4(dg))
        return KDA_ERR_ALIGN;
    const size_t need = kda_gk_chunk_bwd_workspace(B, T, H, dk, dv);
    if (!ws || ws_bytes < need) return KDA_ERR_WORKSPACE;
    if (!aligned16(ws)) return KDA_ERR_ALIGN;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (rows == 0) {   // nothing but the state: dh0 = dhT
        if (!dinitial_state || B == 0) return KDA_OK;
        const size_t n = (size_t)B * H * dk * dv * sizeof(float);
        if (dfinal_state) return launch_status(cudaMemcpyAsync(dinitial_state, dfinal_state, n, cudaMemcpyDeviceToDevice, st));
        return launch_status(cudaMemsetAsync(dinitial_state, 0, n, st));
    }
    size_t o_st = 0, o_dst = 0, o_scr = 0;
    gk_chunk_bwd_layout(B, T, H, dk, &o_st, &o_dst, &o_scr);
    char *w = static_cast<char *>(ws);
    __nv_bfloat16 *fstates = reinterpret_cast<__nv_bfloat16 *>(w + o_st);
    __nv_bfloat16 *bstates = reinterpret_cast<__nv_bfloat16 *>(w + o_dst);
    if (cudaMemsetAsync(ws, 0, sizeof(int) * 2, st) != cudaSuccess) return KDA_ERR_CUDA;
    // the two walks over the chunk maps: the per-channel prep builds them (without g there is
    // no decay and the scalar prep's maps are the same)
    SeqBatch a{};
    a.q = q; a.k = k; a.v = v; a.beta = beta; a.decay = nullptr; a.h0 = initial_state;
    a.gk = g; a.per_channel = g ? 1 : 0;
    a.o = nullptr; a.hT = nullptr; a.cu_seqlens = nullptr; a.nseq = B; a.T = T; a.H = H;
    a.dk = dk; a.dv = dv; a.chunk = 64; a.dtype = DType::BF16;
    a.scale = resolve_scale(scale, dk); a.use_l2 = use_qk_l2norm ? 1 : 0;
    a.decayed_read = decayed_read ? 1 : 0;
    a.ws = static_cast<WsHeader *>(ws);
    a.ws_body = w + kWsHeader;
    a.ws_body_bytes = o_st - kWsHeader;
    cudaError_t e = launch_chunk_tc_walks(a, d_o, dfinal_state, dinitial_state, nullptr, fstates, bstates, st);
    if (e != cudaSuccess) return launch_status(e);
    BwdArgs b{};
    b.q = q; b.k = k; b.v = v; b.dout = d_o; b.beta = beta; b.g = g;
    b.dq = dq; b.dk = dk_out; b.dv = dv_out; b.dbeta = dbeta; b.dg = g ? dg : nullptr;
    b.B = B; b.T = T; b.H = H; b.dkdim = dk; b.dvdim = dv; b.dtype = DType::BF16;
    b.scale = a.scale; b.use_l2 = a.use_l2; b.decayed_read = a.decayed_read;
    if (!g && dg &&   // dg without g: no decay, a zero gradient
        cudaMemsetAsync(dg, 0, (size_t)rows * H * dk * sizeof(float), st) != cudaSuccess)
        return KDA_ERR_CUDA;
    return launch_status(launch_gk_chunk_bwd_grads(b, fstates, bstates, w + o_scr, st));
}
