// chunk_tc_noalloc.cu -- the tensor-core chunked prefill without a caller workspace.
//
// Some callers cannot allocate device memory at the point where they call us: a plugin
// inside a host framework that owns the memory pool and forbids allocations of its own,
// code on a latency-critical path where cudaMalloc / cudaFree would synchronise the
// device, or a caller with no spare memory it can hand over.  For them this file
// provides kda_chunk_fwd_noalloc, which runs the same prep/chain kernels as
// kda_chunk_fwd but places their scratch (error word, the chains' E_c rings and flags) in
// a file-scope __device__ array of fixed size.  It allocates nothing.
//
// The array is 48 MiB and lives on every GPU that loads this library, until the process
// exits.  The prefill's scratch does not grow with the problem (at most kMaxChains chains,
// each with a ring of E_c slots: about 45 MiB at head dim 128), so every supported problem
// fits; the size check below is a guard.  Host code cannot use the array's name as a device
// address (on the host it is only a stand-in), so the device address is looked up once per
// device with cudaGetSymbolAddress, with that device current, on the first call made on
// the device (or on the first kda_query_device_error(NULL, ...) there).
#include <math.h>
#include <mutex>

#include "../../include/kda.h"
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(48) << 20;   // 48 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 128;
std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxDevices];   // device address of g_noalloc_scratch, per device

// Device address of the scratch array on the current device (looked up on first use).
cudaError_t noalloc_scratch(void **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace

// The built-in array's header on the current device (kda_query_device_error with NULL).
cudaError_t noalloc_header(void **out) { return noalloc_scratch(out); }

namespace {

bool aligned16(const void *p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void *p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace
}  // namespace kda

extern "C" kda_status kda_chunk_fwd_noalloc(const void *q, const void *k, const void *v,
                                            const float *beta, const float *decay,
                                            const float *initial_state, void *o,
                                            float *final_state, int B, int T, int H, int dk,
                                            int dv, kda_dtype dtype, float scale, int chunk_size,
                                            int use_qk_l2norm, kda_stream_t stream) {
    using namespace kda;
    if (dtype != KDA_F32 && dtype != KDA_BF16) return KDA_ERR_DTYPE;
    if (B < 0 || T < 0 || H <= 0 || dk <= 0 || dv <= 0) return KDA_ERR_SHAPE;
    if (!chunk_tc_supported(dk, dv, chunk_size, dtype == KDA_BF16 ? DType::BF16 : DType::F32))
        return KDA_ERR_UNSUPPORTED;
    if ((long)B * T > 0 && (!q || !k || !v || !beta || !o)) return KDA_ERR_NULL;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
        !aligned16(initial_state) || !aligned16(final_state) || !aligned4(beta) || !aligned4(decay))
        return KDA_ERR_ALIGN;
    const long rows = (long)B * T;
    if (sizeof(WsHeader) + chunk_tc_scratch_bytes(B, H, dk, false) > kNoAllocScratchBytes)
        return KDA_ERR_WORKSPACE;   // the problem needs more than the built-in array
    if (B == 0) return KDA_OK;
    void *scratch = nullptr;
    if (noalloc_scratch(&scratch) != cudaSuccess) return KDA_ERR_CUDA;

    SeqBatch a{};
    a.q = q; a.k = k; a.v = v; a.beta = beta; a.decay = decay; a.h0 = initial_state;
    a.o = o; a.hT = final_state; a.cu_seqlens = nullptr; a.nseq = B; a.T = T; a.H = H;
    a.dk = dk; a.dv = dv; a.chunk = chunk_size; a.dtype = DType::BF16;
    a.scale = scale > 0.f ? scale : 1.0f / sqrtf((float)dk);
    a.use_l2 = use_qk_l2norm ? 1 : 0;
    a.ws = static_cast<WsHeader *>(scratch);
    a.ws_body = static_cast<char *>(scratch) + sizeof(WsHeader);
    a.ws_body_bytes = kNoAllocScratchBytes - sizeof(WsHeader);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // the array keeps the previous call's contents: the error word must start at zero
    if (cudaMemsetAsync(scratch, 0, sizeof(int) * 2, st) != cudaSuccess) return KDA_ERR_CUDA;
    cudaError_t e = (T == 0) ? launch_state_passthrough(a, st) : launch_chunk_tc(a, rows, st);
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}
