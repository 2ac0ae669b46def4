// scan.cu -- single-token decode and the token-by-token (recurrent) prefill.
//
// Both run the recurrence of ejkernel kda() ("The core recurrence") one token at
// a time with the fp32 state held in registers (key-major [dk, dv] per head here; the
// value-major [dv, dk] layout has its own kernel below):
//     r = S^T k^,  p = S^T q~,  u = beta (v - r),
//     o = alpha p + (k^ . q~) u,  S <- alpha S + k^ u^T,   alpha = exp(decay)
// (o = h_t^T q~ expanded with h_t = alpha S + k^ u^T; with alpha = 1 this is the
// step of TileOPs DeltaNetRecurrentFwdOp).
//
// With a decay per key channel (TileOPs KDAFwdOp, g [.., dk]; GLARecurrentFwdOp:
// diag(exp(gk)) S) alpha becomes the diagonal D = diag(exp(g_t)):
//     r = S^T k^ or (D S)^T k^ (decayed read),  p = (D S)^T q~ = S^T (D q~),
//     o = p + (k^ . q~) u,  S <- D S + k^ u^T,
// i.e. the per-row factor exp(g_t[i]) scales row i of the state, and folds into the
// k and q entries of the two reductions.
//
// One CTA owns one (sequence, head, value-slab) and keeps its [dk x slab] slice of
// the state in registers: thread (rg, cg) holds float4 column group cg of rows
// rg, rg + RG, rg + 2RG, ...  A warp therefore touches consecutive rows of one
// head, i.e. one contiguous stretch of the key-major state: every state access is
// a coalesced 128-bit load or store, and the state crosses HBM exactly once in
// and once out per call.  The two reductions over dk (S^T k and S^T q) are
// in-thread sums followed by one shared-memory pass over the row groups (with many row
// groups, each column summed by a few lanes and a shuffle).
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kThreads = 256;

struct ScanParams {
    const void *q, *k, *v;
    const float *beta, *decay;
    const float *gk;   // per-channel decay [rows, H, DK] (GK kernels only; may be null)
    const float *h0;   // may equal hT (decode updates in place)
    void *o;
    float *hT;
    const int *cu_seqlens;
    int nseq, T, H, DV;
    float scale;
    int use_l2;
    int decayed_read;  // the delta term reads the decayed state (D S, or alpha S)
    const float *A_log, *dt_bias;   // raw gate -> decay (gate_decay); dt_bias [H] or [H, DK]
    int beta_sig, neg_eig;
    int G;             // value heads per q/k head: H counts value heads, q/k have H / G
};

// One token's inputs, each thread its share (k or q entry, g, v entry, beta and decay),
// read from global memory ahead of their use so that the loads' latency overlaps the
// earlier tokens' work; put() converts them, applies the gate and beta transforms and
// fills the shared staging arrays.
template <typename Tin, int DK, int DVS, bool GK>
struct TokenLoad {
    // raw values: no instruction uses a loaded register before put(), so the loads stay in
    // flight until then
    Tin kq{}, v{};
    float g = 0.f, beta = 0.f, decay = 0.f;
    __device__ __forceinline__ void fetch(const ScanParams &p, long row, int h, int col0, int tid) {
        const size_t qk_off = ((size_t)row * (p.H / p.G) + h / p.G) * DK;   // q/k head of value head h
        if (tid < DK) {
            kq = static_cast<const Tin *>(p.k)[qk_off + tid];
            if (GK && p.gk) g = p.gk[((size_t)row * p.H + h) * DK + tid];
        } else if (tid < 2 * DK) {
            kq = static_cast<const Tin *>(p.q)[qk_off + tid - DK];
        }
        if (tid < DVS) v = static_cast<const Tin *>(p.v)[((size_t)row * p.H + h) * p.DV + col0 + tid];
        if (tid == 0) {
            beta = p.beta[(size_t)row * p.H + h];
            decay = p.decay ? p.decay[(size_t)row * p.H + h] : 0.f;
        }
    }
    __device__ __forceinline__ void put(const ScanParams &p, int h, int tid, float *s_k, float *s_q, float *s_a,
                                        float *s_v, float *s_sc) const {
        if (tid < DK) {
            s_k[tid] = to_f32(kq);
            if constexpr (GK) {
                float gv = g;
                if (p.gk && p.A_log)
                    gv = gate_decay(gv, p.A_log[h], p.dt_bias ? p.dt_bias[(size_t)h * DK + tid] : 0.f);
                s_a[tid] = expf(gv);
            }
        } else if (tid < 2 * DK) {
            s_q[tid - DK] = to_f32(kq);
        }
        if (tid < DVS) s_v[tid] = to_f32(v);
        if (tid == 0) {
            s_sc[0] = beta_of(beta, p.beta_sig, p.neg_eig);
            float d = decay;
            if (p.decay && p.A_log) d = gate_decay(d, p.A_log[h], p.dt_bias ? p.dt_bias[h] : 0.f);
            s_sc[1] = d;
        }
    }
};

template <typename Tin, int DK, int DVS, bool GK>
__global__ void __launch_bounds__(kThreads) scan_kernel(ScanParams p) {
    constexpr int TPR = DVS / 4;          // threads per state row (one float4 each)
    constexpr int RG = kThreads / TPR;    // row groups
    constexpr int R = DK / RG;            // rows per thread
    static_assert(R >= 1 && DK % RG == 0, "state slab does not tile the block");
    static_assert(2 * DK <= kThreads && DVS <= kThreads, "staging assumes small heads");

    // the token's staging, double-buffered (token t uses buffer t & 1), so that the next
    // token can be staged while slow threads still read this one: three barriers a token
    __shared__ float s_k2[2][DK], s_q2[2][DK], s_v2[2][DVS];
    __shared__ float s_a2[2][GK ? DK : 1];   // exp(g_t[i]) per key channel
    __shared__ float s_sc2[2][8];
    __shared__ __align__(16) float s_u[DVS];
    __shared__ __align__(16) float s_red[2][RG][DVS];

    const int nslab = p.DV / DVS;
    const int slab = blockIdx.x % nslab;
    const int h = (blockIdx.x / nslab) % p.H;
    const int n = blockIdx.x / (nslab * p.H);
    long start;
    int len;
    if (p.cu_seqlens) {
        start = p.cu_seqlens[n];
        len = p.cu_seqlens[n + 1] - p.cu_seqlens[n];
    } else {
        start = (long)n * p.T;
        len = p.T;
    }
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cg = tid % TPR, rg = tid / TPR;
    const int col0 = slab * DVS;
    Tin *o = static_cast<Tin *>(p.o);

    const size_t sbase = ((size_t)n * p.H + h) * DK * p.DV + col0 + 4 * cg;
    float4 S[R];
#pragma unroll
    for (int m = 0; m < R; ++m) {
        const int i = rg + RG * m;
        S[m] = p.h0 ? __ldcs(reinterpret_cast<const float4 *>(p.h0 + sbase + (size_t)i * p.DV))
                    : make_float4(0.f, 0.f, 0.f, 0.f);
    }

    // this thread's share of the next kAhead tokens, in flight: slot j is refilled as soon as
    // its token is staged (the inner loop is unrolled, so the slots stay in registers).
    // Prefill slabs read the inputs from DRAM and need the depth; decode has one token.
    constexpr int kAhead = DVS <= 64 ? 4 : 1;
    TokenLoad<Tin, DK, DVS, GK> ring[kAhead];
#pragma unroll
    for (int j = 0; j < kAhead; ++j)
        if (j < len) ring[j].fetch(p, start + j, h, col0, tid);
    for (int t0 = 0; t0 < len; t0 += kAhead) {
#pragma unroll
    for (int jj = 0; jj < kAhead; ++jj) {
        const int t = t0 + jj;
        if (t >= len) break;
        const long row = start + t;
        const size_t v_off = ((size_t)row * p.H + h) * p.DV + col0;
        float *s_k = s_k2[t & 1], *s_q = s_q2[t & 1], *s_v = s_v2[t & 1], *s_a = s_a2[t & 1];
        float *s_sc = s_sc2[t & 1];
        ring[jj].put(p, h, tid, s_k, s_q, s_a, s_v, s_sc);
        __syncthreads();
        if (t + kAhead < len) ring[jj].fetch(p, row + kAhead, h, col0, tid);

        if (warp < 3) {  // ||k||^2, ||q||^2, k.q
            float acc = 0.f;
            for (int i = lane; i < DK; i += 32) {
                const float a = (warp == 1) ? s_q[i] : s_k[i];
                const float b = (warp == 0) ? s_k[i] : s_q[i];
                acc = fmaf(a, b, acc);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            if (lane == 0) s_sc[2 + warp] = acc;
        }
        float4 r = make_float4(0.f, 0.f, 0.f, 0.f), pq = r;
#pragma unroll
        for (int m = 0; m < R; ++m) {
            const int i = rg + RG * m;
            float kk = s_k[i], qq = s_q[i];
            if constexpr (GK) {
                const float ai = s_a[i];
                qq *= ai;
                if (p.decayed_read) kk *= ai;
            }
            r.x = fmaf(S[m].x, kk, r.x); r.y = fmaf(S[m].y, kk, r.y);
            r.z = fmaf(S[m].z, kk, r.z); r.w = fmaf(S[m].w, kk, r.w);
            pq.x = fmaf(S[m].x, qq, pq.x); pq.y = fmaf(S[m].y, qq, pq.y);
            pq.z = fmaf(S[m].z, qq, pq.z); pq.w = fmaf(S[m].w, qq, pq.w);
        }
        *reinterpret_cast<float4 *>(&s_red[0][rg][4 * cg]) = r;
        *reinterpret_cast<float4 *>(&s_red[1][rg][4 * cg]) = pq;
        __syncthreads();

        const float kn = p.use_l2 ? 1.f / fmaxf(sqrtf(s_sc[2]), kNormEps) : 1.f;
        const float qn = p.scale * (p.use_l2 ? 1.f / fmaxf(sqrtf(s_sc[3]), kNormEps) : 1.f);
        const float alpha = expf(s_sc[1]);
        if constexpr (RG <= 8) {   // few row groups (whole-width slabs): one thread per column
            if (tid < DVS) {
                float rs = 0.f, ps = 0.f;
#pragma unroll
                for (int g = 0; g < RG; ++g) {
                    rs += s_red[0][g][tid];
                    ps += s_red[1][g][tid];
                }
                const float u = s_sc[0] * (s_v[tid] - kn * ((!GK && p.decayed_read) ? alpha * rs : rs));
                const float out = (GK ? 1.f : alpha) * (qn * ps) + (kn * qn * s_sc[4]) * u;
                s_u[tid] = u;
                o[v_off + tid] = from_f32<Tin>(out);
            }
        } else {   // sums over the RG row groups: P consecutive lanes per column, RG / P terms each
            constexpr int P = kThreads / DVS, PER = RG / P;
            static_assert(P * DVS == kThreads && PER * P == RG && P <= 32, "reduction split");
            const int j = tid / P, part = tid % P;
            float rs = 0.f, ps = 0.f;
#pragma unroll
            for (int e = 0; e < PER; ++e) {
                rs += s_red[0][part * PER + e][j];
                ps += s_red[1][part * PER + e][j];
            }
#pragma unroll
            for (int off = P / 2; off > 0; off >>= 1) {
                rs += __shfl_xor_sync(0xffffffffu, rs, off);
                ps += __shfl_xor_sync(0xffffffffu, ps, off);
            }
            if (part == 0) {
                // the decayed read with one decay per head: r = (alpha S)^T k
                const float u = s_sc[0] * (s_v[j] - kn * ((!GK && p.decayed_read) ? alpha * rs : rs));
                const float out = (GK ? 1.f : alpha) * (qn * ps) + (kn * qn * s_sc[4]) * u;
                s_u[j] = u;
                o[v_off + j] = from_f32<Tin>(out);
            }
        }
        __syncthreads();

        const float4 u4 = *reinterpret_cast<const float4 *>(&s_u[4 * cg]);
#pragma unroll
        for (int m = 0; m < R; ++m) {
            const float kk = kn * s_k[rg + RG * m];
            const float am = GK ? s_a[rg + RG * m] : alpha;
            S[m].x = fmaf(am, S[m].x, kk * u4.x);
            S[m].y = fmaf(am, S[m].y, kk * u4.y);
            S[m].z = fmaf(am, S[m].z, kk * u4.z);
            S[m].w = fmaf(am, S[m].w, kk * u4.w);
        }
    }
    }

    if (p.hT) {
#pragma unroll
        for (int m = 0; m < R; ++m) {
            const int i = rg + RG * m;
            __stcs(reinterpret_cast<float4 *>(p.hT + sbase + (size_t)i * p.DV), S[m]);
        }
    }
}

// ---------------------------------------------------------------------------------
// The same recurrence with a value-major state ([.., dv, dk] per head: TileOPs
// state_v_first).  Lane l of a warp owns key rows [l RPL, (l + 1) RPL) of the warp's CPW
// value columns, so that a column's dk entries are one contiguous run of a warp's loads
// and stores; the reductions over dk are warp shuffles (all lanes end with each column's
// sum).
// ---------------------------------------------------------------------------------
template <typename Tin, int DK, int DVS, bool GK>
__global__ void __launch_bounds__(kThreads) scan_vm_kernel(ScanParams p) {
    constexpr int NW = kThreads / 32;
    constexpr int CPW = DVS / NW;           // value columns per warp
    constexpr int RPL = DK / 32;            // key rows per lane
    static_assert(CPW >= 1 && DVS % NW == 0 && RPL >= 1 && DK % 32 == 0, "slab does not tile the block");
    static_assert(2 * DK <= kThreads && DVS <= kThreads, "staging assumes small heads");

    // double-buffered staging (token t uses buffer t & 1): two barriers a token
    __shared__ __align__(16) float s_k2[2][DK];
    __shared__ __align__(16) float s_q2[2][DK];
    __shared__ __align__(16) float s_a2[2][GK ? DK : 4];
    __shared__ float s_v2[2][DVS];
    __shared__ float s_sc2[2][8];

    const int nslab = p.DV / DVS;
    const int slab = blockIdx.x % nslab;
    const int h = (blockIdx.x / nslab) % p.H;
    const int n = blockIdx.x / (nslab * p.H);
    long start;
    int len;
    if (p.cu_seqlens) {
        start = p.cu_seqlens[n];
        len = p.cu_seqlens[n + 1] - p.cu_seqlens[n];
    } else {
        start = (long)n * p.T;
        len = p.T;
    }
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int col0 = slab * DVS, c0w = warp * CPW;   // the warp's first column in the slab
    Tin *o = static_cast<Tin *>(p.o);

    // S[c][e] = state(i = lane RPL + e, j = col0 + c0w + c), stored at j DK + i
    const size_t vbase = ((size_t)n * p.H + h) * (size_t)p.DV * DK + (size_t)(col0 + c0w) * DK + lane * RPL;
    float S[CPW][RPL];
#pragma unroll
    for (int c = 0; c < CPW; ++c) {
        const float *src = p.h0 + vbase + (size_t)c * DK;
        if (!p.h0) {
#pragma unroll
            for (int e = 0; e < RPL; ++e) S[c][e] = 0.f;
        } else if constexpr (RPL == 4) {
            const float4 x = __ldcs(reinterpret_cast<const float4 *>(src));
            S[c][0] = x.x; S[c][1] = x.y; S[c][2] = x.z; S[c][3] = x.w;
        } else if constexpr (RPL == 2) {
            const float2 x = __ldcs(reinterpret_cast<const float2 *>(src));
            S[c][0] = x.x; S[c][1] = x.y;
        } else {
            S[c][0] = __ldcs(src);
        }
    }

    // the next kAhead tokens' loads in flight, as in scan_kernel
    constexpr int kAhead = DVS <= 64 ? 4 : 1;
    TokenLoad<Tin, DK, DVS, GK> ring[kAhead];
#pragma unroll
    for (int j = 0; j < kAhead; ++j)
        if (j < len) ring[j].fetch(p, start + j, h, col0, tid);
    for (int t0 = 0; t0 < len; t0 += kAhead) {
#pragma unroll
    for (int jj = 0; jj < kAhead; ++jj) {
        const int t = t0 + jj;
        if (t >= len) break;
        const long row = start + t;
        const size_t v_off = ((size_t)row * p.H + h) * p.DV + col0;
        float *s_k = s_k2[t & 1], *s_q = s_q2[t & 1], *s_v = s_v2[t & 1], *s_a = s_a2[t & 1];
        float *s_sc = s_sc2[t & 1];
        ring[jj].put(p, h, tid, s_k, s_q, s_a, s_v, s_sc);
        __syncthreads();
        if (t + kAhead < len) ring[jj].fetch(p, row + kAhead, h, col0, tid);
        if (warp < 3) {  // ||k||^2, ||q||^2, k.q
            float acc = 0.f;
            for (int i = lane; i < DK; i += 32) {
                const float a = (warp == 1) ? s_q[i] : s_k[i];
                const float b = (warp == 0) ? s_k[i] : s_q[i];
                acc = fmaf(a, b, acc);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            if (lane == 0) s_sc[2 + warp] = acc;
        }
        __syncthreads();
        const float kn = p.use_l2 ? 1.f / fmaxf(sqrtf(s_sc[2]), kNormEps) : 1.f;
        const float qn = p.scale * (p.use_l2 ? 1.f / fmaxf(sqrtf(s_sc[3]), kNormEps) : 1.f);
        const float alpha = expf(s_sc[1]), bt = s_sc[0], kq = s_sc[4];
        float kk[RPL], qq[RPL], am[RPL];
#pragma unroll
        for (int e = 0; e < RPL; ++e) {
            const int i = lane * RPL + e;
            am[e] = GK ? s_a[i] : alpha;
            kk[e] = s_k[i];
            qq[e] = s_q[i];
        }
#pragma unroll
        for (int c = 0; c < CPW; ++c) {
            float r = 0.f, pq = 0.f;
#pragma unroll
            for (int e = 0; e < RPL; ++e) {
                // r reads S (or D S with the decayed read); p reads D S
                r = fmaf(S[c][e], (GK && p.decayed_read) ? am[e] * kk[e] : kk[e], r);
                pq = fmaf(S[c][e], GK ? am[e] * qq[e] : qq[e], pq);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                r += __shfl_xor_sync(0xffffffffu, r, off);
                pq += __shfl_xor_sync(0xffffffffu, pq, off);
            }
            const int j = c0w + c;
            const float u = bt * (s_v[j] - kn * ((!GK && p.decayed_read) ? alpha * r : r));
            if (lane == c % 32) o[v_off + j] = from_f32<Tin>((GK ? 1.f : alpha) * (qn * pq) + (kn * qn * kq) * u);
#pragma unroll
            for (int e = 0; e < RPL; ++e) S[c][e] = fmaf(am[e], S[c][e], kn * kk[e] * u);
        }
    }
    }

    if (p.hT) {
#pragma unroll
        for (int c = 0; c < CPW; ++c) {
            float *dst = p.hT + vbase + (size_t)c * DK;
            if constexpr (RPL == 4) __stcs(reinterpret_cast<float4 *>(dst), make_float4(S[c][0], S[c][1], S[c][2], S[c][3]));
            else if constexpr (RPL == 2) __stcs(reinterpret_cast<float2 *>(dst), make_float2(S[c][0], S[c][1]));
            else __stcs(dst, S[c][0]);
        }
    }
}

template <typename Tin, int DK, bool GK, int DVS>
void launch_vm(const ScanParams &p, int grid, bool vm, cudaStream_t s) {
    if (vm) scan_vm_kernel<Tin, DK, DVS, GK><<<grid, kThreads, 0, s>>>(p);
    else scan_kernel<Tin, DK, DVS, GK><<<grid, kThreads, 0, s>>>(p);
}

template <typename Tin, int DK, bool GK>
cudaError_t launch_dk(const ScanParams &p, int dvs, int grid, bool vm, cudaStream_t s) {
    switch (dvs) {
        case 32: launch_vm<Tin, DK, GK, 32>(p, grid, vm, s); break;
        case 64: launch_vm<Tin, DK, GK, 64>(p, grid, vm, s); break;
        case 128: launch_vm<Tin, DK, GK, 128>(p, grid, vm, s); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

template <typename Tin, bool GK>
cudaError_t launch_typed(const ScanParams &p, int dk, int dvs, int grid, bool vm, cudaStream_t s) {
    switch (dk) {
        case 32: return launch_dk<Tin, 32, GK>(p, dvs, grid, vm, s);
        case 64: return launch_dk<Tin, 64, GK>(p, dvs, grid, vm, s);
        case 128: return launch_dk<Tin, 128, GK>(p, dvs, grid, vm, s);
        default: return cudaErrorInvalidValue;
    }
}

// gk selects the per-key-channel kernels (p.gk may still be null: no decay); vm the
// value-major state.
cudaError_t launch_scan(const ScanParams &p, DType dt, int dk, int dvs, bool gk, bool vm, cudaStream_t s) {
    const long grid = (long)p.nseq * p.H * (p.DV / dvs);
    if (grid <= 0) return cudaSuccess;
    if (grid > 0x7fffffffL) return cudaErrorInvalidConfiguration;
    if (gk)
        return dt == DType::BF16 ? launch_typed<__nv_bfloat16, true>(p, dk, dvs, (int)grid, vm, s)
                                 : launch_typed<float, true>(p, dk, dvs, (int)grid, vm, s);
    return dt == DType::BF16 ? launch_typed<__nv_bfloat16, false>(p, dk, dvs, (int)grid, vm, s)
                             : launch_typed<float, false>(p, dk, dvs, (int)grid, vm, s);
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t s) {
    ScanParams p{};
    p.q = a.q; p.k = a.k; p.v = a.v; p.beta = a.beta; p.decay = a.decay;
    p.h0 = a.state; p.hT = a.state; p.o = a.o; p.cu_seqlens = nullptr;
    p.nseq = a.B; p.T = 1; p.H = a.H; p.DV = a.dv; p.scale = a.scale; p.use_l2 = a.use_l2;
    p.gk = a.gk; p.decayed_read = a.decayed_read;
    p.A_log = a.A_log; p.dt_bias = a.dt_bias; p.beta_sig = a.beta_sig; p.neg_eig = a.neg_eig;
    p.G = a.G > 1 ? a.G : 1;
    // one CTA per head, whole value width
    return launch_scan(p, a.dtype, a.dk, a.dv, a.per_channel != 0, a.v_first != 0, s);
}

cudaError_t launch_recurrent(const SeqBatch &a, cudaStream_t s) {
    ScanParams p{};
    p.q = a.q; p.k = a.k; p.v = a.v; p.beta = a.beta; p.decay = a.decay;
    p.h0 = a.h0; p.hT = a.hT; p.o = a.o; p.cu_seqlens = a.cu_seqlens;
    p.nseq = a.nseq; p.T = a.T; p.H = a.H; p.DV = a.dv; p.scale = a.scale; p.use_l2 = a.use_l2;
    p.gk = a.gk; p.decayed_read = a.decayed_read;
    p.A_log = a.A_log; p.dt_bias = a.dt_bias; p.beta_sig = a.beta_sig; p.neg_eig = a.neg_eig;
    p.G = a.G > 1 ? a.G : 1;
    // 32-column slabs: a long prefill is latency-bound per token, so spread the
    // independent value columns over more CTAs.
    return launch_scan(p, a.dtype, a.dk, 32, a.per_channel != 0, a.v_first != 0, s);
}

}  // namespace kda
