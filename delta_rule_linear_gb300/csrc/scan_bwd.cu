// scan_bwd.cu -- gradients of the per-key-channel recurrence, token by token.
//
// The forward (TileOPs KDAFwdOp: D_t = diag(exp g_t); ejkernel kda(), "The core recurrence",
// or the gated delta rule with the decayed read), per (sequence, head):
//     u_t = beta_t (v_t - R_t^T k^_t),  R_t = h_{t-1} or D_t h_{t-1}
//     h_t = D_t h_{t-1} + k^_t u_t^T,   o_t = h_t^T q~_t
// Walking t backwards with dh the gradient of the state after token t (dh_T = the final
// state's gradient), the gradients are (i key rows, j value columns):
//     dh      += q~_t do_t^T
//     du_j     = sum_i dh[i,j] k^_i,          dv_t = beta_t du,   dbeta_t = du . (v_t - r)
//     dq~_i    = sum_j h_t[i,j] do_j
//     dk^_i    = sum_j dh[i,j] u_j - beta_t sum_j R[i,j] du_j
//     dg_i     = a_i (sum_j dh[i,j] h_{t-1}[i,j] - [decayed read] beta_t k^_i sum_j h_{t-1}[i,j] du_j)
//     dh      <- D_t dh - beta_t (k^ or D_t k^) du^T                          (now for h_{t-1})
// with r = R^T k^ and a = exp(g_t).  The states h_{t-1} come back chunk by chunk: a forward
// pass stores the state at every chunk start; the backward pass recomputes one chunk's
// states into a scratch slab and walks it in reverse.  Each CTA owns a slab of value
// columns (everything above is separable in j except the sums over j, which go to fp32
// accumulators by atomic adds).  A last kernel turns the gradients of k^ and q~ into those
// of the raw k and q (through the L2 normalisation and the scale).
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kThreads = 256;
constexpr int kBwdChunk = 32;   // tokens between stored states
constexpr int kSlab = 64;       // value columns per CTA

struct BwdParams {
    const void *q, *k, *v, *dout;
    const float *beta, *gk, *h0, *dhT;
    float *dq, *dk, *dv, *dbeta, *dg, *dh0;   // dq, dk: accumulators of the gradients of q~, k^
    float *ckpt;                              // [nseq, H, nc, DK, DV]
    float *scratch;                           // [grid, kBwdChunk, DK, DVS]
    int nseq, T, H, DV, nc;
    float scale;
    int use_l2, decayed_read;
};

template <int DVS>
struct BwdLayout {
    static constexpr int TPR = DVS / 4;          // threads per state row (float4 each)
    static constexpr int RG = kThreads / TPR;    // row groups
};

// Token staging shared by both passes: k^, q~, exp(g) per key row, beta, v (and do) of the
// slab, and the norms.  Returns nothing; fills the shared arrays and syncs twice.
template <typename Tin, int DK, int DVS>
__device__ __forceinline__ void stage_token(const BwdParams &p, long row, int h, int col0, bool with_do,
                                            float *s_k, float *s_q, float *s_a, float *s_v, float *s_do,
                                            float *s_sc) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const Tin *q = static_cast<const Tin *>(p.q);
    const Tin *k = static_cast<const Tin *>(p.k);
    const Tin *v = static_cast<const Tin *>(p.v);
    const Tin *dout = static_cast<const Tin *>(p.dout);
    const size_t qk_off = ((size_t)row * p.H + h) * DK;
    const size_t v_off = ((size_t)row * p.H + h) * p.DV + col0;
    if (tid < DK) {
        s_k[tid] = to_f32(k[qk_off + tid]);
        s_a[tid] = p.gk ? expf(p.gk[qk_off + tid]) : 1.f;
    } else if (tid < 2 * DK) {
        s_q[tid - DK] = to_f32(q[qk_off + tid - DK]);
    }
    if (tid < DVS) {
        s_v[tid] = to_f32(v[v_off + tid]);
        if (with_do) s_do[tid] = to_f32(dout[v_off + tid]);
    }
    if (tid == 0) s_sc[0] = p.beta[(size_t)row * p.H + h];
    __syncthreads();
    if (warp < 2) {   // ||k||^2, ||q||^2
        const float *x = warp == 0 ? s_k : s_q;
        float acc = 0.f;
        for (int i = lane; i < DK; i += 32) acc = fmaf(x[i], x[i], acc);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (lane == 0) s_sc[1 + warp] = acc;
    }
    __syncthreads();
    // normalise in place (each thread its own entry, read by everyone after the next sync)
    const float kn = p.use_l2 ? 1.f / fmaxf(sqrtf(s_sc[1]), kNormEps) : 1.f;
    const float qn = p.scale * (p.use_l2 ? 1.f / fmaxf(sqrtf(s_sc[2]), kNormEps) : 1.f);
    if (tid < DK) s_k[tid] *= kn;
    else if (tid < 2 * DK) s_q[tid - DK] *= qn;
    __syncthreads();
}

// Forward pass: the state before every chunk, per (sequence, head, slab).
template <typename Tin, int DK, int DVS>
__global__ void __launch_bounds__(kThreads) bwd_ckpt_kernel(BwdParams p) {
    using Ly = BwdLayout<DVS>;
    constexpr int TPR = Ly::TPR, RG = Ly::RG, R = DK / RG;
    __shared__ __align__(16) float s_k[DK], s_q[DK], s_a[DK], s_v[DVS], s_do[DVS];
    __shared__ __align__(16) float s_red[RG][DVS];
    __shared__ float s_u[DVS], s_sc[8];
    const int nslab = p.DV / DVS;
    const int slab = blockIdx.x % nslab, h = (blockIdx.x / nslab) % p.H, n = blockIdx.x / (nslab * p.H);
    const int tid = threadIdx.x, cg = tid % TPR, rg = tid / TPR, col0 = slab * DVS;
    const size_t sb = ((size_t)n * p.H + h) * DK * p.DV + col0 + 4 * cg;
    float4 S[R];
#pragma unroll
    for (int m = 0; m < R; ++m)
        S[m] = p.h0 ? *reinterpret_cast<const float4 *>(p.h0 + sb + (size_t)(rg + RG * m) * p.DV)
                    : make_float4(0.f, 0.f, 0.f, 0.f);
    for (int t = 0; t < p.T; ++t) {
        if (t % kBwdChunk == 0) {   // the state before chunk t / kBwdChunk
            float *dst = p.ckpt + (((size_t)n * p.H + h) * p.nc + t / kBwdChunk) * DK * p.DV + col0 + 4 * cg;
#pragma unroll
            for (int m = 0; m < R; ++m) *reinterpret_cast<float4 *>(dst + (size_t)(rg + RG * m) * p.DV) = S[m];
        }
        stage_token<Tin, DK, DVS>(p, (long)n * p.T + t, h, col0, false, s_k, s_q, s_a, s_v, s_do, s_sc);
        float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int m = 0; m < R; ++m) {
            const int i = rg + RG * m;
            const float kx = p.decayed_read ? s_a[i] * s_k[i] : s_k[i];
            r.x = fmaf(S[m].x, kx, r.x); r.y = fmaf(S[m].y, kx, r.y);
            r.z = fmaf(S[m].z, kx, r.z); r.w = fmaf(S[m].w, kx, r.w);
        }
        *reinterpret_cast<float4 *>(&s_red[rg][4 * cg]) = r;
        __syncthreads();
        if (tid < DVS) {
            float rs = 0.f;
            for (int g2 = 0; g2 < RG; ++g2) rs += s_red[g2][tid];
            s_u[tid] = s_sc[0] * (s_v[tid] - rs);
        }
        __syncthreads();
        const float4 u4 = *reinterpret_cast<const float4 *>(&s_u[4 * cg]);
#pragma unroll
        for (int m = 0; m < R; ++m) {
            const int i = rg + RG * m;
            const float a = s_a[i], kk = s_k[i];
            S[m].x = fmaf(a, S[m].x, kk * u4.x); S[m].y = fmaf(a, S[m].y, kk * u4.y);
            S[m].z = fmaf(a, S[m].z, kk * u4.z); S[m].w = fmaf(a, S[m].w, kk * u4.w);
        }
        __syncthreads();
    }
}

__device__ __forceinline__ float dot4(float4 a, float4 b) {
    return fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, a.w * b.w)));
}
// sum over the TPR threads that share a state row (consecutive lanes)
template <int TPR>
__device__ __forceinline__ float row_sum(float x) {
#pragma unroll
    for (int off = TPR / 2; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

// Backward pass, per (sequence, head, slab).
template <typename Tin, int DK, int DVS>
__global__ void __launch_bounds__(kThreads) bwd_kernel(BwdParams p) {
    using Ly = BwdLayout<DVS>;
    constexpr int TPR = Ly::TPR, RG = Ly::RG, R = DK / RG;
    static_assert(TPR <= 32 && 32 % TPR == 0, "a state row lies within one warp");
    __shared__ __align__(16) float s_k[DK], s_q[DK], s_a[DK], s_v[DVS], s_do[DVS];
    __shared__ __align__(16) float s_red[2][RG][DVS];
    __shared__ __align__(16) float s_u[DVS], s_du[DVS];
    __shared__ float s_sc[8], s_db[kThreads / 32];
    const int nslab = p.DV / DVS;
    const int slab = blockIdx.x % nslab, h = (blockIdx.x / nslab) % p.H, n = blockIdx.x / (nslab * p.H);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cg = tid % TPR, rg = tid / TPR, col0 = slab * DVS;
    const size_t sb = ((size_t)n * p.H + h) * DK * p.DV + col0 + 4 * cg;
    float *scr = p.scratch + (size_t)blockIdx.x * kBwdChunk * DK * DVS + 4 * cg;   // [t][i][j] slab
    float4 dH[R], Hc[R], Hp[R];
#pragma unroll
    for (int m = 0; m < R; ++m)
        dH[m] = p.dhT ? *reinterpret_cast<const float4 *>(p.dhT + sb + (size_t)(rg + RG * m) * p.DV)
                      : make_float4(0.f, 0.f, 0.f, 0.f);

    for (int c = p.nc - 1; c >= 0; --c) {
        const int t0 = c * kBwdChunk, t1 = min(p.T, t0 + kBwdChunk);
        const float *ck = p.ckpt + (((size_t)n * p.H + h) * p.nc + c) * DK * p.DV + col0 + 4 * cg;
#pragma unroll
        for (int m = 0; m < R; ++m) Hp[m] = *reinterpret_cast<const float4 *>(ck + (size_t)(rg + RG * m) * p.DV);
        // recompute the chunk: the state before each token into the scratch slab
        for (int t = t0; t < t1; ++t) {
#pragma unroll
            for (int m = 0; m < R; ++m)
                *reinterpret_cast<float4 *>(scr + ((size_t)(t - t0) * DK + rg + RG * m) * DVS) = Hp[m];
            stage_token<Tin, DK, DVS>(p, (long)n * p.T + t, h, col0, false, s_k, s_q, s_a, s_v, s_do, s_sc);
            float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int m = 0; m < R; ++m) {
                const int i = rg + RG * m;
                const float kx = p.decayed_read ? s_a[i] * s_k[i] : s_k[i];
                r.x = fmaf(Hp[m].x, kx, r.x); r.y = fmaf(Hp[m].y, kx, r.y);
                r.z = fmaf(Hp[m].z, kx, r.z); r.w = fmaf(Hp[m].w, kx, r.w);
            }
            *reinterpret_cast<float4 *>(&s_red[0][rg][4 * cg]) = r;
            __syncthreads();
            if (tid < DVS) {
                float rs = 0.f;
                for (int g2 = 0; g2 < RG; ++g2) rs += s_red[0][g2][tid];
                s_u[tid] = s_sc[0] * (s_v[tid] - rs);
            }
            __syncthreads();
            const float4 u4 = *reinterpret_cast<const float4 *>(&s_u[4 * cg]);
#pragma unroll
            for (int m = 0; m < R; ++m) {
                const int i = rg + RG * m;
                const float a = s_a[i], kk = s_k[i];
                Hp[m].x = fmaf(a, Hp[m].x, kk * u4.x); Hp[m].y = fmaf(a, Hp[m].y, kk * u4.y);
                Hp[m].z = fmaf(a, Hp[m].z, kk * u4.z); Hp[m].w = fmaf(a, Hp[m].w, kk * u4.w);
            }
            __syncthreads();
        }
#pragma unroll
        for (int m = 0; m < R; ++m) Hc[m] = Hp[m];   // the state after the chunk's last token
        // walk the chunk backwards
        for (int t = t1 - 1; t >= t0; --t) {
            const long row = (long)n * p.T + t;
#pragma unroll
            for (int m = 0; m < R; ++m)
                Hp[m] = *reinterpret_cast<const float4 *>(scr + ((size_t)(t - t0) * DK + rg + RG * m) * DVS);
            stage_token<Tin, DK, DVS>(p, row, h, col0, true, s_k, s_q, s_a, s_v, s_do, s_sc);
            const float bt = s_sc[0];
            const float4 do4 = *reinterpret_cast<const float4 *>(&s_do[4 * cg]);
            // dh += q~ do^T;  r = R^T k^;  du = dh^T k^   (both row sums through shared memory)
            float4 r = make_float4(0.f, 0.f, 0.f, 0.f), du = r;
#pragma unroll
            for (int m = 0; m < R; ++m) {
                const int i = rg + RG * m;
                const float qq = s_q[i], kk = s_k[i], kx = p.decayed_read ? s_a[i] * kk : kk;
                dH[m].x = fmaf(qq, do4.x, dH[m].x); dH[m].y = fmaf(qq, do4.y, dH[m].y);
                dH[m].z = fmaf(qq, do4.z, dH[m].z); dH[m].w = fmaf(qq, do4.w, dH[m].w);
                r.x = fmaf(Hp[m].x, kx, r.x); r.y = fmaf(Hp[m].y, kx, r.y);
                r.z = fmaf(Hp[m].z, kx, r.z); r.w = fmaf(Hp[m].w, kx, r.w);
                du.x = fmaf(dH[m].x, kk, du.x); du.y = fmaf(dH[m].y, kk, du.y);
                du.z = fmaf(dH[m].z, kk, du.z); du.w = fmaf(dH[m].w, kk, du.w);
            }
            *reinterpret_cast<float4 *>(&s_red[0][rg][4 * cg]) = r;
            *reinterpret_cast<float4 *>(&s_red[1][rg][4 * cg]) = du;
            __syncthreads();
            float dbp = 0.f;   // this column's share of dbeta
            if (tid < DVS) {
                float rs = 0.f, ds = 0.f;
                for (int g2 = 0; g2 < RG; ++g2) {
                    rs += s_red[0][g2][tid];
                    ds += s_red[1][g2][tid];
                }
                s_u[tid] = bt * (s_v[tid] - rs);
                s_du[tid] = ds;
                p.dv[((size_t)row * p.H + h) * p.DV + col0 + tid] = bt * ds;
                dbp = ds * (s_v[tid] - rs);
            }
            if (warp < (DVS + 31) / 32) {
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) dbp += __shfl_xor_sync(0xffffffffu, dbp, off);
                if (lane == 0) s_db[warp] = dbp;
            }
            __syncthreads();
            if (tid == 0) {
                float s = 0.f;
                for (int w = 0; w < (DVS + 31) / 32; ++w) s += s_db[w];
                atomicAdd(p.dbeta + (size_t)row * p.H + h, s);
            }
            const float4 u4 = *reinterpret_cast<const float4 *>(&s_u[4 * cg]);
            const float4 du4 = *reinterpret_cast<const float4 *>(&s_du[4 * cg]);
            const size_t kd_off = ((size_t)row * p.H + h) * DK;
#pragma unroll
            for (int m = 0; m < R; ++m) {
                const int i = rg + RG * m;
                const float a = s_a[i], kk = s_k[i];
                // sums over this thread's four columns, then over the row's TPR threads
                float dq_i = row_sum<TPR>(dot4(Hc[m], do4));
                const float hu = dot4(Hp[m], du4);   // sum_j h_{t-1}[i,j] du_j
                float dk_i = row_sum<TPR>(dot4(dH[m], u4) - bt * (p.decayed_read ? a : 1.f) * hu);
                float de_i = row_sum<TPR>(dot4(dH[m], Hp[m]) - (p.decayed_read ? bt * kk * hu : 0.f));
                if (cg == 0) {
                    atomicAdd(p.dq + kd_off + i, dq_i);
                    atomicAdd(p.dk + kd_off + i, dk_i);
                    if (p.dg) atomicAdd(p.dg + kd_off + i, a * de_i);
                }
                // dh for the state before token t
                const float kb = bt * (p.decayed_read ? a * kk : kk);
                dH[m].x = fmaf(a, dH[m].x, -kb * du4.x); dH[m].y = fmaf(a, dH[m].y, -kb * du4.y);
                dH[m].z = fmaf(a, dH[m].z, -kb * du4.z); dH[m].w = fmaf(a, dH[m].w, -kb * du4.w);
                Hc[m] = Hp[m];
            }
            __syncthreads();   // the staging arrays are rewritten by the next token
        }
    }
    if (p.dh0) {
#pragma unroll
        for (int m = 0; m < R; ++m) *reinterpret_cast<float4 *>(p.dh0 + sb + (size_t)(rg + RG * m) * p.DV) = dH[m];
    }
}

// dq~, dk^ (accumulated in dq, dk) -> the gradients of the raw q, k, in place:
// x^ = x / max(|x|, eps) gives dx = (dx^ - x^ (x^ . dx^)) / |x| (|x| > eps; dx^ / eps otherwise),
// and q~ = scale q^.
template <typename Tin, int DK>
__global__ void bwd_finish_kernel(BwdParams p, long rows_heads) {
    const int lane = threadIdx.x & 31;
    const long w = (blockIdx.x * (long)blockDim.x + threadIdx.x) >> 5;   // one warp per (row, head)
    if (w >= rows_heads) return;
    const Tin *q = static_cast<const Tin *>(p.q);
    const Tin *k = static_cast<const Tin *>(p.k);
    for (int which = 0; which < 2; ++which) {
        const Tin *x = which ? k : q;
        float *dx = (which ? p.dk : p.dq) + (size_t)w * DK;
        const float mult = which ? 1.f : p.scale;
        float xv[DK / 32], gv[DK / 32], nn = 0.f, xg = 0.f;
#pragma unroll
        for (int e = 0; e < DK / 32; ++e) {
            xv[e] = to_f32(x[(size_t)w * DK + lane + 32 * e]);
            gv[e] = dx[lane + 32 * e] * mult;
            nn = fmaf(xv[e], xv[e], nn);
            xg = fmaf(xv[e], gv[e], xg);
        }
        if (!p.use_l2) {
#pragma unroll
            for (int e = 0; e < DK / 32; ++e) dx[lane + 32 * e] = gv[e];
            continue;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            nn += __shfl_xor_sync(0xffffffffu, nn, off);
            xg += __shfl_xor_sync(0xffffffffu, xg, off);
        }
        const float norm = sqrtf(nn);
        if (norm > kNormEps) {
            const float inv = 1.f / norm, proj = xg * inv * inv;   // (x^ . dx^) / |x|
#pragma unroll
            for (int e = 0; e < DK / 32; ++e) dx[lane + 32 * e] = (gv[e] - xv[e] * proj) * inv;
        } else {
#pragma unroll
            for (int e = 0; e < DK / 32; ++e) dx[lane + 32 * e] = gv[e] / kNormEps;
        }
    }
}

template <typename Tin, int DK>
cudaError_t run_bwd(const BwdParams &p, long rows, cudaStream_t s) {
    const int dvs = p.DV < kSlab ? p.DV : kSlab;
    const long grid = (long)p.nseq * p.H * (p.DV / dvs);
    if (dvs == 64) {
        bwd_ckpt_kernel<Tin, DK, 64><<<(unsigned)grid, kThreads, 0, s>>>(p);
        bwd_kernel<Tin, DK, 64><<<(unsigned)grid, kThreads, 0, s>>>(p);
    } else {
        bwd_ckpt_kernel<Tin, DK, 32><<<(unsigned)grid, kThreads, 0, s>>>(p);
        bwd_kernel<Tin, DK, 32><<<(unsigned)grid, kThreads, 0, s>>>(p);
    }
    const long rh = rows * p.H;
    bwd_finish_kernel<Tin, DK><<<(unsigned)((rh * 32 + 255) / 256), 256, 0, s>>>(p, rh);
    return cudaGetLastError();
}

}  // namespace

size_t gk_bwd_scratch_bytes(int nseq, int T, int H, int dk, int dv) {
    const int nc = (T + kBwdChunk - 1) / kBwdChunk;
    const int dvs = dv < kSlab ? dv : kSlab;
    const size_t ctas = (size_t)nseq * H * (dv / dvs);
    return (size_t)nseq * H * nc * dk * dv * 4 + ctas * kBwdChunk * dk * dvs * 4;
}

cudaError_t launch_gk_bwd(const BwdArgs &a, cudaStream_t s) {
    BwdParams p{};
    p.q = a.q; p.k = a.k; p.v = a.v; p.dout = a.dout;
    p.beta = a.beta; p.gk = a.g; p.h0 = a.h0; p.dhT = a.dhT;
    p.dq = a.dq; p.dk = a.dk; p.dv = a.dv; p.dbeta = a.dbeta; p.dg = a.dg; p.dh0 = a.dh0;
    p.nseq = a.B; p.T = a.T; p.H = a.H; p.DV = a.dvdim;
    p.nc = (a.T + kBwdChunk - 1) / kBwdChunk;
    p.scale = a.scale; p.use_l2 = a.use_l2; p.decayed_read = a.decayed_read;
    p.ckpt = static_cast<float *>(a.ws);
    p.scratch = p.ckpt + (size_t)a.B * a.H * p.nc * a.dkdim * a.dvdim;
    const long rows = (long)a.B * a.T;
    cudaError_t e;
    // the sums over value columns accumulate into these
    const size_t nk = (size_t)rows * a.H * a.dkdim * sizeof(float);
    if ((e = cudaMemsetAsync(a.dq, 0, nk, s)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(a.dk, 0, nk, s)) != cudaSuccess) return e;
    if (a.dg && (e = cudaMemsetAsync(a.dg, 0, nk, s)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(a.dbeta, 0, (size_t)rows * a.H * sizeof(float), s)) != cudaSuccess) return e;
    const bool bf = a.dtype == DType::BF16;
    switch (a.dkdim) {
        case 32: return bf ? run_bwd<__nv_bfloat16, 32>(p, rows, s) : run_bwd<float, 32>(p, rows, s);
        case 64: return bf ? run_bwd<__nv_bfloat16, 64>(p, rows, s) : run_bwd<float, 64>(p, rows, s);
        case 128: return bf ? run_bwd<__nv_bfloat16, 128>(p, rows, s) : run_bwd<float, 128>(p, rows, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace kda
