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
// states into a scratch slab and walks it in reverse.  With one decay per head (D_t = a_t I)
// the same walk runs with every channel's factor equal, and the decay's gradient is the
// channel sum of dg.  Each CTA owns a slab of value
// columns (everything above is separable in j except the sums over j, which go to fp32
// accumulators by atomic adds).  A last kernel turns the gradients of k^ and q~ into those
// of the raw k and q (through the L2 normalisation and the scale).
#include <algorithm>
#include <cstddef>

#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kThreads = 256;
constexpr int kBwdChunk = 32;   // tokens between stored states
constexpr int kSlab = 64;       // value columns per CTA (32 when that leaves SMs idle)
constexpr int kAhead = 4;       // tokens whose loads are in flight in the checkpoint pass

struct BwdParams {
    const void *q, *k, *v, *dout;
    const float *beta, *gk, *h0, *dhT;
    const float *decay;                       // one decay per head [rows, H] (when gk is null)
    float *ddecay;                            // its gradient: the channel sum of dg
    float *dq, *dk, *dv, *dbeta, *dg, *dh0;   // dq, dk: accumulators of the gradients of q~, k^
    float *ckpt;                              // [nseq, H, nc, DK, DV]
    float *scratch;                           // [grid, kBwdChunk, DK, DVS]
    int nseq, T, H, DV, nc;
    // the chunk-parallel walk (bwd_chunk_kernel): the state entering every 64-token chunk and
    // the gradient of the state leaving it, bf16 key-major [nseq, H, nc64, DK, DK], and a bf16
    // scratch [grid, 64, DK, DVS] for the recomputed states
    const __nv_bfloat16 *fstates, *bstates;
    __nv_bfloat16 *scratch16;
    int nc64;
    float scale;
    int use_l2, decayed_read;
};

template <int DVS>
struct BwdLayout {
    static constexpr int TPR = DVS / 4;          // threads per state row (float4 each)
    static constexpr int RG = kThreads / TPR;    // row groups
};

// One token's inputs as this thread fetches them (raw, so the loads stay in flight until the
// token is staged): k (threads [0, DK)) or q (threads [DK, 2 DK)) of one key channel, the
// channel's log decay, v and do of one value column (threads [0, DVS)), beta (thread 0).
template <typename Tin>
struct TokenRegs {
    Tin x, v, d;
    float g, beta;
};

// The staged token: raw k, q, exp(g) per key row, v, do of the slab, beta, and per-warp sums
// of k^2 and q^2 (the norms are finished by each thread from these).
// Aligned so that both buffers of a stage array keep the 16-byte alignment of `d` (read as
// float4).
template <int DK, int DVS>
struct __align__(16) Stage {
    float k[DK], q[DK], a[DK], v[DVS], d[DVS];
    float nk[DK / 32], nq[DK / 32];
    float beta;
};
template <int DK, int DVS>
__host__ __device__ constexpr bool stage_aligned() {
    using S = Stage<DK, DVS>;
    return sizeof(S) % 16 == 0 && offsetof(S, d) % 16 == 0;
}

template <typename Tin, int DK, int DVS>
__device__ __forceinline__ void fetch_token(const BwdParams &p, long row, int h, int col0, bool with_do,
                                            TokenRegs<Tin> &r) {
    const int tid = threadIdx.x;
    const size_t qk_off = ((size_t)row * p.H + h) * DK;
    const size_t v_off = ((size_t)row * p.H + h) * p.DV + col0;
    if (tid < DK) {
        r.x = static_cast<const Tin *>(p.k)[qk_off + tid];
        // one load for either decay layout: per channel [rows, H, DK], or per head [rows, H]
        // (the same element for every channel); the pointer and offset are selected, not
        // the code path
        const float *gsrc = p.gk ? p.gk : p.decay;
        const size_t goff = p.gk ? qk_off + tid : (size_t)row * p.H + h;
        r.g = gsrc ? gsrc[goff] : 0.f;
    } else if (tid < 2 * DK) {
        r.x = static_cast<const Tin *>(p.q)[qk_off + tid - DK];
    }
    if (tid < DVS) {
        r.v = static_cast<const Tin *>(p.v)[v_off + tid];
        if (with_do) r.d = static_cast<const Tin *>(p.dout)[v_off + tid];
    }
    if (tid == 0) r.beta = p.beta[(size_t)row * p.H + h];
}

// Registers -> stage (the caller syncs before anyone reads it).
template <typename Tin, int DK, int DVS>
__device__ __forceinline__ void put_token(const BwdParams &p, const TokenRegs<Tin> &r, bool with_do,
                                          Stage<DK, DVS> &s) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid < 2 * DK) {   // whole warps
        const float x = to_f32(r.x);
        float sq = x * x;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, off);
        if (tid < DK) {
            s.k[tid] = x;
            s.a[tid] = (p.gk || p.decay) ? expf(r.g) : 1.f;
            if (lane == 0) s.nk[warp] = sq;
        } else {
            s.q[tid - DK] = x;
            if (lane == 0) s.nq[warp - DK / 32] = sq;
        }
    }
    if (tid < DVS) {
        s.v[tid] = to_f32(r.v);
        if (with_do) s.d[tid] = to_f32(r.d);
    }
    if (tid == 0) s.beta = r.beta;
}

// The normalisation factors of the staged token: k^ = kn k, q~ = qn q.
template <int DK, int DVS>
__device__ __forceinline__ void token_norms(const BwdParams &p, const Stage<DK, DVS> &s, float &kn, float &qn) {
    float nk = 0.f, nq = 0.f;
#pragma unroll
    for (int w = 0; w < DK / 32; ++w) {
        nk += s.nk[w];
        nq += s.nq[w];
    }
    // 1 / max(|x|, eps) = rsqrt(max(|x|^2, eps^2))
    kn = p.use_l2 ? rsqrtf(fmaxf(nk, kNormEps * kNormEps)) : 1.f;
    qn = p.scale * (p.use_l2 ? rsqrtf(fmaxf(nq, kNormEps * kNormEps)) : 1.f);
}

// A token as the steps read it: raw k, q and exp(g) per key row, v and do of the slab,
// beta, and the normalisation factors (k^ = kn k, q~ = qn q).  StageTok reads a staged
// token (Stage), ChunkTok one token of a chunk staged whole (the chunk-parallel walk).
template <int DK, int DVS>
struct StageTok {
    const Stage<DK, DVS> &s;
    float kn, qn;
    __device__ float k(int i) const { return s.k[i]; }
    __device__ float q(int i) const { return s.q[i]; }
    __device__ float a(int i) const { return s.a[i]; }
    __device__ float v(int j) const { return s.v[j]; }
    __device__ float4 d4(int j0) const { return *reinterpret_cast<const float4 *>(&s.d[j0]); }
    __device__ float beta() const { return s.beta; }
};
template <int DK, int DVS>
__device__ __forceinline__ StageTok<DK, DVS> stage_tok(const BwdParams &p, const Stage<DK, DVS> &s) {
    float kn, qn;
    token_norms(p, s, kn, qn);
    return StageTok<DK, DVS>{s, kn, qn};
}

// Sums over the RG row groups of one or two [RG][DVS] partial arrays.  Column j's sums land
// in its owner thread (returns true there): the first DVS threads with few row groups, else
// P = kThreads / DVS consecutive lanes per column that each add RG / P terms and shuffle.
template <int DVS, int RG, bool TWO>
__device__ __forceinline__ bool column_sums(const float (*a)[DVS], const float (*b)[DVS], int tid, int &j,
                                            float &sa, float &sb) {
    sa = 0.f;
    sb = 0.f;
    if constexpr (RG <= 8) {
        j = tid;
        if (tid >= DVS) return false;
#pragma unroll
        for (int g = 0; g < RG; ++g) {
            sa += a[g][tid];
            if (TWO) sb += b[g][tid];
        }
        return true;
    } else {
        constexpr int P = kThreads / DVS, PER = RG / P;
        static_assert(P * DVS == kThreads && PER * P == RG && P <= 32, "reduction split");
        const int part = tid % P;
        j = tid / P;
#pragma unroll
        for (int e = 0; e < PER; ++e) {
            sa += a[part * PER + e][j];
            if (TWO) sb += b[part * PER + e][j];
        }
#pragma unroll
        for (int off = P / 2; off > 0; off >>= 1) {
            sa += __shfl_xor_sync(0xffffffffu, sa, off);
            if (TWO) sb += __shfl_xor_sync(0xffffffffu, sb, off);
        }
        return part == 0;
    }
}

// One token of the forward recurrence on this thread's rows of the slab (S: the state before
// the token on entry, after it on return).  The stage was synced by the caller; two syncs.
// y_out (optional, DVS floats): the token's v - r, kept for its backward step.
template <int DK, int DVS, int RG, int R, bool DR, typename Tok>
__device__ __forceinline__ void forward_token(const BwdParams &p, const Tok &s, float4 (&S)[R],
                                              float (*s_red)[DVS], float *s_u, float *y_out = nullptr) {
    const int tid = threadIdx.x, cg = tid % (DVS / 4), rg = tid / (DVS / 4);
    const float kn = s.kn;
    float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int m = 0; m < R; ++m) {
        const int i = rg + RG * m;
        const float kk = s.k(i) * kn, kx = DR ? s.a(i) * kk : kk;
        r.x = fmaf(S[m].x, kx, r.x); r.y = fmaf(S[m].y, kx, r.y);
        r.z = fmaf(S[m].z, kx, r.z); r.w = fmaf(S[m].w, kx, r.w);
    }
    *reinterpret_cast<float4 *>(&s_red[rg][4 * cg]) = r;
    __syncthreads();
    {
        int j;
        float rs, unused;
        if (column_sums<DVS, RG, false>(s_red, s_red, tid, j, rs, unused)) {
            const float y = s.v(j) - rs;
            s_u[j] = s.beta() * y;
            if (y_out) y_out[j] = y;
        }
    }
    __syncthreads();
    const float4 u4 = *reinterpret_cast<const float4 *>(&s_u[4 * cg]);
#pragma unroll
    for (int m = 0; m < R; ++m) {
        const int i = rg + RG * m;
        const float a = s.a(i), kk = s.k(i) * kn;
        S[m].x = fmaf(a, S[m].x, kk * u4.x); S[m].y = fmaf(a, S[m].y, kk * u4.y);
        S[m].z = fmaf(a, S[m].z, kk * u4.z); S[m].w = fmaf(a, S[m].w, kk * u4.w);
    }
}

// Forward pass: the state before every chunk, per (sequence, head, slab).  Each token's
// inputs are fetched one token ahead; the stage is double-buffered, so three syncs a token.
// DR: the delta term reads the decayed state (the decayed read), a compile-time choice
template <typename Tin, int DK, int DVS, bool DR>
__global__ void __launch_bounds__(kThreads) bwd_ckpt_kernel(BwdParams p) {
    using Ly = BwdLayout<DVS>;
    constexpr int TPR = Ly::TPR, RG = Ly::RG, R = DK / RG;
    static_assert(stage_aligned<DK, DVS>(), "both stage buffers 16-byte aligned");
    __shared__ __align__(16) Stage<DK, DVS> st[2];
    __shared__ __align__(16) float s_red[RG][DVS];
    __shared__ __align__(16) float s_u[DVS];
    const int nslab = p.DV / DVS;
    const int slab = blockIdx.x % nslab, h = (blockIdx.x / nslab) % p.H, n = blockIdx.x / (nslab * p.H);
    const int tid = threadIdx.x, cg = tid % TPR, rg = tid / TPR, col0 = slab * DVS;
    const size_t sb = ((size_t)n * p.H + h) * DK * p.DV + col0 + 4 * cg;
    float4 S[R];
#pragma unroll
    for (int m = 0; m < R; ++m)
        S[m] = p.h0 ? *reinterpret_cast<const float4 *>(p.h0 + sb + (size_t)(rg + RG * m) * p.DV)
                    : make_float4(0.f, 0.f, 0.f, 0.f);
    // This pass is the first to read the inputs (from DRAM): a ring of kAhead tokens' loads
    // stays in flight, each slot refilled as soon as its token is staged (the ring index is
    // a compile-time constant of the unrolled inner loop, so the slots stay in registers).
    TokenRegs<Tin> ring[kAhead];
#pragma unroll
    for (int j = 0; j < kAhead; ++j)
        if (j < p.T) fetch_token<Tin, DK, DVS>(p, (long)n * p.T + j, h, col0, false, ring[j]);
    for (int t0 = 0; t0 < p.T; t0 += kAhead) {
#pragma unroll
        for (int j = 0; j < kAhead; ++j) {
            const int t = t0 + j;
            if (t >= p.T) break;
            if (t % kBwdChunk == 0) {   // the state before chunk t / kBwdChunk
                float *dst = p.ckpt + (((size_t)n * p.H + h) * p.nc + t / kBwdChunk) * DK * p.DV + col0 + 4 * cg;
#pragma unroll
                for (int m = 0; m < R; ++m) *reinterpret_cast<float4 *>(dst + (size_t)(rg + RG * m) * p.DV) = S[m];
            }
            Stage<DK, DVS> &s = st[j & 1];
            put_token<Tin, DK, DVS>(p, ring[j], false, s);
            __syncthreads();
            if (t + kAhead < p.T) fetch_token<Tin, DK, DVS>(p, (long)n * p.T + t + kAhead, h, col0, false, ring[j]);
            forward_token<DK, DVS, RG, R, DR>(p, stage_tok(p, s), S, s_red, s_u);
        }
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

// One token of the backward walk: the stage holds token `row` (synced by the caller), Hp is
// the state before it and Hc the state after it (Hc becomes Hp on return), dH the gradient
// of the state after it on entry and of the state before it on return.  Writes the token's
// dv columns and adds its shares of dbeta, dq~, dk^, dg and ddecay.  Two syncs.  KY: the
// token's v - r was kept by its forward step (ys, DVS floats) and is not recomputed.
template <int DK, int DVS, int RG, int R, bool DR, bool KY = false, typename Tok>
__device__ __forceinline__ void backward_token(const BwdParams &p, const Tok &s, long row, int h,
                                               int col0, float4 (&dH)[R], float4 (&Hc)[R], const float4 (&Hp)[R],
                                               float (*s_red)[RG][DVS], float *s_u, float *s_du, float *s_db,
                                               const float *ys = nullptr) {
    constexpr int TPR = DVS / 4;
    constexpr int kOwnerWarps = RG <= 8 ? (DVS + 31) / 32 : kThreads / 32;   // warps holding column sums
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cg = tid % TPR, rg = tid / TPR;
    const float kn = s.kn, qn = s.qn;
    const float bt = s.beta();
    const float4 do4 = s.d4(4 * cg);
    // dh += q~ do^T;  r = R^T k^;  du = dh^T k^   (both row sums through shared memory)
    float4 r = make_float4(0.f, 0.f, 0.f, 0.f), du = r;
#pragma unroll
    for (int m = 0; m < R; ++m) {
        const int i = rg + RG * m;
        const float qq = s.q(i) * qn, kk = s.k(i) * kn, kx = DR ? s.a(i) * kk : kk;
        dH[m].x = fmaf(qq, do4.x, dH[m].x); dH[m].y = fmaf(qq, do4.y, dH[m].y);
        dH[m].z = fmaf(qq, do4.z, dH[m].z); dH[m].w = fmaf(qq, do4.w, dH[m].w);
        if (!KY) {
            r.x = fmaf(Hp[m].x, kx, r.x); r.y = fmaf(Hp[m].y, kx, r.y);
            r.z = fmaf(Hp[m].z, kx, r.z); r.w = fmaf(Hp[m].w, kx, r.w);
        }
        du.x = fmaf(dH[m].x, kk, du.x); du.y = fmaf(dH[m].y, kk, du.y);
        du.z = fmaf(dH[m].z, kk, du.z); du.w = fmaf(dH[m].w, kk, du.w);
    }
    if (!KY) *reinterpret_cast<float4 *>(&s_red[0][rg][4 * cg]) = r;
    *reinterpret_cast<float4 *>(&s_red[1][rg][4 * cg]) = du;
    __syncthreads();
    float dbp = 0.f;   // this column's share of dbeta
    {
        int j;
        float rs = 0.f, ds;
        const bool owner = KY ? column_sums<DVS, RG, false>(s_red[1], s_red[1], tid, j, ds, rs)
                              : column_sums<DVS, RG, true>(s_red[0], s_red[1], tid, j, rs, ds);
        if (owner) {
            const float y = KY ? ys[j] : s.v(j) - rs;
            s_u[j] = bt * y;
            s_du[j] = ds;
            p.dv[((size_t)row * p.H + h) * p.DV + col0 + j] = bt * ds;
            dbp = ds * y;
        }
    }
    if (warp < kOwnerWarps) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) dbp += __shfl_xor_sync(0xffffffffu, dbp, off);
        if (lane == 0) s_db[warp] = dbp;
    }
    __syncthreads();
    if (tid == 0) {
        float sum = 0.f;
        for (int w = 0; w < kOwnerWarps; ++w) sum += s_db[w];
        atomicAdd(p.dbeta + (size_t)row * p.H + h, sum);
    }
    const float4 u4 = *reinterpret_cast<const float4 *>(&s_u[4 * cg]);
    const float4 du4 = *reinterpret_cast<const float4 *>(&s_du[4 * cg]);
    const size_t kd_off = ((size_t)row * p.H + h) * DK;
    if constexpr (TPR == 8 && R == 4) {
        // The twelve row sums of this thread's rows (dq, dk, de of each of its four rows) by a
        // transposing reduction over the 8 lanes of the row group: each step halves the values
        // a lane carries (12 shuffles instead of 36), and lanes 2m, 2m + 1 of the group end
        // with row m's three sums.
        float x[12];
#pragma unroll
        for (int m = 0; m < R; ++m) {
            const int i = rg + RG * m;
            const float a = s.a(i), kk = s.k(i) * kn;
            const float hu = dot4(Hp[m], du4);   // sum_j h_{t-1}[i,j] du_j
            x[3 * m] = dot4(Hc[m], do4);
            x[3 * m + 1] = dot4(dH[m], u4) - bt * (DR ? a : 1.f) * hu;
            x[3 * m + 2] = dot4(dH[m], Hp[m]) - (DR ? bt * kk * hu : 0.f);
            // dh for the state before token t
            const float kb = bt * (DR ? a * kk : kk);
            dH[m].x = fmaf(a, dH[m].x, -kb * du4.x); dH[m].y = fmaf(a, dH[m].y, -kb * du4.y);
            dH[m].z = fmaf(a, dH[m].z, -kb * du4.z); dH[m].w = fmaf(a, dH[m].w, -kb * du4.w);
            Hc[m] = Hp[m];
        }
        const bool hi4 = (cg & 4) != 0, hi2 = (cg & 2) != 0;
        float y[6], z[3];
#pragma unroll
        for (int v = 0; v < 6; ++v)   // rows 0, 1 stay with cg < 4, rows 2, 3 with cg >= 4
            y[v] = (hi4 ? x[6 + v] : x[v]) + __shfl_xor_sync(0xffffffffu, hi4 ? x[v] : x[6 + v], 4);
#pragma unroll
        for (int v = 0; v < 3; ++v)   // then the even row with bit 1 clear, the odd one with it set
            z[v] = (hi2 ? y[3 + v] : y[v]) + __shfl_xor_sync(0xffffffffu, hi2 ? y[v] : y[3 + v], 2);
#pragma unroll
        for (int v = 0; v < 3; ++v) z[v] += __shfl_xor_sync(0xffffffffu, z[v], 1);
        const int i = rg + RG * ((cg >> 1) & 3);
        const float a = s.a(i);
        if ((cg & 1) == 0) {
            atomicAdd(p.dq + kd_off + i, z[0]);
            atomicAdd(p.dk + kd_off + i, z[1]);
            if (p.dg) atomicAdd(p.dg + kd_off + i, a * z[2]);
        }
        if (p.ddecay) {   // one decay per head: sum over the warp's rows of a_i de_i
            float dd = (cg & 1) == 0 ? a * z[2] : 0.f;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) dd += __shfl_xor_sync(0xffffffffu, dd, off);
            if (lane == 0) atomicAdd(p.ddecay + (size_t)row * p.H + h, dd);
        }
        return;
    }
    float dd = 0.f;   // one decay per head: sum over this thread's rows of a_i de_i
#pragma unroll
    for (int m = 0; m < R; ++m) {
        const int i = rg + RG * m;
        const float a = s.a(i), kk = s.k(i) * kn;
        // sums over this thread's four columns, then over the row's TPR threads
        float dq_i = row_sum<TPR>(dot4(Hc[m], do4));
        const float hu = dot4(Hp[m], du4);   // sum_j h_{t-1}[i,j] du_j
        float dk_i = row_sum<TPR>(dot4(dH[m], u4) - bt * (DR ? a : 1.f) * hu);
        float de_i = row_sum<TPR>(dot4(dH[m], Hp[m]) - (DR ? bt * kk * hu : 0.f));
        if (cg == 0) {
            atomicAdd(p.dq + kd_off + i, dq_i);
            atomicAdd(p.dk + kd_off + i, dk_i);
            if (p.dg) atomicAdd(p.dg + kd_off + i, a * de_i);
        }
        dd = fmaf(a, de_i, dd);
        // dh for the state before token t
        const float kb = bt * (DR ? a * kk : kk);
        dH[m].x = fmaf(a, dH[m].x, -kb * du4.x); dH[m].y = fmaf(a, dH[m].y, -kb * du4.y);
        dH[m].z = fmaf(a, dH[m].z, -kb * du4.z); dH[m].w = fmaf(a, dH[m].w, -kb * du4.w);
        Hc[m] = Hp[m];
    }
    if (p.ddecay) {   // the row groups of the warp (every lane of a group holds its sum)
#pragma unroll
        for (int off = TPR; off < 32; off <<= 1) dd += __shfl_xor_sync(0xffffffffu, dd, off);
        if (lane == 0) atomicAdd(p.ddecay + (size_t)row * p.H + h, dd);
    }
}

// Backward pass, per (sequence, head, slab).  Inputs fetched one token ahead (forwards in the
// recomputation, backwards in the walk) into a double-buffered stage, as in the forward pass.
template <typename Tin, int DK, int DVS, bool DR>
__global__ void __launch_bounds__(kThreads) bwd_kernel(BwdParams p) {
    using Ly = BwdLayout<DVS>;
    constexpr int TPR = Ly::TPR, RG = Ly::RG, R = DK / RG;
    static_assert(TPR <= 32 && 32 % TPR == 0, "a state row lies within one warp");
    static_assert(stage_aligned<DK, DVS>(), "both stage buffers 16-byte aligned");
    __shared__ __align__(16) Stage<DK, DVS> st[2];
    __shared__ __align__(16) float s_red[2][RG][DVS];
    __shared__ __align__(16) float s_u[DVS];
    __shared__ __align__(16) float s_du[DVS];
    __shared__ float s_db[kThreads / 32];
    const int nslab = p.DV / DVS;
    const int slab = blockIdx.x % nslab, h = (blockIdx.x / nslab) % p.H, n = blockIdx.x / (nslab * p.H);
    const int tid = threadIdx.x;
    const int cg = tid % TPR, rg = tid / TPR, col0 = slab * DVS;
    const size_t sb = ((size_t)n * p.H + h) * DK * p.DV + col0 + 4 * cg;
    float *scr = p.scratch + (size_t)blockIdx.x * kBwdChunk * DK * DVS + 4 * cg;   // [t][i][j] slab
    float4 dH[R], Hc[R], Hp[R];
#pragma unroll
    for (int m = 0; m < R; ++m)
        dH[m] = p.dhT ? *reinterpret_cast<const float4 *>(p.dhT + sb + (size_t)(rg + RG * m) * p.DV)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
    TokenRegs<Tin> cur{}, nxt{};
    int it = 0;   // tokens staged so far: selects the stage buffer

    for (int c = p.nc - 1; c >= 0; --c) {
        const int t0 = c * kBwdChunk, t1 = min(p.T, t0 + kBwdChunk);
        const float *ck = p.ckpt + (((size_t)n * p.H + h) * p.nc + c) * DK * p.DV + col0 + 4 * cg;
#pragma unroll
        for (int m = 0; m < R; ++m) Hp[m] = *reinterpret_cast<const float4 *>(ck + (size_t)(rg + RG * m) * p.DV);
        // recompute the chunk: the state before each token into the scratch slab
        fetch_token<Tin, DK, DVS>(p, (long)n * p.T + t0, h, col0, false, cur);
        for (int t = t0; t < t1; ++t, ++it) {
#pragma unroll
            for (int m = 0; m < R; ++m)
                *reinterpret_cast<float4 *>(scr + ((size_t)(t - t0) * DK + rg + RG * m) * DVS) = Hp[m];
            Stage<DK, DVS> &s = st[it & 1];
            put_token<Tin, DK, DVS>(p, cur, false, s);
            __syncthreads();
            if (t + 1 < t1) fetch_token<Tin, DK, DVS>(p, (long)n * p.T + t + 1, h, col0, false, nxt);
            forward_token<DK, DVS, RG, R, DR>(p, stage_tok(p, s), Hp, s_red[0], s_u);
            cur = nxt;
        }
#pragma unroll
        for (int m = 0; m < R; ++m) Hc[m] = Hp[m];   // the state after the chunk's last token
        // walk the chunk backwards
        fetch_token<Tin, DK, DVS>(p, (long)n * p.T + t1 - 1, h, col0, true, cur);
        for (int t = t1 - 1; t >= t0; --t, ++it) {
            const long row = (long)n * p.T + t;
#pragma unroll
            for (int m = 0; m < R; ++m)
                Hp[m] = *reinterpret_cast<const float4 *>(scr + ((size_t)(t - t0) * DK + rg + RG * m) * DVS);
            Stage<DK, DVS> &s = st[it & 1];
            put_token<Tin, DK, DVS>(p, cur, true, s);
            __syncthreads();
            if (t > t0) fetch_token<Tin, DK, DVS>(p, row - 1, h, col0, true, nxt);
            backward_token<DK, DVS, RG, R, DR>(p, stage_tok(p, s), row, h, col0, dH, Hc, Hp, s_red, s_u, s_du, s_db);
            cur = nxt;
        }
    }
    if (p.dh0) {
#pragma unroll
        for (int m = 0; m < R; ++m) *reinterpret_cast<float4 *>(p.dh0 + sb + (size_t)(rg + RG * m) * p.DV) = dH[m];
    }
}

// Chunk-parallel backward (bf16, dk == dv): the same token walk, but every 64-token chunk on
// its own.  A forward launch on the tensor cores keeps the state entering each chunk, and
// the reverse walk over the chunk maps gives the gradient of the state leaving it (both in
// bf16); with those a unit -- (chunk, sequence, head, value slab) -- depends on no other
// unit.  A unit stages its whole chunk in shared memory, recomputes the chunk's states into
// its scratch (bf16; two tokens per pair of barriers) keeping each token's v - r, and walks
// them in reverse, adding its shares of dq~, dk^, dbeta and dg as the sequential walk does;
// the state before the next token of the reverse walk is loaded one token ahead.
// Persistent CTAs take the units in (chunk, sequence, head, slab) order, so that the CTAs
// running at one time read the same tokens.
constexpr int kUnitTokens = 64;   // the tensor-core chunk
constexpr int kUnitSlab = 32;     // value columns per unit
constexpr int kChunkBwdCtas = 304;   // persistent CTAs (two per SM on 152 SMs)

// 16-byte global -> shared copy (both addresses 16-byte aligned), and the wait for every copy
// this thread has issued
__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;"
                 :: "r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ float4 bf16x4_to_float4(uint2 w) {
    return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u),
                       __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
}
__device__ __forceinline__ float4 ld_bf16x4(const __nv_bfloat16 *src) {
    return bf16x4_to_float4(*reinterpret_cast<const uint2 *>(src));
}
__device__ __forceinline__ void st_bf16x4(__nv_bfloat16 *dst, float4 v) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
    *reinterpret_cast<uint2 *>(dst) = make_uint2(*reinterpret_cast<const uint32_t *>(&a),
                                                 *reinterpret_cast<const uint32_t *>(&b));
}

// One token of the staged chunk, read like a staged token: raw k, q (bf16), exp(g), v and do
// of the slab (bf16), beta and the normalisation factors.
template <int DK, int DVS>
struct ChunkTok {
    const __nv_bfloat16 *kr, *qr, *vr, *dr;
    const float *ar;
    float kn, qn, b;
    __device__ float k(int i) const { return __bfloat162float(kr[i]); }
    __device__ float q(int i) const { return __bfloat162float(qr[i]); }
    __device__ float a(int i) const { return ar[i]; }
    __device__ float v(int j) const { return __bfloat162float(vr[j]); }
    __device__ float4 d4(int j0) const { return ld_bf16x4(dr + j0); }
    __device__ float beta() const { return b; }
};

// The chunk staged whole in shared memory (dynamic): raw k, q rows [64][DK] bf16, exp(g)
// [64][DK] fp32, the v and do columns of the slab [64][DVS] bf16, and beta, kn, qn [64].
template <int DK, int DVS>
struct ChunkStage {
    static constexpr int K = 0, Q = K + kUnitTokens * DK * 2, A = Q + kUnitTokens * DK * 2;
    static constexpr int V = A + kUnitTokens * DK * 4, D = V + kUnitTokens * DVS * 2;
    static constexpr int BETA = D + kUnitTokens * DVS * 2, KN = BETA + kUnitTokens * 4, QN = KN + kUnitTokens * 4;
    static constexpr int CD = QN + kUnitTokens * 4;   // k^_{t-1} . kx_t (kx: k^, or exp(g) k^ with the decayed read)
    static constexpr int BYTES = CD + kUnitTokens * 4;
};

// Two tokens of the forward recurrence (t0, then t1) with two barriers: the state after t0 is
// a_0 S + k^_0 u_0^T, so t1's read-out is S^T (a_0 kx_1) + u_0 (k^_0 . kx_1), and one pass over
// S gives both tokens' column sums.  c01 = k^_0 . kx_1.  S holds the state before t0 on entry
// and after t1 on return; mid receives the state between them (after t0).  y0, y1: the tokens'
// v - r, kept for their backward steps.
template <int DK, int DVS, int RG, int R, bool DR, typename Tok>
__device__ __forceinline__ void forward_pair(const Tok &s0, const Tok &s1, float c01, float4 (&S)[R],
                                             __nv_bfloat16 *mid, float (*s_red)[RG][DVS], float (*s_u2)[DVS],
                                             float *y0, float *y1) {
    const int tid = threadIdx.x, cg = tid % (DVS / 4), rg = tid / (DVS / 4);
    float4 r0 = make_float4(0.f, 0.f, 0.f, 0.f), r1 = r0;
#pragma unroll
    for (int m = 0; m < R; ++m) {
        const int i = rg + RG * m;
        const float k0 = s0.k(i) * s0.kn, kx0 = DR ? s0.a(i) * k0 : k0;
        const float k1 = s1.k(i) * s1.kn, w1 = s0.a(i) * (DR ? s1.a(i) * k1 : k1);
        r0.x = fmaf(S[m].x, kx0, r0.x); r0.y = fmaf(S[m].y, kx0, r0.y);
        r0.z = fmaf(S[m].z, kx0, r0.z); r0.w = fmaf(S[m].w, kx0, r0.w);
        r1.x = fmaf(S[m].x, w1, r1.x); r1.y = fmaf(S[m].y, w1, r1.y);
        r1.z = fmaf(S[m].z, w1, r1.z); r1.w = fmaf(S[m].w, w1, r1.w);
    }
    *reinterpret_cast<float4 *>(&s_red[0][rg][4 * cg]) = r0;
    *reinterpret_cast<float4 *>(&s_red[1][rg][4 * cg]) = r1;
    __syncthreads();
    {
        int j;
        float rs0, rs1;
        if (column_sums<DVS, RG, true>(s_red[0], s_red[1], tid, j, rs0, rs1)) {
            const float ya = s0.v(j) - rs0, ua = s0.beta() * ya;
            const float yb = s1.v(j) - rs1 - c01 * ua;
            s_u2[0][j] = ua;
            s_u2[1][j] = s1.beta() * yb;
            y0[j] = ya;
            y1[j] = yb;
        }
    }
    __syncthreads();
    const float4 u0 = *reinterpret_cast<const float4 *>(&s_u2[0][4 * cg]);
    const float4 u1 = *reinterpret_cast<const float4 *>(&s_u2[1][4 * cg]);
#pragma unroll
    for (int m = 0; m < R; ++m) {
        const int i = rg + RG * m;
        const float a0 = s0.a(i), k0 = s0.k(i) * s0.kn;
        S[m].x = fmaf(a0, S[m].x, k0 * u0.x); S[m].y = fmaf(a0, S[m].y, k0 * u0.y);
        S[m].z = fmaf(a0, S[m].z, k0 * u0.z); S[m].w = fmaf(a0, S[m].w, k0 * u0.w);
        st_bf16x4(mid + (size_t)i * DVS, S[m]);
        const float a1 = s1.a(i), k1 = s1.k(i) * s1.kn;
        S[m].x = fmaf(a1, S[m].x, k1 * u1.x); S[m].y = fmaf(a1, S[m].y, k1 * u1.y);
        S[m].z = fmaf(a1, S[m].z, k1 * u1.z); S[m].w = fmaf(a1, S[m].w, k1 * u1.w);
    }
}

template <int DK, int DVS, bool DR>
__global__ void __launch_bounds__(kThreads, 2) bwd_chunk_kernel(BwdParams p) {
    using Ly = BwdLayout<DVS>;
    using CS = ChunkStage<DK, DVS>;
    constexpr int TPR = Ly::TPR, RG = Ly::RG, R = DK / RG;
    static_assert(TPR <= 32 && 32 % TPR == 0, "a state row lies within one warp");
    extern __shared__ __align__(16) uint8_t chunk_smem[];
    __nv_bfloat16 *ck = reinterpret_cast<__nv_bfloat16 *>(chunk_smem + CS::K);
    __nv_bfloat16 *cq = reinterpret_cast<__nv_bfloat16 *>(chunk_smem + CS::Q);
    float *ca = reinterpret_cast<float *>(chunk_smem + CS::A);
    __nv_bfloat16 *cv = reinterpret_cast<__nv_bfloat16 *>(chunk_smem + CS::V);
    __nv_bfloat16 *cd = reinterpret_cast<__nv_bfloat16 *>(chunk_smem + CS::D);
    float *cbeta = reinterpret_cast<float *>(chunk_smem + CS::BETA);
    float *ckn = reinterpret_cast<float *>(chunk_smem + CS::KN);
    float *cqn = reinterpret_cast<float *>(chunk_smem + CS::QN);
    float *ccd = reinterpret_cast<float *>(chunk_smem + CS::CD);
    __shared__ __align__(16) float s_red[2][RG][DVS];
    __shared__ __align__(16) float s_u[DVS];
    __shared__ __align__(16) float s_du[DVS];
    __shared__ __align__(16) float s_u2[2][DVS];
    __shared__ float s_db[kThreads / 32];
    __shared__ float s_y[kUnitTokens][DVS];   // each token's v - r, from the recomputation
    const int tid = threadIdx.x, cg = tid % TPR, rg = tid / TPR;
    constexpr int nslab = DK / DVS;   // dv == dk
    const long units = (long)p.nc64 * p.nseq * p.H * nslab;
    // this thread's element of the scratch: [token][row][column] of the unit's slab
    __nv_bfloat16 *scr = p.scratch16 + (size_t)blockIdx.x * kUnitTokens * DK * DVS + 4 * cg;
    const __nv_bfloat16 *gq = static_cast<const __nv_bfloat16 *>(p.q);
    const __nv_bfloat16 *gk = static_cast<const __nv_bfloat16 *>(p.k);
    const __nv_bfloat16 *gv = static_cast<const __nv_bfloat16 *>(p.v);
    const __nv_bfloat16 *gdo = static_cast<const __nv_bfloat16 *>(p.dout);
    for (long u = blockIdx.x; u < units; u += gridDim.x) {
        const int slab = (int)(u % nslab);
        const long r = u / nslab;
        const int h = (int)(r % p.H), n = (int)((r / p.H) % p.nseq), c = (int)(r / ((long)p.H * p.nseq));
        const int col0 = slab * DVS;
        const int t0 = c * kUnitTokens, t1 = min(p.T, t0 + kUnitTokens), nv = t1 - t0;
        const long row0 = (long)n * p.T + t0;
        __syncthreads();   // the previous unit's reads of the staged chunk are done
        // the chunk's tokens by 16-byte copies: k, q rows; g rows (exp taken below); the v
        // and do columns of the slab; beta
        {
            constexpr int PK = DK / 8, PG = DK / 4, PV = DVS / 8;   // 16-byte pieces per row
            for (int x = tid; x < 2 * kUnitTokens * PK; x += kThreads) {
                const int isq = x / (kUnitTokens * PK), t = (x / PK) % kUnitTokens, pc = x % PK;
                if (t < nv)
                    cp_async16((isq ? cq : ck) + t * DK + 8 * pc,
                               (isq ? gq : gk) + ((row0 + t) * p.H + h) * DK + 8 * pc);
            }
            if (p.gk)
                for (int x = tid; x < kUnitTokens * PG; x += kThreads) {
                    const int t = x / PG, pc = x % PG;
                    if (t < nv) cp_async16(ca + t * DK + 4 * pc, p.gk + ((row0 + t) * p.H + h) * DK + 4 * pc);
                }
            for (int x = tid; x < 2 * kUnitTokens * PV; x += kThreads) {
                const int isd = x / (kUnitTokens * PV), t = (x / PV) % kUnitTokens, pc = x % PV;
                if (t < nv)
                    cp_async16((isd ? cd : cv) + t * DVS + 8 * pc,
                               (isd ? gdo : gv) + ((row0 + t) * p.H + h) * p.DV + col0 + 8 * pc);
            }
            if (tid < nv) cbeta[tid] = p.beta[(row0 + tid) * p.H + h];
            cp_async_wait_all();
        }
        float4 dH[R], Hp[R];
        const size_t kb = (((size_t)n * p.H + h) * p.nc64 + c) * DK * DK + col0 + 4 * cg;
#pragma unroll
        for (int m = 0; m < R; ++m) {
            Hp[m] = ld_bf16x4(p.fstates + kb + (size_t)(rg + RG * m) * DK);
            dH[m] = ld_bf16x4(p.bstates + kb + (size_t)(rg + RG * m) * DK);
        }
        __syncthreads();
        // exp(g) in place (1 without a decay); the norms of the k and q rows, two threads a row
        for (int x = tid; x < kUnitTokens * DK; x += kThreads)
            ca[x] = p.gk ? expf(ca[x]) : 1.f;
        {
            const int rr = tid >> 1, half = tid & 1, t = rr & (kUnitTokens - 1);
            const __nv_bfloat16 *xr = (rr >= kUnitTokens ? cq : ck) + t * DK + half * (DK / 2);
            float ss = 0.f;
#pragma unroll 8
            for (int i = 0; i < DK / 2; ++i) {
                const float x = __bfloat162float(xr[i]);
                ss = fmaf(x, x, ss);
            }
            ss += __shfl_xor_sync(0xffffffffu, ss, 1);
            if (half == 0 && t < nv) {
                // 1 / max(|x|, eps) = rsqrt(max(|x|^2, eps^2))
                const float inv = p.use_l2 ? rsqrtf(fmaxf(ss, kNormEps * kNormEps)) : 1.f;
                if (rr >= kUnitTokens) cqn[t] = p.scale * inv;
                else ckn[t] = inv;
            }
        }
        __syncthreads();
        {   // k^_{t-1} . kx_t for the token pairs of the recomputation, four threads a dot
            const int t = tid >> 2, part = tid & 3;
            float dot = 0.f;
            if (t > 0 && t < nv) {
                const __nv_bfloat16 *k0 = ck + (t - 1) * DK, *k1 = ck + t * DK;
                const float *a1 = ca + t * DK;
#pragma unroll 8
                for (int i = part; i < DK; i += 4)
                    dot = fmaf(__bfloat162float(k0[i]), DR ? a1[i] * __bfloat162float(k1[i]) : __bfloat162float(k1[i]), dot);
            }
            dot += __shfl_xor_sync(0xffffffffu, dot, 1);
            dot += __shfl_xor_sync(0xffffffffu, dot, 2);
            if (part == 0 && t < nv) ccd[t] = t > 0 ? dot * ckn[t - 1] * ckn[t] : 0.f;
        }
        __syncthreads();
        auto tok = [&](int t) {
            return ChunkTok<DK, DVS>{ck + t * DK, cq + t * DK, cv + t * DVS, cd + t * DVS, ca + t * DK,
                                     ckn[t], cqn[t], cbeta[t]};
        };
        // the chunk's states, each before its token, into the scratch: two tokens per pair of
        // barriers, the last one alone when the chunk is odd
        int t = 0;
        for (; t + 1 < nv; t += 2) {
#pragma unroll
            for (int m = 0; m < R; ++m) st_bf16x4(scr + ((size_t)t * DK + rg + RG * m) * DVS, Hp[m]);
            forward_pair<DK, DVS, RG, R, DR>(tok(t), tok(t + 1), ccd[t + 1], Hp, scr + (size_t)(t + 1) * DK * DVS,
                                             s_red, s_u2, s_y[t], s_y[t + 1]);
        }
        if (t < nv) {
#pragma unroll
            for (int m = 0; m < R; ++m) st_bf16x4(scr + ((size_t)t * DK + rg + RG * m) * DVS, Hp[m]);
            forward_token<DK, DVS, RG, R, DR>(p, tok(t), Hp, s_red[0], s_u, s_y[t]);
        }
        // the walk back (each thread reads back only what it wrote; v - r of every token is
        // read by the thread that kept it).  The states before the next three tokens of the
        // walk are in flight, and the state after the current token is kept, all raw (bf16)
        // until used; the state after the chunk's last token is rounded like the others.
        auto raw_state = [&](int t, uint2 (&w)[R]) {
#pragma unroll
            for (int m = 0; m < R; ++m)
                w[m] = *reinterpret_cast<const uint2 *>(scr + ((size_t)t * DK + rg + RG * m) * DVS);
        };
        uint2 Hc_raw[R], Pa[R], Pb[R], Pc[R];
#pragma unroll
        for (int m = 0; m < R; ++m) {
            const __nv_bfloat162 lo = __floats2bfloat162_rn(Hp[m].x, Hp[m].y), hi = __floats2bfloat162_rn(Hp[m].z, Hp[m].w);
            Hc_raw[m] = make_uint2(*reinterpret_cast<const uint32_t *>(&lo), *reinterpret_cast<const uint32_t *>(&hi));
        }
        raw_state(nv - 1, Pa);
        if (nv > 1) raw_state(nv - 2, Pb);
        if (nv > 2) raw_state(nv - 3, Pc);
        for (int t = nv - 1; t >= 0; --t) {
            float4 Hc[R];
#pragma unroll
            for (int m = 0; m < R; ++m) {
                Hc[m] = bf16x4_to_float4(Hc_raw[m]);
                Hp[m] = bf16x4_to_float4(Pa[m]);
                Hc_raw[m] = Pa[m];   // the state after the next token of the walk
                Pa[m] = Pb[m];
                Pb[m] = Pc[m];
            }
            if (t > 2) raw_state(t - 3, Pc);
            backward_token<DK, DVS, RG, R, DR, true>(p, tok(t), row0 + t, h, col0, dH, Hc, Hp, s_red, s_u, s_du,
                                                     s_db, s_y[t]);
        }
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
    // one CTA per (sequence, head, slab): narrower slabs when the wide ones leave SMs idle
    int dev = 0, nsm = 0;
    cudaError_t e;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    const bool narrow = p.DV < kSlab || (long)p.nseq * p.H * (p.DV / kSlab) < nsm;
    const int dvs = narrow ? 32 : kSlab;
    const long grid = (long)p.nseq * p.H * (p.DV / dvs);
    const bool dr = p.decayed_read != 0;
    if (dvs == 64) {
        if (dr) {
            bwd_ckpt_kernel<Tin, DK, 64, true><<<(unsigned)grid, kThreads, 0, s>>>(p);
            bwd_kernel<Tin, DK, 64, true><<<(unsigned)grid, kThreads, 0, s>>>(p);
        } else {
            bwd_ckpt_kernel<Tin, DK, 64, false><<<(unsigned)grid, kThreads, 0, s>>>(p);
            bwd_kernel<Tin, DK, 64, false><<<(unsigned)grid, kThreads, 0, s>>>(p);
        }
    } else {
        if (dr) {
            bwd_ckpt_kernel<Tin, DK, 32, true><<<(unsigned)grid, kThreads, 0, s>>>(p);
            bwd_kernel<Tin, DK, 32, true><<<(unsigned)grid, kThreads, 0, s>>>(p);
        } else {
            bwd_ckpt_kernel<Tin, DK, 32, false><<<(unsigned)grid, kThreads, 0, s>>>(p);
            bwd_kernel<Tin, DK, 32, false><<<(unsigned)grid, kThreads, 0, s>>>(p);
        }
    }
    const long rh = rows * p.H;
    bwd_finish_kernel<Tin, DK><<<(unsigned)((rh * 32 + 255) / 256), 256, 0, s>>>(p, rh);
    return cudaGetLastError();
}

}  // namespace

size_t gk_bwd_scratch_bytes(int nseq, int T, int H, int dk, int dv) {
    // checkpoints, then one kBwdChunk x dk x (slab) scratch per CTA: nseq*H*dv columns in all,
    // whatever the slab width
    const int nc = (T + kBwdChunk - 1) / kBwdChunk;
    return (size_t)nseq * H * nc * dk * dv * 4 + (size_t)nseq * H * kBwdChunk * dk * dv * 4;
}

cudaError_t launch_gk_bwd(const BwdArgs &a, cudaStream_t s) {
    BwdParams p{};
    p.q = a.q; p.k = a.k; p.v = a.v; p.dout = a.dout;
    p.beta = a.beta; p.gk = a.g; p.h0 = a.h0; p.dhT = a.dhT;
    p.decay = a.g ? nullptr : a.decay;
    p.ddecay = p.decay ? a.ddecay : nullptr;
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
    if (p.ddecay && (e = cudaMemsetAsync(p.ddecay, 0, (size_t)rows * a.H * sizeof(float), s)) != cudaSuccess)
        return e;
    if ((e = cudaMemsetAsync(a.dbeta, 0, (size_t)rows * a.H * sizeof(float), s)) != cudaSuccess) return e;
    const bool bf = a.dtype == DType::BF16;
    switch (a.dkdim) {
        case 32: return bf ? run_bwd<__nv_bfloat16, 32>(p, rows, s) : run_bwd<float, 32>(p, rows, s);
        case 64: return bf ? run_bwd<__nv_bfloat16, 64>(p, rows, s) : run_bwd<float, 64>(p, rows, s);
        case 128: return bf ? run_bwd<__nv_bfloat16, 128>(p, rows, s) : run_bwd<float, 128>(p, rows, s);
        default: return cudaErrorInvalidValue;
    }
}


size_t gk_chunk_bwd_scratch_bytes(int dk) {
    return (size_t)kChunkBwdCtas * kUnitTokens * dk * kUnitSlab * sizeof(__nv_bfloat16);
}

cudaError_t launch_gk_chunk_bwd_grads(const BwdArgs &a, const __nv_bfloat16 *fstates,
                                      const __nv_bfloat16 *bstates, void *scratch, cudaStream_t s) {
    if (a.dtype != DType::BF16 || a.dkdim != a.dvdim || (a.dkdim != 64 && a.dkdim != 128))
        return cudaErrorInvalidValue;
    BwdParams p{};
    p.q = a.q; p.k = a.k; p.v = a.v; p.dout = a.dout;
    p.beta = a.beta; p.gk = a.g; p.h0 = nullptr; p.dhT = nullptr;
    p.decay = nullptr; p.ddecay = nullptr;
    p.dq = a.dq; p.dk = a.dk; p.dv = a.dv; p.dbeta = a.dbeta; p.dg = a.dg; p.dh0 = nullptr;
    p.nseq = a.B; p.T = a.T; p.H = a.H; p.DV = a.dvdim;
    p.scale = a.scale; p.use_l2 = a.use_l2; p.decayed_read = a.decayed_read;
    p.fstates = fstates; p.bstates = bstates;
    p.scratch16 = static_cast<__nv_bfloat16 *>(scratch);
    p.nc64 = (a.T + kUnitTokens - 1) / kUnitTokens;
    const long rows = (long)a.B * a.T;
    cudaError_t e;
    // the sums over value slabs accumulate into these
    const size_t nk = (size_t)rows * a.H * a.dkdim * sizeof(float);
    if ((e = cudaMemsetAsync(a.dq, 0, nk, s)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(a.dk, 0, nk, s)) != cudaSuccess) return e;
    if (a.dg && (e = cudaMemsetAsync(a.dg, 0, nk, s)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(a.dbeta, 0, (size_t)rows * a.H * sizeof(float), s)) != cudaSuccess) return e;
    const long units = (long)p.nc64 * a.B * a.H * (a.dkdim / kUnitSlab);
    const unsigned grid = (unsigned)std::min<long>(units, kChunkBwdCtas);
    const bool dr = p.decayed_read != 0;
    auto go = [&](auto kern, int smem) {
        cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (err != cudaSuccess) return err;
        kern<<<grid, kThreads, smem, s>>>(p);
        return cudaGetLastError();
    };
    if (a.dkdim == 128) {
        constexpr int smem = ChunkStage<128, kUnitSlab>::BYTES;
        e = dr ? go(bwd_chunk_kernel<128, kUnitSlab, true>, smem) : go(bwd_chunk_kernel<128, kUnitSlab, false>, smem);
    } else {
        constexpr int smem = ChunkStage<64, kUnitSlab>::BYTES;
        e = dr ? go(bwd_chunk_kernel<64, kUnitSlab, true>, smem) : go(bwd_chunk_kernel<64, kUnitSlab, false>, smem);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const long rh = rows * a.H;
    if (a.dkdim == 128) bwd_finish_kernel<__nv_bfloat16, 128><<<(unsigned)((rh * 32 + 255) / 256), 256, 0, s>>>(p, rh);
    else bwd_finish_kernel<__nv_bfloat16, 64><<<(unsigned)((rh * 32 + 255) / 256), 256, 0, s>>>(p, rh);
    return cudaGetLastError();
}

}  // namespace kda
