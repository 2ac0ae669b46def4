// chunk_bwd.cu -- the chunk-local gradients of the chunked backward.
//
// The backward of the chunked WY / UT form (one decay per head; the delta term reads
// h_{t-1}, or exp(decay_t) h_{t-1} with decayed_read).  Per chunk of C = 64 tokens entering
// with state S (a forward walk wrote it) and leaving with state gradient dS' (the reverse
// walk wrote it), with the forward's chunk quantities
//
//   k^ = l2(k), q~ = scale l2(q), G_t = sum_{r<=t} decay_r, R_t = G_{t-1} or G_t,
//   L = beta_t (k^ k^^T) (.) E_kk (strict), E_kk[t][s] = exp(R_t - G_s),  T = (I + L)^{-1},
//   W = T diag(beta e^R) K^,  U = T diag(beta) V - W S,
//   A = (q~ k^^T) (.) E_qk (inclusive), E_qk[t][s] = exp(G_t - G_s),  K~ = diag(e^{G_n - G}) K^,
//   O = diag(e^G) Q~ S + A U,   S' = e^{G_n} S + K~^T U,
//
// the adjoint of those lines, in order:
//
//   dU  = A^T dO + K~ dS'           dA  = mask_incl(dO U^T)      dK~ = U dS'^T
//   dW  = -dU S^T                   dT  = dU (diag(beta) V)^T + dW (diag(beta e^R) K^)^T
//   dL  = -mask_strict(T^T dT T^T)  dK^ = diag(beta e^R) T^T dW + P K^ + P^T K^
//                                         + (dA (.) E_qk)^T Q~ + diag(e^{G_n - G}) dK~,
//                                         P = dL (.) beta_t E_kk
//   dQ~ = (dA (.) E_qk) K^ + diag(e^G) dO S^T
//
// with beta and the decay collected from the same terms (the decay through G, R and G_n,
// then a reverse cumulative sum inside the chunk) and the L2 normalisation's adjoint
// dx = (dx^ - x^ (x^ . dx^)) / |x|.  The value gradient and the state gradients come from
// the reverse walk (chunk_tc.cu).
//
// One CTA per chunk at a time (persistent CTAs over the chunks).  Every intermediate is an
// fp32 matrix in the CTA's own scratch region of global memory, where it stays in L2 and
// L1; the states of the two walks are read in place.  The products are warp-level tensor
// MMAs (m16n8k8, tf32 operands, fp32 accumulation) over 16 x 8 output tiles, the warps
// taking tiles in turn; every operand is addressed through (row stride, column stride), so
// transposed operands cost nothing.  Padded rows past a sequence's end act as k = q = v =
// dO = 0, beta = 0, decay = 0 and are never stored.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kC = 64;
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr float kNormEpsB = 1e-12f;


__device__ __forceinline__ uint32_t tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

// d += a b, m16n8k8, tf32 operands, fp32 accumulators
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm volatile("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
                 "{%8, %9}, {%0, %1, %2, %3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// C[M x N] = A B^T with A [M][K] and B [N][K] row-major (both contiguous along the
// contraction; M a multiple of 32, N of 16, K of 16), the warps of the CTA taking output
// tiles of 32 x WN (WN = 32 when the 64-row output has 8 such tiles, else 16) in turn: each
// A fragment serves WN / 8 MMAs and each B fragment two.  epi(r, c, v0, v1) receives
// C[r][c], C[r][c + 1] (lane = 4 g + t4 holds rows g + 8 i, columns 2 t4 + 8 j of its tile)
// and returns a contribution to row r's sum, which is reduced over the lanes of the row and
// added to rowsum[r] (shared memory) when rowsum is given.  Inside a 16-wide k step lane t4
// takes the four consecutive k = 4 t4 .. 4 t4 + 3 for both operands (one 16-byte load each),
// the first two for the first MMA and the last two for the second: the same permutation of
// k on A and B, which leaves the sum unchanged.
template <int WN, typename Epi>
__device__ __forceinline__ void gemm_t(int M, int N, int K, const float *A, int lda, const float *B, int ldb,
                                       Epi epi, float *rowsum) {
    constexpr int NJ = WN / 8;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t4 = lane & 3;
    const int tn = N / WN, tiles = (M / 32) * tn;
    for (int tile = warp; tile < tiles; tile += kWarps) {
        const int m0 = (tile / tn) * 32, n0 = (tile % tn) * WN;
        const float *ap[4], *bp[NJ];
#pragma unroll
        for (int i = 0; i < 4; ++i) ap[i] = A + (size_t)(m0 + g + 8 * i) * lda + 4 * t4;
#pragma unroll
        for (int j = 0; j < NJ; ++j) bp[j] = B + (size_t)(n0 + 8 * j + g) * ldb + 4 * t4;
        float d[2][NJ][4] = {};
#pragma unroll 2
        for (int k0 = 0; k0 < K; k0 += 16) {
            float4 x[4], z[NJ];
#pragma unroll
            for (int i = 0; i < 4; ++i) x[i] = *reinterpret_cast<const float4 *>(ap[i] + k0);
#pragma unroll
            for (int j = 0; j < NJ; ++j) z[j] = *reinterpret_cast<const float4 *>(bp[j] + k0);
#pragma unroll
            for (int mi = 0; mi < 2; ++mi) {
                const uint32_t a[4] = {tf32(x[2 * mi].x), tf32(x[2 * mi + 1].x), tf32(x[2 * mi].y), tf32(x[2 * mi + 1].y)};
                const uint32_t a2[4] = {tf32(x[2 * mi].z), tf32(x[2 * mi + 1].z), tf32(x[2 * mi].w), tf32(x[2 * mi + 1].w)};
#pragma unroll
                for (int j = 0; j < NJ; ++j) {
                    const uint32_t b[2] = {tf32(z[j].x), tf32(z[j].y)};
                    const uint32_t b2[2] = {tf32(z[j].z), tf32(z[j].w)};
                    mma_tf32(d[mi][j], a, b);
                    mma_tf32(d[mi][j], a2, b2);
                }
            }
        }
#pragma unroll
        for (int mi = 0; mi < 2; ++mi)
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                const int r = m0 + 16 * mi + g + 8 * h2;
                float part = 0.f;
#pragma unroll
                for (int j = 0; j < NJ; ++j) part += epi(r, n0 + 8 * j + 2 * t4, d[mi][j][2 * h2], d[mi][j][2 * h2 + 1]);
                if (rowsum) {
                    part += __shfl_xor_sync(0xffffffffu, part, 1);
                    part += __shfl_xor_sync(0xffffffffu, part, 2);
                    if (t4 == 0) atomicAdd(rowsum + r, part);
                }
            }
    }
}
// Operands are copied into shared memory before each product (16-byte cp.async copies,
// many in flight), rows padded to K + 16 floats: the 16-byte fragment loads of a quarter
// warp (rows g, g + 1, columns 4 t4) then fall on distinct banks.
__device__ __forceinline__ void stage(float *dst, const float *src, int rows, int K) {
    const int per_row = K >> 2, pitch = K + 16;
    for (int x = threadIdx.x; x < rows * per_row; x += kThreads) {
        const int r = x / per_row, c4 = x - r * per_row;
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst + r * pitch + 4 * c4)),
                     "l"(src + (size_t)r * K + 4 * c4)
                     : "memory");
    }
}

// C = A B^T for A [M][K], B [N][K] in global memory (row-major, contiguous rows): both staged
// into the CTA's operand buffers sA, sB, then multiplied (see gemm_t).  Starts and ends with
// a barrier of the CTA, so the products of a chunk run in program order.
template <typename Epi>
__device__ __forceinline__ void gemm(float *sA, float *sB, int M, int N, int K, const float *A, const float *B,
                                     Epi epi, float *rowsum = nullptr) {
    __syncthreads();   // the previous product has read the buffers; its outputs are in memory
    stage(sA, A, M, K);
    if (B != A) stage(sB, B, N, K);
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_all;" ::: "memory");
    __syncthreads();
    const float *b = B != A ? sB : sA;
    if (N >= 128) gemm_t<32>(M, N, K, sA, K + 16, b, K + 16, epi, rowsum);
    else gemm_t<16>(M, N, K, sA, K + 16, b, K + 16, epi, rowsum);
    __syncthreads();
}

// The CTA's scratch, in floats: 64 x D matrices, 64 x 64 matrices, per-token scalars.
template <int D>
struct Scr {
    // 64 x D (a "t" suffix: the transposed copy, D x 64)
    enum { Kh, Qh, V, dO, Kt, W, U, dU, dW, dkh, dqh, Kht, Qht, Vt, dOt, dUt, dWt, NBig };
    enum { KKE, L, A, T, Pv, Pk, dA, dT, X, dL, At, Tt, Xt, NSmall };
    enum { St, dSpt, NSq };   // D x D: the transposed states
    enum { beta, G, R, eG, eR, eGnG, kn, qn, knorm, qnorm, dG, dGp, dbeta, NScal };
    static constexpr size_t big(int i) { return (size_t)i * kC * D; }
    static constexpr size_t small(int i) { return (size_t)NBig * kC * D + (size_t)i * kC * kC; }
    static constexpr size_t sq(int i) { return small(NSmall) + (size_t)i * D * D; }
    static constexpr size_t scal(int i) { return sq(NSq) + (size_t)i * kC; }
    static constexpr size_t floats = scal(NScal) + 64;   // + the chunk's G_n terms
};

}  // namespace

namespace {

__device__ __forceinline__ float bf2f(__nv_bfloat16 x) { return __bfloat162float(x); }

template <int D>
__global__ void __launch_bounds__(kThreads, 2) chunk_bwd_kernel(ChunkBwdArgs a) {
    using Sc = Scr<D>;
    constexpr int PL = kC + 1;   // padded rows of the inverse's shared arrays
    // the products' operand buffers: A [64][D + 16], B [D][D + 16]; the inverse's L and T (and
    // the state transposes' tiles) reuse them between products
    extern __shared__ float smem_dyn[];
    float *sA = smem_dyn, *sB = smem_dyn + kC * (D + 16);
    float *sL = sB, *sT = sB + kC * PL;   // (the buffer is sized to hold both)
    __shared__ float red[10 * kC];   // per-token row / column sums
    __shared__ float sGn[2];        // G_n, and the chunk's gradient of G_n
    float *sc = a.scratch + (size_t)blockIdx.x * Sc::floats;
    auto big = [&](int i) { return sc + Sc::big(i); };
    auto sml = [&](int i) { return sc + Sc::small(i); };
    auto scl = [&](int i) { return sc + Sc::scal(i); };
    float *Kh = big(Sc::Kh), *Qh = big(Sc::Qh), *V = big(Sc::V), *dO = big(Sc::dO), *Kt = big(Sc::Kt);
    float *W = big(Sc::W), *U = big(Sc::U), *dU = big(Sc::dU), *dW = big(Sc::dW);
    float *dkh = big(Sc::dkh), *dqh = big(Sc::dqh);
    float *Kht = big(Sc::Kht), *Qht = big(Sc::Qht), *Vt = big(Sc::Vt), *dOt = big(Sc::dOt);
    float *dUt = big(Sc::dUt), *dWt = big(Sc::dWt);
    float *KKE = sml(Sc::KKE), *L = sml(Sc::L), *A = sml(Sc::A);
    float *T = sml(Sc::T), *Pv = sml(Sc::Pv), *Pk = sml(Sc::Pk), *dA = sml(Sc::dA), *dT = sml(Sc::dT);
    float *X = sml(Sc::X), *dL = sml(Sc::dL), *At = sml(Sc::At), *Tt = sml(Sc::Tt), *Xt = sml(Sc::Xt);
    // after dL: P = dL beta_t E_kk and dA (.) E_qk with their transposes reuse X, Xt, dT, Pv
    float *dKK = X, *dKKt = Xt, *dQK = dT, *dQKt = Pv;
    float *St = sc + Sc::sq(Sc::St), *dSpt = sc + Sc::sq(Sc::dSpt);
    float *beta = scl(Sc::beta), *G = scl(Sc::G), *R = scl(Sc::R), *eG = scl(Sc::eG), *eR = scl(Sc::eR);
    float *eGnG = scl(Sc::eGnG), *kn = scl(Sc::kn), *qn = scl(Sc::qn), *knorm = scl(Sc::knorm);
    float *qnorm = scl(Sc::qnorm), *dG = scl(Sc::dG), *dGp = scl(Sc::dGp), *dbeta = scl(Sc::dbeta);
    float *rA = red, *cA = red + kC, *rL = red + 2 * kC, *cL = red + 3 * kC, *rLK = red + 4 * kC;
    float *rqd = red + 5 * kC, *rkd = red + 6 * kC, *rbv = red + 7 * kC, *rbk = red + 8 * kC;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nc = (a.T + kC - 1) / kC;
    const long nchunks = (long)a.B * a.H * nc;
    const __nv_bfloat16 *gq = static_cast<const __nv_bfloat16 *>(a.q);
    const __nv_bfloat16 *gk = static_cast<const __nv_bfloat16 *>(a.k);
    const __nv_bfloat16 *gv = static_cast<const __nv_bfloat16 *>(a.v);
    const __nv_bfloat16 *gdo = static_cast<const __nv_bfloat16 *>(a.d_o);

    for (long ci = blockIdx.x; ci < nchunks; ci += gridDim.x) {
        const int c = (int)(ci % nc), bh = (int)(ci / nc);
        const int h = bh % a.H, b = bh / a.H;
        const long row0 = (long)b * a.T + (long)c * kC;
        const int nv = min(kC, a.T - c * kC);
        const float *S = a.fstates + (size_t)ci * D * D;    // state entering the chunk
        const float *dSp = a.bstates + (size_t)ci * D * D;  // gradient of the state leaving it

        // ---- rows: norms, k^, q~, v, dO (zero past the valid tokens) and their transposes,
        // cleared accumulators
        for (int t = warp; t < kC; t += kWarps) {
            const bool valid = t < nv;
            const size_t gi = ((size_t)(row0 + t) * a.H + h) * D;
            float kk[D / 32], qq[D / 32], ssk = 0.f, ssq = 0.f;
#pragma unroll
            for (int m = 0; m < D / 32; ++m) {
                const int i = lane + 32 * m;
                kk[m] = valid ? bf2f(gk[gi + i]) : 0.f;
                qq[m] = valid ? bf2f(gq[gi + i]) : 0.f;
                ssk = fmaf(kk[m], kk[m], ssk);
                ssq = fmaf(qq[m], qq[m], ssq);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                ssk += __shfl_xor_sync(0xffffffffu, ssk, o);
                ssq += __shfl_xor_sync(0xffffffffu, ssq, o);
            }
            const float nk = sqrtf(ssk), nq = sqrtf(ssq);
            const float fk = a.use_l2 ? 1.f / fmaxf(nk, kNormEpsB) : 1.f;
            const float fq = a.scale * (a.use_l2 ? 1.f / fmaxf(nq, kNormEpsB) : 1.f);
#pragma unroll
            for (int m = 0; m < D / 32; ++m) {
                const int i = lane + 32 * m;
                const float vv = valid ? bf2f(gv[gi + i]) : 0.f, oo = valid ? bf2f(gdo[gi + i]) : 0.f;
                Kh[t * D + i] = kk[m] * fk; Kht[i * kC + t] = kk[m] * fk;
                Qh[t * D + i] = qq[m] * fq; Qht[i * kC + t] = qq[m] * fq;
                V[t * D + i] = vv; Vt[i * kC + t] = vv;
                dO[t * D + i] = oo; dOt[i * kC + t] = oo;
                dkh[t * D + i] = 0.f;
                dqh[t * D + i] = 0.f;
            }
            if (lane == 0) {
                rqd[t] = 0.f; rkd[t] = 0.f; rbv[t] = 0.f; rbk[t] = 0.f;
                kn[t] = fk; qn[t] = fq; knorm[t] = nk; qnorm[t] = nq;
                beta[t] = valid ? a.beta[(row0 + t) * a.H + h] : 0.f;
            }
        }
        // the transposed states, through 32 x 32 tiles in shared memory (the inverse's arrays)
        for (int tile = 0; tile < (D / 32) * (D / 32); ++tile) {
            const int r0 = (tile / (D / 32)) * 32, c0 = (tile % (D / 32)) * 32;
            for (int x = tid; x < 1024; x += kThreads) {
                const int r = x >> 5, cc = x & 31;
                sL[r * 33 + cc] = S[(size_t)(r0 + r) * D + c0 + cc];
                sT[r * 33 + cc] = dSp[(size_t)(r0 + r) * D + c0 + cc];
            }
            __syncthreads();
            for (int x = tid; x < 1024; x += kThreads) {
                const int r = x >> 5, cc = x & 31;
                St[(size_t)(c0 + r) * D + r0 + cc] = sL[cc * 33 + r];
                dSpt[(size_t)(c0 + r) * D + r0 + cc] = sT[cc * 33 + r];
            }
            __syncthreads();
        }
        if (warp == 0) {   // in-chunk cumulative log decay: lane owns tokens 2 lane, 2 lane + 1
            auto dec = [&](int t) { return (t < nv && a.decay) ? a.decay[(row0 + t) * a.H + h] : 0.f; };
            const float d0 = dec(2 * lane), d1 = dec(2 * lane + 1);
            float incl = d0 + d1;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += y;
            }
            const float gn = __shfl_sync(0xffffffffu, incl, 31);
            const float g0 = incl - d1, g1 = incl;   // G_{2 lane}, G_{2 lane + 1}
            const float p0 = g0 - d0, p1 = g0;       // G_{t-1}
            const float r0 = a.decayed_read ? g0 : p0, r1 = a.decayed_read ? g1 : p1;
            G[2 * lane] = g0; G[2 * lane + 1] = g1;
            R[2 * lane] = r0; R[2 * lane + 1] = r1;
            eG[2 * lane] = __expf(g0); eG[2 * lane + 1] = __expf(g1);
            eR[2 * lane] = __expf(r0); eR[2 * lane + 1] = __expf(r1);
            eGnG[2 * lane] = __expf(gn - g0); eGnG[2 * lane + 1] = __expf(gn - g1);
            if (lane == 0) { sGn[0] = gn; sGn[1] = 0.f; }
        }
        __syncthreads();
        for (int x = tid; x < kC * D; x += kThreads) Kt[x] = eGnG[x / D] * Kh[x];

        // ---- Gram products: A = (q~ k^^T) E_qk (inclusive), L = beta_t (k^ k^^T) E_kk (strict);
        // the second product reads one staged operand, so its epilogue may fill the inverse's L
        // in the other buffer
        gemm(sA, sB, kC, kC, D, Qh, Kh, [&](int t, int s, float v0, float v1) -> float {
            const float vv[2] = {v0, v1};
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const float e = (s + u <= t) ? __expf(G[t] - G[s + u]) : 0.f;
                A[t * kC + s + u] = vv[u] * e;
                At[(s + u) * kC + t] = vv[u] * e;
            }
            return 0.f;
        });
        gemm(sA, sB, kC, kC, D, Kh, Kh, [&](int t, int s, float v0, float v1) -> float {
            const float vv[2] = {v0, v1};
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const float e = (s + u < t) ? __expf(R[t] - G[s + u]) : 0.f;
                KKE[t * kC + s + u] = vv[u] * e;
                L[t * kC + s + u] = beta[t] * vv[u] * e;
                sL[t * PL + s + u] = beta[t] * vv[u] * e;
            }
            return 0.f;
        });
        __syncthreads();

        // ---- T = (I + L)^{-1}: four threads per column j (a quarter of the terms each), rows
        // in order; T[r][j] = delta_rj - sum_{s<r} L[r][s] T[s][j]
        {
            const int j = tid >> 2, part = tid & 3;
            for (int r = 0; r < kC; ++r) {
                float acc = 0.f;
                for (int s = part; s < r; s += 4) acc = fmaf(sL[r * PL + s], sT[s * PL + j], acc);
                acc += __shfl_xor_sync(0xffffffffu, acc, 1);
                acc += __shfl_xor_sync(0xffffffffu, acc, 2);
                if (part == 0) sT[r * PL + j] = (r == j ? 1.f : 0.f) - (r > j ? acc : 0.f);
                __syncwarp();
            }
        }
        __syncthreads();
        for (int x = tid; x < kC * kC; x += kThreads) {
            const int t = x / kC, s = x % kC;
            const float tv = sT[t * PL + s];
            T[x] = tv;
            Tt[s * kC + t] = tv;
            Pv[x] = tv * beta[s];
            Pk[x] = tv * beta[s] * eR[s];
        }
        __syncthreads();

        // ---- forward quantities: W = T diag(beta e^R) K^, U = T diag(beta) V - W S;  dU = A^T dO
        gemm(sA, sB, kC, D, kC, Pk, Kht, [&](int t, int j, float v0, float v1) -> float {
            W[t * D + j] = v0; W[t * D + j + 1] = v1;
            return 0.f;
        });
        gemm(sA, sB, kC, D, kC, Pv, Vt, [&](int t, int j, float v0, float v1) -> float {
            U[t * D + j] = v0; U[t * D + j + 1] = v1;
            return 0.f;
        });
        gemm(sA, sB, kC, D, kC, At, dOt, [&](int s, int j, float v0, float v1) -> float {
            dU[s * D + j] = v0; dU[s * D + j + 1] = v1;
            return 0.f;
        });
        __syncthreads();
        // U -= W S;  dU += K~ dS' (and its transpose);  DOS = dO S^T  (each output element stays
        // with one thread across the products that write it)
        gemm(sA, sB, kC, D, D, W, St, [&](int t, int j, float v0, float v1) -> float {
            U[t * D + j] -= v0; U[t * D + j + 1] -= v1;
            return 0.f;
        });
        gemm(sA, sB, kC, D, D, Kt, dSpt, [&](int s, int j, float v0, float v1) -> float {
            const float u0 = dU[s * D + j] + v0, u1 = dU[s * D + j + 1] + v1;
            dU[s * D + j] = u0; dU[s * D + j + 1] = u1;
            dUt[j * kC + s] = u0; dUt[(j + 1) * kC + s] = u1;
            return 0.f;
        });
        gemm(sA, sB, kC, D, D, dO, S, [&](int t, int i, float v0, float v1) -> float {   // dO S^T
            dqh[t * D + i] += eG[t] * v0; dqh[t * D + i + 1] += eG[t] * v1;
            return v0 * Qh[t * D + i] + v1 * Qh[t * D + i + 1];
        }, rqd);
        __syncthreads();

        // ---- dA = mask_incl(dO U^T),  dK~ = U dS'^T,  dW = -dU S^T
        gemm(sA, sB, kC, kC, D, dO, U, [&](int t, int s, float v0, float v1) -> float {
            dA[t * kC + s] = s <= t ? v0 : 0.f;
            dA[t * kC + s + 1] = s + 1 <= t ? v1 : 0.f;
            return 0.f;
        });
        gemm(sA, sB, kC, D, D, U, dSp, [&](int s, int i, float v0, float v1) -> float {   // dK~
            dkh[s * D + i] += eGnG[s] * v0; dkh[s * D + i + 1] += eGnG[s] * v1;
            return v0 * Kt[s * D + i] + v1 * Kt[s * D + i + 1];
        }, rkd);
        gemm(sA, sB, kC, D, D, dU, S, [&](int s, int i, float v0, float v1) -> float {
            dW[s * D + i] = -v0; dW[s * D + i + 1] = -v1;
            dWt[i * kC + s] = -v0; dWt[(i + 1) * kC + s] = -v1;
            return 0.f;
        });
        __syncthreads();

        // ---- dT = dU (diag(beta) V)^T + dW (diag(beta e^R) K^)^T;  dBv = T^T dU;  dBk = T^T dW,
        // dK^ += diag(beta e^R) dBk
        gemm(sA, sB, kC, kC, D, dU, V, [&](int t, int s, float v0, float v1) -> float {
            dT[t * kC + s] = v0 * beta[s];
            dT[t * kC + s + 1] = v1 * beta[s + 1];
            return 0.f;
        });
        gemm(sA, sB, kC, D, kC, Tt, dUt, [&](int s, int j, float v0, float v1) -> float {   // dBv
            return v0 * V[s * D + j] + v1 * V[s * D + j + 1];
        }, rbv);
        gemm(sA, sB, kC, kC, D, dW, Kh, [&](int t, int s, float v0, float v1) -> float {
            dT[t * kC + s] += v0 * beta[s] * eR[s];
            dT[t * kC + s + 1] += v1 * beta[s + 1] * eR[s + 1];
            return 0.f;
        });
        gemm(sA, sB, kC, D, kC, Tt, dWt, [&](int s, int i, float v0, float v1) -> float {   // dBk
            const float w = beta[s] * eR[s];
            dkh[s * D + i] += w * v0; dkh[s * D + i + 1] += w * v1;
            return v0 * Kh[s * D + i] + v1 * Kh[s * D + i + 1];
        }, rbk);
        __syncthreads();

        // ---- dL = -mask_strict(T^T dT T^T)
        gemm(sA, sB, kC, kC, kC, dT, T, [&](int t, int s, float v0, float v1) -> float {
            X[t * kC + s] = v0; X[t * kC + s + 1] = v1;
            Xt[s * kC + t] = v0; Xt[(s + 1) * kC + t] = v1;
            return 0.f;
        });
        __syncthreads();
        gemm(sA, sB, kC, kC, kC, Tt, Xt, [&](int t, int s, float v0, float v1) -> float {
            dL[t * kC + s] = s < t ? -v0 : 0.f;
            dL[t * kC + s + 1] = s + 1 < t ? -v1 : 0.f;
            return 0.f;
        });
        __syncthreads();

        // ---- row and column sums of dA (.) A and dL (.) L, dL (.) KKE; P = dL beta_t E_kk and
        // dA (.) E_qk, with their transposes
        if (tid < kC) {
            const int t = tid;
            float sa = 0.f, sl = 0.f, slk = 0.f;
            for (int s = 0; s < kC; ++s) {
                sa = fmaf(dA[t * kC + s], A[t * kC + s], sa);
                sl = fmaf(dL[t * kC + s], L[t * kC + s], sl);
                slk = fmaf(dL[t * kC + s], KKE[t * kC + s], slk);
            }
            rA[t] = sa; rL[t] = sl; rLK[t] = slk;
        } else if (tid < 2 * kC) {
            const int s = tid - kC;
            float sa = 0.f, sl = 0.f;
            for (int t = 0; t < kC; ++t) {
                sa = fmaf(dA[t * kC + s], A[t * kC + s], sa);
                sl = fmaf(dL[t * kC + s], L[t * kC + s], sl);
            }
            cA[s] = sa; cL[s] = sl;
        }
        for (int x = tid; x < kC * kC; x += kThreads) {
            const int t = x / kC, s = x % kC;
            const float ekk = s < t ? __expf(R[t] - G[s]) : 0.f, eqk = s <= t ? __expf(G[t] - G[s]) : 0.f;
            const float p = dL[x] * beta[t] * ekk, qk = dA[x] * eqk;
            dKK[x] = p; dKKt[s * kC + t] = p;
            dQK[x] = qk; dQKt[s * kC + t] = qk;
        }
        __syncthreads();
        // dK^ += P K^ + P^T K^ + (dA E_qk)^T Q~;  dQ~ += (dA E_qk) K^
        gemm(sA, sB, kC, D, kC, dKK, Kht, [&](int t, int i, float v0, float v1) -> float {
            dkh[t * D + i] += v0; dkh[t * D + i + 1] += v1;
            return 0.f;
        });
        gemm(sA, sB, kC, D, kC, dKKt, Kht, [&](int s, int i, float v0, float v1) -> float {
            dkh[s * D + i] += v0; dkh[s * D + i + 1] += v1;
            return 0.f;
        });
        gemm(sA, sB, kC, D, kC, dQKt, Qht, [&](int s, int i, float v0, float v1) -> float {
            dkh[s * D + i] += v0; dkh[s * D + i + 1] += v1;
            return 0.f;
        });
        gemm(sA, sB, kC, D, kC, dQK, Kht, [&](int t, int i, float v0, float v1) -> float {
            dqh[t * D + i] += v0; dqh[t * D + i + 1] += v1;
            return 0.f;
        });
        __syncthreads();

        // ---- per token: dG, dR, dbeta (the dots of q~ . dO S^T, dK~ . K~, dBv . v, dBk . k^ came
        // from the products' epilogues)
        if (tid < kC) {
            const int t = tid;
            const float dr = rL[t] + beta[t] * eR[t] * rbk[t];
            float dg = eG[t] * rqd[t] + rA[t] - cA[t] - cL[t] - rkd[t];
            float dgp = 0.f;
            if (a.decayed_read) dg += dr; else dgp = dr;
            dG[t] = dg;
            dGp[t] = dgp;
            dbeta[t] = rbv[t] + eR[t] * rbk[t] + rLK[t];
            atomicAdd(&sGn[1], rkd[t]);
        }
        {   // e^{G_n} sum(S (.) dS')
            float acc = 0.f;
            for (int x = tid; x < D * D; x += kThreads) acc = fmaf(S[x], dSp[x], acc);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
            if (lane == 0) atomicAdd(&sGn[1], __expf(sGn[0]) * acc);
        }
        __syncthreads();

        // ---- decay gradient: the chunk's G_n is G at its last token (padded decays are 0);
        // ddecay_r = sum_{t >= r} dG_t + sum_{t > r} dGp_t
        if (warp == 0) {
            const int t0 = 2 * lane, t1 = 2 * lane + 1;
            const float g0 = dG[t0], g1 = dG[t1] + (t1 == kC - 1 ? sGn[1] : 0.f);
            const float p0 = dGp[t0], p1 = dGp[t1];
            // reverse inclusive sums over the 64 tokens: suffix scan by lanes from the top
            float sg = g0 + g1, sp = p0 + p1;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float yg = __shfl_down_sync(0xffffffffu, sg, off);
                const float yp = __shfl_down_sync(0xffffffffu, sp, off);
                if (lane + off < 32) { sg += yg; sp += yp; }
            }
            // sg, sp: sums over tokens >= 2 lane
            const float dd0 = sg + (sp - p0), dd1 = (sg - g0) + (sp - p0 - p1);
            if (a.ddecay) {
                if (t0 < nv) a.ddecay[(row0 + t0) * a.H + h] = dd0;
                if (t1 < nv) a.ddecay[(row0 + t1) * a.H + h] = dd1;
            }
            if (t0 < nv) a.dbeta[(row0 + t0) * a.H + h] = dbeta[t0];
            if (t1 < nv) a.dbeta[(row0 + t1) * a.H + h] = dbeta[t1];
        }
        // ---- dq, dk through the normalisation: dx = f (dx^ - x^ (x^ . dx^)) for |x| > eps
        for (int t = warp; t < nv; t += kWarps) {
            float kdot = 0.f, qdot = 0.f;
#pragma unroll
            for (int m = 0; m < D / 32; ++m) {
                const int x = t * D + lane + 32 * m;
                kdot = fmaf(Kh[x], dkh[x], kdot);
                qdot = fmaf(Qh[x], dqh[x], qdot);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                kdot += __shfl_xor_sync(0xffffffffu, kdot, o);
                qdot += __shfl_xor_sync(0xffffffffu, qdot, o);
            }
            const bool pk = a.use_l2 && knorm[t] > kNormEpsB, pq = a.use_l2 && qnorm[t] > kNormEpsB;
            const float qs = a.scale * a.scale;
            const size_t gi = ((size_t)(row0 + t) * a.H + h) * D;
#pragma unroll
            for (int m = 0; m < D / 32; ++m) {
                const int i = lane + 32 * m, x = t * D + i;
                a.dk[gi + i] = kn[t] * (dkh[x] - (pk ? Kh[x] * kdot : 0.f));
                a.dq[gi + i] = qn[t] * (dqh[x] - (pq ? Qh[x] * qdot / qs : 0.f));
            }
        }
        __syncthreads();   // the scratch is rewritten by the next chunk
    }
}

}  // namespace

size_t chunk_bwd_scratch_floats(int D) {
    return D == 128 ? Scr<128>::floats : Scr<64>::floats;
}

// Persistent CTAs of the gradient kernel: a fixed number, so that the workspace query needs
// no device (each CTA has its own scratch region).
int chunk_bwd_ctas() { return 304; }

template <int D>
cudaError_t launch_grads(const ChunkBwdArgs &a, cudaStream_t st) {
    const int smem = (int)sizeof(float) * max((kC + D) * (D + 16), kC * (D + 16) + 2 * kC * (kC + 1));
    cudaError_t e = cudaFuncSetAttribute(chunk_bwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    chunk_bwd_kernel<D><<<a.ctas, kThreads, smem, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_chunk_bwd_grads(const ChunkBwdArgs &a, cudaStream_t st) {
    if (a.D == 128) return launch_grads<128>(a, st);
    if (a.D == 64) return launch_grads<64>(a, st);
    return cudaErrorInvalidValue;
}

}  // namespace kda
