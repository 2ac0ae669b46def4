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

// element (r, c) of an fp32 matrix at p[r * rs + c * cs]
struct Mat {
    const float *p;
    int rs, cs;
    __device__ __forceinline__ float operator()(int r, int c) const { return p[(size_t)r * rs + (size_t)c * cs]; }
};

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

// C[M x N] = A[M x K] B[K x N] (M a multiple of 16, N of 8, K of 8), the warps of the CTA
// taking the 16 x 8 output tiles in turn; epi(r, c, v0, v1) receives C[r][c], C[r][c + 1]
// (lane = 4 g + t4 holds rows g and g + 8, columns 2 t4 and 2 t4 + 1 of its tile).
template <typename Epi>
__device__ __forceinline__ void gemm(int M, int N, int K, Mat A, Mat B, Epi epi) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t4 = lane & 3;
    const int tn = N >> 3, tiles = (M >> 4) * tn;
    for (int tile = warp; tile < tiles; tile += kWarps) {
        const int m0 = (tile / tn) << 4, n0 = (tile % tn) << 3;
        float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
        for (int k0 = 0; k0 < K; k0 += 8) {
            const uint32_t a[4] = {tf32(A(m0 + g, k0 + t4)), tf32(A(m0 + g + 8, k0 + t4)),
                                   tf32(A(m0 + g, k0 + t4 + 4)), tf32(A(m0 + g + 8, k0 + t4 + 4))};
            const uint32_t b[2] = {tf32(B(k0 + t4, n0 + g)), tf32(B(k0 + t4 + 4, n0 + g))};
            mma_tf32(d, a, b);
        }
        epi(m0 + g, n0 + 2 * t4, d[0], d[1]);
        epi(m0 + g + 8, n0 + 2 * t4, d[2], d[3]);
    }
}

// The CTA's scratch, in floats: 64 x D matrices, 64 x 64 matrices, per-token scalars.
template <int D>
struct Scr {
    enum { Kh, Qh, V, dO, Kt, W, U, dU, dW, dKt, DOS, dBv, dBk, dkh, dqh, NBig };
    enum { KKE, Ekk, L, A, Eqk, T, Pv, Pk, dA, dT, X, dL, dKK, NSmall };
    enum { beta, G, R, eG, eR, eGnG, kn, qn, knorm, qnorm, dG, dGp, dbeta, NScal };
    static constexpr size_t big(int i) { return (size_t)i * kC * D; }
    static constexpr size_t small(int i) { return (size_t)NBig * kC * D + (size_t)i * kC * kC; }
    static constexpr size_t scal(int i) { return small(NSmall) + (size_t)i * kC; }
    static constexpr size_t floats = scal(NScal) + 64;   // + the chunk's G_n terms
};

}  // namespace

namespace {

__device__ __forceinline__ float bf2f(__nv_bfloat16 x) { return __bfloat162float(x); }

template <int D>
__global__ void __launch_bounds__(kThreads) chunk_bwd_kernel(ChunkBwdArgs a) {
    using Sc = Scr<D>;
    constexpr int PL = kC + 1;   // padded rows of the inverse's shared arrays
    __shared__ float sL[kC * PL], sT[kC * PL];
    __shared__ float red[8 * kC];   // per-token row / column sums
    __shared__ float sGn[2];        // G_n, and the chunk's gradient of G_n
    float *sc = a.scratch + (size_t)blockIdx.x * Sc::floats;
    auto big = [&](int i) { return sc + Sc::big(i); };
    auto sml = [&](int i) { return sc + Sc::small(i); };
    auto scl = [&](int i) { return sc + Sc::scal(i); };
    float *Kh = big(Sc::Kh), *Qh = big(Sc::Qh), *V = big(Sc::V), *dO = big(Sc::dO), *Kt = big(Sc::Kt);
    float *W = big(Sc::W), *U = big(Sc::U), *dU = big(Sc::dU), *dW = big(Sc::dW), *dKt = big(Sc::dKt);
    float *DOS = big(Sc::DOS), *dBv = big(Sc::dBv), *dBk = big(Sc::dBk), *dkh = big(Sc::dkh), *dqh = big(Sc::dqh);
    float *KKE = sml(Sc::KKE), *Ekk = sml(Sc::Ekk), *L = sml(Sc::L), *A = sml(Sc::A), *Eqk = sml(Sc::Eqk);
    float *T = sml(Sc::T), *Pv = sml(Sc::Pv), *Pk = sml(Sc::Pk), *dA = sml(Sc::dA), *dT = sml(Sc::dT);
    float *X = sml(Sc::X), *dL = sml(Sc::dL), *dKK = sml(Sc::dKK);
    float *beta = scl(Sc::beta), *G = scl(Sc::G), *R = scl(Sc::R), *eG = scl(Sc::eG), *eR = scl(Sc::eR);
    float *eGnG = scl(Sc::eGnG), *kn = scl(Sc::kn), *qn = scl(Sc::qn), *knorm = scl(Sc::knorm);
    float *qnorm = scl(Sc::qnorm), *dG = scl(Sc::dG), *dGp = scl(Sc::dGp), *dbeta = scl(Sc::dbeta);
    float *rA = red, *cA = red + kC, *rL = red + 2 * kC, *cL = red + 3 * kC, *rLK = red + 4 * kC;

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

        // ---- rows: norms, k^, q~, v, dO (zero past the valid tokens), cleared accumulators
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
                Kh[t * D + i] = kk[m] * fk;
                Qh[t * D + i] = qq[m] * fq;
                V[t * D + i] = valid ? bf2f(gv[gi + i]) : 0.f;
                dO[t * D + i] = valid ? bf2f(gdo[gi + i]) : 0.f;
                dkh[t * D + i] = 0.f;
                dqh[t * D + i] = 0.f;
            }
            if (lane == 0) {
                kn[t] = fk; qn[t] = fq; knorm[t] = nk; qnorm[t] = nq;
                beta[t] = valid ? a.beta[(row0 + t) * a.H + h] : 0.f;
            }
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

        // ---- Gram products: L = beta_t (k^ k^^T) E_kk (strict), A = (q~ k^^T) E_qk (inclusive)
        gemm(kC, kC, D, Mat{Kh, D, 1}, Mat{Kh, 1, D}, [&](int t, int s, float v0, float v1) {
            const float vv[2] = {v0, v1};
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const float e = (s + u < t) ? __expf(R[t] - G[s + u]) : 0.f;
                KKE[t * kC + s + u] = vv[u] * e;
                Ekk[t * kC + s + u] = e;
                L[t * kC + s + u] = beta[t] * vv[u] * e;
                sL[t * PL + s + u] = beta[t] * vv[u] * e;
            }
        });
        gemm(kC, kC, D, Mat{Qh, D, 1}, Mat{Kh, 1, D}, [&](int t, int s, float v0, float v1) {
            const float vv[2] = {v0, v1};
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const float e = (s + u <= t) ? __expf(G[t] - G[s + u]) : 0.f;
                A[t * kC + s + u] = vv[u] * e;
                Eqk[t * kC + s + u] = e;
            }
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
            Pv[x] = tv * beta[s];
            Pk[x] = tv * beta[s] * eR[s];
        }
        __syncthreads();

        // ---- forward quantities: W = T diag(beta e^R) K^, U = T diag(beta) V - W S
        gemm(kC, D, kC, Mat{Pk, kC, 1}, Mat{Kh, D, 1}, [&](int t, int j, float v0, float v1) {
            W[t * D + j] = v0; W[t * D + j + 1] = v1;
        });
        gemm(kC, D, kC, Mat{Pv, kC, 1}, Mat{V, D, 1}, [&](int t, int j, float v0, float v1) {
            U[t * D + j] = v0; U[t * D + j + 1] = v1;
        });
        // dU = A^T dO (same output tiles as U: the dU writes do not race the U writes)
        gemm(kC, D, kC, Mat{A, 1, kC}, Mat{dO, D, 1}, [&](int s, int j, float v0, float v1) {
            dU[s * D + j] = v0; dU[s * D + j + 1] = v1;
        });
        __syncthreads();
        gemm(kC, D, D, Mat{W, D, 1}, Mat{S, D, 1}, [&](int t, int j, float v0, float v1) {
            U[t * D + j] -= v0; U[t * D + j + 1] -= v1;
        });
        // dU += K~ dS';  DOS = dO S^T
        gemm(kC, D, D, Mat{Kt, D, 1}, Mat{dSp, D, 1}, [&](int s, int j, float v0, float v1) {
            dU[s * D + j] += v0; dU[s * D + j + 1] += v1;
        });
        gemm(kC, D, D, Mat{dO, D, 1}, Mat{S, 1, D}, [&](int t, int i, float v0, float v1) {
            DOS[t * D + i] = v0; DOS[t * D + i + 1] = v1;
        });
        __syncthreads();

        // ---- dA = mask_incl(dO U^T),  dK~ = U dS'^T,  dW = -dU S^T
        gemm(kC, kC, D, Mat{dO, D, 1}, Mat{U, 1, D}, [&](int t, int s, float v0, float v1) {
            dA[t * kC + s] = s <= t ? v0 : 0.f;
            dA[t * kC + s + 1] = s + 1 <= t ? v1 : 0.f;
        });
        gemm(kC, D, D, Mat{U, D, 1}, Mat{dSp, 1, D}, [&](int s, int i, float v0, float v1) {
            dKt[s * D + i] = v0; dKt[s * D + i + 1] = v1;
        });
        gemm(kC, D, D, Mat{dU, D, 1}, Mat{S, 1, D}, [&](int s, int i, float v0, float v1) {
            dW[s * D + i] = -v0; dW[s * D + i + 1] = -v1;
        });
        __syncthreads();

        // ---- dT = dU (diag(beta) V)^T + dW (diag(beta e^R) K^)^T;  dBv = T^T dU;  dBk = T^T dW,
        // dK^ += diag(beta e^R) dBk
        gemm(kC, kC, D, Mat{dU, D, 1}, Mat{V, 1, D}, [&](int t, int s, float v0, float v1) {
            dT[t * kC + s] = v0 * beta[s];
            dT[t * kC + s + 1] = v1 * beta[s + 1];
        });
        gemm(kC, D, kC, Mat{T, 1, kC}, Mat{dU, D, 1}, [&](int s, int j, float v0, float v1) {
            dBv[s * D + j] = v0; dBv[s * D + j + 1] = v1;
        });
        gemm(kC, kC, D, Mat{dW, D, 1}, Mat{Kh, 1, D}, [&](int t, int s, float v0, float v1) {
            dT[t * kC + s] += v0 * beta[s] * eR[s];
            dT[t * kC + s + 1] += v1 * beta[s + 1] * eR[s + 1];
        });
        gemm(kC, D, kC, Mat{T, 1, kC}, Mat{dW, D, 1}, [&](int s, int i, float v0, float v1) {
            dBk[s * D + i] = v0; dBk[s * D + i + 1] = v1;
            const float w = beta[s] * eR[s];
            dkh[s * D + i] += w * v0; dkh[s * D + i + 1] += w * v1;
        });
        __syncthreads();

        // ---- dL = -mask_strict(T^T dT T^T)
        gemm(kC, kC, kC, Mat{dT, kC, 1}, Mat{T, 1, kC}, [&](int t, int s, float v0, float v1) {
            X[t * kC + s] = v0; X[t * kC + s + 1] = v1;
        });
        __syncthreads();
        gemm(kC, kC, kC, Mat{T, 1, kC}, Mat{X, kC, 1}, [&](int t, int s, float v0, float v1) {
            dL[t * kC + s] = s < t ? -v0 : 0.f;
            dL[t * kC + s + 1] = s + 1 < t ? -v1 : 0.f;
        });
        __syncthreads();

        // ---- row and column sums of dA (.) A and dL (.) L, dL (.) KKE; P = dL beta_t E_kk,
        // dA (.) E_qk (into X)
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
            const int t = x / kC;
            dKK[x] = dL[x] * beta[t] * Ekk[x];
            X[x] = dA[x] * Eqk[x];
        }
        __syncthreads();
        // dK^ += P K^ + P^T K^ + (dA E_qk)^T Q~;  dQ~ += (dA E_qk) K^  (each element of dkh and
        // dqh stays with one thread across these products)
        gemm(kC, D, kC, Mat{dKK, kC, 1}, Mat{Kh, D, 1}, [&](int t, int i, float v0, float v1) {
            dkh[t * D + i] += v0; dkh[t * D + i + 1] += v1;
        });
        gemm(kC, D, kC, Mat{dKK, 1, kC}, Mat{Kh, D, 1}, [&](int s, int i, float v0, float v1) {
            dkh[s * D + i] += v0; dkh[s * D + i + 1] += v1;
        });
        gemm(kC, D, kC, Mat{X, 1, kC}, Mat{Qh, D, 1}, [&](int s, int i, float v0, float v1) {
            dkh[s * D + i] += v0; dkh[s * D + i + 1] += v1;
        });
        gemm(kC, D, kC, Mat{X, kC, 1}, Mat{Kh, D, 1}, [&](int t, int i, float v0, float v1) {
            dqh[t * D + i] += v0; dqh[t * D + i + 1] += v1;
        });
        __syncthreads();

        // ---- per token: dG, dR, dbeta; dK^ += e^{G_n - G} dK~;  dQ~ += e^G dO S^T
        for (int t = warp; t < kC; t += kWarps) {
            float qd = 0.f, kd = 0.f, bv = 0.f, bk = 0.f;
            const float et = eG[t], en = eGnG[t];
#pragma unroll
            for (int m = 0; m < D / 32; ++m) {
                const int x = t * D + lane + 32 * m;
                qd = fmaf(Qh[x], DOS[x], qd);
                kd = fmaf(dKt[x], Kt[x], kd);
                bv = fmaf(dBv[x], V[x], bv);
                bk = fmaf(dBk[x], Kh[x], bk);
                dkh[x] += en * dKt[x];
                dqh[x] += et * DOS[x];
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                qd += __shfl_xor_sync(0xffffffffu, qd, o);
                kd += __shfl_xor_sync(0xffffffffu, kd, o);
                bv += __shfl_xor_sync(0xffffffffu, bv, o);
                bk += __shfl_xor_sync(0xffffffffu, bk, o);
            }
            if (lane == 0) {
                const float dr = rL[t] + beta[t] * eR[t] * bk;
                float dg = et * qd + rA[t] - cA[t] - cL[t] - kd;
                float dgp = 0.f;
                if (a.decayed_read) dg += dr; else dgp = dr;
                dG[t] = dg;
                dGp[t] = dgp;
                dbeta[t] = bv + eR[t] * bk + rLK[t];
                atomicAdd(&sGn[1], kd);
            }
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
int chunk_bwd_ctas() { return 160; }

cudaError_t launch_chunk_bwd_grads(const ChunkBwdArgs &a, cudaStream_t st) {
    if (a.D == 128) chunk_bwd_kernel<128><<<a.ctas, kThreads, 0, st>>>(a);
    else if (a.D == 64) chunk_bwd_kernel<64><<<a.ctas, kThreads, 0, st>>>(a);
    else return cudaErrorInvalidValue;
    return cudaGetLastError();
}

}  // namespace kda
