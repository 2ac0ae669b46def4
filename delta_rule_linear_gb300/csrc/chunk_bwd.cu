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
//   dV  = diag(beta) T^T dU
//   dL  = -mask_strict(T^T dT T^T)  dK^ = diag(beta e^R) T^T dW + P K^ + P^T K^
//                                         + (dA (.) E_qk)^T Q~ + diag(e^{G_n - G}) dK~,
//                                         P = dL (.) beta_t E_kk
//   dQ~ = (dA (.) E_qk) K^ + diag(e^G) dO S^T
//
// with beta and the decay collected from the same terms (the decay through G, R and G_n,
// then a reverse cumulative sum inside the chunk) and the L2 normalisation's adjoint
// dx = (dx^ - x^ (x^ . dx^)) / |x|.  The state gradients (dS' of every chunk) come from the
// reverse walk (chunk_tc.cu).
//
// One CTA per chunk at a time (persistent CTAs over the chunks, two per SM).  The chunk's
// fp32 intermediates live in the CTA's own scratch region of global memory (L2); the states
// of the two walks are read in place; the per-token scalars and the row / column sums live in
// shared memory.  A product is one or more passes over (A, B) operand pairs into register
// accumulators: each pass stages both operands into shared memory with cp.async (one round
// trip for the whole operand), as they lie in memory -- contraction index along rows or along
// columns, the fragment loads read either form, so no transposed copy is ever written -- and
// runs warp-level tensor MMAs (m16n8k8, tf32 operands, fp32 accumulation) over one 32 x 32 or
// 32 x 16 output tile per warp.  The epilogue first issues every read it needs from memory,
// then stores; the dot products the gradients of beta and the decay take over a product's
// output are its row and column sums, reduced in the epilogue.  Padded rows past a
// sequence's end act as k = q = v = dO = 0, beta = 0, decay = 0 and are never stored.
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

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
// 16-byte copy that reads src_bytes (0 or 16) and zero-fills the rest
__device__ __forceinline__ void cp_async16z(void *dst, const void *src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async8(void *dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_all;" ::: "memory");
}
__device__ __forceinline__ void st2(float *p, float x, float y) { *reinterpret_cast<float2 *>(p) = make_float2(x, y); }
__device__ __forceinline__ float rtf(float x) { return __uint_as_float(tf32(x)); }   // rounded to tf32
// stores an operand of the tensor cores, rounded to tf32 as they would round it
__device__ __forceinline__ void st2r(float *p, float x, float y) { st2(p, rtf(x), rtf(y)); }
__device__ __forceinline__ float2 ld2(const float *p) { return *reinterpret_cast<const float2 *>(p); }

// Operand layouts in shared memory, for an operand with w rows on its side of the product
// (M for A, N for B) and contraction length K.  kRow: element (m, k) at m (K + 16) + k, k
// contiguous -- a quarter warp's 16-byte loads at rows g, g + 1 and columns 4 t4 fall on
// distinct banks since K + 16 = 16 mod 32.  kCol: element (m, k) at k (w + 2) + m, m contiguous
// -- the warp's 4-byte loads at rows 4 t4 + j and columns g fall on distinct banks since
// 4 (w + 2) = 8 mod 32; its rows keep 8-byte alignment only, so it is staged with 8-byte copies.
// kRowH, kColH: the same with bf16 elements (an input read in place: v, dO), pitches K + 16
// and w + 2 in elements -- a half warp's 8-byte loads at rows g .. g + 3 fall on distinct bank
// groups since (K + 16) / 2 = 8 mod 32, and the 2-byte loads at rows 4 t4 + j, columns g on
// distinct banks since 2 (w + 2) = 4 mod 32; bf16 values enter the MMA as they are (exact in
// tf32).  Sizes in floats.
enum Lay { kRow = 0, kCol = 1, kRowH = 2, kColH = 3 };
template <Lay L>
__host__ __device__ constexpr int lay_pitch(int w, int K) { return (L == kRow || L == kRowH) ? K + 16 : w + 2; }
template <Lay L>
__host__ __device__ constexpr int lay_floats(int w, int K) {
    return L == kRow ? w * (K + 16) : L == kCol ? K * (w + 2) : L == kRowH ? w * (K + 16) / 2 : K * (w + 2) / 2;
}
template <Lay L>
__host__ __device__ constexpr bool lay_bf16() { return L == kRowH || L == kColH; }

__device__ __forceinline__ void cp_async4z(void *dst, const void *src, int src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
                 : "memory");
}

// Copies an operand from global memory, where it lies as [w][K] (kRow, kRowH) or [K][w]
// (kCol, kColH) with row stride ld elements, into dst in the layout above.  Rows of memory
// from `valid` on are zeros (bf16 layouts: an input's rows past the sequence's end).
template <Lay L, int w, int K>
__device__ __forceinline__ void stage(float *dst, const void *src, int ld, int valid) {
    if constexpr (L == kRow) {
        const float *sf = static_cast<const float *>(src);
        constexpr int per = K / 4, p = K + 16;
        for (int x = threadIdx.x; x < w * per; x += kThreads) {
            const int r = x / per, c = x % per;
            cp_async16(dst + r * p + 4 * c, sf + (size_t)r * ld + 4 * c);
        }
    } else if constexpr (L == kCol) {
        const float *sf = static_cast<const float *>(src);
        constexpr int per = w / 2, p = w + 2;
        for (int x = threadIdx.x; x < K * per; x += kThreads) {
            const int r = x / per, c = x % per;
            cp_async8(dst + r * p + 2 * c, sf + (size_t)r * ld + 2 * c);
        }
    } else if constexpr (L == kRowH) {
        const __nv_bfloat16 *sh = static_cast<const __nv_bfloat16 *>(src);
        __nv_bfloat16 *dh = reinterpret_cast<__nv_bfloat16 *>(dst);
        constexpr int per = K / 8, p = K + 16;
        for (int x = threadIdx.x; x < w * per; x += kThreads) {
            const int r = x / per, c = x % per;
            const bool in = r < valid;
            cp_async16z(dh + r * p + 8 * c, sh + (size_t)(in ? r : 0) * ld + 8 * c, in ? 16 : 0);
        }
    } else {
        const __nv_bfloat16 *sh = static_cast<const __nv_bfloat16 *>(src);
        __nv_bfloat16 *dh = reinterpret_cast<__nv_bfloat16 *>(dst);
        constexpr int per = w / 2, p = w + 2;
        for (int x = threadIdx.x; x < K * per; x += kThreads) {
            const int r = x / per, c = x % per;
            const bool in = r < valid;
            cp_async4z(dh + r * p + 2 * c, sh + (size_t)(in ? r : 0) * ld + 2 * c, in ? 4 : 0);
        }
    }
}

// The four elements (m, k .. k + 3) of a staged operand.
template <Lay L, int P>
__device__ __forceinline__ void frag4(float (&v)[4], const float *s, int m, int k) {
    if constexpr (L == kRow) {
        const float4 x = *reinterpret_cast<const float4 *>(s + m * P + k);
        v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
    } else if constexpr (L == kCol) {
#pragma unroll
        for (int j = 0; j < 4; ++j) v[j] = s[(k + j) * P + m];
    } else if constexpr (L == kRowH) {
        const uint2 u = *reinterpret_cast<const uint2 *>(reinterpret_cast<const __nv_bfloat16 *>(s) + m * P + k);
        v[0] = __uint_as_float(u.x << 16); v[1] = __uint_as_float(u.x & 0xffff0000u);
        v[2] = __uint_as_float(u.y << 16); v[3] = __uint_as_float(u.y & 0xffff0000u);
    } else {
        const unsigned short *h = reinterpret_cast<const unsigned short *>(s);
#pragma unroll
        for (int j = 0; j < 4; ++j) v[j] = __uint_as_float((uint32_t)h[(k + j) * P + m] << 16);
    }
}

// A 64 x N product's accumulators: warp w owns the output tile of rows 32 (w / 4) ..,
// columns WN (w % 4) .. (WN = 32 for N = 128, 16 for N = 64; eight warps, eight tiles).
// Lane 4 g + t4 holds rows g + 8 i, columns 2 t4 + 8 j (+ 1) of the tile.
template <int N>
struct Acc {
    static constexpr int WN = N / 4, NJ = WN / 8;
    float d[2][NJ][4];
    __device__ __forceinline__ void zero() {
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < NJ; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) d[i][j][e] = 0.f;
    }
};

// acc += A B^T from operands already staged at sa, sb (layouts LA, LB).  Every operand's values
// are tf32 already (stored rounded by their producers, or bf16), so they enter the MMA as
// they are.  Inside a 16-wide k
// step lane t4 takes the four consecutive k = 4 t4 .. 4 t4 + 3 on both operands, the first two
// for one MMA and the last two for the other: the same permutation of k on A and B, which
// leaves the sum unchanged.
template <Lay LA, Lay LB, int N, int K>
__device__ __forceinline__ void mma_staged(Acc<N> &acc, const float *sa, const float *bb) {
    auto ca = [](float x) { return __float_as_uint(x); };
    auto cb = [](float x) { return __float_as_uint(x); };
    constexpr int PA = lay_pitch<LA>(kC, K), PB = lay_pitch<LB>(N, K), NJ = Acc<N>::NJ;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t4 = lane & 3;
    const int m0 = (warp >> 2) * 32, n0 = (warp & 3) * Acc<N>::WN;
#pragma unroll 2
    for (int k0 = 0; k0 < K; k0 += 16) {
        float xa[4][4], zb[NJ][4];
#pragma unroll
        for (int i = 0; i < 4; ++i) frag4<LA, PA>(xa[i], sa, m0 + g + 8 * i, k0 + 4 * t4);
#pragma unroll
        for (int j = 0; j < NJ; ++j) frag4<LB, PB>(zb[j], bb, n0 + 8 * j + g, k0 + 4 * t4);
#pragma unroll
        for (int mi = 0; mi < 2; ++mi) {
            const uint32_t a[4] = {ca(xa[2 * mi][0]), ca(xa[2 * mi + 1][0]), ca(xa[2 * mi][1]), ca(xa[2 * mi + 1][1])};
            const uint32_t a2[4] = {ca(xa[2 * mi][2]), ca(xa[2 * mi + 1][2]), ca(xa[2 * mi][3]), ca(xa[2 * mi + 1][3])};
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
                const uint32_t b[2] = {cb(zb[j][0]), cb(zb[j][1])};
                const uint32_t b2[2] = {cb(zb[j][2]), cb(zb[j][3])};
                mma_tf32(acc.d[mi][j], a, b);
                mma_tf32(acc.d[mi][j], a2, b2);
            }
        }
    }
}

// One pass: acc += A B^T over a contraction of length K, A(m, k) for m < 64 and B(n, k) for
// n < N given in global memory in layouts LA, LB (row strides lda, ldb).  A null pointer
// reuses what the previous pass staged in that buffer (same layout and sizes); B == A stages
// the operand once and reads it on both sides; va, vb: the valid rows of a bf16 operand.  Begins with a barrier of the CTA, so the
// stores of the previous epilogue are visible and the previous pass has finished reading the
// buffers.
template <Lay LA, Lay LB, int N, int K>
__device__ __forceinline__ void pass(Acc<N> &acc, float *sA, float *sB, const void *A, int lda, const void *B,
                                     int ldb, int va = 1 << 30, int vb = 1 << 30) {
    const bool same = (A != nullptr && B == A);
    __syncthreads();
    if (A) stage<LA, kC, K>(sA, A, lda, va);
    if (B && !same) stage<LB, N, K>(sB, B, ldb, vb);
    cp_async_wait_all();
    __syncthreads();
    mma_staged<LA, LB, N, K>(acc, sA, same ? sA : sB);
}

// The epilogue over a product's accumulators (one or two products of the same shape, e.g. two
// terms that the output weighs by different per-column factors).  For each half of the warp's
// tile it first calls pre(r, c) for every element pair (r, c), (r, c + 1) it holds -- the reads
// from memory the epilogue needs, all issued before any store -- then
// epi(r, c, x0, x1, y0, y1, aux, cs) with the accumulated values (x from acc, y from acc2 or
// 0), which stores the outputs, returns a contribution to row r's sum and adds the columns'
// contributions to cs[0], cs[1] (and a second pair of column sums to cs[2], cs[3]).  Row sums
// are reduced over the four lanes of a row and added to rowsum[r]; column sums over the warp's
// rows and added to colsum[c], colsum2[c] (shared memory, each when given).  Ends with a
// barrier of the CTA.
template <int N, typename Pre, typename Epi>
__device__ __forceinline__ void finish2(const Acc<N> &acc, const Acc<N> *acc2, Pre pre, Epi epi, float *rowsum,
                                        float *colsum, float *colsum2) {
    constexpr int NJ = Acc<N>::NJ;
    using Aux = decltype(pre(0, 0));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t4 = lane & 3;
    const int m0 = (warp >> 2) * 32, n0 = (warp & 3) * Acc<N>::WN;
    float cs[NJ][4] = {};
#pragma unroll
    for (int mi = 0; mi < 2; ++mi) {
        Aux aux[2][NJ];
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
            for (int j = 0; j < NJ; ++j) aux[h2][j] = pre(m0 + 16 * mi + g + 8 * h2, n0 + 8 * j + 2 * t4);
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
            const int r = m0 + 16 * mi + g + 8 * h2;
            float part = 0.f;
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
                const float y0 = acc2 ? acc2->d[mi][j][2 * h2] : 0.f, y1 = acc2 ? acc2->d[mi][j][2 * h2 + 1] : 0.f;
                part += epi(r, n0 + 8 * j + 2 * t4, acc.d[mi][j][2 * h2], acc.d[mi][j][2 * h2 + 1], y0, y1, aux[h2][j],
                            cs[j]);
            }
            if (rowsum) {
                part += __shfl_xor_sync(0xffffffffu, part, 1);
                part += __shfl_xor_sync(0xffffffffu, part, 2);
                if (t4 == 0) atomicAdd(rowsum + r, part);
            }
        }
    }
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        float *dst = q == 0 ? colsum : colsum2;
        if (!dst) continue;
#pragma unroll
        for (int j = 0; j < NJ; ++j)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                float v = cs[j][2 * q + e];
                v += __shfl_xor_sync(0xffffffffu, v, 4);
                v += __shfl_xor_sync(0xffffffffu, v, 8);
                v += __shfl_xor_sync(0xffffffffu, v, 16);
                if (g == 0) atomicAdd(dst + n0 + 8 * j + 2 * t4 + e, v);
            }
    }
    __syncthreads();
}

template <int N, typename Pre, typename Epi>
__device__ __forceinline__ void finish(const Acc<N> &acc, Pre pre, Epi epi, float *rowsum = nullptr,
                                       float *colsum = nullptr) {
    finish2<N>(acc, nullptr, pre, epi, rowsum, colsum, nullptr);
}

// The CTA's scratch, in floats: 64 x D and 64 x 64 matrices (row-major).
template <int D>
struct Scr {
    enum { Kh, Qh, Kt, U, dU, dW, dkh, dqh, NBig };   // (v and dO are read in place)
    enum { KKE, A, T, Pv, Pk, P, dQK, NSmall };      // (-W, dT and X go straight to shared memory)
    static constexpr size_t big(int i) { return (size_t)i * kC * D; }
    static constexpr size_t small(int i) { return (size_t)NBig * kC * D + (size_t)i * kC * kC; }
    static constexpr size_t floats = small(NSmall);
};

// Shared memory of the kernel (dynamic part, floats): the two operand buffers, large enough
// for either layout of every operand the products stage; between products the inverse's two
// padded 64 x 64 arrays and the chunk's bf16 input rows reuse them.
template <int D>
struct Smem {
    static constexpr int a_floats = lay_floats<kRow>(kC, D) > lay_floats<kCol>(kC, D) ? lay_floats<kRow>(kC, D)
                                                                                        : lay_floats<kCol>(kC, D);
    static constexpr int b_floats = lay_floats<kRow>(D, D) > lay_floats<kCol>(D, D) ? lay_floats<kRow>(D, D)
                                                                                      : lay_floats<kCol>(D, D);
    static constexpr int inv_floats = 2 * kC * (kC + 1);
    static constexpr int floats = a_floats + (b_floats > inv_floats ? b_floats : inv_floats);
    static_assert(2 * kC * D / 2 <= floats, "bf16 input rows fit the operand buffers");
};

}  // namespace

namespace {

// E consecutive bf16 values (E = 2 or 4) from shared memory, widened exactly.
template <int E>
__device__ __forceinline__ void ld_bf16(float (&f)[E], const __nv_bfloat16 *p) {
    auto lo = [](uint32_t u) { return __uint_as_float(u << 16); };
    auto hi = [](uint32_t u) { return __uint_as_float(u & 0xffff0000u); };
    if constexpr (E == 4) {
        const uint2 u = *reinterpret_cast<const uint2 *>(p);
        f[0] = lo(u.x); f[1] = hi(u.x); f[2] = lo(u.y); f[3] = hi(u.y);
    } else {
        const uint32_t u = *reinterpret_cast<const uint32_t *>(p);
        f[0] = lo(u); f[1] = hi(u);
    }
}
template <int E, bool ROUND = false>
__device__ __forceinline__ void st_row(float *p, const float (&f)[E], float scale) {
    auto r = [&](float x) { return ROUND ? rtf(scale * x) : scale * x; };
    if constexpr (E == 4) *reinterpret_cast<float4 *>(p) = make_float4(r(f[0]), r(f[1]), r(f[2]), r(f[3]));
    else *reinterpret_cast<float2 *>(p) = make_float2(r(f[0]), r(f[1]));
}

template <int D>
__global__ void __launch_bounds__(kThreads, 2) chunk_bwd_kernel(ChunkBwdArgs a) {
    using Sc = Scr<D>;
    constexpr int PL = kC + 1;   // padded rows of the inverse's shared arrays
    extern __shared__ __align__(16) float smem_dyn[];
    float *sA = smem_dyn, *sB = smem_dyn + Smem<D>::a_floats;
    float *sL = sB, *sT = sB + kC * PL;
    __nv_bfloat16 *sIn = reinterpret_cast<__nv_bfloat16 *>(smem_dyn);   // q, k rows: [2][64][D]
    // per-token scalars, then the products' row and column sums, then G_n and its gradient
    __shared__ float sv[18 * kC + 2];
    float *beta = sv, *G = sv + kC, *R = sv + 2 * kC, *eG = sv + 3 * kC, *eR = sv + 4 * kC;
    float *eGnG = sv + 5 * kC, *kn = sv + 6 * kC, *qn = sv + 7 * kC;
    float *rA = sv + 8 * kC, *cA = sv + 9 * kC, *cL = sv + 10 * kC, *rLK = sv + 11 * kC, *rqd = sv + 12 * kC;
    float *rkd = sv + 13 * kC, *rbv = sv + 14 * kC, *rbk = sv + 15 * kC, *kdot = sv + 16 * kC, *qdot = sv + 17 * kC;
    float *sGn = sv + 18 * kC;
    // once the per-token gradients are formed they replace the sums they came from
    float *dG = rA, *dGp = cA, *dbeta = cL;

    float *sc = a.scratch + (size_t)blockIdx.x * Sc::floats;
    auto big = [&](int i) { return sc + Sc::big(i); };
    auto sml = [&](int i) { return sc + Sc::small(i); };
    float *Kh = big(Sc::Kh), *Qh = big(Sc::Qh), *Kt = big(Sc::Kt);
    float *U = big(Sc::U), *dU = big(Sc::dU), *dW = big(Sc::dW);
    float *dkh = big(Sc::dkh), *dqh = big(Sc::dqh);
    float *KKE = sml(Sc::KKE), *A = sml(Sc::A), *T = sml(Sc::T), *Pv = sml(Sc::Pv), *Pk = sml(Sc::Pk);
    float *P = sml(Sc::P), *dQK = sml(Sc::dQK);
    auto nopre = [](int, int) { return 0; };

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
        const __nv_bfloat16 *S = a.fstates + (size_t)ci * D * D;    // state entering the chunk
        const __nv_bfloat16 *dSp = a.bstates + (size_t)ci * D * D;  // gradient of the state leaving it

        // the chunk's rows of v and dO, read in place by the products (bf16, row stride H D)
        const __nv_bfloat16 *V = gv + ((size_t)row0 * a.H + h) * D, *dO = gdo + ((size_t)row0 * a.H + h) * D;
        const int ldt = a.H * D;

        // ---- the chunk's rows of q, k (bf16) into shared memory, zeros past the valid tokens;
        // beta, the in-chunk cumulative log decay, cleared sums
        {
            constexpr int per = D / 8;   // 16-byte pieces of a row
            for (int x = tid; x < 2 * kC * per; x += kThreads) {
                const int arr = x / (kC * per), t = (x / per) % kC, p = x % per;
                const bool valid = t < nv;
                const __nv_bfloat16 *src = arr == 0 ? gq : gk;
                const size_t gi = ((size_t)(row0 + (valid ? t : 0)) * a.H + h) * D + 8 * p;
                cp_async16z(sIn + ((size_t)arr * kC + t) * D + 8 * p, src + gi, valid ? 16 : 0);
            }
            asm volatile("cp.async.commit_group;" ::: "memory");
        }
        if (warp == 0) {   // lane owns tokens 2 lane, 2 lane + 1
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
        } else if (warp == 1) {
            for (int t = lane; t < kC; t += 32) beta[t] = t < nv ? a.beta[(row0 + t) * a.H + h] : 0.f;
        }
        for (int x = tid; x < 10 * kC; x += kThreads) rA[x] = 0.f;
        asm volatile("cp.async.wait_all;" ::: "memory");
        __syncthreads();

        // ---- rows: norms; k^, q~ and K~ = diag(e^{G_n - G}) k^ into the scratch (fp32)
        for (int t = warp; t < kC; t += kWarps) {
            constexpr int E = D / 32;   // consecutive elements per lane
            float fq_[E], fk_[E];
            ld_bf16<E>(fq_, sIn + (size_t)(0 * kC + t) * D + E * lane);
            ld_bf16<E>(fk_, sIn + (size_t)(1 * kC + t) * D + E * lane);
            float ssk = 0.f, ssq = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) {
                ssk = fmaf(fk_[e], fk_[e], ssk);
                ssq = fmaf(fq_[e], fq_[e], ssq);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                ssk += __shfl_xor_sync(0xffffffffu, ssk, o);
                ssq += __shfl_xor_sync(0xffffffffu, ssq, o);
            }
            const float nk = sqrtf(ssk), nq = sqrtf(ssq);
            const float fk = a.use_l2 ? 1.f / fmaxf(nk, kNormEpsB) : 1.f;
            const float fqn = a.use_l2 ? 1.f / fmaxf(nq, kNormEpsB) : 1.f;
            const size_t o = (size_t)t * D + E * lane;
            st_row<E, true>(Kh + o, fk_, fk);
            st_row<E, true>(Kt + o, fk_, fk * eGnG[t]);
            st_row<E, true>(Qh + o, fq_, a.scale * fqn);
            if (lane == 0) {   // the normalisation factors, negative where its adjoint is the identity
                kn[t] = (a.use_l2 && nk > kNormEpsB) ? fk : -fk;
                qn[t] = (a.use_l2 && nq > kNormEpsB) ? fqn : -fqn;
            }
        }

        // ---- A = (q~ k^^T) (.) E_qk (inclusive);  (k^ k^^T) (.) E_kk (strict), kept, and
        // L = beta_t (k^ k^^T) (.) E_kk into the inverse's array: both from one staging of q~, k^
        {
            Acc<kC> acc, acck;
            acc.zero();
            acck.zero();
            pass<kRow, kRow, kC, D>(acc, sA, sB, Qh, D, Kh, D);
            mma_staged<kRow, kRow, kC, D>(acck, sB, sB);
            finish<kC>(acc, nopre, [&](int t, int s, float x0, float x1, float, float, int, float *) -> float {
                const float e0 = s <= t ? __expf(G[t] - G[s]) : 0.f, e1 = s + 1 <= t ? __expf(G[t] - G[s + 1]) : 0.f;
                st2r(A + t * kC + s, x0 * e0, x1 * e1);
                return 0.f;
            });
            // (every warp is past both products: the staged k^ may be overwritten)
            finish<kC>(acck, nopre, [&](int t, int s, float x0, float x1, float, float, int, float *) -> float {
                const float e0 = s < t ? __expf(R[t] - G[s]) : 0.f, e1 = s + 1 < t ? __expf(R[t] - G[s + 1]) : 0.f;
                st2(KKE + t * kC + s, x0 * e0, x1 * e1);
                sL[t * PL + s] = beta[t] * x0 * e0;
                sL[t * PL + s + 1] = beta[t] * x1 * e1;
                return 0.f;
            });
        }

        // ---- T = (I + L)^{-1} in 32 x 32 blocks.  The diagonal blocks by substitution: warp w
        // takes block w, lane j its column j, held in registers; once row s of the column is final
        // its term is subtracted from every later row.  Meanwhile the other warps clear the upper
        // block and sum S (.) dS'.  Then T_BA = -T_BB (L_BA T_AA), L_BA T_AA kept in the L array's unused upper
        // block.
        if (warp < 2) {
            const int o = 32 * warp;
            float tc[32];
#pragma unroll
            for (int r = 0; r < 32; ++r) tc[r] = r == lane ? 1.f : 0.f;
#pragma unroll
            for (int s = 0; s < 31; ++s)
#pragma unroll
                for (int r = s + 1; r < 32; ++r) tc[r] = fmaf(-sL[(o + r) * PL + o + s], tc[s], tc[r]);
#pragma unroll
            for (int r = 0; r < 32; ++r) sT[(o + r) * PL + o + lane] = tc[r];
        } else {
            for (int x = tid - 64; x < 32 * 32; x += kThreads - 64) sT[(x >> 5) * PL + 32 + (x & 31)] = 0.f;
            // e^{G_n} sum(S (.) dS'), a term of the gradient of G_n
            const uint4 *s8 = reinterpret_cast<const uint4 *>(S), *d8 = reinterpret_cast<const uint4 *>(dSp);
            auto lo = [](uint32_t u) { return __uint_as_float(u << 16); };
            auto hi = [](uint32_t u) { return __uint_as_float(u & 0xffff0000u); };
            float acc = 0.f;
#pragma unroll 4
            for (int x = tid - 64; x < D * D / 8; x += kThreads - 64) {   // 8 bf16 at a time
                const uint4 u = s8[x], w = d8[x];
                const uint32_t uu[4] = {u.x, u.y, u.z, u.w}, ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) acc = fmaf(lo(uu[e]), lo(ww[e]), fmaf(hi(uu[e]), hi(ww[e]), acc));
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
            if (lane == 0) atomicAdd(&sGn[1], __expf(sGn[0]) * acc);
        }
        __syncthreads();
        {
            float y[4] = {};
#pragma unroll 8
            for (int s = 0; s < 32; ++s) {
                const float tv = sT[s * PL + lane];
#pragma unroll
                for (int q = 0; q < 4; ++q) y[q] = fmaf(sL[(32 + warp + 8 * q) * PL + s], tv, y[q]);
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) sL[(warp + 8 * q) * PL + 32 + lane] = y[q];
        }
        __syncthreads();
        {
            float y[4] = {};
#pragma unroll 8
            for (int s = 0; s < 32; ++s) {
                const float lv = sL[s * PL + 32 + lane];
#pragma unroll
                for (int q = 0; q < 4; ++q) y[q] = fmaf(sT[(32 + warp + 8 * q) * PL + 32 + s], lv, y[q]);
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) sT[(32 + warp + 8 * q) * PL + lane] = -y[q];
        }
        __syncthreads();
        // T, and T with its columns scaled: Pv = T diag(beta), Pk = T diag(beta e^R), stored
        // rounded to tf32 like every operand of the products (k^, q~, A and the epilogues' st2r
        // outputs; the walks store the states rounded)
        for (int x = tid; x < kC * kC; x += kThreads) {
            const int t = x / kC, s = x % kC;
            const float tv = sT[t * PL + s];
            T[x] = rtf(tv);
            Pv[x] = rtf(tv * beta[s]);
            Pk[x] = rtf(tv * beta[s] * eR[s]);
        }

        // ---- forward quantities: W = Pk K^, negated straight into the A buffer of the next
        // product (once every warp is done reading it), U = -W S + Pv V
        {
            Acc<D> acc;
            acc.zero();
            pass<kRow, kCol, D, kC>(acc, sA, sB, Pk, kC, Kh, D);
            __syncthreads();
            finish<D>(acc, nopre, [&](int t, int j, float x0, float x1, float, float, int, float *) -> float {
                st2r(sA + t * (D + 16) + j, -x0, -x1);   // kRow, contraction D
                return 0.f;
            });
        }
        {
            Acc<D> acc;
            acc.zero();
            pass<kRow, kColH, D, D>(acc, sA, sB, nullptr, D, S, D);   // -W is staged
            pass<kRow, kColH, D, kC>(acc, sA, sB, Pv, kC, V, ldt, 1 << 30, nv);
            finish<D>(acc, nopre, [&](int t, int j, float x0, float x1, float, float, int, float *) -> float {
                st2r(U + t * D + j, x0, x1);
                return 0.f;
            });
        }
        // ---- dU = A^T dO + K~ dS'
        {
            Acc<D> acc;
            acc.zero();
            pass<kCol, kColH, D, kC>(acc, sA, sB, A, kC, dO, ldt, 1 << 30, nv);
            pass<kRow, kColH, D, D>(acc, sA, sB, Kt, D, dSp, D);
            finish<D>(acc, nopre, [&](int s, int j, float x0, float x1, float, float, int, float *) -> float {
                st2r(dU + s * D + j, x0, x1);
                return 0.f;
            });
        }
        // ---- dV = diag(beta) T^T dU, written out (fp32)
        {
            Acc<D> acc;
            acc.zero();
            pass<kCol, kCol, D, kC>(acc, sA, sB, T, kC, dU, D);
            finish<D>(acc, nopre, [&](int s, int j, float x0, float x1, float, float, int, float *) -> float {
                if (s < nv) st2(a.dv + ((size_t)(row0 + s) * a.H + h) * D + j, beta[s] * x0, beta[s] * x1);
                return 0.f;
            });
        }
        // ---- dq~ = diag(e^G) dO S^T (its first term); row sums q~ . dO S^T
        {
            Acc<D> acc;
            acc.zero();
            pass<kRowH, kRowH, D, D>(acc, sA, sB, dO, ldt, S, D, nv);
            finish<D>(acc, [&](int t, int i) { return ld2(Qh + t * D + i); },
                      [&](int t, int i, float x0, float x1, float, float, float2 q, float *) -> float {
                          st2(dqh + t * D + i, eG[t] * x0, eG[t] * x1);
                          return x0 * q.x + x1 * q.y;
                      },
                      rqd);
        }
        // ---- dW = -dU S^T
        {
            Acc<D> acc;
            acc.zero();
            pass<kRow, kRowH, D, D>(acc, sA, sB, dU, D, nullptr, D);   // S is still staged
            finish<D>(acc, nopre, [&](int s, int i, float x0, float x1, float, float, int, float *) -> float {
                st2r(dW + s * D + i, -x0, -x1);
                return 0.f;
            });
        }
        // ---- dT = diag(beta) applied to the columns of dU V^T, plus diag(beta e^R) to those of
        // dW K^^T; the column sums of T (.) (dU V^T) and T (.) (dW K^^T) are (T^T dU) . v and
        // (T^T dW) . k^, the terms of beta's gradient through V and through K^
        {
            Acc<kC> acc, acc2;
            acc.zero();
            acc2.zero();
            pass<kRow, kRowH, kC, D>(acc, sA, sB, nullptr, D, V, ldt, 1 << 30, nv);   // dU is still staged
            pass<kRow, kRow, kC, D>(acc2, sA, sB, dW, D, Kh, D);
            __syncthreads();   // dT goes straight into the A buffer of X = dT T^T
            finish2<kC>(acc, &acc2, [&](int t, int s) { return ld2(T + t * kC + s); },
                        [&](int t, int s, float x0, float x1, float y0, float y1, float2 tv, float *cs) -> float {
                            const float b0 = beta[s], b1 = beta[s + 1];
                            st2r(sA + t * (kC + 16) + s, b0 * (x0 + eR[s] * y0), b1 * (x1 + eR[s + 1] * y1));
                            cs[0] += tv.x * x0;
                            cs[1] += tv.y * x1;
                            cs[2] += tv.x * y0;
                            cs[3] += tv.y * y1;
                            return 0.f;
                        },
                        nullptr, rbv, rbk);
        }
        // ---- X = dT T^T;  dL = -mask_strict(T^T X) -> P = dL (.) beta_t E_kk, with the row sums
        // of dL (.) (k^ k^^T) E_kk and the column sums of dL (.) L
        {
            Acc<kC> acc;
            acc.zero();
            pass<kRow, kRow, kC, kC>(acc, sA, sB, nullptr, kC, T, kC);   // dT is staged
            __syncthreads();   // X goes straight into the B buffer of T^T X (kCol: X[r][s] at r (64 + 2) + s)
            finish<kC>(acc, nopre, [&](int t, int s, float x0, float x1, float, float, int, float *) -> float {
                sB[t * (kC + 2) + s] = rtf(x0);
                sB[t * (kC + 2) + s + 1] = rtf(x1);
                return 0.f;
            });
        }
        {
            Acc<kC> acc;
            acc.zero();
            pass<kCol, kCol, kC, kC>(acc, sA, sB, T, kC, nullptr, kC);   // X is staged
            finish<kC>(acc, [&](int t, int s) { return ld2(KKE + t * kC + s); },
                       [&](int t, int s, float x0, float x1, float, float, float2 kk, float *cs) -> float {
                           const float l0 = s < t ? -x0 : 0.f, l1 = s + 1 < t ? -x1 : 0.f;
                           const float e0 = s < t ? __expf(R[t] - G[s]) : 0.f;
                           const float e1 = s + 1 < t ? __expf(R[t] - G[s + 1]) : 0.f;
                           const float bt = beta[t];
                           st2r(P + t * kC + s, l0 * bt * e0, l1 * bt * e1);
                           const float p0 = l0 * kk.x, p1 = l1 * kk.y;
                           cs[0] += bt * p0;
                           cs[1] += bt * p1;
                           return p0 + p1;
                       },
                       rLK, cL);
        }
        // ---- dA = mask_incl(dO U^T) -> dA (.) E_qk; row and column sums of dA (.) A
        {
            Acc<kC> acc;
            acc.zero();
            pass<kRowH, kRow, kC, D>(acc, sA, sB, dO, ldt, U, D, nv);
            finish<kC>(acc, [&](int t, int s) { return ld2(A + t * kC + s); },
                       [&](int t, int s, float x0, float x1, float, float, float2 av, float *cs) -> float {
                           const float e0 = s <= t ? __expf(G[t] - G[s]) : 0.f;
                           const float e1 = s + 1 <= t ? __expf(G[t] - G[s + 1]) : 0.f;
                           const float d0 = s <= t ? x0 : 0.f, d1 = s + 1 <= t ? x1 : 0.f;
                           st2r(dQK + t * kC + s, d0 * e0, d1 * e1);
                           const float p0 = d0 * av.x, p1 = d1 * av.y;
                           cs[0] += p0;
                           cs[1] += p1;
                           return p0 + p1;
                       },
                       rA, cA);
        }
        // ---- dK~ = U dS'^T: dk^ = diag(e^{G_n - G}) dK~ (its first term); row sums K~ . dK~
        {
            Acc<D> acc;
            acc.zero();
            pass<kRow, kRowH, D, D>(acc, sA, sB, U, D, dSp, D);
            finish<D>(acc, [&](int s, int i) { return ld2(Kh + s * D + i); },
                      [&](int s, int i, float x0, float x1, float, float, float2 k, float *) -> float {
                          const float w = eGnG[s];
                          st2(dkh + s * D + i, w * x0, w * x1);
                          return w * (x0 * k.x + x1 * k.y);
                      },
                      rkd);
        }
        // ---- dk^ += Pk^T dW + P K^ + P^T K^ + (dA (.) E_qk)^T Q~  (Pk^T dW = diag(beta e^R) T^T dW);
        // row sums k^ . dk^
        {
            Acc<D> acc;
            acc.zero();
            pass<kCol, kCol, D, kC>(acc, sA, sB, Pk, kC, dW, D);
            pass<kRow, kCol, D, kC>(acc, sA, sB, P, kC, Kh, D);
            pass<kCol, kCol, D, kC>(acc, sA, sB, P, kC, nullptr, D);   // K^ is still staged
            pass<kCol, kCol, D, kC>(acc, sA, sB, dQK, kC, Qh, D);
            finish<D>(acc,
                      [&](int s, int i) {
                          const float2 o = ld2(dkh + s * D + i), k = ld2(Kh + s * D + i);
                          return make_float4(o.x, o.y, k.x, k.y);
                      },
                      [&](int s, int i, float x0, float x1, float, float, float4 ok, float *) -> float {
                          const float d0 = ok.x + x0, d1 = ok.y + x1;
                          st2(dkh + s * D + i, d0, d1);
                          return d0 * ok.z + d1 * ok.w;
                      },
                      kdot);
        }
        // ---- dq~ += (dA (.) E_qk) K^;  row sums q~ . dq~
        {
            Acc<D> acc;
            acc.zero();
            pass<kRow, kCol, D, kC>(acc, sA, sB, dQK, kC, Kh, D);
            finish<D>(acc,
                      [&](int t, int i) {
                          const float2 o = ld2(dqh + t * D + i), q = ld2(Qh + t * D + i);
                          return make_float4(o.x, o.y, q.x, q.y);
                      },
                      [&](int t, int i, float x0, float x1, float, float, float4 oq, float *) -> float {
                          const float d0 = oq.x + x0, d1 = oq.y + x1;
                          st2(dqh + t * D + i, d0, d1);
                          return d0 * oq.z + d1 * oq.w;
                      },
                      qdot);
        }

        // ---- per token: the gradients of G, of R (through G_{t-1} or G_t) and of beta
        if (tid < kC) {
            const int t = tid;
            const float dr = beta[t] * rLK[t] + beta[t] * eR[t] * rbk[t];
            float dg = eG[t] * rqd[t] + rA[t] - cA[t] - cL[t] - rkd[t];
            float dgp = 0.f;
            if (a.decayed_read) dg += dr; else dgp = dr;
            const float db = rbv[t] + eR[t] * rbk[t] + rLK[t];
            atomicAdd(&sGn[1], rkd[t]);
            dG[t] = dg;
            dGp[t] = dgp;
            dbeta[t] = db;
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
        // ---- dq, dk through the normalisation: dx = f (dx^ - x^ (x^ . dx^)) where |x| > eps
        {
            constexpr int per = D / 4, iters = kC * per / kThreads;   // float4 pieces
            const float qs = a.scale * a.scale;
#pragma unroll
            for (int u0 = 0; u0 < iters; u0 += 4) {
                float4 kh[4], gk[4], qh[4], gq[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int x = tid + (u0 + u) * kThreads;
                    kh[u] = reinterpret_cast<const float4 *>(Kh)[x];
                    gk[u] = reinterpret_cast<const float4 *>(dkh)[x];
                    qh[u] = reinterpret_cast<const float4 *>(Qh)[x];
                    gq[u] = reinterpret_cast<const float4 *>(dqh)[x];
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int x = tid + (u0 + u) * kThreads, t = x / per, i = 4 * (x % per);
                    if (t >= nv) continue;
                    const float fk = fabsf(kn[t]), ck = kn[t] > 0.f ? kdot[t] : 0.f;
                    const float fq = a.scale * fabsf(qn[t]), cq = qn[t] > 0.f ? qdot[t] / qs : 0.f;
                    const size_t gi = ((size_t)(row0 + t) * a.H + h) * D + i;
                    *reinterpret_cast<float4 *>(a.dk + gi) =
                        make_float4(fk * (gk[u].x - kh[u].x * ck), fk * (gk[u].y - kh[u].y * ck),
                                    fk * (gk[u].z - kh[u].z * ck), fk * (gk[u].w - kh[u].w * ck));
                    *reinterpret_cast<float4 *>(a.dq + gi) =
                        make_float4(fq * (gq[u].x - qh[u].x * cq), fq * (gq[u].y - qh[u].y * cq),
                                    fq * (gq[u].z - qh[u].z * cq), fq * (gq[u].w - qh[u].w * cq));
                }
            }
        }
        __syncthreads();   // the scratch and the shared arrays are rewritten by the next chunk
    }
}

}  // namespace

size_t chunk_bwd_scratch_floats(int D) {
    return D == 128 ? Scr<128>::floats : Scr<64>::floats;
}

// Persistent CTAs of the gradient kernel for `nchunks` (chunk, head) items: at most 304 (two
// per SM on a 152-SM part), as few as keep the same number of waves, so that every CTA takes
// the same number of chunks (1024 chunks: 256 CTAs of four, 0.889 ms for the whole backward
// against 0.948 ms with 304 CTAs, of which 112 ran a fourth wave).  It depends on the shape
// alone, so that the workspace query needs no device (each CTA has its own scratch region).
int chunk_bwd_ctas(long nchunks) {
    constexpr long kMaxCtas = 304;
    if (nchunks < 1) return 1;
    const long waves = (nchunks + kMaxCtas - 1) / kMaxCtas;
    return (int)((nchunks + waves - 1) / waves);
}

template <int D>
cudaError_t launch_grads(const ChunkBwdArgs &a, cudaStream_t st) {
    const int smem = (int)sizeof(float) * Smem<D>::floats;
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
