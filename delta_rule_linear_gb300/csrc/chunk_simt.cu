// chunk_simt.cu -- chunked prefill on CUDA cores, all arithmetic in fp32.
//
// Chunked mode of ejkernel kda() ("Algorithm Modes": parallel inside a chunk,
// sequential across chunks) in the WY / UT-transform form (the representation
// TileOPs DeltaNetChunkFwdOp computes with prepare_wy_repr -> w, u).  For a chunk
// of n <= C tokens entering with state S, G_t the inclusive in-chunk sum of decay, and
// R_t = G_{t-1} (the delta term reads h_{t-1}) or G_t (it reads the decayed memory):
//
//   L[t][s]  = beta_t (k^_t . k^_s) exp(R_t - G_s)               s < t
//   T        = (I + L)^{-1}                                      forward substitution
//   W        = T diag(beta_s exp(R_s)) K^                        [C, dk]
//   U0       = T diag(beta_s) V                                  [C, dv-tile]
//   U        = U0 - W S                                          (the delta terms u_t)
//   Aqk[t][s] = (q~_t . k^_s) exp(G_t - G_s)                     s <= t
//   O        = diag(exp G_t) Q~ S + Aqk U
//   S_next   = exp(G_n) S + sum_s exp(G_n - G_s) k^_s u_s^T
//
// No floating-point tensor-core instruction is used: an fp32 caller gets fp32
// arithmetic throughout (TileOPs DeltaNetRecurrentFwdOp: the fp32 path avoids
// TF32 mantissa truncation).  One CTA owns one (sequence, head, value tile) and
// walks its chunks in order; everything lives in shared memory.  Rows past the
// end of a sequence are zero keys with beta = 0 and decay = 0, which leaves the
// state and the valid outputs unchanged; their outputs are not stored.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kThreads = 256;
constexpr int kCMax = 64;

template <int DK, int DVT>
struct SimtLayout {
    static constexpr int KP = DK + 1;   // padded rows: conflict-free column walks
    static constexpr int CP = kCMax + 1;
    static constexpr int oK = 0;                     // k^   [C][KP]
    static constexpr int oQ = oK + kCMax * KP;       // q~   [C][KP]
    static constexpr int oW = oQ + kCMax * KP;       // W    [C][KP]
    static constexpr int oL = oW + kCMax * KP;       // L    [C][CP]
    static constexpr int oT = oL + kCMax * CP;       // T    [C][CP]
    static constexpr int oA = oT + kCMax * CP;       // Aqk  [C][CP]
    static constexpr int oV = oA + kCMax * CP;       // V -> U0 -> U  [C][DVT]
    static constexpr int oS = oV + kCMax * DVT;      // S    [DK][DVT]
    static constexpr int ob = oS + DK * DVT;         // beta
    static constexpr int oG = ob + kCMax;            // G (inclusive)
    static constexpr int oGp = oG + kCMax;           // G_{t-1}
    static constexpr int obg = oGp + kCMax;          // beta_t exp(G_{t-1})
    static constexpr int okd = obg + kCMax;          // exp(G_n - G_t)
    static constexpr int oeg = okd + kCMax;          // exp(G_t)
    static constexpr int total = oeg + kCMax;
    static constexpr size_t bytes = sizeof(float) * total;
};

template <typename Tin, int DK, int DVT>
__global__ void __launch_bounds__(kThreads) chunk_simt_kernel(SeqBatch p) {
    using Lay = SimtLayout<DK, DVT>;
    constexpr int KP = Lay::KP, CP = Lay::CP;
    constexpr int EPL = DK / 32;                        // key elements per lane
    constexpr int RU = (kCMax * DVT + kThreads - 1) / kThreads;
    extern __shared__ float smem[];
    float *sK = smem + Lay::oK, *sQ = smem + Lay::oQ, *sW = smem + Lay::oW;
    float *sL = smem + Lay::oL, *sT = smem + Lay::oT, *sA = smem + Lay::oA;
    float *sV = smem + Lay::oV, *sS = smem + Lay::oS;
    float *sb = smem + Lay::ob, *sG = smem + Lay::oG, *sGp = smem + Lay::oGp;
    float *sbg = smem + Lay::obg, *skd = smem + Lay::okd, *seg = smem + Lay::oeg;

    const int C = p.chunk;
    const int DV = p.dv, H = p.H;
    const int ntile = DV / DVT;
    const int tile = blockIdx.x % ntile;
    const int h = (blockIdx.x / ntile) % H;
    const int n = blockIdx.x / (ntile * H);
    const int col0 = tile * DVT;
    long start;
    int len;
    seq_range(p, n, start, len);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const Tin *q = static_cast<const Tin *>(p.q);
    const Tin *k = static_cast<const Tin *>(p.k);
    const Tin *v = static_cast<const Tin *>(p.v);
    Tin *o = static_cast<Tin *>(p.o);
    // element (i, j) of the state: key-major at i DV + j, value-major at j DK + i
    const size_t st_head = ((size_t)n * H + h) * DK * DV;
    const auto st_at = [&](int i, int j) -> size_t {
        return p.v_first ? st_head + (size_t)(col0 + j) * DK + i : st_head + (size_t)i * DV + col0 + j;
    };

    for (int idx = tid; idx < DK * DVT; idx += kThreads) {
        const int i = p.v_first ? idx % DK : idx / DVT, j = p.v_first ? idx / DK : idx % DVT;
        sS[i * DVT + j] = p.h0 ? p.h0[st_at(i, j)] : 0.f;
    }

    for (int c0 = 0; c0 < len; c0 += C) {
        const int nrow = min(C, len - c0);
        // --- rows of the chunk: normalised keys, scaled queries, values, beta, decay
        for (int t = warp; t < C; t += kThreads / 32) {
            float kv[EPL], qv[EPL];
            float sk = 0.f, sq = 0.f;
            const int G = p.G > 1 ? p.G : 1;   // q/k head h / G of value head h
            const size_t off = ((size_t)(start + c0 + t) * (H / G) + h / G) * DK;
#pragma unroll
            for (int e = 0; e < EPL; ++e) {
                kv[e] = t < nrow ? to_f32(k[off + lane + 32 * e]) : 0.f;
                qv[e] = t < nrow ? to_f32(q[off + lane + 32 * e]) : 0.f;
                sk = fmaf(kv[e], kv[e], sk);
                sq = fmaf(qv[e], qv[e], sq);
            }
#pragma unroll
            for (int x = 16; x > 0; x >>= 1) {
                sk += __shfl_xor_sync(0xffffffffu, sk, x);
                sq += __shfl_xor_sync(0xffffffffu, sq, x);
            }
            const float kn = p.use_l2 ? 1.f / fmaxf(sqrtf(sk), kNormEps) : 1.f;
            const float qn = p.scale * (p.use_l2 ? 1.f / fmaxf(sqrtf(sq), kNormEps) : 1.f);
#pragma unroll
            for (int e = 0; e < EPL; ++e) {
                sK[t * KP + lane + 32 * e] = kv[e] * kn;
                sQ[t * KP + lane + 32 * e] = qv[e] * qn;
            }
        }
        for (int idx = tid; idx < C * DVT; idx += kThreads) {
            const int t = idx / DVT, j = idx % DVT;
            sV[idx] = t < nrow ? to_f32(v[((size_t)(start + c0 + t) * H + h) * DV + col0 + j]) : 0.f;
        }
        if (tid < C) {
            const size_t g = (size_t)(start + c0 + tid) * H + h;
            sb[tid] = tid < nrow ? beta_of(p.beta[g], p.beta_sig, p.neg_eig) : 0.f;
            float d = (tid < nrow && p.decay) ? p.decay[g] : 0.f;  // decay; cumsum below
            if (tid < nrow && p.decay && p.A_log) d = gate_decay(d, p.A_log[h], p.dt_bias ? p.dt_bias[h] : 0.f);
            sG[tid] = d;
        }
        __syncthreads();
        if (tid == 0) {
            float run = 0.f;
            for (int t = 0; t < C; ++t) {
                sGp[t] = run;
                run += sG[t];
                sG[t] = run;
            }
        }
        __syncthreads();
        const float gn = sG[C - 1];   // = G at the last valid row (padded decay is 0)
        // the delta term reads h_{t-1} (R_t = G_{t-1}) or the decayed memory (R_t = G_t)
        const float *sR = p.decayed_read ? sG : sGp;
        if (tid < C) {
            sbg[tid] = sb[tid] * expf(sR[tid]);
            skd[tid] = expf(gn - sG[tid]);
            seg[tid] = expf(sG[tid]);
        }
        // --- L (strictly lower) and Aqk (lower, diagonal included)
        for (int idx = tid; idx < C * C; idx += kThreads) {
            const int t = idx / C, s = idx % C;
            float kk = 0.f, qk = 0.f;
#pragma unroll 8
            for (int i = 0; i < DK; ++i) {
                const float ks = sK[s * KP + i];
                kk = fmaf(sK[t * KP + i], ks, kk);
                qk = fmaf(sQ[t * KP + i], ks, qk);
            }
            sL[t * CP + s] = s < t ? sb[t] * kk * expf(sR[t] - sG[s]) : 0.f;
            sA[t * CP + s] = s <= t ? qk * expf(sG[t] - sG[s]) : 0.f;
        }
        __syncthreads();
        // --- T = (I + L)^{-1}: thread j solves column j by forward substitution
        if (tid < C) {
            const int j = tid;
            for (int t = 0; t < j; ++t) sT[t * CP + j] = 0.f;
            sT[j * CP + j] = 1.f;
            for (int t = j + 1; t < C; ++t) {
                float x = 0.f;
                for (int s = j; s < t; ++s) x = fmaf(-sL[t * CP + s], sT[s * CP + j], x);
                sT[t * CP + j] = x;
            }
        }
        __syncthreads();
        // --- W = T diag(beta exp R) K^ ;  U0 = T diag(beta) V
        for (int idx = tid; idx < C * DK; idx += kThreads) {
            const int t = idx / DK, i = idx % DK;
            float acc = 0.f;
            for (int s = 0; s <= t; ++s) acc = fmaf(sT[t * CP + s] * sbg[s], sK[s * KP + i], acc);
            sW[t * KP + i] = acc;
        }
        float reg[RU];
#pragma unroll
        for (int r = 0; r < RU; ++r) {
            const int idx = tid + r * kThreads;
            float acc = 0.f;
            if (idx < C * DVT) {
                const int t = idx / DVT, j = idx % DVT;
                for (int s = 0; s <= t; ++s) acc = fmaf(sT[t * CP + s] * sb[s], sV[s * DVT + j], acc);
            }
            reg[r] = acc;
        }
        __syncthreads();
#pragma unroll
        for (int r = 0; r < RU; ++r) {
            const int idx = tid + r * kThreads;
            if (idx < C * DVT) sV[idx] = reg[r];
        }
        __syncthreads();
        // --- U = U0 - W S  and  P = Q~ S  (P kept in registers for the output)
        float pq[RU];
#pragma unroll
        for (int r = 0; r < RU; ++r) {
            const int idx = tid + r * kThreads;
            float aw = 0.f, aq = 0.f;
            if (idx < C * DVT) {
                const int t = idx / DVT, j = idx % DVT;
#pragma unroll 8
                for (int i = 0; i < DK; ++i) {
                    const float s_ij = sS[i * DVT + j];
                    aw = fmaf(sW[t * KP + i], s_ij, aw);
                    aq = fmaf(sQ[t * KP + i], s_ij, aq);
                }
                reg[r] = sV[idx] - aw;
            }
            pq[r] = aq;
        }
        __syncthreads();
#pragma unroll
        for (int r = 0; r < RU; ++r) {
            const int idx = tid + r * kThreads;
            if (idx < C * DVT) sV[idx] = reg[r];
        }
        __syncthreads();
        // --- O = diag(exp G) Q~ S + Aqk U   (valid rows only)
#pragma unroll
        for (int r = 0; r < RU; ++r) {
            const int idx = tid + r * kThreads;
            if (idx < C * DVT) {
                const int t = idx / DVT, j = idx % DVT;
                if (t < nrow) {
                    float acc = seg[t] * pq[r];
                    for (int s = 0; s <= t; ++s) acc = fmaf(sA[t * CP + s], sV[s * DVT + j], acc);
                    o[((size_t)(start + c0 + t) * H + h) * DV + col0 + j] = from_f32<Tin>(acc);
                }
            }
        }
        // --- S <- exp(G_n) S + sum_s exp(G_n - G_s) k^_s u_s^T
        const float egn = expf(gn);
        for (int idx = tid; idx < DK * DVT; idx += kThreads) {
            const int i = idx / DVT, j = idx % DVT;
            float acc = egn * sS[idx];
            for (int s = 0; s < C; ++s) acc = fmaf(skd[s] * sK[s * KP + i], sV[s * DVT + j], acc);
            sS[idx] = acc;
        }
        __syncthreads();
    }

    if (p.hT) {
        for (int idx = tid; idx < DK * DVT; idx += kThreads) {
            const int i = p.v_first ? idx % DK : idx / DVT, j = p.v_first ? idx / DK : idx % DVT;
            p.hT[st_at(i, j)] = sS[i * DVT + j];
        }
    }
}

template <typename Tin, int DK, int DVT>
cudaError_t launch_one(const SeqBatch &p, int grid, cudaStream_t s) {
    using Lay = SimtLayout<DK, DVT>;
    // Set on every call: the attribute belongs to the function on the current
    // device, and the call is cheap next to the kernel.
    cudaError_t e = cudaFuncSetAttribute(chunk_simt_kernel<Tin, DK, DVT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)Lay::bytes);
    if (e != cudaSuccess) return e;
    chunk_simt_kernel<Tin, DK, DVT><<<grid, kThreads, Lay::bytes, s>>>(p);
    return cudaGetLastError();
}

template <typename Tin, int DK>
cudaError_t launch_dk(const SeqBatch &p, int dvt, int grid, cudaStream_t s) {
    return dvt == 64 ? launch_one<Tin, DK, 64>(p, grid, s) : launch_one<Tin, DK, 32>(p, grid, s);
}

template <typename Tin>
cudaError_t launch_typed(const SeqBatch &p, int dvt, int grid, cudaStream_t s) {
    switch (p.dk) {
        case 32: return launch_dk<Tin, 32>(p, dvt, grid, s);
        case 64: return launch_dk<Tin, 64>(p, dvt, grid, s);
        case 128: return launch_dk<Tin, 128>(p, dvt, grid, s);
        default: return cudaErrorInvalidValue;
    }
}

int value_tile(int dv) { return dv >= 64 ? 64 : 32; }

}  // namespace

size_t chunk_simt_smem_bytes(int dk, int dv, int /*chunk*/) {
    const int dvt = value_tile(dv);
    switch (dk * 1000 + dvt) {
        case 32032: return SimtLayout<32, 32>::bytes;
        case 32064: return SimtLayout<32, 64>::bytes;
        case 64032: return SimtLayout<64, 32>::bytes;
        case 64064: return SimtLayout<64, 64>::bytes;
        case 128032: return SimtLayout<128, 32>::bytes;
        case 128064: return SimtLayout<128, 64>::bytes;
        default: return 0;
    }
}

cudaError_t launch_chunk_simt(const SeqBatch &p, cudaStream_t s) {
    if (p.chunk < 1 || p.chunk > kCMax) return cudaErrorInvalidValue;
    const int dvt = value_tile(p.dv);
    const long grid = (long)p.nseq * p.H * (p.dv / dvt);
    if (grid <= 0) return cudaSuccess;
    if (grid > 0x7fffffffL) return cudaErrorInvalidConfiguration;
    return p.dtype == DType::BF16 ? launch_typed<__nv_bfloat16>(p, dvt, (int)grid, s)
                                  : launch_typed<float>(p, dvt, (int)grid, s);
}

}  // namespace kda
