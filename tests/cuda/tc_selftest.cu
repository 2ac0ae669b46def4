// tc_selftest.cu -- test-only kernels that pin the encodings the tensor-core prefill
// relies on: the tcgen05 shared-memory / instruction descriptors, the canonical
// 128-byte-swizzle operand layouts (K-major and MN-major), and the claim that a TMA
// load with 128-byte swizzle writes exactly that layout.  Built and run by
// tests/test_gpu_tc_selftest.py; not part of libkda.so.
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../delta_rule_linear_gb300/csrc/tc_ptx.cuh"
#include "../../delta_rule_linear_gb300/csrc/tma_host.cuh"

using namespace kda::ptx;

namespace {

constexpr uint64_t kWaitNs = 1000000000ull;  // 1 s

__device__ uint8_t *align1024(uint8_t *p) {
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

uint32_t tmem_cols_for(int n) {
    uint32_t c = 32;
    while ((int)c < n) c <<= 1;
    return c;
}

// D[128][N] = A[128][K] * B[K][N]; operands staged by plain stores into the canonical
// layout selected by a_mn / b_mn; one CTA of 128 threads.
__global__ void gemm_plain_kernel(const __nv_bfloat16 *A, const __nv_bfloat16 *B, float *D, int N,
                                  int K, int a_mn, int b_mn, uint32_t tcols, int *status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    // a 128-byte-swizzle K-major row is 128 bytes wide even when K < 64
    const int kp = ((K + 63) / 64) * 64;
    uint8_t *sA = smem;
    uint8_t *sB = sA + 128 * kp * 2;
    __shared__ uint64_t bar;
    __shared__ uint32_t tbase;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    for (int idx = tid; idx < 128 * K; idx += blockDim.x) {
        const int r = idx / K, k = idx % K;
        const uint32_t off = a_mn ? mnmajor_sw128_offset(K, r, k) : kmajor_sw128_offset(128, r, k);
        *reinterpret_cast<__nv_bfloat16 *>(sA + off) = A[idx];
    }
    for (int idx = tid; idx < K * N; idx += blockDim.x) {
        const int k = idx / N, n = idx % N;
        const uint32_t off = b_mn ? mnmajor_sw128_offset(K, n, k) : kmajor_sw128_offset(N, n, k);
        *reinterpret_cast<__nv_bfloat16 *>(sB + off) = B[idx];
    }
    fence_proxy_async();
    if (warp == 0) {
        tmem_alloc(&tbase, tcols);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = tbase;
    if (tid == 0) {
        const uint32_t idesc = idesc_bf16_f32(128, N, a_mn != 0, b_mn != 0);
        const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
        for (int ks = 0; ks < K / 16; ++ks) {
            const uint64_t ad = a_mn ? desc_mnmajor_sw128(a0, K, ks) : desc_kmajor_sw128(a0, 128, ks);
            const uint64_t bd = b_mn ? desc_mnmajor_sw128(b0, K, ks) : desc_kmajor_sw128(b0, N, ks);
            mma_bf16_ss(tm, ad, bd, idesc, ks > 0 ? 1u : 0u);
        }
        mma_commit(&bar);
    }
    const bool ok = mbar_wait(&bar, 0, kWaitNs);
    if (!ok && lane == 0) atomicExch(status, 1);
    tc_fence_after();
    if (ok) {
        for (int c0 = 0; c0 < N; c0 += 16) {
            uint32_t r[16];
            tmem_ld16(tm + ((uint32_t)(32 * warp) << 16) + (uint32_t)c0, r);
            tmem_ld_wait();
            for (int j = 0; j < 16; ++j) D[(32 * warp + lane) * N + c0 + j] = __uint_as_float(r[j]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, tcols);
}

// dst[r][c] = element (r, c) read back from a TMA-loaded 128B-swizzled tile, using the
// layout's offset function.  src/dst: [R][C] bf16, C a multiple of 64, R <= 256.
__global__ void tma_roundtrip_kernel(const __grid_constant__ CUtensorMap map, __nv_bfloat16 *dst,
                                     int R, int C, int *status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    __shared__ uint64_t bar;
    const int tid = threadIdx.x;
    if (tid == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0) {
        mbar_expect_tx(&bar, (uint32_t)(R * C * 2));
        for (int cb = 0; cb < C / 64; ++cb) tma_load_2d(smem + cb * R * 128, &map, &bar, cb * 64, 0);
    }
    const bool ok = mbar_wait(&bar, 0, kWaitNs);
    if (!ok) {
        if (tid == 0) atomicExch(status, 1);
        return;
    }
    for (int idx = tid; idx < R * C; idx += blockDim.x) {
        const int r = idx / C, c = idx % C;
        dst[idx] = *reinterpret_cast<const __nv_bfloat16 *>(smem + kmajor_sw128_offset(R, r, c));
    }
}

// D[128][N] = A[128][K] * B[K][N] with both operands TMA-loaded in their natural
// row-major layouts: A as K-major (boxes of 64 K x 128 rows), B as MN-major (boxes of
// 64 N x K rows).  This is how the prefill feeds q/k (contract over d) and k/v
// (contract over tokens).
__global__ void gemm_tma_kernel(const __grid_constant__ CUtensorMap mapA,
                                const __grid_constant__ CUtensorMap mapB, float *D, int N, int K,
                                uint32_t tcols, int *status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    uint8_t *sA = smem;
    uint8_t *sB = sA + 128 * K * 2;
    __shared__ uint64_t bar_ld, bar_mma;
    __shared__ uint32_t tbase;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (warp == 0) {
        tmem_alloc(&tbase, tcols);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&bar_ld, 1);
        mbar_init(&bar_mma, 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = tbase;
    const int nblk = (N + 63) / 64;
    if (tid == 0) {
        mbar_expect_tx(&bar_ld, (uint32_t)(128 * K * 2 + K * nblk * 64 * 2));
        for (int kb = 0; kb < K / 64; ++kb) tma_load_2d(sA + kb * 128 * 128, &mapA, &bar_ld, kb * 64, 0);
        for (int nb = 0; nb < nblk; ++nb) tma_load_2d(sB + nb * K * 128, &mapB, &bar_ld, nb * 64, 0);
    }
    bool ok = mbar_wait(&bar_ld, 0, kWaitNs);
    if (ok && tid == 0) {
        tc_fence_after();
        const uint32_t idesc = idesc_bf16_f32(128, N, false, true);
        const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
        for (int ks = 0; ks < K / 16; ++ks)
            mma_bf16_ss(tm, desc_kmajor_sw128(a0, 128, ks), desc_mnmajor_sw128(b0, K, ks), idesc,
                        ks > 0 ? 1u : 0u);
        mma_commit(&bar_mma);
    }
    if (ok) ok = mbar_wait(&bar_mma, 0, kWaitNs);
    if (!ok && lane == 0) atomicExch(status, 1);
    tc_fence_after();
    if (ok) {
        for (int c0 = 0; c0 < N; c0 += 16) {
            uint32_t r[16];
            tmem_ld16(tm + ((uint32_t)(32 * warp) << 16) + (uint32_t)c0, r);
            tmem_ld_wait();
            for (int j = 0; j < 16; ++j) D[(32 * warp + lane) * N + c0 + j] = __uint_as_float(r[j]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, tcols);
}

// Probe of the TMEM placement of an M=64 result and of MN-major sub-block addressing:
// D = A[64][K] * B[K][N0..N0+N) where B is staged as an MN-major SW128 tile 64 elements
// wide and the descriptor starts n_off elements (a multiple of 8) into each row.
// Every one of the 128 TMEM lanes x N columns is copied to D[128][N], so the host can
// see which lanes hold the 64 result rows.
__global__ void gemm_m64_probe_kernel(const __nv_bfloat16 *A, const __nv_bfloat16 *B, float *D,
                                      int N, int K, int n_off, uint32_t tcols, int *status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    const int kp = ((K + 63) / 64) * 64;
    uint8_t *sA = smem;                 // K-major, 64 rows
    uint8_t *sB = sA + 64 * kp * 2;     // MN-major, one 64-wide block
    __shared__ uint64_t bar;
    __shared__ uint32_t tbase;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    for (int idx = tid; idx < 64 * K; idx += blockDim.x) {
        const int r = idx / K, k = idx % K;
        *reinterpret_cast<__nv_bfloat16 *>(sA + kmajor_sw128_offset(64, r, k)) = A[idx];
    }
    for (int idx = tid; idx < K * 64; idx += blockDim.x) {
        const int k = idx / 64, n = idx % 64;
        *reinterpret_cast<__nv_bfloat16 *>(sB + mnmajor_sw128_offset(K, n, k)) = B[idx];
    }
    fence_proxy_async();
    if (warp == 0) {
        tmem_alloc(&tbase, tcols);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = tbase;
    // clear every lane of the N columns first so that untouched lanes read as zero
    {
        uint32_t z[16];
        for (int j = 0; j < 16; ++j) z[j] = 0u;
        for (int c0 = 0; c0 < N; c0 += 16) {
            asm volatile(
                "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
                "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
                    tm + ((uint32_t)(32 * warp) << 16) + (uint32_t)c0),
                "r"(z[0]), "r"(z[1]), "r"(z[2]), "r"(z[3]), "r"(z[4]), "r"(z[5]), "r"(z[6]),
                "r"(z[7]), "r"(z[8]), "r"(z[9]), "r"(z[10]), "r"(z[11]), "r"(z[12]), "r"(z[13]),
                "r"(z[14]), "r"(z[15])
                : "memory");
        }
        tmem_st_wait();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {
        const uint32_t idesc = idesc_bf16_f32(64, N, false, true);
        const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB) + (uint32_t)n_off * 2u;
        for (int ks = 0; ks < K / 16; ++ks)
            mma_bf16_ss(tm, desc_kmajor_sw128(a0, 64, ks), desc_mnmajor_sw128(b0, K, ks), idesc,
                        ks > 0 ? 1u : 0u);
        mma_commit(&bar);
    }
    const bool ok = mbar_wait(&bar, 0, kWaitNs);
    if (!ok && lane == 0) atomicExch(status, 1);
    tc_fence_after();
    if (ok) {
        for (int c0 = 0; c0 < N; c0 += 16) {
            uint32_t r[16];
            tmem_ld16(tm + ((uint32_t)(32 * warp) << 16) + (uint32_t)c0, r);
            tmem_ld_wait();
            for (int j = 0; j < 16; ++j) D[(32 * warp + lane) * N + c0 + j] = __uint_as_float(r[j]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, tcols);
}

bool map2d(CUtensorMap *m, const void *base, int rows, int cols, int box_rows) {
    const uint64_t dims[2] = {(uint64_t)cols, (uint64_t)rows};
    const uint64_t strides[1] = {(uint64_t)cols * 2};
    const uint32_t box[2] = {64u, (uint32_t)box_rows};
    return kda::make_tensor_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box,
                                true);
}

int finish(int *status_dev) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return 1000 + (int)e;
    int st = 0;
    cudaMemcpy(&st, status_dev, sizeof(int), cudaMemcpyDeviceToHost);
    cudaFree(status_dev);
    return st ? 2 : 0;
}

}  // namespace

extern "C" int selftest_gemm_plain(const void *A, const void *B, float *D, int N, int K, int a_mn,
                                   int b_mn) {
    if (K % 16 || K > 256 || N % 16 || N > 256 || N < 16) return -1;
    if (b_mn && N % 64 && N > 64) return -1;
    int *st;
    cudaMalloc(&st, sizeof(int));
    cudaMemset(st, 0, sizeof(int));
    const int kp = ((K + 63) / 64) * 64;
    const size_t bbytes = b_mn ? (size_t)K * (((N + 63) / 64) * 64) * 2 : (size_t)N * kp * 2;
    const size_t smem = 1024 + (size_t)128 * kp * 2 + bbytes;
    cudaFuncSetAttribute(gemm_plain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    gemm_plain_kernel<<<1, 128, smem>>>(static_cast<const __nv_bfloat16 *>(A),
                                        static_cast<const __nv_bfloat16 *>(B), D, N, K, a_mn, b_mn,
                                        tmem_cols_for(N), st);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return 1000 + (int)e;
    return finish(st);
}

extern "C" int selftest_tma_roundtrip(const void *src, void *dst, int R, int C) {
    if (C % 64 || R > 256 || R < 1) return -1;
    CUtensorMap m;
    if (!map2d(&m, src, R, C, R)) return -2;
    int *st;
    cudaMalloc(&st, sizeof(int));
    cudaMemset(st, 0, sizeof(int));
    const size_t smem = 1024 + (size_t)R * C * 2;
    cudaFuncSetAttribute(tma_roundtrip_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    tma_roundtrip_kernel<<<1, 256, smem>>>(m, static_cast<__nv_bfloat16 *>(dst), R, C, st);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return 1000 + (int)e;
    return finish(st);
}

extern "C" int selftest_gemm_tma(const void *A, const void *B, float *D, int N, int K) {
    if (K % 64 || K > 256 || N % 64 || N > 256) return -1;
    CUtensorMap ma, mb;
    if (!map2d(&ma, A, 128, K, 128)) return -2;
    if (!map2d(&mb, B, K, N, K)) return -2;
    int *st;
    cudaMalloc(&st, sizeof(int));
    cudaMemset(st, 0, sizeof(int));
    const size_t smem = 1024 + (size_t)128 * K * 2 + (size_t)K * N * 2;
    cudaFuncSetAttribute(gemm_tma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    gemm_tma_kernel<<<1, 128, smem>>>(ma, mb, D, N, K, tmem_cols_for(N), st);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return 1000 + (int)e;
    return finish(st);
}

extern "C" int selftest_gemm_m64_probe(const void *A, const void *B, float *D, int N, int K,
                                       int n_off) {
    if (K % 16 || K > 256 || N % 16 || N < 16 || n_off % 8 || n_off + N > 64) return -1;
    int *st;
    cudaMalloc(&st, sizeof(int));
    cudaMemset(st, 0, sizeof(int));
    const int kp = ((K + 63) / 64) * 64;
    const size_t smem = 1024 + (size_t)64 * kp * 2 + (size_t)K * 64 * 2;
    cudaFuncSetAttribute(gemm_m64_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)smem);
    gemm_m64_probe_kernel<<<1, 128, smem>>>(static_cast<const __nv_bfloat16 *>(A),
                                            static_cast<const __nv_bfloat16 *>(B), D, N, K, n_off,
                                            tmem_cols_for(N), st);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return 1000 + (int)e;
    return finish(st);
}
