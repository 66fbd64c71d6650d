// GPU unit check of MN-major (transposed) shared-memory operands for tcgen05.mma: B (or A)
// stored as [K][N] (N contiguous) in 128-byte-swizzled atoms, described with explicit
// leading / stride byte offsets. Test-only.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "tc.cuh"

using namespace la::tc;

// mode 1: bf16, A K-major [128][K] smem, B MN-major [K][N]
// mode 2: bf16, A MN-major [K][128] smem, B K-major [N][K]
// mode 4: bf16, A in TMEM (two per column), B MN-major [K][N]
// Bt / At are given row-major as [K][N] / [K][128].
__global__ void __launch_bounds__(128, 1)
probe_mn_kernel(const float *A, const float *B, float *D, int N, int K, int mode, int swap,
                int *err) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    __shared__ uint64_t bar;
    __shared__ uint32_t tmem_base_sh;
    const int M = 128;
    unsigned char *sm = (unsigned char *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int tid = threadIdx.x, warp = tid >> 5;
    const uint32_t es = 2;
    unsigned char *As = sm;
    unsigned char *Bs = sm + M * K * es;
    // A: mode 1 K-major [128][K]; mode 2 MN-major stored as tile [K rows][128 cols]
    if (mode == 1 || mode == 4) {
        for (int i = tid; i < M * K; i += 128) {
            int r = i / K, k = i % K;
            *(__nv_bfloat16 *)(As + sw128_offset(r, k, M, 2)) = __float2bfloat16_rn(A[i]);
        }
    } else if (mode == 2) {
        for (int i = tid; i < K * M; i += 128) {  // A given as [K][128]
            int k = i / M, m = i % M;
            *(__nv_bfloat16 *)(As + sw128_offset(k, m, K, 2)) = __float2bfloat16_rn(A[i]);
        }
    }
    if (mode == 2) {  // B K-major [N][K]
        for (int i = tid; i < N * K; i += 128) {
            int r = i / K, k = i % K;
            *(__nv_bfloat16 *)(Bs + sw128_offset(r, k, N, 2)) = __float2bfloat16_rn(B[i]);
        }
    } else {  // mode 1: B MN-major, given as [K][N]
        for (int i = tid; i < K * N; i += 128) {
            int k = i / N, n = i % N;
            *(__nv_bfloat16 *)(Bs + sw128_offset(k, n, K, 2)) = __float2bfloat16_rn(B[i]);
        }
    }
    if (tid == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&tmem_base_sh, 512);
        tmem_relinquish();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tbase = tmem_base_sh;
    const uint32_t lane = tmem_lane_base(warp);
    if (mode == 4) {  // A row tid -> TMEM lane tid, columns 256.. (packed pairs)
        for (int g = 0; g < K / 32; ++g) {
            float v[16];
            for (int i = 0; i < 16; ++i) {
                const __nv_bfloat162 p = __floats2bfloat162_rn(A[tid * K + g * 32 + 2 * i],
                                                               A[tid * K + g * 32 + 2 * i + 1]);
                v[i] = *reinterpret_cast<const float *>(&p);
            }
            tmem_st16(tmem_addr(tbase, lane, 256 + g * 16), v);
        }
        tmem_wait_st();
    }
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    if (tid == 0) {
        fence_after_sync();
        const uint32_t kstep = 16;
        // MN-major tile [K rows][X cols]: atoms of 128 B along X, each K*128 bytes; 8-row groups
        // along K 1024 bytes apart. swap exchanges the two offsets (to detect a misreading).
        for (uint32_t kk = 0; kk < (uint32_t)K / kstep; ++kk) {
            const uint32_t k0 = kk * kstep;
            if (mode == 4) {
                uint32_t lbo = K * 128, sbo = 1024;
                if (swap) { uint32_t t = lbo; lbo = sbo; sbo = t; }
                const uint64_t bd = sdesc_sw128_mn(smem_u32(Bs) + k0 * 128, lbo, sbo);
                mma_bf16_ts(tbase, tbase + 256 + k0 / 2, bd, idesc(M, N, FMT_BF16, false, true), kk > 0);
            } else if (mode == 1) {
                uint32_t lbo = K * 128, sbo = 1024;
                if (swap) { uint32_t t = lbo; lbo = sbo; sbo = t; }
                const uint32_t per_atom = 64, atom = k0 / per_atom, inner = (k0 % per_atom) * 2;
                const uint64_t ad = sdesc_sw128(smem_u32(As) + atom * M * 128 + inner);
                const uint64_t bd = sdesc_sw128_mn(smem_u32(Bs) + k0 * 128, lbo, sbo);
                mma_bf16_ss(tbase, ad, bd, idesc(M, N, FMT_BF16, false, true), kk > 0);
            } else {
                uint32_t lbo = K * 128, sbo = 1024;
                if (swap) { uint32_t t = lbo; lbo = sbo; sbo = t; }
                const uint32_t per_atom = 64, atom = k0 / per_atom, inner = (k0 % per_atom) * 2;
                const uint64_t ad = sdesc_sw128_mn(smem_u32(As) + k0 * 128, lbo, sbo);
                const uint64_t bd = sdesc_sw128(smem_u32(Bs) + atom * N * 128 + inner);
                mma_bf16_ss(tbase, ad, bd, idesc(M, N, FMT_BF16, true, false), kk > 0);
            }
        }
        mma_commit(&bar);
    }
    __syncwarp();
    const bool ok = mbar_wait(&bar, 0, 1000000000ull);
    if (!ok && (tid & 31) == 0) atomicExch(err, 1);
    fence_after_sync();
    if (ok) {
        for (int g = 0; g < N / 16; ++g) {
            float v[16];
            tmem_ld16(tmem_addr(tbase, lane, g * 16), v);
            tmem_wait_ld();
            for (int i = 0; i < 16; ++i) D[tid * N + g * 16 + i] = v[i];
        }
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, 512);
}

extern "C" int probe_mn_run(const float *A, const float *B, float *D, int N, int K, int mode,
                            int swap, int *err) {
    if (mode != 1 && mode != 2 && mode != 4) return -4;
    const size_t es = 2;
    const size_t smem = (128 + N) * K * es + 1024;
    if (cudaFuncSetAttribute(probe_mn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
        return -1;
    probe_mn_kernel<<<1, 128, smem>>>(A, B, D, N, K, mode, swap, err);
    if (cudaGetLastError() != cudaSuccess) return -2;
    return cudaDeviceSynchronize() == cudaSuccess ? 0 : -3;
}
