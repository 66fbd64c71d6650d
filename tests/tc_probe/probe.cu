// GPU unit check of the library's tcgen05 helpers (tc.cuh): one CTA computes
// D[128][N] = A[128][K] * B[N][K]^T with operands staged in the 128-byte-swizzled K-major
// shared-memory layout (or A in tensor memory), read back through tcgen05.ld. Test-only.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "tc.cuh"

using namespace la::tc;

// mode 0: bf16 A,B from smem; 1: tf32 A,B from smem; 2: tf32 A from TMEM, B from smem;
// 3: bf16 A from TMEM (two elements per 32-bit column, the lower k in the low half), B bf16
// from smem
__global__ void __launch_bounds__(128, 1)
probe_kernel(const float *A, const float *B, float *D, int N, int K, int mode, int *err) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    __shared__ uint64_t bar;
    __shared__ uint32_t tmem_base_sh;
    const int M = 128;
    unsigned char *sm = (unsigned char *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int tid = threadIdx.x, warp = tid >> 5;
    const bool bf = (mode == 0 || mode == 3);
    const uint32_t es = bf ? 2 : 4;
    unsigned char *As = sm;
    unsigned char *Bs = sm + M * K * es;
    for (int i = tid; i < M * K; i += 128) {
        int r = i / K, k = i % K;
        if (bf) *(__nv_bfloat16 *)(As + sw128_offset(r, k, M, 2)) = __float2bfloat16_rn(A[i]);
        else *(float *)(As + sw128_offset(r, k, M, 4)) = to_tf32(A[i]);
    }
    for (int i = tid; i < N * K; i += 128) {
        int r = i / K, k = i % K;
        if (bf) *(__nv_bfloat16 *)(Bs + sw128_offset(r, k, N, 2)) = __float2bfloat16_rn(B[i]);
        else *(float *)(Bs + sw128_offset(r, k, N, 4)) = to_tf32(B[i]);
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
    if (mode == 2) {
        for (int g = 0; g < K / 16; ++g) {
            float v[16];
            for (int i = 0; i < 16; ++i) v[i] = to_tf32(A[tid * K + g * 16 + i]);
            tmem_st16(tmem_addr(tbase, lane, 256 + g * 16), v);
        }
        tmem_wait_st();
    } else if (mode == 3) {
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
        const uint32_t kstep = bf ? 16 : 8;
        const uint32_t per_atom = 128 / es;
        const uint32_t id = idesc(M, N, bf ? FMT_BF16 : FMT_TF32);
        for (uint32_t kk = 0; kk < (uint32_t)K / kstep; ++kk) {
            const uint32_t k0 = kk * kstep;
            const uint32_t atom = k0 / per_atom, inner = (k0 % per_atom) * es;
            const uint64_t bd = sdesc_sw128(smem_u32(Bs) + atom * N * 128 + inner);
            if (mode == 2) {
                mma_tf32_ts(tbase, tbase + 256 + k0, bd, id, kk > 0);
            } else if (mode == 3) {
                mma_bf16_ts(tbase, tbase + 256 + k0 / 2, bd, id, kk > 0);
            } else {
                const uint64_t ad = sdesc_sw128(smem_u32(As) + atom * M * 128 + inner);
                if (bf) mma_bf16_ss(tbase, ad, bd, id, kk > 0);
                else mma_tf32_ss(tbase, ad, bd, id, kk > 0);
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

extern "C" int probe_run(const float *A, const float *B, float *D, int N, int K, int mode,
                         int *err) {
    const size_t es = mode == 0 ? 2 : 4;
    const size_t smem = (128 + N) * K * es + 1024;
    if (cudaFuncSetAttribute(probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
        return -1;
    probe_kernel<<<1, 128, smem>>>(A, B, D, N, K, mode, err);
    if (cudaGetLastError() != cudaSuccess) return -2;
    return cudaDeviceSynchronize() == cudaSuccess ? 0 : -3;
}
