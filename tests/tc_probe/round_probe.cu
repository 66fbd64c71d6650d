// Exhaustive check of la::tc::to_tf32 (and of la::tc::to_tf32_operand as the tensor core reads
// it, low 13 bits ignored) against the hardware conversion cvt.rna.tf32.f32 over every fp32 bit
// pattern that is not a NaN: counts the patterns whose results differ and records the smallest.
#include <cstdint>

#include "tc.cuh"

__global__ void round_kernel(unsigned long long *count, unsigned int *first) {
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < (1ull << 32); i += stride) {
        const uint32_t b = (uint32_t)i;
        if ((b & 0x7F800000u) == 0x7F800000u && (b & 0x007FFFFFu) != 0u) continue;  // NaN
        const float x = __uint_as_float(b);
        const uint32_t mine = __float_as_uint(la::tc::to_tf32(x));
        const uint32_t operand = __float_as_uint(la::tc::to_tf32_operand(x)) & 0xFFFFE000u;
        uint32_t ref;
        asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(ref) : "f"(x));
        if (mine != ref || operand != ref) {
            atomicAdd(count, 1ull);
            atomicMin(first, b);
        }
    }
}

// count, first: device pointers (one element each), initialised by the caller.
extern "C" int round_run(unsigned long long *count, unsigned int *first) {
    round_kernel<<<152 * 8, 256>>>(count, first);
    return (int)cudaDeviceSynchronize();
}
