// Blackwell (sm_100 family, here sm_103a) tensor-core helpers: tcgen05 MMA, tensor memory
// (TMEM), shared-memory matrix descriptors and bounded mbarrier waits, as inline PTX.
//
// Layout conventions used by every kernel of this library:
//  - MMA computes D[M][N] (+)= A[M][K] * B[N][K]^T with both operands K-major.
//  - Shared-memory operands use the 128-byte swizzle: a tile of R rows is stored as
//    K-atoms of 128 bytes per row (64 bf16 or 32 tf32 elements); atom a occupies R*128
//    bytes at offset a*R*128; inside an atom row r sits at r*128 and its 16-byte chunk j is
//    stored at chunk position j ^ (r % 8). Tile bases are 1024-byte aligned.
//  - TMEM: D of an M=128 MMA puts row m in lane m and column n in column (base + n).
//    A tf32 A-operand in TMEM holds row m in lane m and element k in column (base + k).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace la {
namespace tc {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- swizzled tile addressing
// Byte offset of element (row r, element k) of a K-major SW128 tile with R rows and
// elements of `esize` bytes.
__host__ __device__ __forceinline__ uint32_t sw128_offset(uint32_t r, uint32_t k, uint32_t R,
                                                          uint32_t esize) {
    const uint32_t per_atom = 128u / esize;  // elements per 128-byte atom row
    const uint32_t atom = k / per_atom;
    const uint32_t byte = (k % per_atom) * esize;  // byte within the 128-byte row
    const uint32_t chunk = (byte >> 4) ^ (r & 7u);
    return atom * R * 128u + r * 128u + (chunk << 4) + (byte & 15u);
}

// ---------------------------------------------------------------- descriptors
// Shared-memory matrix descriptor, K-major, 128-byte swizzle: start address, leading byte
// offset (unused by this layout, encoded 1), stride byte offset 1024 (8 rows x 128 B),
// descriptor version 1 (bits 46-48 = 0b001), swizzle mode 2 (bits 61-63).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(1u) << 16;
    d |= static_cast<uint64_t>(1024u >> 4) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    d |= static_cast<uint64_t>(2u) << 61;
    return d;
}

// Same with explicit leading / stride byte offsets. For an MN-major operand in the 128-byte
// swizzle (128-byte atoms along M/N, 8 rows of K per atom), `lbo` is the byte distance between
// atoms along M/N and `sbo` the distance between 8-row groups along K.
__device__ __forceinline__ uint64_t sdesc_sw128_mn(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo & 0x3FFFFu) >> 4) << 16;
    d |= static_cast<uint64_t>((sbo & 0x3FFFFu) >> 4) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    d |= static_cast<uint64_t>(2u) << 61;
    return d;
}

enum : uint32_t { FMT_BF16 = 1, FMT_TF32 = 2 };

// Instruction descriptor for kind::f16 / kind::tf32 with fp32 accumulation; A and B K-major
// unless a_mn / b_mn select the MN-major (transposed) form.
__host__ __device__ constexpr uint32_t idesc(uint32_t M, uint32_t N, uint32_t fmt,
                                             bool a_mn = false, bool b_mn = false) {
    return (1u << 4)                     // D format: f32
           | (fmt << 7)                  // A format
           | (fmt << 10)                 // B format
           | ((a_mn ? 1u : 0u) << 15)    // A major-ness
           | ((b_mn ? 1u : 0u) << 16)    // B major-ness
           | ((N >> 3) << 17)            // N / 8
           | ((M >> 4) << 24);           // M / 16
}

// ---------------------------------------------------------------- MMA
// A and B from shared memory, kind::f16 (bf16 operands).
__device__ __forceinline__ void mma_bf16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t id, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(id), "r"(accumulate));
}
// A and B from shared memory, kind::tf32.
__device__ __forceinline__ void mma_tf32_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t id, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(id), "r"(accumulate));
}
// A from tensor memory (two bf16 per 32-bit column, the lower k in the low half), B from
// shared memory, kind::f16 with bf16 operands.
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t id, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(id), "r"(accumulate));
}
// A from tensor memory, B from shared memory, kind::tf32.
__device__ __forceinline__ void mma_tf32_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t id, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(id), "r"(accumulate));
}
// Arrive once on `bar` when every MMA issued so far by this thread has completed.
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// ---------------------------------------------------------------- fences
__device__ __forceinline__ void fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Make this thread's generic-proxy shared-memory writes visible to the tensor core.
__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- TMEM allocation (one warp)
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

// ---------------------------------------------------------------- TMEM <-> registers
// Lane quadrant of the calling warp: warp w may only touch lanes 32*(w%4) .. 32*(w%4)+31.
__device__ __forceinline__ uint32_t tmem_lane_base(uint32_t warp) { return (warp & 3u) * 32u; }
__device__ __forceinline__ uint32_t tmem_addr(uint32_t base, uint32_t lane, uint32_t col) {
    return base + (lane << 16) + col;
}

// 32 lanes x 16 consecutive 32-bit columns: thread i gets lane (quadrant + i), columns col..col+15.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float *v) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float *v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15]))
        : "memory");
}
// 32 lanes x 8 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float *v) {
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const float *v) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(
                     taddr),
                 "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
                 "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
                 "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7]))
                 : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- mbarriers (bounded waits)
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// The same test with a suspend-time hint: a thread whose phase is not complete sleeps until it
// completes or `hint_ns` nanoseconds have passed, instead of returning at once (waiting threads
// then take no issue slots from the others).
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}
// Waits for phase `parity` of `bar` to complete, giving up after `limit_ns` nanoseconds.
// Returns false on timeout (the caller records an error and unwinds). With `sleep_ns` > 0 the
// waiting thread sleeps between tests (for threads that wait long while others work: the
// GEMM's epilogue warps during a tile's main loop); without, it polls (the recurrence's waits,
// which are short and on its critical path: there the sleep form was slower).
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint64_t limit_ns,
                                          uint32_t sleep_ns = 0) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (sleep_ns ? mbar_try_wait_sleep(bar, parity, sleep_ns) : mbar_try_wait(bar, parity))
            return true;
        if ((i & (sleep_ns ? 3u : 63u)) == 0 && globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// Arrival that also expects `bytes` of asynchronous copies (TMA) to complete on this phase.
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
// 2-D tiled TMA load of the box at (x = inner coordinate, y) into shared memory, completing
// `bar`'s transaction count. `map` is a CUtensorMap in parameter, constant or global memory.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *map, int x, int y,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// 2^x on the special-function unit (ex2.approx.ftz: relative error below 2^-22; +inf above
// the float range, 0 below its normal range).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// One lane of a converged warp (elect.sync): MMAs are issued by the elected lane of a fully
// converged warp so that their descriptor operands stay warp-uniform.
__device__ __forceinline__ bool elect_one() {
    uint32_t pred = 0;
    asm volatile(
        "{\n\t.reg .pred P;\n\telect.sync _|P, 0xffffffff;\n\tselp.u32 %0, 1, 0, P;\n\t}\n"
        : "=r"(pred));
    return pred != 0;
}

// fp32 -> tf32 (kept in a 32-bit container), rounded to nearest with ties away from zero: tf32
// keeps the sign, the 8 exponent bits and the top 10 of the 23 fraction bits, so adding half a
// unit of the 11th kept bit (0x1000) to the sign-magnitude pattern and clearing the 13 dropped
// bits rounds the magnitude (a carry out of the fraction moves to the next binade, and past the
// largest finite value to infinity). Two integer operations: with them in place of the
// conversion instruction the tensor-core recurrence runs 5-6% faster on sm_103a. Not for NaN
// inputs, which do not reach it.
__device__ __forceinline__ float to_tf32(float x) {
    return __uint_as_float((__float_as_uint(x) + 0x1000u) & 0xFFFFE000u);
}
// The same rounding for a value that only ever reaches the tensor core as a tf32 MMA operand:
// the MMA reads the top 19 bits of the 32-bit pattern and ignores the 13 low ones (a GPU test
// checks this for operands in shared and in tensor memory), so the add alone rounds and the
// clearing step is left out. Anything else that reads the value sees it unrounded, low bits
// and all.
__device__ __forceinline__ float to_tf32_operand(float x) {
    return __uint_as_float(__float_as_uint(x) + 0x1000u);
}

}  // namespace tc
}  // namespace la
