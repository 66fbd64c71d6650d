// Chunked gated delta rule on the 5th-generation tensor cores (tcgen05 + TMEM), bf16
// activations, head dim 128, GDN (scalar gate) and KDA (per-channel gate).
//
// Pages: "glm5next_kda/prefill.rs", Glm5NextKdaLayer::prefill_with_pad_fill — chunk_prepare
// (cumulative gate, WY factors per chunk) then chunk_scan (one block per head walking the
// chunks, state updated in place); "split_prefill.rs", prefill_gdn_full_batched and
// prefill_gdn_full_batched_fla_varlen (streams through a device array of h-state pointers,
// cu_seqlens). Here prepare and scan are fused in one persistent block per SM that claims
// (stream, v-head) units, longest stream first.
//
// Per chunk of C = 64 tokens (t, i: tokens; c: k-channel; d: v-channel; S = H^T [d][c], fp32,
// resident in TMEM for the whole unit; gc: inclusive cumulative log-gate, pad rows g = 0):
//   D1 = [K ; Q] K^T                     tensor core (GDN: bf16 inputs as loaded;
//                                        KDA: tf32, with the decays split per factor:
//                                        [K e^gc ; Q e^gc] (K e^{-gc})^T)
//   A  = strictly-lower(beta_t e^{gc_t-gc_i} D1_KK),  P = lower(e^{gc_t-gc_i} D1_QK)
//   T  = (I + A)^{-1}                    CUDA cores, forward substitution per column
//   D2 = S [K e^gc ; Q e^gc]^T           tensor core (KDA: tf32, S read from TMEM; GDN: S as
//                                        two bf16 terms in TMEM against the raw bf16 tile,
//                                        the decays applied to the result)
//   R^T = beta (V^T - D2[:, :64])        CUDA cores -> TMEM
//   U'^T = R^T T^T                       tensor core
//   O^T = D2[:, 64:] + U'^T P^T          tensor core (U'^T P^T), summed in the epilogue
//   S  <- S diag(e^{gc_L}) + U'^T (K e^{gc_L - gc})     tensor core, accumulating into S
//                                        (GDN: Ud = U' e^{gc_L - gc} as two bf16 terms
//                                        against the raw K rows)
//   o  = scale O                          epilogue
// which is the token recurrence S_t = S_{t-1} diag(a_t)(I - b_t k_t k_t^T) + b_t v_t k_t^T,
// o_t = scale S_t q_t, unrolled over the chunk. Every exponent is <= 0 except the two split
// decays of D1 (GDN: at the mid row, KDA: e^{-gc}), whose range is checked per chunk; a chunk
// whose decay exceeds e^80 (GDN: in either half, KDA: in some channel over the whole chunk)
// takes an exact pairwise-exponent path for D1 on the CUDA cores.
//
// Fused front end (FRONT): the block also computes its q, k and v tiles, chunk by chunk, from
// the pre-conv rows x — causal depthwise conv over the carried conv state, SiLU, and the L2
// norm of each q and k row ("glm5next_kda/prefill.rs", conv_prefill and l2 launches) — so the
// conv output never reaches HBM. The next chunk's raw rows (64 + 3 halo) are copied into the
// buffer of the tf32 K|Q tile once D2 has read it, and turned into the bf16 tiles while the
// tensor core runs the state update. Arithmetic and reduction order are those of
// the conv and L2 kernels, so both paths give identical bits. The conv state of a stream is
// advanced by the blocks that read it: v channels by their unit, q|k channels by the last of
// the units sharing that k-head to read the old state (a per-(stream, k-head) count).
//
// Precision: operands that are raw bf16 inputs use kind::f16; operands derived from fp32
// values (state, T, U', decayed keys) use kind::tf32 with round-to-nearest conversion, except
// the two intermediate products of the block substitution (U'0 and Z, inside U' = R T^T),
// which the next MMA reads from TMEM without that rounding step, and GDN's state and Ud, which
// enter kind::f16 MMAs as two bf16 terms each (within 2^-18 of the fp32 value);
// accumulation is fp32. Rows at or past a stream's end are removed by selects.
#include <cuda.h>

#include <mutex>

#include "chunk_tiles.cuh"
#include "common.cuh"
#include "launch.h"
#include "tc.cuh"

namespace la {

namespace {

using namespace tiles;

constexpr int TC_C = 64;         // chunk
constexpr int TC_D = 128;        // dk = dv
constexpr int TC_THREADS = 512;  // 16 warps: warp w owns TMEM lanes 32*(w%4).. and column quarter w/4
constexpr int NQ = TC_THREADS / 128;  // column parts per TMEM lane
constexpr uint64_t WAIT_NS = 2000000000ull;

// TMEM columns. D1 (K K^T | Q K^T) and D6 (U'0^T | Z^T of the block substitution) share
// columns: D1 is consumed before D6 is produced. U'1^T lands in the P U' accumulator columns
// before MMA4 overwrites them. V^T (identity MMA, with D2) lands in the U'd^T columns (KDA) or
// in D1's (GDN, D1 consumed by then); GDN's D2 operand S_hi | S_lo (bf16, two per column) sits
// in the R^T | U'd^T columns until D2 has read it, and its state-update operand Ud_hi | Ud_lo
// in the U'd^T columns.
constexpr uint32_t COL_S = 0, COL_D2 = 128, COL_RU = 256, COL_RUD = 320, COL_D1 = 384,
                   COL_D6 = 384, COL_D4 = 448, COL_SHI = COL_RU, COL_SLO = COL_RUD;
constexpr uint32_t TMEM_COLS = 512;

// shared memory layout (bytes from a 1024-aligned base)
constexpr uint32_t SM_KQ = 0;                    // bf16 SW128 [128 rows: K | Q][128]
constexpr uint32_t SM_V = SM_KQ + 32768;         // bf16 SW128 [64][128]
constexpr uint32_t SM_KQG = SM_V + 16384;        // tf32 SW128 [128 rows: K | Q][128], KDA's decayed tile
constexpr uint32_t SM_KDT = SM_KQG + 65536;      // tf32 SW128 [128 c][64 t]: Kdec^T (KDA)
constexpr uint32_t SM_KQ1 = SM_KDT;              // GDN: the K|Q tile of odd chunks (bf16, as SM_KQ)
constexpr uint32_t SM_P = SM_KDT + 32768;        // tf32 SW128 [64 t][64 i]
constexpr uint32_t SM_T00 = SM_P + 16384;        // tf32 SW128 [32 t][32 i]  (I + A00)^{-1}
constexpr uint32_t SM_T11 = SM_T00 + 4096;       // tf32 SW128 [32 t][32 i]  (I + A11)^{-1}
constexpr uint32_t SM_NA10 = SM_T11 + 4096;      // tf32 SW128 [32 t][32 i]  -A[32 + t][i]
constexpr uint32_t SM_ID = SM_NA10 + 8192;       // bf16 SW128 [64][64] identity (1024-aligned)
constexpr uint32_t AT_LD = 68;                   // 64 x AT_LD fp32: the space of the output tile
constexpr uint32_t SM_AT = SM_ID + 8192;         // bf16 O tile [64 t][O_LD]
constexpr uint32_t O_LD = 136;                   // padded row (bf16) of the output staging tile
constexpr uint32_t SM_SMALL = SM_AT + 64 * AT_LD * 4;
// small region (floats)
constexpr uint32_t SF_GC = 0, SF_GC2 = 64, SF_BETA = 128, SF_EG = 192, SF_EGL = 256,
                   SF_GL = 320, SF_EL = 448, SF_CARRY = 704 /* [NQ][128] */,
                   SF_WARP = 704 + 128 * NQ, SF_RF = SF_WARP + 8, SF_CF = SF_RF + 64,
                   SF_END = SF_CF + 64;
constexpr uint32_t SM_BARS = SM_SMALL + SF_END * 4;  // mbarriers, flags, tmem base (128 B)
// fused front end: conv taps (fp32 [4 taps][3 x 128 channels], leading taps zero when
// kernel < 4) and bias of the unit's q | k | v channels; the raw rows share the tf32 K|Q buffer
constexpr uint32_t SM_CW = SM_BARS + 128;
constexpr uint32_t SM_CB = SM_CW + 3 * TC_D * 16;
constexpr uint32_t SM_RAW = SM_KQG;             // bf16 [67 rows][384 channels]
constexpr int RAW_ROWS = TC_C + 3;              // chunk + halo of the longest conv (4 taps)
constexpr uint32_t RAW_LD = 3 * TC_D * 2;       // bytes per raw row
static_assert(RAW_ROWS * RAW_LD <= 65536, "raw rows fit the K|Q staging buffer");
// the two 32 x 32 diagonal blocks of A, transposed (fp32 [2][32 i][AD_LD]), the triangular
// solves' input: apart from the output tile, whose previous chunk's copy is still being stored
constexpr uint32_t AD_LD = 36;
constexpr uint32_t SM_AD = SM_CB + 3 * TC_D * 4;
constexpr uint32_t SM_BYTES = SM_AD + 2 * 32 * AD_LD * 4;
constexpr size_t TC_SMEM = SM_BYTES + 1024;                // alignment slack
static_assert(TC_SMEM <= 227 * 1024, "the block's shared memory fits an SM");
static_assert(TC_C * O_LD * 2 <= TC_C * AT_LD * 4, "the output tile fits its space");
constexpr float LOG2E = 1.4426950408889634f;

struct TcParams {
    RecArgs a;
    const int32_t *perm;  // streams sorted by decreasing length
    int *counter;         // unit claim counter (zeroed by the order kernel)
    int *conv_readers;    // fused front end: [B][Hk] readers of the old conv state so far
    int num_units;
    // Plain recurrence calls: the K, Q and V tiles arrive by TMA, boxes of 64 rows x 64
    // channels of [tokens][heads x 128] (rows past the last token read as zero); otherwise
    // (fused front end, segmented scan) by 16-byte async copies.
    int tma;
    CUtensorMap map_k, map_q, map_v;
};

// Issue the K, Q (k-head kh) and V (v-head j) rows of one chunk as 16-byte async copies into
// the swizzled tiles; rows >= n are zero-filled (their source is never read).
__device__ __forceinline__ void load_kq(const RecArgs &a, unsigned char *sm, int tok0, int n,
                                        int kh, int tid, uint32_t kqo = SM_KQ) {
    const __nv_bfloat16 *kp = reinterpret_cast<const __nv_bfloat16 *>(a.k) + (int64_t)kh * TC_D;
    const __nv_bfloat16 *qp = reinterpret_cast<const __nv_bfloat16 *>(a.q) + (int64_t)kh * TC_D;
    const uint32_t base = tc::smem_u32(sm + kqo);
#pragma unroll
    for (int m = 0; m < 2048 / TC_THREADS; ++m) {
        const int idx = tid + TC_THREADS * m;  // 0..2047
        const int which = idx >> 10, rem = idx & 1023;
        const int row = rem >> 4, ch = rem & 15;
        const bool valid = row < n;
        const int srow = tok0 + (valid ? row : 0);
        const __nv_bfloat16 *src =
            (which ? qp : kp) + (int64_t)srow * (which ? a.q_stride : a.k_stride) + ch * 8;
        cp_async16(base + tc::sw128_offset(which * 64 + row, ch * 8, 128, 2), src, valid);
    }
}
__device__ __forceinline__ void load_v(const RecArgs &a, unsigned char *sm, int tok0, int n,
                                       int j, int tid, bool alt) {
    const __nv_bfloat16 *vp =
        reinterpret_cast<const __nv_bfloat16 *>(alt ? a.v_alt : a.v) + (int64_t)j * TC_D;
    const int64_t vs = alt ? 0 : a.v_stride;
    const uint32_t base = tc::smem_u32(sm + SM_V);
#pragma unroll
    for (int m = 0; m < 1024 / TC_THREADS; ++m) {
        const int idx = tid + TC_THREADS * m;  // 0..1023
        const int row = idx >> 4, ch = idx & 15;
        const bool valid = row < n;
        const int srow = tok0 + (valid ? row : 0);
        cp_async16(base + tc::sw128_offset(row, ch * 8, 64, 2),
                   vp + (int64_t)srow * vs + ch * 8, valid);
    }
}

// ---- fused front end
// First channel of section sec (0 q, 1 k, 2 v) of a unit within a packed x row.
__device__ __forceinline__ int front_channel(const RecArgs &a, int sec, int kh, int j) {
    return sec == 0 ? kh * TC_D : sec == 1 ? (a.Hk + kh) * TC_D : (2 * a.Hk + j) * TC_D;
}

// Conv taps and bias of the unit's 384 channels -> shared memory (fp32, tap-major, taps
// right-aligned: tap m of a kernel-K conv sits at row m + 4 - K).
__device__ __forceinline__ void load_conv_weights(const RecArgs &a, unsigned char *sm, int kh,
                                                  int j, int tid) {
    const __nv_bfloat16 *w = reinterpret_cast<const __nv_bfloat16 *>(a.conv_w);
    const __nv_bfloat16 *b = reinterpret_cast<const __nv_bfloat16 *>(a.conv_bias);
    const int K = a.conv_k;
    float *cw = reinterpret_cast<float *>(sm + SM_CW);
    for (int idx = tid; idx < 3 * TC_D; idx += TC_THREADS) {
        const int ch = front_channel(a, idx / TC_D, kh, j) + idx % TC_D;
#pragma unroll
        for (int m = 0; m < 4; ++m)
            cw[m * 3 * TC_D + idx] = m >= 4 - K ? __bfloat162float(w[(int64_t)ch * K + m - (4 - K)]) : 0.f;
        reinterpret_cast<float *>(sm + SM_CB)[idx] = b ? __bfloat162float(b[ch]) : 0.f;
    }
}

// Raw rows of the chunk starting at stream row rel0: raw row rho holds stream row
// rel0 - 3 + rho of [conv state ; x] (rows before the stream come from the carried state,
// rows past its end and before the state are zero-filled), q | k | v channels of the unit.
__device__ __forceinline__ void load_raw(const RecArgs &a, unsigned char *sm,
                                         const __nv_bfloat16 *state, int t0, int len, int rel0,
                                         int kh, int j, int tid) {
    const __nv_bfloat16 *x = reinterpret_cast<const __nv_bfloat16 *>(a.x);
    const int64_t cd = (int64_t)(2 * a.Hk + a.Hv) * TC_D;
    const int K1 = a.conv_k - 1;
    // thread t < 480 copies 16-byte piece t % 48 (16 per section) of raw rows t / 48 + 10 m
    if (tid >= 480) return;
    const int cc = tid % 48, rho0 = tid / 48;
    const int ch = front_channel(a, cc >> 4, kh, j) + (cc & 15) * 8;
    const uint32_t dst = tc::smem_u32(sm + SM_RAW) + rho0 * RAW_LD + cc * 16;
    const int64_t xs = a.x_stride;
#pragma unroll
    for (int m = 0; m < 7; ++m) {
        const int rho = rho0 + 10 * m;
        if (rho < RAW_ROWS) {
            const int r = rel0 - 3 + rho;
            const __nv_bfloat16 *src = x;
            bool valid;
            if (r >= 0) {
                valid = r < len;
                if (valid) src = x + (int64_t)(t0 + r) * xs + ch;
            } else {
                valid = state != nullptr && K1 + r >= 0;
                if (valid) src = state + (int64_t)(K1 + r) * cd + ch;
            }
            cp_async16(dst + 10 * m * RAW_LD, src, valid);
        }
    }
}

// bf16 pair (low half = first element) widened to an fp32 pair
__device__ __forceinline__ uint64_t bf2_to_f2(uint32_t w) {
    return pk2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// q, k, v tiles of a chunk from its raw rows: out[t][c] = SiLU(b[c] + sum_m w[c][m] xh[t-3+m][c])
// rounded to bf16, then q and k rows scaled by 1/sqrt(sum of squares + eps) and rounded again.
// Warp w takes rows 4w..4w+3, lane l the channel quad 4l..4l+3 of each section: a section row
// is one warp, reduced with xor-shuffles in the order of the L2 kernel. Rows >= n get pad (q, k)
// or zero (v). K4: a 4-tap conv (no leading zero taps to skip).
template <bool K4>
__device__ __forceinline__ void conv_tile(const RecArgs &a, unsigned char *sm, int n, float pad,
                                          int warp, int lane, uint32_t kqo) {
    const float *cw = reinterpret_cast<const float *>(sm + SM_CW);
    const float *cb = reinterpret_cast<const float *>(sm + SM_CB);
    const int m0 = K4 ? 0 : 4 - a.conv_k;  // first tap that is not zero
    const int tau0 = 4 * warp;
    const __nv_bfloat162 pf2 = __float2bfloat162_rn(pad);
    const uint32_t pfw = *reinterpret_cast<const uint32_t *>(&pf2);
#pragma unroll 1
    for (int sec = 0; sec < 3; ++sec) {
        const int c0 = sec * TC_D + 4 * lane;
        uint64_t w01[4], w23[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const float4 wv = *reinterpret_cast<const float4 *>(cw + m * 3 * TC_D + c0);
            w01[m] = pk2(wv.x, wv.y);
            w23[m] = pk2(wv.z, wv.w);
        }
        const float4 bv = *reinterpret_cast<const float4 *>(cb + c0);
        uint64_t x01[7], x23[7];
#pragma unroll
        for (int i = 0; i < 7; ++i) {
            const uint2 raw = *reinterpret_cast<const uint2 *>(sm + SM_RAW + (tau0 + i) * RAW_LD + c0 * 2);
            x01[i] = bf2_to_f2(raw.x);
            x23[i] = bf2_to_f2(raw.y);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int tau = tau0 + q;
            uint64_t a01 = pk2(bv.x, bv.y), a23 = pk2(bv.z, bv.w);
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                if (K4 || m >= m0) {
                    a01 = fma2(w01[m], x01[q + m], a01);
                    a23 = fma2(w23[m], x23[q + m], a23);
                }
            }
            float y[4];
            upk2(silu2(a01), y[0], y[1]);
            upk2(silu2(a23), y[2], y[3]);
            __nv_bfloat162 lo = __floats2bfloat162_rn(y[0], y[1]);
            __nv_bfloat162 hi = __floats2bfloat162_rn(y[2], y[3]);
            if (sec < 2) {
                // the conv output as stored (bf16), then the L2 of the row
                uint32_t wl = *reinterpret_cast<const uint32_t *>(&lo);
                uint32_t wh = *reinterpret_cast<const uint32_t *>(&hi);
                const uint64_t r01 = bf2_to_f2(wl), r23 = bf2_to_f2(wh);
                upk2(r01, y[0], y[1]);
                upk2(r23, y[2], y[3]);
                float ss = 0.f;
#pragma unroll
                for (int e = 0; e < 4; ++e) ss = fmaf(y[e], y[e], ss);
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
                const float inv = rsqrtf(ss + a.l2_eps);
                const uint64_t iv = pk2(inv, inv);
                upk2(mul2(r01, iv), y[0], y[1]);
                upk2(mul2(r23, iv), y[2], y[3]);
                lo = __floats2bfloat162_rn(y[0], y[1]);
                hi = __floats2bfloat162_rn(y[2], y[3]);
            }
            uint2 packed = make_uint2(*reinterpret_cast<const uint32_t *>(&lo),
                                      *reinterpret_cast<const uint32_t *>(&hi));
            if (tau >= n) packed = sec < 2 ? make_uint2(pfw, pfw) : make_uint2(0u, 0u);
            const uint32_t off = sec == 2 ? SM_V + tc::sw128_offset(tau, 4 * lane, 64, 2)
                                          : kqo + tc::sw128_offset((sec == 0 ? 64 : 0) + tau, 4 * lane, 128, 2);
            *reinterpret_cast<uint2 *>(sm + off) = packed;
        }
    }
}
__device__ __forceinline__ void conv_tile_any(const RecArgs &a, unsigned char *sm, int n,
                                              float pad, int warp, int lane, uint32_t kqo) {
    if (a.conv_k == 4) conv_tile<true>(a, sm, n, pad, warp, lane, kqo);
    else conv_tile<false>(a, sm, n, pad, warp, lane, kqo);
}

// New conv state of a stream, rows i < kernel - 1 = stream rows len - (kernel - 1) + i of
// [old state ; x], for the sections in [sec0, sec1): from the first chunk's raw rows when the
// stream fits one chunk, else from x.
__device__ __forceinline__ void write_conv_state(const RecArgs &a, const unsigned char *sm,
                                                 __nv_bfloat16 *state, int t0, int len, int kh,
                                                 int j, int sec0, int sec1, int tid) {
    const __nv_bfloat16 *x = reinterpret_cast<const __nv_bfloat16 *>(a.x);
    const int64_t cd = (int64_t)(2 * a.Hk + a.Hv) * TC_D;
    const int K1 = a.conv_k - 1;
    const int per = (sec1 - sec0) * 16;
    for (int idx = tid; idx < K1 * per; idx += TC_THREADS) {
        const int i = idx / per, cc = sec0 * 16 + idx % per;
        const int ch = front_channel(a, cc >> 4, kh, j) + (cc & 15) * 8;
        const int r = len - K1 + i;
        const uint4 v = len <= TC_C
                            ? *reinterpret_cast<const uint4 *>(sm + SM_RAW + (r + 3) * RAW_LD + cc * 16)
                            : *reinterpret_cast<const uint4 *>(x + (int64_t)(t0 + r) * a.x_stride + ch);
        *reinterpret_cast<uint4 *>(state + (int64_t)i * cd + ch) = v;
    }
}

// A gate value read once: through the non-coherent path without allocating in L1 (the block's
// shared memory leaves L1 little room, and the tile is not read again).
__device__ __forceinline__ float ld_gate(const float *p) {
    float v;
    asm volatile("ld.global.nc.L1::no_allocate.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}

// Block-wide barrier that also reports whether any thread raised the local error flag. All
// threads take the same branch: the flag is raised only by a wait that has run out, i.e. at
// least the wait limit (1 ms or more) after that thread left this barrier, long after every
// thread has read the flag here. (A reduction barrier, __syncthreads_or, made the KDA
// recurrence 10% slower.)
__device__ __forceinline__ bool sync_ok(volatile int *flag) {
    __syncthreads();
    return *flag == 0;
}

template <bool KDA, bool FRONT>
__global__ void __launch_bounds__(TC_THREADS, 1) chunk_tc_kernel(const __grid_constant__ TcParams P) {
    const RecArgs &a = P.a;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm =
        reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                          ~static_cast<uintptr_t>(1023));
    float *sf = reinterpret_cast<float *>(sm + SM_SMALL);
    float *adp = reinterpret_cast<float *>(sm + SM_AD);
    uint64_t *bar_a = reinterpret_cast<uint64_t *>(sm + SM_BARS);
    uint64_t *bar_b = bar_a + 1;
    uint64_t *bar_c = reinterpret_cast<uint64_t *>(sm + SM_BARS + 40);  // state update done
    uint64_t *bar_d = reinterpret_cast<uint64_t *>(sm + SM_BARS + 48);  // block-substitution steps
    uint64_t *bar_e = reinterpret_cast<uint64_t *>(sm + SM_BARS + 56);  // final drain of the MMAs
    uint64_t *bar_kq = reinterpret_cast<uint64_t *>(sm + SM_BARS + 64);  // K|Q tile by TMA
    uint64_t *bar_v = reinterpret_cast<uint64_t *>(sm + SM_BARS + 72);   // V tile by TMA
    volatile int *err = reinterpret_cast<volatile int *>(sm + SM_BARS + 16);
    volatile int *unit_sh = err + 1;
    volatile int *slow_sh = err + 2;
    volatile int *qk_sh = err + 3;
    uint32_t *tmem_sh = reinterpret_cast<uint32_t *>(sm + SM_BARS + 32);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    constexpr uint32_t COL_VT = KDA ? COL_RUD : COL_D1;  // V^T from the identity MMA
    const uint32_t lq = tc::tmem_lane_base(warp);  // this warp's TMEM lane quadrant
    // TMEM row (= k-channel c when staging, = v-channel d in the state phases) and which of the
    // NQ parts of the columns (or of the chunk's rows) this thread takes.
    const int row = tid & 127;
    const int part = tid >> 7;
    constexpr int C16 = TC_C / NQ;   // chunk rows / 64-column slices per part
    constexpr int D32 = TC_D / NQ;   // 128-column slices per part

    if (tid == 0) {
        *err = 0;
        tc::mbar_init(bar_a, 1);
        tc::mbar_init(bar_b, 1);
        tc::mbar_init(bar_c, 1);
        tc::mbar_init(bar_d, 1);
        tc::mbar_init(bar_e, 1);
        tc::mbar_init(bar_kq, 1);
        tc::mbar_init(bar_v, 1);
        tc::fence_mbar_init();
    }
    // identity tile (bf16, K-major 64x64) for the transposing MMAs
    for (int idx = tid; idx < 64 * 64; idx += TC_THREADS) {
        const int r = idx >> 6, k = idx & 63;
        *reinterpret_cast<__nv_bfloat16 *>(sm + SM_ID + tc::sw128_offset(r, k, 64, 2)) =
            __float2bfloat16_rn(r == k ? 1.f : 0.f);
    }
    tc::fence_async_smem();
    if (warp == 0) {
        tc::tmem_alloc(tmem_sh, TMEM_COLS);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tm = *tmem_sh;
    const uint32_t sb = tc::smem_u32(sm);  // shared-window address of the tile area (uniform)
    uint32_t phase_a = 0, phase_b = 0, phase_c = 0;
    bool pend_c = false;  // a state-update MMA group not yet waited for

    const uint64_t wait_ns = a.wait_ns ? a.wait_ns : WAIT_NS;
    auto wait_bar = [&](uint64_t *bar, uint32_t &ph) {
        const bool ok = tc::mbar_wait(bar, ph, wait_ns);
        ph ^= 1u;
        if (!ok) *err = 1;
        tc::fence_after_sync();
    };
    // The state update of a chunk completes on bar_c, after the output MMA (bar_b): the output
    // epilogue and the next chunk's prologue run meanwhile. Wait for it before anything reads S
    // or rewrites the operands it reads (the transposed key tile, the U' columns).
    auto wait_state = [&]() {
        if (pend_c) {
            wait_bar(bar_c, phase_c);
            pend_c = false;
        }
    };

    // TMA loads of the K|Q and V tiles (plain calls): one thread issues the boxes of a chunk, one
    // load per tile and chunk in flight at most; every thread waits for a tile's phase before
    // its first use (par_*: parity of the next load to be consumed; fly_*: the issuing thread's
    // record of a load that has not been consumed, drained on exit)
    const bool use_tma = !FRONT && P.tma != 0;
    uint32_t par_kq = 0, par_v = 0;
    bool fly_kq = false, fly_v = false;
    auto tma_kq = [&](int kh_, int tok, uint32_t kqo, int issuer = 0) {
        if (tid == issuer) {
            tc::fence_async_smem();  // earlier generic accesses of the tile come first
            tc::mbar_expect_tx(bar_kq, 32768u);
            const int x = kh_ * TC_D;
            tc::tma_load_2d(sb + kqo, &P.map_k, x, tok, bar_kq);           // K, channels 0-63
            tc::tma_load_2d(sb + kqo + 16384, &P.map_k, x + 64, tok, bar_kq);  // K, 64-127
            tc::tma_load_2d(sb + kqo + 8192, &P.map_q, x, tok, bar_kq);    // Q rows 64.. of the tile
            tc::tma_load_2d(sb + kqo + 24576, &P.map_q, x + 64, tok, bar_kq);
            fly_kq = true;
        }
    };
    auto tma_v = [&](int j_, int tok) {
        if (tid == 0) {
            tc::fence_async_smem();
            tc::mbar_expect_tx(bar_v, 16384u);
            const int x = j_ * TC_D;
            tc::tma_load_2d(sb + SM_V, &P.map_v, x, tok, bar_v);
            tc::tma_load_2d(sb + SM_V + 8192, &P.map_v, x + 64, tok, bar_v);
            fly_v = true;
        }
    };
    auto tma_wait = [&](uint64_t *bar, uint32_t par) {
        if (!tc::mbar_wait(bar, par, wait_ns)) *err = 1;
    };

    ColWalk w_kq, w_kqg, w_kr;
    w_kq.init(SM_KQ, row, 128, 2);    // column c of the bf16 K|Q tile
    w_kqg.init(SM_KQG, row, 128, 4);  // column c of the tf32 K|Q tile
    w_kr.init(SM_P, row, 64, 4);      // column c of the tf32 Kinv tile (KDA; D1's B operand
                                      // in the P | T00 | T11 | -A10 space, free until D1)

    const float scale = a.scale;
    const int Hv = a.Hv, group = a.Hv / a.Hk;
    // q|k pad rows of the fused front end: pad_fill (KDA); zero for GDN, whose k tile is also
    // contracted over tokens by the transposing MMA, where a NaN row would reach every column
    const float pad_qk = KDA ? a.pad_fill : 0.f;

    for (;;) {
        __syncthreads();  // everyone has read the previous unit index
        if (tid == 0) *unit_sh = atomicAdd(P.counter, 1);
        if (!sync_ok(err)) break;
        const int u = *unit_sh;
        if (u >= P.num_units) break;
        const int s = P.perm[u / Hv];
        const int j = u % Hv;
        const int kh = j / group;
        const bool alt = a.use_alt && s >= a.alt_from;  // segmented scan: a transition run
        int t0, len;
        if (!(alt ? stream_range(a.cu_alt, s - a.alt_from, 0, a.total, a.max_seqlen, a.status, t0, len)
                  : stream_range(a.cu, s, a.T_each, a.total, a.max_seqlen, a.status, t0, len)))
            continue;
        if (len <= 0) continue;
        const int nch = (len + TC_C - 1) / TC_C;
        float *hg = reinterpret_cast<float *>(a.h_ptrs[s]) + (int64_t)j * TC_D * TC_D;
        __nv_bfloat16 *og = reinterpret_cast<__nv_bfloat16 *>(alt ? a.out_alt : a.out) + (int64_t)j * TC_D;

        __nv_bfloat16 *conv_state =
            FRONT && a.conv_k > 1 ? reinterpret_cast<__nv_bfloat16 *>(a.conv_state_ptrs[s]) : nullptr;
        if (FRONT) {
            load_conv_weights(a, sm, kh, j, tid);
            load_raw(a, sm, conv_state, t0, len, 0, kh, j, tid);
        } else if (use_tma && !alt) {
            tma_kq(kh, t0, SM_KQ);
            tma_v(j, t0);
        } else {
            load_kq(a, sm, t0, min(TC_C, len), kh, tid);
            load_v(a, sm, t0, min(TC_C, len), j, tid, alt);
        }
        cp_async_commit();
        // S[d][c] = H[c][d]: thread (d, part) loads columns c in [D32*part, D32*part + D32)
#pragma unroll
        for (int g = 0; g < D32 / 16; ++g) {
            float v[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = hg[(int64_t)(D32 * part + g * 16 + i) * TC_D + row];
            tc::tmem_st16(tc::tmem_addr(tm, lq, COL_S + D32 * part + g * 16), v);
        }
        tc::tmem_wait_st();
        if (FRONT) {  // first chunk's q, k, v tiles; advance the conv state
            cp_async_wait_all();
            __syncthreads();
            if (conv_state) {
                // v channels belong to this unit alone; q|k channels are written by the last
                // unit of the k-head group to have read the old state
                if (tid == 0) {
                    __threadfence();
                    *qk_sh = atomicAdd(P.conv_readers + s * a.Hk + kh, 1) == group - 1;
                    __threadfence();
                }
                __syncthreads();
                write_conv_state(a, sm, conv_state, t0, len, kh, j, *qk_sh ? 0 : 2, 3, tid);
            }
            conv_tile_any(a, sm, min(TC_C, len), pad_qk, warp, lane, SM_KQ);
            tc::fence_async_smem();
        }

        // gates and beta of the chunk being computed are fetched one chunk ahead: GDN and beta
        // by threads < 64, the KDA gate tile by every thread (16 rows of its channel)
        float pre_g = 0.f, pre_b = 0.f;
        float pre_gk[KDA ? C16 : 1];
        auto fetch_gates = [&](int tok, int nn) {
            if (tid < TC_C) {
                pre_b = tid < nn ? a.beta[(int64_t)(tok + tid) * Hv + j] : 0.f;
                if (!KDA) pre_g = tid < nn ? a.g[(int64_t)(tok + tid) * Hv + j] : 0.f;
            }
        };
        fetch_gates(t0, min(TC_C, len));
        if (KDA) {
            const int nn = min(TC_C, len);
            const float *gp = a.g + ((int64_t)t0 * Hv + j) * TC_D + row;
#pragma unroll
            for (int t = 0; t < C16; ++t) {
                const int tt = C16 * part + t;
                pre_gk[t] = tt < nn ? gp[(int64_t)tt * Hv * TC_D] : 0.f;
            }
        }
        // KDA: a chunk's cumulative gates in base-2 units, gc[C16*part + t][c] log2(e) (c = row),
        // are formed in pre_gk one chunk ahead, in two halves around a barrier of the chunk
        // before (the partial sums of the four row parts meet in shared memory); the chunk
        // itself then starts from them without a barrier of its own. gates_sum: this thread's
        // 16 rows; gates_carry: the earlier parts' totals, gc_L and e^{gc_L}, beta.
        auto gates_sum = [&]() {
            float acc = 0.f;
#pragma unroll
            for (int t = 0; t < C16; ++t) {
                acc = fmaf(pre_gk[t], LOG2E, acc);
                pre_gk[t] = acc;
            }
            sf[SF_CARRY + part * 128 + row] = acc;
        };
        auto gates_carry = [&]() {
            float carry = 0.f;
#pragma unroll
            for (int pp = 0; pp < NQ - 1; ++pp)
                if (pp < part) carry += sf[SF_CARRY + pp * 128 + row];
#pragma unroll
            for (int t = 0; t < C16; ++t) pre_gk[t] += carry;
            if (part == NQ - 1) {
                sf[SF_GL + row] = pre_gk[C16 - 1];  // base 2
                sf[SF_EL + row] = tc::ex2(pre_gk[C16 - 1]);
            }
            if (tid < TC_C) sf[SF_BETA + tid] = pre_b;
        };
        if (KDA) {  // the first chunk's
            gates_sum();
            __syncthreads();
            gates_carry();
        }

        // Global stores of a chunk's output tile, staged as bf16 [t][d] in the A^T buffer; they
        // are issued in the next chunk (or after the last chunk) by warps w0 .. w0 + nw - 1.
        // Within the chunk loop: in GDN's recurrence-only launch by warps 1-7 while warps 8-15
        // solve and warp 0 issues D2 (their wait for D2 has nothing else to overlap); in KDA's
        // by warps 1-15 while D1 runs (warp 0 issues it and writes part of A00 next; there the
        // later placement was slower); in the fused launch by all warps while D1 runs.
        auto store_o = [&](int tok0s, int ns, int w0, int nw) {
            const __nv_bfloat16 *os = reinterpret_cast<const __nv_bfloat16 *>(sm + SM_AT);
            auto store_piece = [&](int idx) {  // row idx / 16, channels 8 (idx % 16) ..
                const int t = idx >> 4, cj = idx & 15;
                __nv_bfloat16 *dst = og + (int64_t)(tok0s + t) * Hv * TC_D + cj * 8;
                if (a.z) {
                    // gated RMSNorm of the stored (bf16) o row: 16 lanes x 8 channels, the
                    // order of the separate gated-norm kernel
                    float ov[8];
                    Vec16<__nv_bfloat16>::load(os + t * O_LD + cj * 8, ov);
                    float ss = 0.f;
#pragma unroll
                    for (int e = 0; e < 8; ++e) ss = fmaf(ov[e], ov[e], ss);
#pragma unroll
                    for (int off = 8; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
                    if (t < ns) {
                        float zv[8], wv[8];
                        Vec16<__nv_bfloat16>::load(reinterpret_cast<const __nv_bfloat16 *>(a.z) +
                                                       ((int64_t)(tok0s + t) * Hv + j) * TC_D + cj * 8, zv);
                        Vec16<__nv_bfloat16>::load(reinterpret_cast<const __nv_bfloat16 *>(a.norm_w) + cj * 8, wv);
                        const float inv = rsqrtf(ss * (1.f / TC_D) + a.norm_eps);
#pragma unroll
                        for (int e = 0; e < 8; ++e) ov[e] = ov[e] * inv * wv[e] * silu(zv[e]);
                        Vec16<__nv_bfloat16>::store(dst, ov);
                    }
                } else if (t < ns) {
                    const uint4 ov = *reinterpret_cast<const uint4 *>(os + t * O_LD + cj * 8);
                    if (FRONT) *reinterpret_cast<uint4 *>(dst) = ov;
                    else __stcs(reinterpret_cast<uint4 *>(dst), ov);  // streamed: not read again here
                }
            };
            if (nw == TC_THREADS / 32) {
#pragma unroll
                for (int m = 0; m < 1024 / TC_THREADS; ++m) store_piece(tid + TC_THREADS * m);
            } else if (warp >= w0 && warp < w0 + nw) {  // whole warps: 16-lane groups aligned
                for (int idx = tid - 32 * w0; idx < 1024; idx += 32 * nw) store_piece(idx);
            }
        };
        int pend_tok0 = 0, pend_n = 0;  // output tile staged, not yet stored

        for (int ch = 0; ch < nch; ++ch) {
            const int tok0 = t0 + ch * TC_C;
            const int n = min(TC_C, len - ch * TC_C);
            const bool last = (ch + 1 == nch);
            // K|Q tile of this chunk and of the next: GDN alternates two buffers by chunk parity
            // (the state update reads the tile at the end of the chunk, after the next one's
            // load has been issued); KDA reads it only until D1 and keeps one
            const uint32_t kqo = (KDA || !(ch & 1)) ? SM_KQ : SM_KQ1;
            const uint32_t kqo_next = (KDA || (ch & 1)) ? SM_KQ : SM_KQ1;

            // ---------------- gates (KDA: formed one chunk ahead; every decay factor below is one
            //                  ex2 of them)
            float gcr[KDA ? C16 : 1];
            if (KDA) {
#pragma unroll
                for (int t = 0; t < C16; ++t) gcr[t] = pre_gk[t];
                if (tid == 0) *slow_sh = 0;
            }
            if (!KDA && tid < TC_C) {
                const int t = tid;
                sf[SF_BETA + t] = pre_b;
                float x = pre_g;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const float y = __shfl_up_sync(0xffffffffu, x, off);
                    if (lane >= off) x += y;
                }
                if (lane == 31) sf[SF_WARP + warp] = x;
                sf[SF_GC + t] = x;  // warp-local; carried below
            }
            cp_async_wait_all();
            if (use_tma) {  // this chunk's K|Q and V tiles (the K|Q may have been waited already)
                tma_wait(bar_kq, par_kq);
                tma_wait(bar_v, par_v);
                par_kq ^= 1u;
                par_v ^= 1u;
                fly_kq = fly_v = false;
            }
            tc::fence_async_smem();
            if (a.debug_stall) {  // test knob: a wait on a barrier nothing completes runs out
                uint32_t never = 0;
                wait_bar(bar_e, never);
            }
            if (!KDA && !sync_ok(err)) break;  // GDN: the scalar gates meet in shared memory
            // this chunk's scalar gates are in shared memory: fetch the next chunk's
            if (!last) fetch_gates(tok0 + TC_C, min(TC_C, len - (ch + 1) * TC_C));
            if (!KDA && tid < TC_C) {
                // gc_t, and the chunk's decay factors from it: gc at rows 31 and 63 are the two
                // warps' totals (so no barrier is needed before the factors)
                const float w0t = sf[SF_WARP];
                const float gct = sf[SF_GC + tid] + (tid >= 32 ? w0t : 0.f);
                const float gL = w0t + sf[SF_WARP + 1], gm = w0t;
                sf[SF_GC + tid] = gct;
                sf[SF_GC2 + tid] = gct * LOG2E;
                sf[SF_EG + tid] = __expf(gct);
                sf[SF_EGL + tid] = __expf(gL - gct);
                // e^{gc_t - gc_i} = e^{gc_t - gc_m} e^{gc_m - gc_i} (m = row 31): both factors
                // are bounded by the half-chunk decay range, checked below
                sf[SF_RF + tid] = __expf(gct - gm);
                sf[SF_CF + tid] = __expf(gm - gct);
            }
            // Pad rows of the K|Q tile carry pad_fill; every consumer removes them by select.
            // The V tile's pad rows are zero: it is contracted over tokens by the transposing
            // MMA, where a NaN row would reach every column even through an exact zero weight.
            // (Async copies zero-fill those rows; a TMA box brings the next stream's rows,
            // rewritten here before any use.)
            if (!FRONT && n < TC_C && (use_tma || a.pad_fill != 0.f)) {
                const __nv_bfloat16 pf = __float2bfloat16_rn(a.pad_fill);
                for (int idx = tid; idx < (TC_C - n) * TC_D; idx += TC_THREADS) {
                    const int r = n + idx / TC_D, c = idx % TC_D;
                    *reinterpret_cast<__nv_bfloat16 *>(sm + kqo + tc::sw128_offset(r, c, 128, 2)) = pf;
                    *reinterpret_cast<__nv_bfloat16 *>(sm + kqo + tc::sw128_offset(64 + r, c, 128, 2)) = pf;
                    if (use_tma && !alt)
                        *reinterpret_cast<__nv_bfloat16 *>(sm + SM_V + tc::sw128_offset(r, c, 64, 2)) =
                            __float2bfloat16_rn(0.f);
                }
                tc::fence_async_smem();
            }
            if (KDA && !sync_ok(err)) break;  // KDA's first barrier of the chunk (GDN: the
                                              // barrier before D1 follows)

            // ---------------- D1 = [K;Q] K^T (KDA: tf32, decays split per factor)
            bool slow = false;
            if (KDA) wait_state();  // the key tile below is the previous state update's operand
            if (KDA) {
                // One pass over the chunk's keys and queries, thread per (channel, row part):
                //  - [K e^gc ; Q e^gc] (D1's A operand, then the state MMA's);
                //  - Kinv = K e^{-gc} (D1's B operand): D1 = [K;Q] K^T with e^{gc_t - gc_i} split
                //    as e^{gc_t} e^{-gc_i}, valid while the chunk's decay e^{-gc_L} stays below
                //    e^80 (else the exact path below);
                //  - (K e^{gc_L - gc})^T, the state update's key tile, with e^{gc_L - gc} formed
                //    as e^{gc_L} e^{-gc} (directly where e^{-gc} could overflow).
                // Rows >= n are zero in all three.
                const int c = row;
                const float gLc = sf[SF_GL + c], eLc = sf[SF_EL + c];
                const bool steep = -gLc > 80.f * LOG2E;
                if (part == NQ - 1 && steep) *slow_sh = 1;
                float kd[4];
#pragma unroll
                for (int t = 0; t < C16; ++t) {
                    const int tt = C16 * part + t;
                    const bool valid = tt < n;
                    // pad rows are zeroed on input: every factor below is finite (e^{-gc} is
                    // bounded by e^80 where the product form is used)
                    const float kv = valid ? ld_bf16(sm, w_kq.at(tt)) : 0.f;
                    const float qv = valid ? ld_bf16(sm, w_kq.at(64 + tt)) : 0.f;
                    const float eg = tc::ex2(gcr[t]), ei = tc::ex2(-gcr[t]);
                    st_tf32(sm, w_kqg.at(tt), kv * eg);
                    st_tf32(sm, w_kqg.at(64 + tt), qv * eg);
                    st_tf32(sm, w_kr.at(tt), kv * ei);
                    const float egl = steep ? tc::ex2(gLc - gcr[t]) : eLc * ei;  // <= 1
                    kd[t & 3] = tc::to_tf32_operand(kv * egl);
                    if ((t & 3) == 3) {
                        *reinterpret_cast<float4 *>(sm + SM_KDT + tc::sw128_offset(c, tt - 3, 128, 4)) =
                            make_float4(kd[0], kd[1], kd[2], kd[3]);
                    }
                }
                tc::fence_async_smem();
                tc::fence_before_sync();
                __syncthreads();
                slow = *slow_sh != 0;
            } else {
                tc::fence_before_sync();
                __syncthreads();
            }
            if (!slow && warp == 0 && tc::elect_one()) {
                tc::fence_after_sync();
                if (KDA) {
                    constexpr uint32_t id = tc::idesc(128, 64, tc::FMT_TF32);
#pragma unroll
                    for (uint32_t kk = 0; kk < 16; ++kk) {
                        const uint32_t off = (kk & 3u) * 32u;
                        const uint64_t ad = tc::sdesc_sw128((sb + SM_KQG) + (kk >> 2) * 16384u + off);
                        const uint64_t bd = tc::sdesc_sw128((sb + SM_P) + (kk >> 2) * 8192u + off);
                        tc::mma_tf32_ss(tm + COL_D1, ad, bd, id, kk > 0);
                    }
                } else {
                    constexpr uint32_t id = tc::idesc(128, 64, tc::FMT_BF16);
#pragma unroll
                    for (uint32_t kk = 0; kk < 8; ++kk) {
                        const uint32_t addr = (sb + kqo) + (kk >> 2) * 16384u + (kk & 3u) * 32u;
                        tc::mma_bf16_ss(tm + COL_D1, tc::sdesc_sw128(addr), tc::sdesc_sw128(addr), id, kk > 0);
                    }
                }
                tc::mma_commit(bar_a);
            }

            // D2 = S [K;Q]^T and V^T (identity MMA). KDA: tf32, A (S) from TMEM, B the decayed
            // [K;Q] tile. GDN: the raw bf16 K|Q tile against S split into two bf16 terms in TMEM
            // (S = S_hi + S_lo within 2^-18; staged below), two kind::f16 groups accumulating
            // into D2. Issued by warp 0 while warps 8-15 solve the triangular blocks: the issuing
            // lane is held for as long as the tensor core takes to run the group, and warp 0 has
            // no share in that solve (the barrier before it made the staged operands visible).
            auto issue_mma2 = [&]() {
                if (warp == 0 && tc::elect_one()) {
                    tc::fence_after_sync();
                    if (KDA) {
                        constexpr uint32_t id = tc::idesc(128, 128, tc::FMT_TF32);
#pragma unroll
                        for (uint32_t kk = 0; kk < 16; ++kk) {
                            const uint64_t bd = tc::sdesc_sw128((sb + SM_KQG) + (kk >> 2) * 16384u + (kk & 3u) * 32u);
                            tc::mma_tf32_ts(tm + COL_D2, tm + COL_S + kk * 8, bd, id, kk > 0);
                        }
                    } else {
                        constexpr uint32_t id = tc::idesc(128, 128, tc::FMT_BF16);
#pragma unroll
                        for (uint32_t h = 0; h < 2; ++h) {
#pragma unroll
                            for (uint32_t kk = 0; kk < 8; ++kk) {
                                const uint64_t bd = tc::sdesc_sw128((sb + kqo) + (kk >> 2) * 16384u + (kk & 3u) * 32u);
                                tc::mma_bf16_ts(tm + COL_D2, tm + (h ? COL_SLO : COL_SHI) + kk * 8, bd, id,
                                                (h | kk) > 0);
                            }
                        }
                    }
                    constexpr uint32_t idv = tc::idesc(128, 64, tc::FMT_BF16, true, false);
#pragma unroll
                    for (uint32_t kk = 0; kk < 4; ++kk) {
                        const uint64_t ad = tc::sdesc_sw128_mn((sb + SM_V) + kk * 2048u, 64u * 128u, 1024u);
                        const uint64_t bd = tc::sdesc_sw128((sb + SM_ID) + kk * 32u);
                        tc::mma_bf16_ss(tm + COL_VT, ad, bd, idv, kk > 0);
                    }
                    tc::mma_commit(bar_b);
                }
            };

            if (!KDA) {
                // the previous state update is complete: S may be read, and the K|Q buffer it
                // read takes the next chunk's tile
                wait_state();
                if (!FRONT && !last && !(use_tma && !alt)) {  // (a TMA tile: after the A/P pass)
                    load_kq(a, sm, tok0 + TC_C, min(TC_C, len - (ch + 1) * TC_C), kh, tid, kqo_next);
                    cp_async_commit();
                }
                // S -> S_hi = bf16(S), S_lo = bf16(S - S_hi), packed two per column, D2's A
                // operand, while D1 is computed: thread (lane, part) takes its 32
                // columns; warp 0 issues D1, so warp 4 (its TMEM lane quadrant) takes its columns
                auto split_cols = [&](int c0) {  // columns c0 .. c0 + 31 of this warp's lanes
                    float sv[D32], hi[D32 / 2], lo[D32 / 2];
#pragma unroll
                    for (int g = 0; g < D32 / 16; ++g)
                        tc::tmem_ld16(tc::tmem_addr(tm, lq, COL_S + c0 + 16 * g), sv + 16 * g);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < D32 / 2; ++i) {
                        const __nv_bfloat162 h2 = __floats2bfloat162_rn(sv[2 * i], sv[2 * i + 1]);
                        const uint32_t hu = *reinterpret_cast<const uint32_t *>(&h2);
                        const __nv_bfloat162 l2 = __floats2bfloat162_rn(
                            sv[2 * i] - __uint_as_float(hu << 16),
                            sv[2 * i + 1] - __uint_as_float(hu & 0xFFFF0000u));
                        hi[i] = __uint_as_float(hu);
                        lo[i] = *reinterpret_cast<const float *>(&l2);
                    }
                    tc::tmem_st16(tc::tmem_addr(tm, lq, COL_SHI + c0 / 2), hi);
                    tc::tmem_st16(tc::tmem_addr(tm, lq, COL_SLO + c0 / 2), lo);
                };
                if (warp != 0) {
                    split_cols(D32 * part);
                    if (warp == 4) split_cols(0);
                    tc::tmem_wait_st();
                    tc::fence_before_sync();
                }
            }

            if (KDA && !last) {
                // the next chunk's gate tile while D1 is computed: 16 loads per thread, 32 KB per
                // chunk, issued where the SM has nothing else in flight (issued later, with the
                // loads of every warp at once, they hold the block for about 2.8k cycles)
                const int nn = min(TC_C, len - (ch + 1) * TC_C);
                const float *gp = a.g + ((int64_t)(tok0 + TC_C) * Hv + j) * TC_D + row;
#pragma unroll
                for (int t = 0; t < C16; ++t) {
                    const int tt = C16 * part + t;
                    pre_gk[t] = tt < nn ? ld_gate(gp + (int64_t)tt * Hv * TC_D) : 0.f;
                }
            }
            if ((FRONT || KDA) && pend_n > 0) {  // previous chunk's output while D1 is computed
                store_o(pend_tok0, pend_n, FRONT ? 0 : 1, FRONT ? TC_THREADS / 32 : TC_THREADS / 32 - 1);
                pend_n = 0;
            }

            // ---------------- D1 ready (or computed exactly on CUDA cores, KDA fallback)
            if (!slow) {
                wait_bar(bar_a, phase_a);
            } else if (KDA) {
                float *gct = reinterpret_cast<float *>(sm + SM_P);  // [64][128] fp32, base 2 (Kinv's space)
#pragma unroll
                for (int t = 0; t < C16; ++t) gct[(C16 * part + t) * TC_D + row] = gcr[t];
                __syncthreads();
                if (part == 0) {  // warps 0-3: thread = D1 row
                    const int r = row & 63;
                    const bool isq = row >= 64;
                    for (int g = 0; g < 4; ++g) {
                        float v[16];
                        for (int ii = 0; ii < 16; ++ii) {
                            const int i = g * 16 + ii;
                            float acc = 0.f;
                            if (i <= r) {
                                for (int c = 0; c < TC_D; ++c) {
                                    const float lv = ld_bf16(sm, SM_KQ + tc::sw128_offset((isq ? 64 : 0) + r, c, 128, 2));
                                    const float kv = ld_bf16(sm, SM_KQ + tc::sw128_offset(i, c, 128, 2));
                                    acc = fmaf(lv * kv, tc::ex2(gct[r * TC_D + c] - gct[i * TC_D + c]), acc);
                                }
                            }
                            v[ii] = acc;
                        }
                        tc::tmem_st16(tc::tmem_addr(tm, lq, COL_D1 + g * 16), v);
                    }
                    tc::tmem_wait_st();
                }
                tc::fence_before_sync();
                __syncthreads();
                tc::fence_after_sync();
            }
            // no barrier: each thread reads D1 after its own wait, and the tiles written below
            // (A's diagonal blocks, P, -A10) have no reader left from before
            // KDA: K|Q tile consumed (the staging pass or the exact D1): the next chunk's in
            // flight (a TMA tile is issued after the A/P pass, below)
            if (KDA && !FRONT && !last && !(use_tma && !alt)) {
                load_kq(a, sm, tok0 + TC_C, min(TC_C, len - (ch + 1) * TC_C), kh, tid);
                cp_async_commit();
            }

            // ---------------- A^T (fp32) and P (tf32) from D1
            {
                const int r = row & 63;
                const bool isq = row >= 64;
                const float bt = sf[SF_BETA + r];
                const bool rv = r < n;
                const int i0 = C16 * part;
                // GDN decays: row factor x column factor when the half-chunk range allows it
                // (uniform per chunk), else the exact exponential of the difference
                const float gm_ = KDA ? 0.f : sf[SF_GC + TC_C / 2 - 1];
                const bool split_ok = KDA || (-gm_ <= 80.f && gm_ - sf[SF_GC + TC_C - 1] <= 80.f);
                const float gct2 = KDA ? 0.f : sf[SF_GC2 + r];
                const float rowf = (KDA ? 1.f : sf[SF_RF + r]) * (isq ? 1.f : bt);
                float v[16];
                tc::tmem_ld16(tc::tmem_addr(tm, lq, COL_D1 + i0), v);
                tc::tmem_wait_ld();
                if (KDA || split_ok) {
#pragma unroll
                    for (int ii = 0; ii < 16; ++ii) {
                        const int i = i0 + ii;
                        const float f = KDA ? rowf : rowf * sf[SF_CF + i];
                        const bool keep = rv && (isq ? i <= r : i < r);
                        v[ii] = keep ? f * v[ii] : 0.f;
                    }
                } else {
#pragma unroll
                    for (int ii = 0; ii < 16; ++ii) {
                        const int i = i0 + ii;
                        const float dec = tc::ex2(fminf(gct2 - sf[SF_GC2 + i], 0.f));
                        v[ii] = isq ? ((rv && i <= r) ? dec * v[ii] : 0.f)
                                    : ((rv && i < r) ? bt * dec * v[ii] : 0.f);
                    }
                }
                if (isq) {
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4)
                        *reinterpret_cast<float4 *>(sm + SM_P + tc::sw128_offset(r, i0 + q4 * 4, 64, 4)) =
                            make_float4(tc::to_tf32_operand(v[q4 * 4]), tc::to_tf32_operand(v[q4 * 4 + 1]),
                                        tc::to_tf32_operand(v[q4 * 4 + 2]), tc::to_tf32_operand(v[q4 * 4 + 3]));
                } else {
                    if ((i0 >> 5) == (r >> 5)) {  // a diagonal block: A00 or A11, transposed
                        float *adb = adp + (r >> 5) * 32 * AD_LD;
#pragma unroll
                        for (int ii = 0; ii < 16; ++ii) adb[((i0 & 31) + ii) * AD_LD + (r & 31)] = v[ii];
                    }
                    if (r >= 32 && i0 < 32) {  // -A10, the coupling of the two 32-token halves
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4)
                            *reinterpret_cast<float4 *>(sm + SM_NA10 + tc::sw128_offset(r - 32, i0 + q4 * 4, 32, 4)) =
                                make_float4(tc::to_tf32_operand(-v[q4 * 4]), tc::to_tf32_operand(-v[q4 * 4 + 1]),
                                            tc::to_tf32_operand(-v[q4 * 4 + 2]), tc::to_tf32_operand(-v[q4 * 4 + 3]));
                    }
                }
            }
            tc::fence_before_sync();
            // Each reader waits for its own writers only (hardware barriers 1-3): A00 is written by
            // warps 0 and 4 and solved by warps 8-11; A11 is written by warps 9 and 13 and solved
            // by warps 12-15; warp 0 issues D2 once every warp has read D1 (GDN's V^T lands in
            // D1's columns). P and -A10 are read by MMAs issued after the barriers that end R^T
            // (their proxy fence is there, when these stores have long drained).
            if (warp == 0 || warp == 4) named_arrive(1, 6 * 32);
            if (warp == 9) named_arrive(2, 5 * 32);
            if (warp != 0) named_arrive(3, TC_THREADS);
            // The next K|Q tile by TMA, from warp 7: it has no share in the solves and waits for
            // D2 next, while warp 0 (an A00 writer) goes straight on to D2's issue
            if (!FRONT && !last && use_tma && !alt) tma_kq(kh, tok0 + TC_C, kqo_next, 7 * 32);

            // ---------------- T00 = (I + A00)^{-1}, T11 = (I + A11)^{-1} (the two 32-token
            //   diagonal blocks of (I + A)^{-1}), fp32 forward substitution on CUDA cores by
            //   warps 8-15, 4 lanes per column (rows 4m + p); meanwhile warp 0 issues D2. The
            //   coupling block is applied by the tensor core as a block substitution:
            //   U'0 = R0 T00^T, U'1 = (R1 - U'0 A10^T) T11^T.
            if (warp >= 8) {
                const int w8 = warp - 8, b = w8 >> 2;
                named_sync(1 + b, b == 0 ? 6 * 32 : 5 * 32);  // this block of A is written
                const int jj = 8 * (w8 & 3) + (lane >> 2), p = lane & 3;
                float x[8];
#pragma unroll
                for (int m = 0; m < 8; ++m) x[m] = (4 * m + p == jj) ? 1.f : 0.f;
                const float *ab = adp + b * 32 * AD_LD + p;  // ab[i*AD_LD + 4m] = A[32b+4m+p][32b+i]
#pragma unroll
                for (int i = 0; i < 31; ++i) {
                    const int m0 = i >> 2;
                    const float xi = __shfl_sync(0xffffffffu, x[m0], (lane & ~3) | (i & 3));
                    {
                        const float nx = fmaf(-ab[i * AD_LD + 4 * m0], xi, x[m0]);
                        x[m0] = (p > (i & 3)) ? nx : x[m0];
                    }
#pragma unroll
                    for (int m = m0 + 1; m < 8; ++m) x[m] = fmaf(-ab[i * AD_LD + 4 * m], xi, x[m]);
                }
                const uint32_t tile = b == 0 ? SM_T00 : SM_T11;
#pragma unroll
                for (int m = 0; m < 8; ++m)
                    st_tf32(sm, tile + tc::sw128_offset(4 * m + p, jj, 32, 4), x[m]);
            } else if (warp == 0) {
                named_sync(3, TC_THREADS);  // every warp has read D1
                issue_mma2();
            } else if (!FRONT && !KDA && pend_n > 0) {  // previous chunk's output (warps 1-7)
                store_o(pend_tok0, pend_n, 1, 7);
            }
            if (!FRONT && !KDA) pend_n = 0;
            // the T blocks are read by the chain's MMAs, issued after the barriers that end R^T
            // (the proxy fence before them covers these stores)

            // ------ D2, V^T ready: R^T = beta (V^T - e^gc D2[:, :64]) -> TMEM
            // every thread reads D2 and V^T only after its own wait, and this phase writes no
            // shared memory: a timed-out wait is caught at the next checked barrier
            wait_bar(bar_b, phase_b);
            if (!last) {  // V tile consumed by the identity MMA: the next chunk's in flight (FRONT:
                          // the raw rows, into the tf32 K|Q buffer, which D2 has read)
                if (FRONT) load_raw(a, sm, nullptr, t0, len, (ch + 1) * TC_C, kh, j, tid);
                else if (use_tma && !alt) tma_v(j, tok0 + TC_C);
                else load_v(a, sm, tok0 + TC_C, min(TC_C, len - (ch + 1) * TC_C), j, tid, alt);
                cp_async_commit();
            }
            {
                const int t0c = C16 * part;
                float v[16], vt[16];
                tc::tmem_ld16(tc::tmem_addr(tm, lq, COL_D2 + t0c), v);
                tc::tmem_ld16(tc::tmem_addr(tm, lq, COL_VT + t0c), vt);
                tc::tmem_wait_ld();
#pragma unroll
                for (int ii = 0; ii < 16; ++ii) {
                    const int t = t0c + ii;
                    const float kh_t = KDA ? v[ii] : sf[SF_EG + t] * v[ii];
                    v[ii] = t < n ? tc::to_tf32(sf[SF_BETA + t] * (vt[ii] - kh_t)) : 0.f;
                }
                tc::tmem_st16(tc::tmem_addr(tm, lq, COL_RU + t0c), v);
                if (t0c >= 32) tc::tmem_st16(tc::tmem_addr(tm, lq, COL_D6 + t0c), v);  // Z = R1
                tc::tmem_wait_st();
            }
            tc::fence_async_smem();  // P, -A10 and the T blocks, for the MMAs after these barriers
            tc::fence_before_sync();
            // The chain's first product reads R0^T (written by warps 0-7) and T00 (warps 8-11),
            // its second and third R1^T (warps 8-15) and T11 (warps 12-15): warp 0 waits for
            // each group on its own hardware barrier (4, then 5). The other warps go on to the
            // state decay below, which touches nothing the chain reads: GDN's at once, KDA's
            // once warps 1-15 have all arrived (barrier 6; its decay and gate sums, started
            // early, take issue slots from the warps the chain waits for).
            if (warp >= 1 && warp < 12) named_arrive(4, 12 * 32);
            if (warp >= 8) named_arrive(5, 9 * 32);
            if (KDA && warp >= 1) named_sync(6, 15 * 32);

            // ---------------- block substitution, one thread: U'0^T = R0^T T00^T;
            //   Z^T = R1^T - U'0^T A10^T (accumulated onto R1^T); U'1^T = Z^T T11^T (into the
            //   P U' accumulator columns 0..31). Each product reads the previous one as its
            //   A operand straight from TMEM, without the rounding step; MMAs into
            //   different accumulators are not ordered, so the issuing thread waits on bar_d
            //   (two completions per chunk: parities 0, then 1) between them.
            constexpr uint32_t id32 = tc::idesc(128, 32, tc::FMT_TF32);
            auto issue_t00 = [&]() {  // U'0^T = R0^T T00^T
                tc::fence_after_sync();
#pragma unroll
                for (uint32_t kk = 0; kk < 4; ++kk)
                    tc::mma_tf32_ts(tm + COL_D6, tm + COL_RU + kk * 8,
                                    tc::sdesc_sw128((sb + SM_T00) + kk * 32u), id32, kk > 0);
                tc::mma_commit(bar_d);
            };
            if (warp == 0) {
                named_sync(4, 12 * 32);
                if (tc::elect_one()) issue_t00();
                __syncwarp();
                named_sync(5, 9 * 32);
            }
            if (warp == 0 && tc::elect_one()) {
                tc::fence_after_sync();
                bool ok = tc::mbar_wait(bar_d, 0, wait_ns);
                tc::fence_after_sync();
                if (ok) {
#pragma unroll
                    for (uint32_t kk = 0; kk < 4; ++kk)
                        tc::mma_tf32_ts(tm + COL_D6 + 32, tm + COL_D6 + kk * 8,
                                        tc::sdesc_sw128((sb + SM_NA10) + kk * 32u), id32, 1);
                    tc::mma_commit(bar_d);
                    ok = tc::mbar_wait(bar_d, 1, wait_ns);
                    tc::fence_after_sync();
                }
                if (ok) {
#pragma unroll
                    for (uint32_t kk = 0; kk < 4; ++kk)
                        tc::mma_tf32_ts(tm + COL_D4, tm + COL_D6 + 32 + kk * 8,
                                        tc::sdesc_sw128((sb + SM_T11) + kk * 32u), id32, kk > 0);
                } else {
                    *err = 1;
                }
                tc::mma_commit(bar_b);
            }
            // S <- S diag(e^{gc_L}) while the tensor core works (the chain above reads none of
            // the state columns; the state MMA is issued after the barriers below). Warp 0 runs
            // the chain, so warps 4 and 8 (the same TMEM lane quadrant) take its 32 columns.
            if (warp != 0) {
                const int c0 = D32 * part;
                float sv[D32];
#pragma unroll
                for (int g = 0; g < D32 / 16; ++g)
                    tc::tmem_ld16(tc::tmem_addr(tm, lq, COL_S + c0 + 16 * g), sv + 16 * g);
                tc::tmem_wait_ld();
                const float egL = KDA ? 0.f : sf[SF_EG + TC_C - 1];
#pragma unroll
                for (int ii = 0; ii < D32; ++ii) sv[ii] *= KDA ? sf[SF_EL + c0 + ii] : egL;
#pragma unroll
                for (int g = 0; g < D32 / 16; ++g)
                    tc::tmem_st16(tc::tmem_addr(tm, lq, COL_S + c0 + 16 * g), sv + 16 * g);
                if (warp == 4 || warp == 8) {  // warp 0's columns, 16 each
                    const int cs = warp == 4 ? 0 : 16;
                    float sx[16];
                    tc::tmem_ld16(tc::tmem_addr(tm, lq, COL_S + cs), sx);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int ii = 0; ii < 16; ++ii) sx[ii] *= KDA ? sf[SF_EL + cs + ii] : egL;
                    tc::tmem_st16(tc::tmem_addr(tm, lq, COL_S + cs), sx);
                }
                tc::tmem_wait_st();
            }
            if (KDA && !last) gates_sum();  // the next chunk's (its loads issued during D1)
            wait_bar(bar_b, phase_b);  // each thread reads the chain's results after its own wait

            // ------ U'^T -> TMEM (tf32); GDN also Ud^T = U'^T diag(e^{gc_L - gc}) for the state
            //        update, as two bf16 terms (Ud = Ud_hi + Ud_lo within 2^-18) packed two per
            //        column: hi in the U'd columns 0..31, lo in 32..63
            {
                const int t0c = C16 * part;  // 16 columns: U'0 (in D6) or U'1 (in D4)
                float v[16];
                if (t0c < 32) tc::tmem_ld16(tc::tmem_addr(tm, lq, COL_D6 + t0c), v);
                else tc::tmem_ld16(tc::tmem_addr(tm, lq, COL_D4 + t0c - 32), v);
                tc::tmem_wait_ld();
                if (!KDA) {
                    float hi[8], lo[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float w0 = v[2 * i] * sf[SF_EGL + t0c + 2 * i];
                        const float w1 = v[2 * i + 1] * sf[SF_EGL + t0c + 2 * i + 1];
                        const __nv_bfloat162 h2 = __floats2bfloat162_rn(w0, w1);
                        const uint32_t hu = *reinterpret_cast<const uint32_t *>(&h2);
                        const __nv_bfloat162 l2 = __floats2bfloat162_rn(w0 - __uint_as_float(hu << 16),
                                                                        w1 - __uint_as_float(hu & 0xFFFF0000u));
                        hi[i] = __uint_as_float(hu);
                        lo[i] = *reinterpret_cast<const float *>(&l2);
                    }
                    tc::tmem_st8(tc::tmem_addr(tm, lq, COL_RUD + t0c / 2), hi);
                    tc::tmem_st8(tc::tmem_addr(tm, lq, COL_RUD + 32 + t0c / 2), lo);
                }
#pragma unroll
                for (int ii = 0; ii < 16; ++ii) v[ii] = tc::to_tf32_operand(v[ii]);
                tc::tmem_st16(tc::tmem_addr(tm, lq, COL_RU + t0c), v);
            }
            tc::tmem_wait_st();
            if (FRONT && !last) cp_async_wait_all();  // next chunk's raw rows
            tc::fence_before_sync();
            __syncthreads();

            // ---------------- D4 = U'^T P^T ; S += Ud^T K (GDN) or U'^T Kdec (KDA)
            if (warp == 0 && tc::elect_one()) {
                tc::fence_after_sync();
                constexpr uint32_t id64 = tc::idesc(128, 64, tc::FMT_TF32);
#pragma unroll
                for (uint32_t kk = 0; kk < 8; ++kk) {
                    const uint64_t bp = tc::sdesc_sw128((sb + SM_P) + (kk >> 2) * 8192u + (kk & 3u) * 32u);
                    tc::mma_tf32_ts(tm + COL_D4, tm + COL_RU + kk * 8, bp, id64, kk > 0);
                }
                tc::mma_commit(bar_b);  // the output MMA: the epilogue may start
                if (KDA) {
                    constexpr uint32_t id128 = tc::idesc(128, 128, tc::FMT_TF32);
#pragma unroll
                    for (uint32_t kk = 0; kk < 8; ++kk) {
                        const uint64_t bk = tc::sdesc_sw128((sb + SM_KDT) + (kk >> 2) * 16384u + (kk & 3u) * 32u);
                        tc::mma_tf32_ts(tm + COL_S, tm + COL_RU + kk * 8, bk, id128, 1);
                    }
                } else {
                    // B = the chunk's K rows [t][c] read MN-major (two 64-channel atoms 16 KB
                    // apart, 8-token groups 1024 bytes apart); A = Ud_hi, then Ud_lo
                    constexpr uint32_t idk = tc::idesc(128, 128, tc::FMT_BF16, false, true);
#pragma unroll
                    for (uint32_t h = 0; h < 2; ++h) {
#pragma unroll
                        for (uint32_t kk = 0; kk < 4; ++kk) {
                            const uint64_t bk = tc::sdesc_sw128_mn((sb + kqo) + kk * 2048u, 128u * 128u, 1024u);
                            tc::mma_bf16_ts(tm + COL_S, tm + COL_RUD + 32 * h + kk * 8, bk, idk, 1);
                        }
                    }
                }
                tc::mma_commit(bar_c);
            }
            pend_c = true;
            // the next chunk's gates, second half: this chunk's beta, gc_L and e^{gc_L} were last
            // read before the barrier above
            if (KDA && !last) gates_carry();
            if (FRONT && !last) {  // next chunk's q, k, v tiles while the tensor core works
                conv_tile_any(a, sm, min(TC_C, len - (ch + 1) * TC_C), pad_qk, warp, lane, kqo_next);
                tc::fence_async_smem();
            }
            wait_bar(bar_b, phase_b);  // each thread reads D4 after its own wait

            // ---------------- o = scale (e^gc (Q H) + P U'): staged as bf16 [t][d] in shared
            //                  memory; written with 16-byte stores (rows < n) in the next chunk.
            //                  In the recurrence-only launch warp 0, held while the tensor core
            //                  takes the state update, hands its 16 tokens (GDN: 8 of them) to
            //                  warp 12 (the same TMEM lane quadrant).
            {
                __nv_bfloat16 *os = reinterpret_cast<__nv_bfloat16 *>(sm + SM_AT);
                auto epi = [&](const int t0c, const int nt) {  // tokens t0c .. t0c + nt - 1 (16 or 8)
                    float vq[16], vp[16];
                    if (nt == 16) {
                        tc::tmem_ld16(tc::tmem_addr(tm, lq, COL_D2 + 64 + t0c), vq);
                        tc::tmem_ld16(tc::tmem_addr(tm, lq, COL_D4 + t0c), vp);
                    } else {
                        tc::tmem_ld8(tc::tmem_addr(tm, lq, COL_D2 + 64 + t0c), vq);
                        tc::tmem_ld8(tc::tmem_addr(tm, lq, COL_D4 + t0c), vp);
                    }
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int ii = 0; ii < 16; ii += 2) {
                        if (ii >= nt) break;
                        const int t = t0c + ii;
                        const float o0 = KDA ? vq[ii] + vp[ii] : fmaf(sf[SF_EG + t], vq[ii], vp[ii]);
                        const float o1 = KDA ? vq[ii + 1] + vp[ii + 1] : fmaf(sf[SF_EG + t + 1], vq[ii + 1], vp[ii + 1]);
                        const __nv_bfloat162 pr = __floats2bfloat162_rn(scale * o0, scale * o1);
                        os[t * O_LD + row] = pr.x;
                        os[(t + 1) * O_LD + row] = pr.y;
                    }
                };
                // GDN: warp 0 keeps 8 of its 16 tokens (warp 12, taking all 16, ended last)
                if (FRONT || warp != 0) epi(C16 * part, 16);
                if (!FRONT && !KDA && warp == 0) epi(0, 8);
                if (!FRONT && warp == 12) epi(KDA ? 0 : 8, KDA ? 16 : 8);
                pend_tok0 = tok0;
                pend_n = n;
            }
            // no barrier here: the staged tile is read (store_o) after the next chunk's first
            // checked barrier, and nothing before that barrier writes what this epilogue reads
        }
        if (!sync_ok(err)) break;
        if (pend_n > 0) {  // the last chunk's output (staged before the barrier above)
            store_o(pend_tok0, pend_n, 0, TC_THREADS / 32);
            pend_n = 0;
        }

        wait_state();
        if (!sync_ok(err)) break;
        // state back: H[c][d] = S[d][c]
#pragma unroll
        for (int g = 0; g < D32 / 16; ++g) {
            float v[16];
            tc::tmem_ld16(tc::tmem_addr(tm, lq, COL_S + D32 * part + g * 16), v);
            tc::tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) hg[(int64_t)(D32 * part + g * 16 + i) * TC_D + row] = v[i];
        }
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
    }

    cp_async_wait_all();
    // a TMA load still in flight after an error lands before the block exits
    if (fly_kq) tc::mbar_wait(bar_kq, par_kq, WAIT_NS);  // by the thread that issued it
    if (fly_v) tc::mbar_wait(bar_v, par_v, WAIT_NS);
    // Every MMA of this block has completed before its TMEM is released, also after a wait gave
    // up: the issuing lane commits once more (a commit tracks all earlier MMAs of its thread)
    // and waits for that commit with the full limit.
    if (warp == 0) {
        __syncwarp();
        if (tc::elect_one()) {
            tc::mma_commit(bar_e);
            if (!tc::mbar_wait(bar_e, 0, WAIT_NS)) *err = 1;
        }
        __syncwarp();
    }
    tc::fence_before_sync();
    __syncthreads();
    if (*err && tid == 0) raise_status(a.status, LA_DEV_TIMEOUT);
    if (warp == 0) tc::tmem_dealloc(tm, TMEM_COLS);
}

// Orders the streams by decreasing length (stable) so that the longest units start first,
// and zeroes the unit counter (and the conv-state reader counts). One thread per stream ranks
// it against all B lengths, read from shared memory (each block stages them first) when B fits,
// else from cu_seqlens; blocks of ORDER_THREADS streams run side by side. Equal lengths (the
// batched call) keep their order.
constexpr int kOrderStaged = 8192;
constexpr int ORDER_THREADS = 256;
__global__ void __launch_bounds__(ORDER_THREADS)
order_streams_kernel(const int32_t *cu, int B, int T_each, int32_t *perm, int *counter,
                     int *conv_readers, int n_readers) {
    __shared__ int lens[kOrderStaged];
    if (blockIdx.x == 0) {
        for (int i = threadIdx.x; i < n_readers; i += blockDim.x) conv_readers[i] = 0;
        if (threadIdx.x == 0) *counter = 0;
    }
    const int s = blockIdx.x * ORDER_THREADS + threadIdx.x;
    if (!cu) {
        if (s < B) perm[s] = s;
        return;
    }
    const bool staged = B <= kOrderStaged;
    if (staged)
        for (int o = threadIdx.x; o < B; o += blockDim.x) lens[o] = cu[o + 1] - cu[o];
    __syncthreads();
    if (s >= B) return;
    const int ls = staged ? lens[s] : cu[s + 1] - cu[s];
    int rank = 0;
    for (int o = 0; o < B; ++o) {
        const int lo = staged ? lens[o] : cu[o + 1] - cu[o];
        rank += (lo > ls) || (lo == ls && o < s);
    }
    perm[rank] = s;
}

int sm_count() {
    static int cached[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return 148;
    if (!cached[dev]) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cached[dev] = n > 0 ? n : 148;
    }
    return cached[dev];
}

}  // namespace

// Workspace: stream order [B] | conv-state reader counts [B * Hk] | 256 B holding the unit
// counter (the last 256 bytes).
static size_t order_bytes(int B) { return (size_t)((B + 64 + 63) / 64) * 64 * sizeof(int32_t); }
static size_t readers_bytes(int B, int Hk) {
    return (size_t)(((int64_t)B * Hk + 63) / 64) * 64 * sizeof(int32_t);
}
size_t chunk_tc_workspace_bytes(int B, int Hk) {
    return order_bytes(B) + readers_bytes(B, Hk) + 256;
}

// ---- Fixed, library-owned scratch for callers that cannot hand the library a workspace.
// It lives in this file's device memory image: every GPU that loads the library holds it until
// the process exits, and every call through it shares it (the previous call's contents stay;
// the stream-order kernel rewrites the order and zeroes the counter at the start of each call).
constexpr int kStaticScratchStreams = 4096;
constexpr size_t kStaticScratchBytes =
    (size_t)((kStaticScratchStreams + 64 + 63) / 64) * 64 * sizeof(int32_t) + 256;
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

int chunk_tc_static_scratch_max_streams() { return kStaticScratchStreams; }

// Device address of the scratch array for the current device, looked up once per device (with
// that device current). Host code may not pass the array's name to a kernel: on the host it is
// only a stand-in symbol, not a device address.
cudaError_t chunk_tc_static_scratch(void **ptr, size_t *bytes) {
    constexpr int kMaxDev = 64;
    static void *cached[kMaxDev] = {nullptr};
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!cached[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess) return e;
        cached[dev] = p;
    }
    *ptr = cached[dev];
    *bytes = kStaticScratchBytes;
    return cudaSuccess;
}

bool chunk_tc_supported(const RecArgs &a) {
    return a.dtype == LA_BF16 && a.dk == TC_D && a.dv == TC_D;
}

cudaError_t launch_chunk_tc(const RecArgs &a, cudaStream_t st) {
    unsigned char *ws = reinterpret_cast<unsigned char *>(a.workspace);
    int32_t *perm = reinterpret_cast<int32_t *>(ws);
    int *readers = a.front ? reinterpret_cast<int *>(ws + order_bytes(a.B)) : nullptr;
    int *counter = reinterpret_cast<int *>(ws + chunk_tc_workspace_bytes(a.B, a.front ? a.Hk : 0) - 256);
    order_streams_kernel<<<(a.B + ORDER_THREADS - 1) / ORDER_THREADS, ORDER_THREADS, 0, st>>>(
        a.cu, a.B, a.T_each, perm, counter, readers, a.front ? a.B * a.Hk : 0);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    TcParams P;
    P.a = a;
    P.perm = perm;
    P.counter = counter;
    P.conv_readers = readers;
    P.num_units = a.B * a.Hv;
    // K, Q, V by TMA for the plain calls (2-D maps over [tokens][heads x 128], 64 x 64 boxes,
    // 128-byte swizzle); the async-copy path stays for the fused front end and the segmented
    // scan, and in case a map cannot be encoded
    P.tma = !a.front && !a.use_alt &&
            make_map_bf16_2d(&P.map_k, a.k, a.total, (int64_t)a.Hk * TC_D, a.k_stride, 64, 64, true) &&
            make_map_bf16_2d(&P.map_q, a.q, a.total, (int64_t)a.Hk * TC_D, a.q_stride, 64, 64, true) &&
            make_map_bf16_2d(&P.map_v, a.v, a.total, (int64_t)a.Hv * TC_D, a.v_stride, 64, 64, true);
    const int grid = min(P.num_units, sm_count());
    auto kern = a.kda ? (a.front ? chunk_tc_kernel<true, true> : chunk_tc_kernel<true, false>)
                      : (a.front ? chunk_tc_kernel<false, true> : chunk_tc_kernel<false, false>);
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)TC_SMEM);
    if (e != cudaSuccess) return e;
    kern<<<grid, TC_THREADS, TC_SMEM, st>>>(P);
    return cudaGetLastError();
}

}  // namespace la
