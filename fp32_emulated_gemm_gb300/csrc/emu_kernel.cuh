// emu_kernel.cuh -- the emulated-SGEMM kernel for sm_103a.
//
// Method: blog "Unlocking Tensor Core performance for machine-learning
// interatomic potentials", section "How Tensor Core FP32 bridges the hardware
// gap": split each FP32 operand into low-precision components (BF16x9: three
// BF16 components, Fig. 1; TF32x3: hi and lo TF32 components, Fig. 2), let the
// tensor cores evaluate the selected component products, and accumulate in
// FP32 (BF16x9: along five anti-diagonal bands; TF32x3: Eq. 1, lo*lo dropped).
//
// One persistent kernel, warp-specialised, one CTA per SM:
//   warp 0      TMA producer: FP32 tiles of op(A) and op(B), 32 k-values per
//               stage, into a ring of shared-memory stages (zero fill beyond
//               the matrix edges).
//   warp 1      MMA issuer: owns TMEM; for every stage issues the component
//               products (18 BF16 MMAs of K=16, or 12 TF32 MMAs of K=8) into
//               a fresh TMEM accumulator, smallest band first.
//   warps 2-9   split warps: read the FP32 stage and write the components in
//               the tensor cores' K-major swizzled layout (transposing when
//               the operand is MN-major in memory).
//   warps 10-17 epilogue: after every stage, read the stage's partial sum
//               from TMEM and add it into FP32 registers (round to nearest),
//               then apply alpha, beta and the bias and store the tile.
//
// Promoting each 32-k partial out of TMEM keeps the tensor core's truncating
// block additions confined to short chains that start from zero, so the
// result is as accurate as the blog's claim requires (BF16x9 at least as
// accurate as native FP32 against an FP64 reference, "Limitations and
// decision criteria").
#pragma once

#include <cstdint>
#include <cuda.h>

#include "ptx.cuh"

namespace emu {

enum Mode : int { MODE_BF16X9 = 0, MODE_TF32X3 = 1 };

constexpr int BM = 128;  // rows of op(A) per tile (TMEM lanes)
constexpr int BN = 128;  // columns of op(B) per tile (TMEM columns per accumulator)
constexpr int BK = 32;   // k-values per pipeline stage
constexpr int NUM_THREADS = 576;
constexpr int WARP_PRODUCER = 0;
constexpr int WARP_MMA = 1;
constexpr int WARP_SPLIT0 = 2;
constexpr int NUM_SPLIT_WARPS = 8;
constexpr int WARP_EPI0 = WARP_SPLIT0 + NUM_SPLIT_WARPS;  // 10
constexpr int NUM_EPI_WARPS = 8;
constexpr uint32_t TMEM_COLS = 2 * BN;  // two accumulators, double-buffered

// FP32 stage: op(A) tile then op(B) tile, 128 rows x 128 bytes each.
constexpr uint32_t FP32_TILE_BYTES = 128 * BK * 4;       // 16 KB
constexpr uint32_t FP32_STAGE_BYTES = 2 * FP32_TILE_BYTES;  // 32 KB

template <int MODE> struct Cfg;
template <> struct Cfg<MODE_BF16X9> {
    static constexpr int NCOMP = 3;                  // components per operand
    static constexpr uint32_t ROW_BYTES = BK * 2;    // 64: one BF16 row of a stage
    static constexpr uint32_t COMP_TILE = 128 * ROW_BYTES;          // 8 KB
    static constexpr uint32_t SLICE_STAGE = 2 * NCOMP * COMP_TILE;  // 48 KB
    static constexpr int NF = 3;                     // FP32 stages
    static constexpr int NS = 2;                     // component stages
    static constexpr uint32_t IDESC = make_idesc(1, BM, BN);
};
template <> struct Cfg<MODE_TF32X3> {
    static constexpr int NCOMP = 2;
    static constexpr uint32_t ROW_BYTES = BK * 4;    // 128
    static constexpr uint32_t COMP_TILE = 128 * ROW_BYTES;          // 16 KB
    static constexpr uint32_t SLICE_STAGE = 2 * NCOMP * COMP_TILE;  // 64 KB
    static constexpr int NF = 2;
    static constexpr int NS = 2;
    static constexpr uint32_t IDESC = make_idesc(2, BM, BN);
};

template <int MODE>
constexpr uint32_t smem_bytes() {
    return 1024 /* alignment slack */ + Cfg<MODE>::NF * FP32_STAGE_BYTES +
           Cfg<MODE>::NS * Cfg<MODE>::SLICE_STAGE + 1024 /* barriers and flags */;
}

struct Params {
    CUtensorMap tmA;  // FP32 op(A): K-major box {32, 128} or MN-major box {32, 32}
    CUtensorMap tmB;  // FP32 op(B): same
    int M, N, K;
    int a_mn_major, b_mn_major;
    int tiles_m, tiles_n, num_tiles, k_stages;
    float alpha, beta;
    const float* c_old;  // read only when beta != 0
    float* c;
    long long ldc;
    const float* bias;   // may be null
    unsigned long long wait_budget_ns;
};

// ----------------------------------------------------------- the splits ----
// Byte offset of element (row, k) of an FP32 tile stored K-major with
// 128-byte rows and the 128-byte swizzle (16-byte chunk index XOR row % 8).
__device__ __forceinline__ uint32_t off_f32_kmajor(uint32_t row, uint32_t k) {
    return row * 128u + ((((k >> 2) ^ row) & 7u) << 4) + ((k & 3u) << 2);
}
// Same for an MN-major FP32 tile: four 32-wide MN blocks of 32 k-rows each.
__device__ __forceinline__ uint32_t off_f32_mnmajor(uint32_t mn, uint32_t k) {
    return (mn >> 5) * 4096u + k * 128u + (((((mn & 31u) >> 2) ^ k) & 7u) << 4) + ((mn & 3u) << 2);
}
// Offset of the 16-byte chunk holding k-values [8g, 8g+8) of BF16 row `row`
// in a K-major tile with 64-byte rows and the 64-byte swizzle (chunk index
// XOR (row / 2) % 4).
__device__ __forceinline__ uint32_t off_bf16_chunk(uint32_t row, uint32_t g) {
    return row * 64u + (((g ^ (row >> 1)) & 3u) << 4);
}
// Offset of the 16-byte chunk holding k-values [4c, 4c+4) of an FP32/TF32
// row in a K-major tile with 128-byte rows and the 128-byte swizzle.
__device__ __forceinline__ uint32_t off_f32_chunk(uint32_t row, uint32_t c) {
    return row * 128u + (((c ^ row) & 7u) << 4);
}

__device__ __forceinline__ uint32_t pack_hi16(uint32_t lo_elem, uint32_t hi_elem) {
    return __byte_perm(lo_elem, hi_elem, 0x7632);
}

// BF16x9 split of 8 values into three BF16 components in natural magnitude:
// c0 = x truncated to BF16, c1 = (x - c0) truncated to BF16, c2 = the rest.
// Both subtractions are exact.  Component i equals the blog's scaled
// component times 2^-8i, so every product c_i * c_j already carries its band
// scale 2^-8(i+j) and all nine products can share one FP32 accumulator.
__device__ __forceinline__ void split_bf16x9_8(const float (&x)[8], uint4& s0, uint4& s1, uint4& s2) {
    uint32_t w0[8], w1[8], w2[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t u = __float_as_uint(x[i]);
        const float r1 = __fsub_rn(x[i], __uint_as_float(u & 0xFFFF0000u));
        const uint32_t v = __float_as_uint(r1);
        const float r2 = __fsub_rn(r1, __uint_as_float(v & 0xFFFF0000u));
        w0[i] = u;
        w1[i] = v;
        w2[i] = __float_as_uint(r2);
    }
    s0 = make_uint4(pack_hi16(w0[0], w0[1]), pack_hi16(w0[2], w0[3]), pack_hi16(w0[4], w0[5]), pack_hi16(w0[6], w0[7]));
    s1 = make_uint4(pack_hi16(w1[0], w1[1]), pack_hi16(w1[2], w1[3]), pack_hi16(w1[4], w1[5]), pack_hi16(w1[6], w1[7]));
    s2 = make_uint4(pack_hi16(w2[0], w2[1]), pack_hi16(w2[2], w2[3]), pack_hi16(w2[4], w2[5]), pack_hi16(w2[6], w2[7]));
}

// Round an FP32 word to the nearest TF32 number, ties to even (Inf and NaN
// unchanged).
__device__ __forceinline__ uint32_t tf32_rn_bits(uint32_t u) {
    const uint32_t r = (u + 0x0FFFu + ((u >> 13) & 1u)) & 0xFFFFE000u;
    return ((u & 0x7F800000u) == 0x7F800000u) ? u : r;
}

// TF32x3 split of one value: hi = nearest TF32, lo = nearest TF32 of x - hi.
__device__ __forceinline__ void split_tf32x3_1(float x, uint32_t& hi, uint32_t& lo) {
    hi = tf32_rn_bits(__float_as_uint(x));
    lo = tf32_rn_bits(__float_as_uint(__fsub_rn(x, __uint_as_float(hi))));
}

// Split one operand tile (128 rows x 32 k) of a stage.  `src` is the FP32
// tile, `dst` the first component tile (components follow at COMP_TILE
// strides).  `t` is the thread's index among the 256 split threads.
template <int MODE>
__device__ __forceinline__ void split_operand(const uint8_t* src, uint8_t* dst, bool mn_major, uint32_t t) {
    using C = Cfg<MODE>;
    const uint32_t lane = t & 31u, warp = t >> 5;
    if (!mn_major) {
        // item = (row, 8-k group): lanes cover 8 rows x 4 groups per warp
#pragma unroll
        for (int it = 0; it < 2; ++it) {
            const uint32_t item = it * 256u + warp * 32u + lane;
            const uint32_t row = (item >> 5) * 8u + ((item & 31u) >> 2);
            const uint32_t g = item & 3u;
            const float4 lo4 = *reinterpret_cast<const float4*>(src + off_f32_chunk(row, 2 * g));
            const float4 hi4 = *reinterpret_cast<const float4*>(src + off_f32_chunk(row, 2 * g + 1));
            const float x[8] = {lo4.x, lo4.y, lo4.z, lo4.w, hi4.x, hi4.y, hi4.z, hi4.w};
            if constexpr (MODE == MODE_BF16X9) {
                uint4 s0, s1, s2;
                split_bf16x9_8(x, s0, s1, s2);
                const uint32_t o = off_bf16_chunk(row, g);
                *reinterpret_cast<uint4*>(dst + o) = s0;
                *reinterpret_cast<uint4*>(dst + C::COMP_TILE + o) = s1;
                *reinterpret_cast<uint4*>(dst + 2 * C::COMP_TILE + o) = s2;
            } else {
                uint32_t h[8], l[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) split_tf32x3_1(x[i], h[i], l[i]);
                const uint32_t o0 = off_f32_chunk(row, 2 * g), o1 = off_f32_chunk(row, 2 * g + 1);
                *reinterpret_cast<uint4*>(dst + o0) = make_uint4(h[0], h[1], h[2], h[3]);
                *reinterpret_cast<uint4*>(dst + o1) = make_uint4(h[4], h[5], h[6], h[7]);
                *reinterpret_cast<uint4*>(dst + C::COMP_TILE + o0) = make_uint4(l[0], l[1], l[2], l[3]);
                *reinterpret_cast<uint4*>(dst + C::COMP_TILE + o1) = make_uint4(l[4], l[5], l[6], l[7]);
            }
        }
    } else {
        // item = (mn, 8-k group): 32 consecutive mn per warp, so that both the
        // column reads of the MN-major tile and the row writes are conflict-free
#pragma unroll
        for (int it = 0; it < 2; ++it) {
            const uint32_t item = it * 256u + warp * 32u + lane;
            const uint32_t mn = item & 127u;
            const uint32_t g = item >> 7;
            float x[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                x[i] = *reinterpret_cast<const float*>(src + off_f32_mnmajor(mn, 8 * g + i));
            if constexpr (MODE == MODE_BF16X9) {
                uint4 s0, s1, s2;
                split_bf16x9_8(x, s0, s1, s2);
                const uint32_t o = off_bf16_chunk(mn, g);
                *reinterpret_cast<uint4*>(dst + o) = s0;
                *reinterpret_cast<uint4*>(dst + C::COMP_TILE + o) = s1;
                *reinterpret_cast<uint4*>(dst + 2 * C::COMP_TILE + o) = s2;
            } else {
                uint32_t h[8], l[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) split_tf32x3_1(x[i], h[i], l[i]);
                const uint32_t o0 = off_f32_chunk(mn, 2 * g), o1 = off_f32_chunk(mn, 2 * g + 1);
                *reinterpret_cast<uint4*>(dst + o0) = make_uint4(h[0], h[1], h[2], h[3]);
                *reinterpret_cast<uint4*>(dst + o1) = make_uint4(h[4], h[5], h[6], h[7]);
                *reinterpret_cast<uint4*>(dst + C::COMP_TILE + o0) = make_uint4(l[0], l[1], l[2], l[3]);
                *reinterpret_cast<uint4*>(dst + C::COMP_TILE + o1) = make_uint4(l[4], l[5], l[6], l[7]);
            }
        }
    }
}

// Issue the tensor-core products of one stage into TMEM accumulator `d`,
// starting from zero.  BF16x9: bands 4, 3, 2, 1, 0 (i + j), each over the two
// K=16 steps of the stage.  TF32x3: lo*hi, hi*lo, hi*hi over four K=8 steps.
template <int MODE>
__device__ __forceinline__ void issue_stage_mmas(uint32_t d, uint32_t a_base, uint32_t b_base) {
    using C = Cfg<MODE>;
    uint32_t acc = 0;
    if constexpr (MODE == MODE_BF16X9) {
        // (i, j) pairs, smallest band first
        constexpr int PI[9] = {2, 1, 2, 0, 1, 2, 0, 1, 0};
        constexpr int PJ[9] = {2, 2, 1, 2, 1, 0, 1, 0, 0};
#pragma unroll
        for (int p = 0; p < 9; ++p) {
#pragma unroll
            for (int ks = 0; ks < BK / 16; ++ks) {
                const uint64_t ad = sdesc_kmajor(a_base + PI[p] * C::COMP_TILE + ks * 32, C::ROW_BYTES);
                const uint64_t bd = sdesc_kmajor(b_base + PJ[p] * C::COMP_TILE + ks * 32, C::ROW_BYTES);
                mma_bf16(d, ad, bd, C::IDESC, acc);
                acc = 1;
            }
        }
    } else {
        constexpr int PI[3] = {1, 0, 0};  // 0 = hi, 1 = lo
        constexpr int PJ[3] = {0, 1, 0};
#pragma unroll
        for (int p = 0; p < 3; ++p) {
#pragma unroll
            for (int ks = 0; ks < BK / 8; ++ks) {
                const uint64_t ad = sdesc_kmajor(a_base + PI[p] * C::COMP_TILE + ks * 32, C::ROW_BYTES);
                const uint64_t bd = sdesc_kmajor(b_base + PJ[p] * C::COMP_TILE + ks * 32, C::ROW_BYTES);
                mma_tf32(d, ad, bd, C::IDESC, acc);
                acc = 1;
            }
        }
    }
}

template <int MODE>
__global__ void __launch_bounds__(NUM_THREADS, 1) emu_gemm_kernel(const __grid_constant__ Params p) {
    using C = Cfg<MODE>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* fp32_ring = smem;
    uint8_t* slice_ring = smem + C::NF * FP32_STAGE_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(slice_ring + C::NS * C::SLICE_STAGE);
    uint64_t* fp32_full = bars;
    uint64_t* fp32_empty = fp32_full + C::NF;
    uint64_t* slice_full = fp32_empty + C::NF;
    uint64_t* slice_empty = slice_full + C::NS;
    uint64_t* acc_full = slice_empty + C::NS;
    uint64_t* acc_empty = acc_full + 2;
    uint64_t* drain = acc_empty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31u;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::NF; ++s) { mbar_init(&fp32_full[s], 1); mbar_init(&fp32_empty[s], NUM_SPLIT_WARPS); }
        for (int s = 0; s < C::NS; ++s) { mbar_init(&slice_full[s], NUM_SPLIT_WARPS); mbar_init(&slice_empty[s], 1); }
        for (int b = 0; b < 2; ++b) { mbar_init(&acc_full[b], 1); mbar_init(&acc_empty[b], NUM_EPI_WARPS); }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == WARP_PRODUCER && lane == 0) {
        tma_prefetch_desc(&p.tmA);
        tma_prefetch_desc(&p.tmB);
    }
    if (warp == WARP_MMA) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const uint64_t budget = p.wait_budget_ns;

    if (warp == WARP_PRODUCER) {
        // ------------------------------------------------------ producer ----
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            uint32_t issued_mask = 0;  // stages holding a load of the current lap
            uint32_t issued_parity = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
                const int m0 = (tile / p.tiles_n) * BM, n0 = (tile % p.tiles_n) * BN;
                for (int ks = 0; ks < p.k_stages; ++ks) {
                    if (!mbar_wait(&fp32_empty[s], ph ^ 1u, abort_flag, budget, 1)) { ok = false; break; }
                    uint64_t* full = &fp32_full[s];
                    mbar_arrive_expect_tx(full, FP32_STAGE_BYTES);
                    uint8_t* dA = fp32_ring + s * FP32_STAGE_BYTES;
                    uint8_t* dB = dA + FP32_TILE_BYTES;
                    const int k0 = ks * BK;
                    if (!p.a_mn_major) tma_load_2d(dA, &p.tmA, full, k0, m0);
                    else for (int j = 0; j < 4; ++j) tma_load_2d(dA + j * 4096, &p.tmA, full, m0 + 32 * j, k0);
                    if (!p.b_mn_major) tma_load_2d(dB, &p.tmB, full, k0, n0);
                    else for (int j = 0; j < 4; ++j) tma_load_2d(dB + j * 4096, &p.tmB, full, n0 + 32 * j, k0);
                    issued_mask |= 1u << s;
                    issued_parity = (issued_parity & ~(1u << s)) | (ph << s);
                    if (++s == C::NF) { s = 0; ph ^= 1u; }
                }
            }
            if (!ok) {
                // give every load already in flight time to land before the CTA exits
                for (int t = 0; t < C::NF; ++t)
                    if (issued_mask & (1u << t)) {
                        volatile int never = 0;
                        mbar_wait(&fp32_full[t], (issued_parity >> t) & 1u, &never, 50000000ull, 1);
                    }
            }
        }
        __syncwarp();
    } else if (warp == WARP_MMA) {
        // ---------------------------------------------------- MMA issuer ----
        if (lane == 0) {
            int s = 0, b = 0;
            uint32_t ph = 0, bph = 0;
            bool ok = true, issued = false;
            const uint32_t slice_base = smem_u32(slice_ring);
            for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
                for (int ks = 0; ks < p.k_stages; ++ks) {
                    if (!mbar_wait(&acc_empty[b], bph ^ 1u, abort_flag, budget, 2)) { ok = false; break; }
                    if (!mbar_wait(&slice_full[s], ph, abort_flag, budget, 2)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a_base = slice_base + s * C::SLICE_STAGE;
                    const uint32_t b_base = a_base + C::NCOMP * C::COMP_TILE;
                    issue_stage_mmas<MODE>(tmem_base + b * BN, a_base, b_base);
                    issued = true;
                    mma_commit(&slice_empty[s]);
                    mma_commit(&acc_full[b]);
                    if (++s == C::NS) { s = 0; ph ^= 1u; }
                    if (++b == 2) { b = 0; bph ^= 1u; }
                }
            }
            if (!ok && issued) {
                // let the products in flight finish before TMEM is released
                mma_commit(drain);
                volatile int never = 0;
                mbar_wait(drain, 0, &never, 50000000ull, 2);
            }
        }
        __syncwarp();
    } else if (warp < WARP_EPI0) {
        // ---------------------------------------------------- split warps ---
        const uint32_t t = threadIdx.x - WARP_SPLIT0 * 32;
        int fs = 0, ss = 0;
        uint32_t fph = 0, sph = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
            for (int ks = 0; ks < p.k_stages; ++ks) {
                if (!mbar_wait_warp(&fp32_full[fs], fph, abort_flag, budget, 3)) { ok = false; break; }
                if (!mbar_wait_warp(&slice_empty[ss], sph ^ 1u, abort_flag, budget, 3)) { ok = false; break; }
                const uint8_t* src = fp32_ring + fs * FP32_STAGE_BYTES;
                uint8_t* dst = slice_ring + ss * C::SLICE_STAGE;
                split_operand<MODE>(src, dst, p.a_mn_major != 0, t);
                split_operand<MODE>(src + FP32_TILE_BYTES, dst + C::NCOMP * C::COMP_TILE, p.b_mn_major != 0, t);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&fp32_empty[fs]);
                    mbar_arrive(&slice_full[ss]);
                }
                if (++fs == C::NF) { fs = 0; fph ^= 1u; }
                if (++ss == C::NS) { ss = 0; sph ^= 1u; }
            }
        }
    } else {
        // ------------------------------------------------------- epilogue ---
        const uint32_t e = warp - WARP_EPI0;
        const uint32_t quarter = warp & 3u;      // TMEM lanes this warp may read
        const uint32_t half = e >> 2;            // which 64 columns of the tile
        const uint32_t lane_base = (quarter * 32u) << 16;
        int b = 0;
        uint32_t bph = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
            float acc[64];
#pragma unroll
            for (int i = 0; i < 64; ++i) acc[i] = 0.0f;
            for (int ks = 0; ks < p.k_stages; ++ks) {
                if (!mbar_wait_warp(&acc_full[b], bph, abort_flag, budget, 4)) { ok = false; break; }
                tc_fence_after();
                const uint32_t col = tmem_base + b * BN + half * 64;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    float v[16];
                    tmem_ld16(col + lane_base + c * 16, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 16; ++i) acc[c * 16 + i] = __fadd_rn(acc[c * 16 + i], v[i]);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&acc_empty[b]);
                if (++b == 2) { b = 0; bph ^= 1u; }
            }
            if (!ok) break;
            // C = alpha * acc + beta * C_old + bias
            const int m0 = (tile / p.tiles_n) * BM, n0 = (tile % p.tiles_n) * BN;
            const int row = m0 + static_cast<int>(quarter * 32u + lane);
            const int col0 = n0 + static_cast<int>(half * 64u);
            if (row < p.M) {
                float* crow = p.c + static_cast<long long>(row) * p.ldc;
                const float* orow = p.c_old + static_cast<long long>(row) * p.ldc;
#pragma unroll
                for (int j = 0; j < 64; j += 4) {
                    const int col = col0 + j;
                    if (col + 3 < p.N) {
                        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
                        if (p.beta != 0.0f) o = *reinterpret_cast<const float4*>(orow + col);
                        float4 bb = make_float4(0.f, 0.f, 0.f, 0.f);
                        if (p.bias) bb = *reinterpret_cast<const float4*>(p.bias + col);
                        float4 r;
                        r.x = __fadd_rn(__fmaf_rn(p.alpha, acc[j + 0], p.beta != 0.0f ? __fmul_rn(p.beta, o.x) : 0.0f), bb.x);
                        r.y = __fadd_rn(__fmaf_rn(p.alpha, acc[j + 1], p.beta != 0.0f ? __fmul_rn(p.beta, o.y) : 0.0f), bb.y);
                        r.z = __fadd_rn(__fmaf_rn(p.alpha, acc[j + 2], p.beta != 0.0f ? __fmul_rn(p.beta, o.z) : 0.0f), bb.z);
                        r.w = __fadd_rn(__fmaf_rn(p.alpha, acc[j + 3], p.beta != 0.0f ? __fmul_rn(p.beta, o.w) : 0.0f), bb.w);
                        *reinterpret_cast<float4*>(crow + col) = r;
                    } else {
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            if (col + q < p.N) {
                                const float bc = p.beta != 0.0f ? __fmul_rn(p.beta, orow[col + q]) : 0.0f;
                                const float bi = p.bias ? p.bias[col + q] : 0.0f;
                                crow[col + q] = __fadd_rn(__fmaf_rn(p.alpha, acc[j + q], bc), bi);
                            }
                        }
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == WARP_MMA) tmem_dealloc(tmem_base, TMEM_COLS);
}

}  // namespace emu
