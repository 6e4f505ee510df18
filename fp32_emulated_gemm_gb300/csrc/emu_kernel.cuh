// emu_kernel.cuh -- the emulated-SGEMM kernel for sm_103a.
//
// Method: blog "Unlocking Tensor Core performance for machine-learning
// interatomic potentials", section "How Tensor Core FP32 bridges the hardware
// gap": split each FP32 operand into low-precision components (BF16x9: three
// BF16 components, Fig. 1; TF32x3: hi and lo TF32 components, Fig. 2), let the
// tensor cores evaluate the selected component products, and accumulate in
// FP32 (BF16x9: along five anti-diagonal bands; TF32x3: Eq. 1, lo*lo dropped).
//
// One persistent kernel on CTA pairs (clusters of 2, one CTA per SM).  A pair
// computes a 256 x TN tile of C (TN = 256 or 128) with 2-SM tensor-core MMAs
// (cta_group::2): CTA r of the pair holds rows [128r, 128r+128) of the
// tile's op(A) block and rows [r TN/2, (r+1) TN/2) of its op(B)^T block; each
// SM's tensor core reads its own A half and both B halves, and writes its
// 128 x TN half of the accumulator to its own TMEM.  Per CTA (16 warps):
//   warp 0      TMA producer: FP32 tiles (128 x 32 of op(A), TN/2 x 32 of
//               op(B)) into a ring of shared-memory stages, zero fill beyond
//               the matrix edges.
//   warp 1      TMEM owner; in the leader CTA also the MMA issuer: for every
//               32-k stage it issues the component products (18 BF16 MMAs of
//               K=16, or 12 TF32 MMAs of K=8) into a fresh TMEM accumulator,
//               smallest band first.
//   warps 2-7   split warps: read the FP32 stage and write the components in
//               the tensor cores' K-major swizzled layout (transposing when
//               the operand is MN-major in memory).
//   warps 8-15  epilogue: after every stage, read the stage's partial sums
//               from TMEM and add them into FP32 registers (round to
//               nearest); at the end apply alpha, beta and the bias and store.
//
// Promoting each 32-k partial out of TMEM confines the tensor core's
// truncating block additions to short chains that start from zero, so the
// result is at least as accurate as native FP32 against an FP64 reference,
// as the blog reports for BF16x9 ("Limitations and decision criteria").
//
// Split-K: when there are too few tiles to fill the GPU, a tile's k-range is
// cut into S pieces processed by different pairs at the same time.  The
// pieces reduce-scatter through a workspace: each publishes the parts of its
// partial tile that the others own, and sums and stores its own part, adding
// the S partials in a fixed order (the owner's first, then the others by
// piece index) -- the result does not depend on timing.  The pieces count
// their arrivals on epoch-tagged counters (one new epoch per launch), so no
// count left by an earlier launch can be taken for this one's.
//
// Chained plans (more tiles than pairs, not a whole number of waves): the
// tiles' k-stages, taken tile by tile, are cut into one contiguous run per
// pair of equal length (to one stage), so every pair has the same work.  A
// run boundary that falls inside a tile cuts it in two pieces on
// neighbouring pairs: the pair whose run starts there takes the tile's low
// k-stages first and publishes its running FP32 sum; the pair whose run ends
// there takes the high k-stages last and starts its running sum from the
// published one.  The sum over stages is then the same sequence of roundings
// as in an uncut tile, so chained plans give the unsplit result bit for bit.
#pragma once

#include <cstdint>
#include <cuda.h>

#include "ptx.cuh"

namespace emu {

// BF16x9 and TF32x3 are the method; BF16x6 (bands 0-2) and one-pass TF32
// (hi*hi) are the faster, less accurate comparators.
enum Mode : int { MODE_BF16X9 = 0, MODE_TF32X3 = 1, MODE_TF32X1 = 2, MODE_BF16X6 = 3 };

constexpr int TILE_M = 256;       // rows of a pair tile (128 per CTA)
constexpr int HALF = 128;         // rows of op(A) held by one CTA (= TMEM lanes)
constexpr int BK = 32;            // k-values per pipeline stage
constexpr int NUM_THREADS = 512;
constexpr int WARP_PRODUCER = 0;
constexpr int WARP_MMA = 1;
constexpr int WARP_SPLIT0 = 2;
constexpr int NUM_SPLIT_WARPS = 6;
constexpr int NUM_SPLIT_THREADS = NUM_SPLIT_WARPS * 32;
constexpr int WARP_EPI0 = 8;
constexpr int NUM_EPI_WARPS = 8;
constexpr uint32_t TMEM_COLS = 512;         // all of TMEM: 512 / TN accumulators of TN columns
constexpr int kMaxChainPairs = 160;         // CTA pairs a chained plan can use
constexpr uint32_t EPI_BARRIER = 1;         // named barrier of the 256 epilogue threads
constexpr uint32_t SPLIT_BARRIER = 2;       // named barrier of the split threads

// FP32 op(A) half-tile of one CTA and stage (its op(B) part follows it).
constexpr uint32_t FP32_TILE_BYTES = HALF * BK * 4;           // 16 KB

// Per mode: components per operand, their row geometry, the MMA kind and
// the (i, j) component products of a stage, smallest first (for BF16: band
// i + j descending; for TF32: 0 = hi, 1 = lo).  COMP_TILE is one component
// of the op(A) half-tile (128 rows).
template <int MODE> struct Cfg;
struct CfgBF16 {
    static constexpr bool TF32 = false;
    static constexpr int NCOMP = 3;                  // components per operand
    static constexpr uint32_t ROW_BYTES = BK * 2;    // 64: one BF16 row of a stage
    static constexpr uint32_t COMP_TILE = HALF * ROW_BYTES;         // 8 KB
    static constexpr int KIND = 1;                   // instruction-descriptor operand format
    static constexpr int KSTEP = 16;                 // k per BF16 MMA
};
struct CfgTF32 {
    static constexpr bool TF32 = true;
    static constexpr uint32_t ROW_BYTES = BK * 4;    // 128
    static constexpr uint32_t COMP_TILE = HALF * ROW_BYTES;         // 16 KB
    static constexpr int KIND = 2;
    static constexpr int KSTEP = 8;                  // k per TF32 MMA
};
template <> struct Cfg<MODE_BF16X9> : CfgBF16 {
    static constexpr int NPROD = 9;
    __host__ __device__ static constexpr int pi(int p) { constexpr int v[9] = {2, 1, 2, 0, 1, 2, 0, 1, 0}; return v[p]; }
    __host__ __device__ static constexpr int pj(int p) { constexpr int v[9] = {2, 2, 1, 2, 1, 0, 1, 0, 0}; return v[p]; }
};
template <> struct Cfg<MODE_BF16X6> : CfgBF16 {
    static constexpr int NPROD = 6;
    __host__ __device__ static constexpr int pi(int p) { constexpr int v[6] = {0, 1, 2, 0, 1, 0}; return v[p]; }
    __host__ __device__ static constexpr int pj(int p) { constexpr int v[6] = {2, 1, 0, 1, 0, 0}; return v[p]; }
};
template <> struct Cfg<MODE_TF32X3> : CfgTF32 {
    static constexpr int NCOMP = 2;
    static constexpr int NPROD = 3;
    __host__ __device__ static constexpr int pi(int p) { constexpr int v[3] = {1, 0, 0}; return v[p]; }
    __host__ __device__ static constexpr int pj(int p) { constexpr int v[3] = {0, 1, 0}; return v[p]; }
};
template <> struct Cfg<MODE_TF32X1> : CfgTF32 {
    static constexpr int NCOMP = 1;
    static constexpr int NPROD = 1;
    __host__ __device__ static constexpr int pi(int) { return 0; }
    __host__ __device__ static constexpr int pj(int) { return 0; }
};

// Tile width and pipeline shape, chosen per launch.  TN is the pair tile's
// width (the MMA's N; each CTA holds TN / 2 rows of op(B)^T); TMEM holds
// 512 / TN accumulators of TN columns, so the MMA can run that many stages
// ahead of the epilogue.  Shared memory cannot hold both deep rings and wide
// staging blocks, so there are two shapes:
//   PIPE_SHORT_K  more FP32 stages and 32-column staging blocks: fastest when
//                 a work unit has few k-stages and the output stores come
//                 often;
//   PIPE_LONG_K   three component stages, 16-column blocks: fastest in long
//                 k-loops.
// TF32x3's larger components leave room for only one shape.  A 128-wide
// tile (four accumulators, so the output stores hide behind the next tile)
// was measured slower on every workload: the kernel is bound by
// shared-memory bandwidth (about 90 bytes per clock per SM sustained), and
// halving the tile width raises the operand bytes per product by half.
enum Pipe : int { PIPE_SHORT_K = 0, PIPE_LONG_K = 1, PIPE_SHORT_K_PACKED = 2, PIPE_LONG_K_PACKED = 3 };
constexpr bool pipe_packed(int pipe) { return pipe >= PIPE_SHORT_K_PACKED; }
// The *_PACKED shapes take op(B) already split (emu_pack_b): its component
// tiles come by TMA straight into a ring of their own (NB stages, refilled as
// soon as a stage's MMAs are done, so they arrive well ahead); the FP32 ring
// holds op(A) alone, the component ring op(A)'s components, and the split
// warps split op(A) alone.
template <int MODE, int PIPE> struct PipeCfg;
template <> struct PipeCfg<MODE_BF16X9, PIPE_SHORT_K> {
    static constexpr int TN = 256, NF = 3, NS = 2, NB = 0, OUT_COLS = 32;
    static constexpr bool PACKED = false;
};
template <> struct PipeCfg<MODE_BF16X9, PIPE_LONG_K> {
    static constexpr int TN = 256, NF = 2, NS = 3, NB = 0, OUT_COLS = 16;
    static constexpr bool PACKED = false;
};
template <> struct PipeCfg<MODE_BF16X9, PIPE_SHORT_K_PACKED> {
    static constexpr int TN = 256, NF = 3, NS = 3, NB = 3, OUT_COLS = 32;
    static constexpr bool PACKED = true;
};
template <> struct PipeCfg<MODE_BF16X9, PIPE_LONG_K_PACKED> {
    static constexpr int TN = 256, NF = 2, NS = 3, NB = 4, OUT_COLS = 16;
    static constexpr bool PACKED = true;
};
template <int PIPE> struct PipeCfg<MODE_BF16X6, PIPE> : PipeCfg<MODE_BF16X9, PIPE> {};
template <int PIPE> struct PipeCfg<MODE_TF32X3, PIPE> {
    static constexpr bool PACKED = pipe_packed(PIPE);
    static constexpr int TN = 256, NF = 2, NS = 2, NB = PACKED ? 3 : 0, OUT_COLS = 32;
};
template <int PIPE> struct PipeCfg<MODE_TF32X1, PIPE> {
    static constexpr bool PACKED = pipe_packed(PIPE);
    static constexpr int TN = 256, NF = 3, NS = 3, NB = PACKED ? 4 : 0, OUT_COLS = 32;
};

// Everything the kernel derives from (mode, shape).
template <int MODE, int PIPE> struct KCfg {
    using C = Cfg<MODE>;
    using P = PipeCfg<MODE, PIPE>;
    static constexpr int TN = P::TN;
    static constexpr int BH = TN / 2;                  // rows of op(B)^T per CTA
    static constexpr int NACC = TMEM_COLS / TN;        // TMEM accumulators
    static constexpr int ACC = TN / 2;                 // accumulator registers per epilogue thread
    static constexpr int NF = P::NF, NS = P::NS, NB = P::NB, OUT_COLS = P::OUT_COLS;
    static constexpr bool PACKED = P::PACKED;
    static constexpr uint32_t FP32_B_BYTES = BH * BK * 4;
    static constexpr uint32_t FP32_STAGE = FP32_TILE_BYTES + (PACKED ? 0u : FP32_B_BYTES);
    static constexpr uint32_t COMP_A = C::COMP_TILE;                  // one component of op(A)
    static constexpr uint32_t COMP_B = BH * C::ROW_BYTES;             // one component of op(B)
    // component ring stage: op(A)'s components, then op(B)'s (unpacked shapes)
    static constexpr uint32_t SLICE_STAGE = C::NCOMP * (COMP_A + (PACKED ? 0u : COMP_B));
    static constexpr uint32_t BCOMP_BYTES = C::NCOMP * COMP_B;        // op(B)'s components of a stage
    static constexpr uint32_t IDESC = make_idesc(C::KIND, TILE_M, TN);
    static constexpr uint32_t STAGE_OUT = 32 * OUT_COLS * 4;          // one epilogue warp's staging block
    static constexpr uint32_t SMEM = 1024 /* alignment slack */ + NF * FP32_STAGE + NS * SLICE_STAGE +
                                     NB * BCOMP_BYTES + NUM_EPI_WARPS * STAGE_OUT + 1024 /* barriers and flags */;
    static_assert(SMEM <= 227 * 1024, "shared memory per CTA");
    static_assert(NACC * TN == (int)TMEM_COLS && NACC <= 4, "TMEM accumulators");
};

template <int MODE, int PIPE>
constexpr uint32_t smem_bytes() { return KCfg<MODE, PIPE>::SMEM; }

struct Params {
    CUtensorMap tmA;  // FP32 op(A): K-major box {32, 128} or MN-major box {32, 32}
    CUtensorMap tmB;  // FP32 op(B): K-major box {32, TN / 2} or MN-major box {32, 32};
                      // packed shapes: op(B)^T's component planes, box {32, TN / 2, 1}
    int M, N, K;
    int a_mn_major, b_mn_major;
    int tiles_m, tiles_n, num_tiles, k_stages;
    // Work units: the first tiles_a tiles in split_a pieces each, then the
    // remaining tiles in split_b pieces each (1 = the whole tile).  Units are
    // numbered tile by tile, pieces in k order; CTA pair c takes units c,
    // c + pairs, c + 2 pairs, ...
    int tiles_a, split_a, split_b;
    int num_units;
    // 1: chained plan (every tile whole in the fields above; the pairs'
    // stage runs decide the units, see walk_of): pair c runs the stages
    // [b_c, b_c+1) of the tile-by-tile sequence, b_c = c U / pairs +
    // chain_delta[c] (U = num_tiles * k_stages; |chain_delta| <= 2), with
    // c U / pairs = c chain_q + (c chain_r) / pairs (U = chain_q pairs +
    // chain_r), which needs no 64-bit division
    int chain;
    int chain_r;
    long long chain_q;
    signed char chain_delta[kMaxChainPairs + 1];
    float alpha, beta;
    const float* c_old;  // read only when beta != 0
    float* c;
    long long ldc;
    const float* bias;   // may be null
    float* workspace;    // split tiles: S partial tiles of 256 x TN each (thread-major);
                         // chained plans: one running sum per run boundary (pairs - 1)
    unsigned long long* counters;  // split tiles: 2 per tile (pieces arrived, per CTA half), epoch-tagged
    unsigned long long epoch;      // this launch's epoch on the counters (> 0, new for every launch)
    unsigned long long wait_budget_ns;
};

// ----------------------------------------------------------- the splits ----
// Byte offset of element (mn, k) of an MN-major FP32 tile: four 32-wide MN
// blocks of 32 k-rows of 128 bytes, 128-byte swizzle (chunk XOR k % 8).
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

// Write the components of 8 consecutive k-values of one row; component c of
// the tile starts at dst + c * CSTRIDE.
template <int MODE, uint32_t CSTRIDE>
__device__ __forceinline__ void store_components(uint8_t* dst, uint32_t row, uint32_t g, const float (&x)[8]) {
    using C = Cfg<MODE>;
    if constexpr (!C::TF32) {
        uint4 s0, s1, s2;
        split_bf16x9_8(x, s0, s1, s2);
        const uint32_t o = off_bf16_chunk(row, g);
        *reinterpret_cast<uint4*>(dst + o) = s0;
        *reinterpret_cast<uint4*>(dst + CSTRIDE + o) = s1;
        *reinterpret_cast<uint4*>(dst + 2 * CSTRIDE + o) = s2;
    } else if constexpr (C::NCOMP == 1) {
        uint32_t h[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) h[i] = tf32_rn_bits(__float_as_uint(x[i]));
        const uint32_t o0 = off_f32_chunk(row, 2 * g), o1 = off_f32_chunk(row, 2 * g + 1);
        *reinterpret_cast<uint4*>(dst + o0) = make_uint4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<uint4*>(dst + o1) = make_uint4(h[4], h[5], h[6], h[7]);
    } else {
        uint32_t h[8], l[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) split_tf32x3_1(x[i], h[i], l[i]);
        const uint32_t o0 = off_f32_chunk(row, 2 * g), o1 = off_f32_chunk(row, 2 * g + 1);
        *reinterpret_cast<uint4*>(dst + o0) = make_uint4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<uint4*>(dst + o1) = make_uint4(h[4], h[5], h[6], h[7]);
        *reinterpret_cast<uint4*>(dst + CSTRIDE + o0) = make_uint4(l[0], l[1], l[2], l[3]);
        *reinterpret_cast<uint4*>(dst + CSTRIDE + o1) = make_uint4(l[4], l[5], l[6], l[7]);
    }
}

// Split one operand tile (ROWS rows x 32 k, ROWS = 128 or 64) of a stage.
// `src` is the FP32 tile, `dst` the first component tile (components follow
// at ROWS * ROW_BYTES strides).  `t` is the thread's index among NT split
// threads (NT a multiple of 32).  Work items are (row, 8-k group) pairs,
// 4 * ROWS per tile.
template <int MODE, int NT, int ROWS>
__device__ __forceinline__ void split_operand(const uint8_t* src, uint8_t* dst, bool mn_major, uint32_t t) {
    static_assert(ROWS == 128 || ROWS == 64, "tile rows");
    constexpr uint32_t ITEMS = 4 * ROWS;
    constexpr uint32_t CSTRIDE = ROWS * Cfg<MODE>::ROW_BYTES;
    if (!mn_major) {
        // lanes cover 8 rows x 4 groups, so both the 16-byte reads and the
        // 16-byte writes of a warp fall on distinct banks
        for (uint32_t item = t; item < ITEMS; item += NT) {
            const uint32_t row = (item >> 5) * 8u + ((item & 31u) >> 2);
            const uint32_t g = item & 3u;
            const float4 lo4 = *reinterpret_cast<const float4*>(src + off_f32_chunk(row, 2 * g));
            const float4 hi4 = *reinterpret_cast<const float4*>(src + off_f32_chunk(row, 2 * g + 1));
            const float x[8] = {lo4.x, lo4.y, lo4.z, lo4.w, hi4.x, hi4.y, hi4.z, hi4.w};
            store_components<MODE, CSTRIDE>(dst, row, g, x);
        }
    } else {
        // 32 consecutive mn per warp: the column reads of the MN-major tile and
        // the row writes are both conflict-free
        for (uint32_t item = t; item < ITEMS; item += NT) {
            const uint32_t mn = item % ROWS;
            const uint32_t g = item / ROWS;
            float x[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                x[i] = *reinterpret_cast<const float*>(src + off_f32_mnmajor(mn, 8 * g + i));
            store_components<MODE, CSTRIDE>(dst, mn, g, x);
        }
    }
}

// Issue the pair products of one stage into TMEM accumulator `d`, starting
// from zero: the mode's (i, j) component products, smallest first (BF16x9:
// bands 4, 3, 2, 1, 0; TF32x3: lo*hi, hi*lo, hi*hi), each over the K steps of
// the stage (two of 16 for BF16, four of 8 for TF32).
template <int MODE, int PIPE>
__device__ __forceinline__ void issue_stage_mmas(uint32_t d, uint32_t a_base, uint32_t b_base) {
    using C = Cfg<MODE>;
    using KC = KCfg<MODE, PIPE>;
    uint32_t acc = 0;
#pragma unroll
    for (int p = 0; p < C::NPROD; ++p) {
#pragma unroll
        for (int ks = 0; ks < BK / C::KSTEP; ++ks) {
            const uint64_t ad = sdesc_kmajor(a_base + C::pi(p) * KC::COMP_A + ks * 32, C::ROW_BYTES);
            const uint64_t bd = sdesc_kmajor(b_base + C::pj(p) * KC::COMP_B + ks * 32, C::ROW_BYTES);
            if constexpr (C::TF32) mma_tf32_pair(d, ad, bd, KC::IDESC, acc);
            else mma_bf16_pair(d, ad, bd, KC::IDESC, acc);
            acc = 1;
        }
    }
}

// What the epilogue does with a unit's sums besides adding its stages:
// ROLE_TILE  a whole tile, or a piece of a reduce-scatter split tile;
// ROLE_HEAD  chained plans: the low k-stages of a cut tile, whose running sum
//            is published for the pair that finishes the tile;
// ROLE_TAIL  chained plans: the high k-stages of a cut tile, whose running
//            sum starts from the published one; stored like a whole tile.
enum Role : int { ROLE_TILE = 0, ROLE_HEAD = 1, ROLE_TAIL = 2 };

struct Unit {
    int tile, piece, pieces, kb, ke, role;
    long long slot;  // first workspace partial tile of a split tile; chained plans: the running sum's slot
};
__device__ __forceinline__ Unit unit_of(const Params& p, int u) {
    Unit w;
    w.role = ROLE_TILE;
    const int units_a = p.tiles_a * p.split_a;
    const long long slots_a = p.split_a > 1 ? static_cast<long long>(units_a) : 0;
    if (u < units_a) {
        w.pieces = p.split_a;
        w.tile = u / p.split_a;
        w.piece = u - w.tile * p.split_a;
        w.slot = static_cast<long long>(w.tile) * p.split_a;
    } else {
        const int v = u - units_a;
        const int t = v / p.split_b;
        w.pieces = p.split_b;
        w.tile = p.tiles_a + t;
        w.piece = v - t * p.split_b;
        w.slot = slots_a + static_cast<long long>(t) * p.split_b;
    }
    // (piece + 1) * k_stages < 32 * 2^26 fits 32 unsigned bits: no 64-bit division
    const uint32_t ks = static_cast<uint32_t>(p.k_stages), np = static_cast<uint32_t>(w.pieces);
    w.kb = static_cast<int>(static_cast<uint32_t>(w.piece) * ks / np);
    w.ke = static_cast<int>(static_cast<uint32_t>(w.piece + 1) * ks / np);
    return w;
}

// The units one CTA pair runs, in order: u = first, first + step, ... < last.
// Other plans: every unit index c, c + pairs, ...  Chained plans: the pair's
// run [s, e) of the tile-major stage sequence (tile t's stages are t * KS ..
// t * KS + KS - 1, taken in DEcreasing k order, so that a run that starts
// inside a tile holds its low k-stages); the units are the tiles the run
// touches, in increasing order.  The planner gives every pair a non-empty run
// that is not strictly inside one tile, so no tile is cut twice.
struct Walk {
    int first, last, step;
    int lo, hi;  // chained plans: the run covers positions [lo, KS) of tile `first`, [0, hi) of tile last - 1
};
__device__ __forceinline__ Walk walk_of(const Params& p, int cid, int ncl) {
    Walk k;
    if (!p.chain) {
        k.first = cid; k.last = p.num_units; k.step = ncl; k.lo = 0; k.hi = 0;
        return k;
    }
    const long long s = cid * p.chain_q + (cid * p.chain_r) / ncl + p.chain_delta[cid];
    const long long e = (cid + 1) * p.chain_q + ((cid + 1) * p.chain_r) / ncl + p.chain_delta[cid + 1];  // e > s
    if (e <= 0x7FFFFFFFll) {  // the usual case: 32-bit divisions (a 64-bit one is a long software routine)
        const uint32_t ks = static_cast<uint32_t>(p.k_stages);
        k.first = static_cast<int>(static_cast<uint32_t>(s) / ks);
        k.last = static_cast<int>(static_cast<uint32_t>(e - 1) / ks) + 1;
    } else {
        k.first = static_cast<int>(s / p.k_stages);
        k.last = static_cast<int>((e - 1) / p.k_stages) + 1;
    }
    k.step = 1;
    k.lo = static_cast<int>(s - static_cast<long long>(k.first) * p.k_stages);
    k.hi = static_cast<int>(e - static_cast<long long>(k.last - 1) * p.k_stages);
    return k;
}
__device__ __forceinline__ Unit unit_at(const Params& p, const Walk& k, int cid, int u) {
    if (!p.chain) return unit_of(p, u);
    Unit w;
    const int lo = u == k.first ? k.lo : 0;                 // the run covers positions
    const int hi = u == k.last - 1 ? k.hi : p.k_stages;     // [lo, hi) of tile u
    w.tile = u; w.piece = 0; w.pieces = 1;
    w.kb = p.k_stages - hi;
    w.ke = p.k_stages - lo;
    // the boundary between pairs c - 1 and c owns running-sum slot c - 1
    if (lo > 0) { w.role = ROLE_HEAD; w.slot = cid - 1; }
    else if (hi < p.k_stages) { w.role = ROLE_TAIL; w.slot = cid; }
    else { w.role = ROLE_TILE; w.slot = 0; }
    return w;
}

// STAGED: split tiles of many pieces read the other pieces' partials through
// the output staging area (see the epilogue); a separate instantiation, so
// that plans with few pieces keep the register-only reduction's code.
template <int MODE, int PIPE, bool STAGED = false>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
emu_gemm_kernel(const __grid_constant__ Params p) {
    using C = Cfg<MODE>;
    using KC = KCfg<MODE, PIPE>;
    constexpr int NF = KC::NF, NS = KC::NS, NB = KC::NB, OUT_COLS = KC::OUT_COLS;
    constexpr int TN = KC::TN, BH = KC::BH, NACC = KC::NACC, ACC = KC::ACC;
    constexpr bool PACKED = KC::PACKED;
    constexpr uint32_t STAGE_OUT_BYTES = KC::STAGE_OUT;  // one epilogue warp's 32 x OUT_COLS block
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // pointer arithmetic on the shared array (not an integer round trip) keeps
    // the shared address space visible to the compiler: shared stores then do
    // not alias global loads, which it can hoist
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t* fp32_ring = smem;
    uint8_t* slice_ring = smem + NF * KC::FP32_STAGE;
    uint8_t* bcomp_ring = slice_ring + NS * KC::SLICE_STAGE;  // packed shapes: op(B)'s components
    uint8_t* out_stage = bcomp_ring + NB * KC::BCOMP_BYTES;    // one block per epilogue warp
    uint64_t* bars = reinterpret_cast<uint64_t*>(out_stage + NUM_EPI_WARPS * STAGE_OUT_BYTES);
    uint64_t* fp32_full = bars;
    uint64_t* fp32_empty = fp32_full + NF;
    uint64_t* slice_full = fp32_empty + NF;   // leader: both CTAs' split warps
    uint64_t* slice_empty = slice_full + NS;  // multicast commit
    uint64_t* acc_full = slice_empty + NS;    // multicast commit
    uint64_t* acc_empty = acc_full + NACC;    // leader: both CTAs' epilogue warps
    uint64_t* drain = acc_empty + NACC;
    uint64_t* bcomp_full = drain + 1;          // packed shapes: a stage's op(B) components landed
    uint64_t* bcomp_empty = bcomp_full + NB;   // packed shapes: multicast commit
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bcomp_empty + NB);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* last_flag = reinterpret_cast<volatile int*>(tmem_slot + 2);
    // this pair's walk (first, last, step, lo, hi), for the epilogue to read
    // at each unit instead of holding it in registers across the k-loops
    volatile int* walk_sh = reinterpret_cast<volatile int*>(tmem_slot + 4);

    const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31u;
    const uint32_t rank = cluster_ctarank();
    const uint32_t cid = cluster_id_x(), ncl = num_clusters_x();

    // The next GEMM in the stream may start its own set-up (barriers, TMEM,
    // the pair barrier) on SMs this grid has left; it touches global memory
    // only after this grid has completed (griddep_wait).
    if (threadIdx.x == 0) griddep_launch_dependents();

    // The producer's TMA loads for the first FP32 stages need nothing but this
    // CTA's own barriers, so they go out before the pair synchronises and
    // allocates TMEM (the load latency overlaps the set-up).  Like every
    // global access of this kernel they wait for the grids this launch
    // depends on.
    // (m0, n0): this CTA's first row of op(A) and of op(B)^T in the tile
    auto issue_load_at = [&](int s, int m0, int n0, int ks) {
        uint64_t* full = &fp32_full[s];
        mbar_arrive_expect_tx(full, KC::FP32_STAGE);
        uint8_t* dA = fp32_ring + s * KC::FP32_STAGE;
        uint8_t* dB = dA + FP32_TILE_BYTES;
        const int k0 = ks * BK;
        if (!p.a_mn_major) tma_load_2d(dA, &p.tmA, full, k0, m0);
        else for (int j = 0; j < HALF / 32; ++j) tma_load_2d(dA + j * 4096, &p.tmA, full, m0 + 32 * j, k0);
        if constexpr (!PACKED) {
            if (!p.b_mn_major) tma_load_2d(dB, &p.tmB, full, k0, n0);
            else for (int j = 0; j < BH / 32; ++j) tma_load_2d(dB + j * 4096, &p.tmB, full, n0 + 32 * j, k0);
        }
    };
    auto issue_load = [&](int s, int tile, int ks) {
        issue_load_at(s, (tile / p.tiles_n) * TILE_M + HALF * rank, (tile % p.tiles_n) * TN + BH * rank, ks);
    };
    // packed shapes: op(B)'s component tiles of a stage, straight into the
    // component ring (box {32 k, BH rows, 1 component} per component)
    auto issue_bload_at = [&](int bslot, int n0, int ks) {
        uint64_t* full = &bcomp_full[bslot];
        mbar_arrive_expect_tx(full, KC::BCOMP_BYTES);
        uint8_t* dst = bcomp_ring + bslot * KC::BCOMP_BYTES;
        for (int c = 0; c < C::NCOMP; ++c) tma_load_3d(dst + c * KC::COMP_B, &p.tmB, full, ks * BK, n0, c);
    };
    auto issue_bload = [&](int bslot, int tile, int ks) {
        issue_bload_at(bslot, (tile % p.tiles_n) * TN + BH * rank, ks);
    };
    int early = 0, early_b = 0;  // stages already issued by thread 0 (warp 0 lane 0, the producer)
    if (threadIdx.x == 0) {
        tma_prefetch_desc(&p.tmA);
        tma_prefetch_desc(&p.tmB);
        for (int s = 0; s < NF; ++s) { mbar_init(&fp32_full[s], 1); mbar_init(&fp32_empty[s], 1); }
        for (int s = 0; s < NS; ++s) { mbar_init(&slice_full[s], 2); mbar_init(&slice_empty[s], 1); }
        for (int b = 0; b < NACC; ++b) { mbar_init(&acc_full[b], 1); mbar_init(&acc_empty[b], 2); }
        mbar_init(drain, 1);
        for (int s = 0; s < NB; ++s) { mbar_init(&bcomp_full[s], 1); mbar_init(&bcomp_empty[s], 1); }
        *abort_flag = 0;
        // this pair's walk, worked out once for all roles
        const Walk wk = walk_of(p, static_cast<int>(cid), static_cast<int>(ncl));
        walk_sh[0] = wk.first; walk_sh[1] = wk.last; walk_sh[2] = wk.step; walk_sh[3] = wk.lo; walk_sh[4] = wk.hi;
        fence_mbar_init();
        // Where the first stages come from depends on the parameters alone:
        // it is worked out before waiting for the previous grid, so that the
        // unit arithmetic and the parameter reads (about a microsecond) do
        // not delay the first loads.
        constexpr int NE = PACKED && NB > NF ? NB : NF;
        int e_m0[NE], e_n0[NE], e_ks[NE], ne = 0;
        {
            int u = wk.first, ks = 0, ke = 0, m0 = 0, n0 = 0;
#pragma unroll
            for (int i = 0; i < NE; ++i) {
                while (ks >= ke && u < wk.last) {
                    const Unit w = unit_at(p, wk, static_cast<int>(cid), u);
                    const int tm = w.tile / p.tiles_n;
                    m0 = tm * TILE_M + HALF * rank;
                    n0 = (w.tile - tm * p.tiles_n) * TN + BH * rank;
                    ks = w.kb; ke = w.ke;
                    u += wk.step;
                }
                if (ks < ke) {
                    e_m0[i] = m0;
                    e_n0[i] = n0;
                    e_ks[i] = ks++;
                    ne = i + 1;
                }
            }
        }
        // the first stage's operands are prefetched into L2 while the
        // previous grid finishes (L2 is coherent, so nothing stale is read);
        // the later stages' loads go out right after the wait anyway, and
        // each prefetch costs this thread issue time when nothing is waited
        // for
        if (ne > 0) {
            const int k0 = e_ks[0] * BK;
            if (!p.a_mn_major) tma_prefetch_l2_2d(&p.tmA, k0, e_m0[0]);
            else for (int j = 0; j < HALF / 32; ++j) tma_prefetch_l2_2d(&p.tmA, e_m0[0] + 32 * j, k0);
            if constexpr (!PACKED) {
                if (!p.b_mn_major) tma_prefetch_l2_2d(&p.tmB, k0, e_n0[0]);
                else for (int j = 0; j < BH / 32; ++j) tma_prefetch_l2_2d(&p.tmB, e_n0[0] + 32 * j, k0);
            } else {
                for (int c = 0; c < C::NCOMP; ++c) tma_prefetch_l2_3d(&p.tmB, k0, e_n0[0], c);
            }
        }
        griddep_wait();
#pragma unroll
        for (int i = 0; i < NE; ++i) {
            if (i < ne) {
                if (i < NF) issue_load_at(i, e_m0[i], e_n0[i], e_ks[i]);
                if (PACKED && i < NB) issue_bload_at(i, e_n0[i], e_ks[i]);
            }
        }
        early = ne < NF ? ne : NF;
        early_b = PACKED ? (ne < NB ? ne : NB) : 0;
    }
    if (warp == WARP_MMA) {
        tmem_alloc_pair(tmem_slot, TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();          // this CTA's barriers and TMEM address visible to all its threads
    cluster_sync_relaxed();   // the peer's barriers initialised before any arrival on them
    tc_fence_after();
    griddep_wait();           // inputs, C, workspace and counters are the previous grids' to finish
    const uint32_t tmem_base = *tmem_slot;
    const uint64_t budget = p.wait_budget_ns;
    Walk walk;  // (thread 0's, from shared memory)
    walk.first = walk_sh[0]; walk.last = walk_sh[1]; walk.step = walk_sh[2]; walk.lo = walk_sh[3]; walk.hi = walk_sh[4];

    if (warp == WARP_PRODUCER) {
        // ------------------------------------------------------ producer ----
        setmaxnreg_dec72();
        if (lane == 0) {
            int s = 0, n = 0, bs = 0;
            uint32_t ph = 0, issued_mask = 0, issued_parity = 0;
            uint32_t bph = 0, bissued_mask = 0, bissued_parity = 0;
            bool ok = true;
            for (int u = walk.first; ok && u < walk.last; u += walk.step) {
                const Unit w = unit_at(p, walk, static_cast<int>(cid), u);
                for (int ks = w.kb; ks < w.ke; ++ks, ++n) {
                    if (n >= early) {  // the first `early` loads went out before the pair sync
                        if (!mbar_wait(&fp32_empty[s], ph ^ 1u, abort_flag, budget, 1)) { ok = false; break; }
                        issue_load(s, w.tile, ks);
                    }
                    issued_mask |= 1u << s;
                    issued_parity = (issued_parity & ~(1u << s)) | (ph << s);
                    if (++s == NF) { s = 0; ph ^= 1u; }
                    if constexpr (PACKED) {
                        if (n >= early_b) {  // the slot is free once its stage's MMAs are done
                            if (!mbar_wait(&bcomp_empty[bs], bph ^ 1u, abort_flag, budget, 1)) { ok = false; break; }
                            issue_bload(bs, w.tile, ks);
                        }
                        bissued_mask |= 1u << bs;
                        bissued_parity = (bissued_parity & ~(1u << bs)) | (bph << bs);
                        if (++bs == NB) { bs = 0; bph ^= 1u; }
                    }
                }
            }
            if (!ok) {
                // give every load already in flight time to land before the CTA exits
                for (int t = 0; t < NF; ++t)
                    if (issued_mask & (1u << t)) {
                        volatile int never = 0;
                        mbar_wait(&fp32_full[t], (issued_parity >> t) & 1u, &never, 50000000ull, 1);
                    }
                for (int t = 0; t < NB; ++t)
                    if (bissued_mask & (1u << t)) {
                        volatile int never = 0;
                        mbar_wait(&bcomp_full[t], (bissued_parity >> t) & 1u, &never, 50000000ull, 1);
                    }
            }
        }
        __syncwarp();
    } else if (warp == WARP_MMA) {
        // ---------------------------------------------- MMA issuer (leader) -
        setmaxnreg_dec72();
        if (lane == 0 && rank == 0) {
            int s = 0, b = 0, bs = 0;
            uint32_t ph = 0, bph = 0;
            bool ok = true, issued = false;
            const uint32_t slice_base = smem_u32(slice_ring), bcomp_base = smem_u32(bcomp_ring);
            for (int u = walk.first; ok && u < walk.last; u += walk.step) {
                const Unit w = unit_at(p, walk, static_cast<int>(cid), u);
                for (int ks = w.kb; ks < w.ke; ++ks) {
                    if (!mbar_wait(&acc_empty[b], bph ^ 1u, abort_flag, budget, 2)) { ok = false; break; }
                    if (!mbar_wait(&slice_full[s], ph, abort_flag, budget, 2)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a_base = slice_base + s * KC::SLICE_STAGE;
                    const uint32_t b_base = PACKED ? bcomp_base + bs * KC::BCOMP_BYTES : a_base + C::NCOMP * KC::COMP_A;
                    issue_stage_mmas<MODE, PIPE>(tmem_base + b * TN, a_base, b_base);
                    issued = true;
                    mma_commit_pair_multicast(&slice_empty[s], 0x3);
                    if constexpr (PACKED) {
                        mma_commit_pair_multicast(&bcomp_empty[bs], 0x3);
                        if (++bs == NB) bs = 0;
                    }
                    mma_commit_pair_multicast(&acc_full[b], 0x3);
                    if (++s == NS) { s = 0; ph ^= 1u; }
                    if (++b == NACC) { b = 0; bph ^= 1u; }
                }
            }
            if (!ok && issued) {
                // let the products in flight finish before TMEM is released
                mma_commit_pair(drain);
                volatile int never = 0;
                mbar_wait(drain, 0, &never, 50000000ull, 2);
            }
        }
        __syncwarp();
    } else if (warp < WARP_EPI0) {
        // ---------------------------------------------------- split warps ---
        setmaxnreg_dec72();
        const uint32_t t = threadIdx.x - WARP_SPLIT0 * 32;
        int fs = 0, ss = 0, bs = 0;
        uint32_t fph = 0, sph = 0, bph = 0;
        bool ok = true;
        for (int u = walk.first; ok && u < walk.last; u += walk.step) {
            const Unit w = unit_at(p, walk, static_cast<int>(cid), u);
            for (int ks = w.kb; ks < w.ke; ++ks) {
                if (!mbar_wait_warp(&fp32_full[fs], fph, abort_flag, budget, 3)) { ok = false; break; }
                if (!mbar_wait_warp(&slice_empty[ss], sph ^ 1u, abort_flag, budget, 3)) { ok = false; break; }
                const uint8_t* src = fp32_ring + fs * KC::FP32_STAGE;
                uint8_t* dst = slice_ring + ss * KC::SLICE_STAGE;
                split_operand<MODE, NUM_SPLIT_THREADS, HALF>(src, dst, p.a_mn_major != 0, t);
                if constexpr (!PACKED) {
                    split_operand<MODE, NUM_SPLIT_THREADS, BH>(src + FP32_TILE_BYTES, dst + C::NCOMP * KC::COMP_A,
                                                               p.b_mn_major != 0, t);
                } else {  // op(B)'s components come by TMA into their own ring
                    if (!mbar_wait_warp(&bcomp_full[bs], bph, abort_flag, budget, 3)) { ok = false; break; }
                    if (++bs == NB) { bs = 0; bph ^= 1u; }
                }
                // one signal per CTA: the split threads meet, then a single
                // thread releases the stage (a cluster-scope arrive is costly)
                fence_proxy_async_smem();
                named_bar_sync(SPLIT_BARRIER, NUM_SPLIT_THREADS);
                if (t == 0) {
                    mbar_arrive(&fp32_empty[fs]);
                    if (rank == 0) mbar_arrive(&slice_full[ss]);
                    else mbar_arrive_cluster(&slice_full[ss], 0);
                }
                if (++fs == NF) { fs = 0; fph ^= 1u; }
                if (++ss == NS) { ss = 0; sph ^= 1u; }
            }
        }
    } else {
        // ------------------------------------------------------- epilogue ---
        setmaxnreg_inc184();
        const uint32_t e = warp - WARP_EPI0;      // 0..7
        const uint32_t quarter = warp & 3u;       // TMEM lanes this warp may read
        const uint32_t half = e >> 2;             // which TN / 2 columns of the tile
        const uint32_t lane_base = (quarter * 32u) << 16;
        int b = 0;
        uint32_t bph = 0;
        bool ok = true;
        for (int u = walk_sh[0]; ok && u < walk_sh[1]; u += walk_sh[2]) {
            Walk wk;
            wk.first = walk_sh[0]; wk.last = walk_sh[1]; wk.step = walk_sh[2]; wk.lo = walk_sh[3]; wk.hi = walk_sh[4];
            const Unit w = unit_at(p, wk, static_cast<int>(cid), u);
            // a chained tile's running sum: one 256 x TN slot per run boundary,
            // thread-major like the split-K partials below (worked out where it
            // is used, so that it holds no registers during the k-loop)
            auto chain_sum = [&](long long slot) {
                return p.workspace + static_cast<size_t>(slot) * (static_cast<size_t>(TILE_M) * TN) +
                       (static_cast<size_t>(rank) * NUM_EPI_WARPS + e) * (32u * ACC) + lane * 4u;
            };
            float acc[ACC];
            if (!STAGED && w.role == ROLE_TAIL) {
                // Start from the running sum of the tile's low k-stages, which
                // the next pair publishes at the start of its run.  Each warp
                // waits for it on its own; all its loads go out at once,
                // straight into the sums' registers, while the tensor cores
                // work on this unit's first stages.
                const unsigned long long* ctr = p.counters + static_cast<size_t>(w.tile) * 2 + rank;
                if (!warp_wait_epoch(ctr, p.epoch, 1u, abort_flag, budget, 7)) { ok = false; break; }
                const float* head = chain_sum(w.slot);
#pragma unroll
                for (int j = 0; j < ACC / 4; ++j) {
                    const float4 x = __ldcg(reinterpret_cast<const float4*>(head + j * 128));
                    acc[4 * j] = x.x; acc[4 * j + 1] = x.y; acc[4 * j + 2] = x.z; acc[4 * j + 3] = x.w;
                }
            } else {
#pragma unroll
                for (int i = 0; i < ACC; ++i) acc[i] = 0.0f;
            }
            for (int ks = w.kb; ks < w.ke; ++ks) {
                if (!mbar_wait_warp(&acc_full[b], bph, abort_flag, budget, 4)) { ok = false; break; }
                tc_fence_after();
                const uint32_t col = tmem_base + lane_base + b * TN + half * ACC;
#pragma unroll
                for (int c = 0; c < ACC / 16; c += 2) {
                    float v0[16], v1[16];
                    tmem_ld16(col + c * 16, v0);
                    tmem_ld16(col + (c + 1) * 16, v1);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        acc[c * 16 + i] = __fadd_rn(acc[c * 16 + i], v0[i]);
                        acc[(c + 1) * 16 + i] = __fadd_rn(acc[(c + 1) * 16 + i], v1[i]);
                    }
                }
                tc_fence_before();
                named_bar_sync(EPI_BARRIER, NUM_EPI_WARPS * 32);
                if (e == 0 && lane == 0) {
                    if (rank == 0) mbar_arrive(&acc_empty[b]);
                    else mbar_arrive_cluster(&acc_empty[b], 0);
                }
                if (++b == NACC) { b = 0; bph ^= 1u; }
            }
            if (!ok) break;
            if (!STAGED && w.role == ROLE_HEAD) {
                // publish this tile's running sum for the pair that runs its
                // high k-stages; nothing is stored to C here
                float* head = chain_sum(w.slot);
#pragma unroll
                for (int j = 0; j < ACC / 4; ++j)
                    __stcg(reinterpret_cast<float4*>(head + j * 128),
                           make_float4(acc[4 * j], acc[4 * j + 1], acc[4 * j + 2], acc[4 * j + 3]));
                __threadfence();
                named_bar_sync(EPI_BARRIER, NUM_EPI_WARPS * 32);
                if (e == 0 && lane == 0) epoch_arrive(p.counters + static_cast<size_t>(w.tile) * 2 + rank, p.epoch);
                continue;
            }
            // Split tiles: a reduce-scatter over the tile's S pieces, which all
            // run at the same time (the plan keeps a tile's pieces in one wave
            // of units).  Chunk q = 4e + c (32 columns of
            // warp e's block) of this CTA's half-tile belongs to piece q mod S.
            // Each piece publishes the chunks that other pieces own, waits until
            // all S pieces have published, and sums the chunks it owns -- its own
            // partial, then the other pieces' in increasing piece order, a fixed
            // order for every chunk -- and stores only those: the result does not
            // depend on timing.
            const int S = w.pieces;
            auto owns = [&](int c) { return S == 1 || static_cast<int>(4 * e + c) % S == w.piece; };
            if (S > 1) {
                const size_t per_piece = static_cast<size_t>(TILE_M) * TN;
                const size_t warp_off = (static_cast<size_t>(rank) * NUM_EPI_WARPS + e) * (32u * ACC) + lane * 4u;
                float* tile_ws = p.workspace + static_cast<size_t>(w.slot) * per_piece + warp_off;
                float* part = tile_ws + static_cast<size_t>(w.piece) * per_piece;
                // (thread-major: float4 j of every lane of a warp is 512
                // contiguous bytes; chunk c is j in [8c, 8c + 8))
#pragma unroll
                for (int j = 0; j < ACC / 4; ++j)
                    if (!owns(j / 8))
                        __stcg(reinterpret_cast<float4*>(part + j * 128),
                               make_float4(acc[4 * j], acc[4 * j + 1], acc[4 * j + 2], acc[4 * j + 3]));
                __threadfence();
                named_bar_sync(EPI_BARRIER, NUM_EPI_WARPS * 32);
                unsigned long long* ctr = p.counters + static_cast<size_t>(w.tile) * 2 + rank;
                if (e == 0 && lane == 0) {
                    epoch_arrive(ctr, p.epoch);
                    *last_flag = wait_epoch_count(ctr, p.epoch, static_cast<unsigned>(S), abort_flag, budget, 6) ? 1 : 0;
                }
                named_bar_sync(EPI_BARRIER, NUM_EPI_WARPS * 32);
                const int published = *last_flag;
                named_bar_sync(EPI_BARRIER, NUM_EPI_WARPS * 32);  // flag read before the next unit rewrites it
                if (!published) { ok = false; break; }
                __threadfence();
                // the owner's own partial first, then the other pieces in
                // increasing order, added in place (a fixed order per chunk).
                // The more bytes in flight, the fewer round trips to L2: in
                // the STAGED build, when few warps own chunks (many pieces:
                // three or more staging blocks per owner), the owners borrow
                // the whole output staging area (idle until the stores below)
                // and copy several pieces' blocks into it at once with
                // cp.async, which holds no registers while the copies fly;
                // otherwise each owner reads two pieces' blocks at a time
                // into registers.
                int n_owners = 0, my_slot0 = 0;
                if constexpr (STAGED) {
#pragma unroll 1
                    for (int e2 = 0; e2 < NUM_EPI_WARPS; ++e2) {
                        bool any = false;
                        for (int c = 0; c < ACC / 32; ++c) any = any || (4 * e2 + c) % S == w.piece;
                        if (any) {
                            if (e2 < static_cast<int>(e)) ++my_slot0;
                            ++n_owners;
                        }
                    }
                }
                constexpr int STAGED_BLOCKS = NUM_EPI_WARPS * STAGE_OUT_BYTES / 4096;  // 4 KB blocks of staging
                const int G = STAGED && n_owners > 0 ? STAGED_BLOCKS / n_owners : 0;  // blocks per owner warp
                if (STAGED && G >= 3) {
                    uint8_t* slots = out_stage + static_cast<uint32_t>(my_slot0 * G) * 4096u + lane * 16u;
#pragma unroll
                    for (int c = 0; c < ACC / 32; ++c) {
                        if (!owns(c)) continue;
                        for (int qi0 = 0; qi0 < S - 1; qi0 += G) {
                            const int n = S - 1 - qi0 < G ? S - 1 - qi0 : G;
                            for (int t = 0; t < n; ++t) {
                                const int qi = qi0 + t, q = qi + (qi >= w.piece ? 1 : 0);
                                const float* src = tile_ws + static_cast<size_t>(q) * per_piece + c * 1024;
#pragma unroll
                                for (int j = 0; j < 8; ++j) cp_async16(slots + t * 4096 + j * 512, src + j * 128);
                            }
                            cp_async_wait_all();  // each lane reads back only what it copied
                            for (int t = 0; t < n; ++t) {
#pragma unroll
                                for (int j = 0; j < 8; ++j) {
                                    const float4 x = *reinterpret_cast<const float4*>(slots + t * 4096 + j * 512);
                                    acc[32 * c + 4 * j] = __fadd_rn(acc[32 * c + 4 * j], x.x);
                                    acc[32 * c + 4 * j + 1] = __fadd_rn(acc[32 * c + 4 * j + 1], x.y);
                                    acc[32 * c + 4 * j + 2] = __fadd_rn(acc[32 * c + 4 * j + 2], x.z);
                                    acc[32 * c + 4 * j + 3] = __fadd_rn(acc[32 * c + 4 * j + 3], x.w);
                                }
                            }
                        }
                    }
                } else {
#pragma unroll
                for (int c = 0; c < ACC / 32; ++c) {
                    if (!owns(c)) continue;
                    // two pieces' blocks in flight at once, added in piece order
                    for (int qi = 0; qi < S - 1; qi += 2) {
                        const int qa = qi + (qi >= w.piece ? 1 : 0);
                        const bool two = qi + 1 < S - 1;
                        const int qb = qi + 1 + (qi + 1 >= w.piece ? 1 : 0);
                        const float* sa = tile_ws + static_cast<size_t>(qa) * per_piece + c * 1024;
                        const float* sb = tile_ws + static_cast<size_t>(two ? qb : qa) * per_piece + c * 1024;
                        float4 x[8], y[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j) x[j] = __ldcg(reinterpret_cast<const float4*>(sa + j * 128));
#pragma unroll
                        for (int j = 0; j < 8; ++j) y[j] = __ldcg(reinterpret_cast<const float4*>(sb + j * 128));
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            acc[32 * c + 4 * j] = __fadd_rn(acc[32 * c + 4 * j], x[j].x);
                            acc[32 * c + 4 * j + 1] = __fadd_rn(acc[32 * c + 4 * j + 1], x[j].y);
                            acc[32 * c + 4 * j + 2] = __fadd_rn(acc[32 * c + 4 * j + 2], x[j].z);
                            acc[32 * c + 4 * j + 3] = __fadd_rn(acc[32 * c + 4 * j + 3], x[j].w);
                        }
                        if (two) {
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                acc[32 * c + 4 * j] = __fadd_rn(acc[32 * c + 4 * j], y[j].x);
                                acc[32 * c + 4 * j + 1] = __fadd_rn(acc[32 * c + 4 * j + 1], y[j].y);
                                acc[32 * c + 4 * j + 2] = __fadd_rn(acc[32 * c + 4 * j + 2], y[j].z);
                                acc[32 * c + 4 * j + 3] = __fadd_rn(acc[32 * c + 4 * j + 3], y[j].w);
                            }
                        }
                    }
                }
                }
                // the staged reads may use other warps' staging blocks: all
                // done before any warp stages its output below
                named_bar_sync(EPI_BARRIER, NUM_EPI_WARPS * 32);
            }
            // (the tile's origin is worked out here, not before the split-tile
            // reduction, so that it holds no registers there)
            const int row0 = (w.tile / p.tiles_n) * TILE_M + static_cast<int>(HALF * rank + quarter * 32u);
            const int col0 = (w.tile % p.tiles_n) * TN + static_cast<int>(half * ACC);
            // ACC / OUT_COLS blocks of 32 rows x OUT_COLS columns: each lane stages
            // its row's sums in shared memory (rows of OUT_COLS * 4 bytes, 16-byte
            // chunks XOR-swizzled by row); the warp then reads them back as whole
            // row segments, applies C = alpha * acc + beta * C_old + bias and
            // stores the rows contiguously (coalesced), clipping rows and columns
            // outside C.
            constexpr int CPR = OUT_COLS / 4;   // 16-byte chunks per staged row
            constexpr int RPP = 32 / CPR;       // rows per read-back pass
            uint8_t* stage = out_stage + e * STAGE_OUT_BYTES;
            const float alpha = p.alpha, beta = p.beta;
            const uint32_t q = lane % CPR;
            auto chunk_off = [](uint32_t r, uint32_t j) {
                return OUT_COLS == 32 ? off_f32_chunk(r, j) : off_bf16_chunk(r, j);
            };
#pragma unroll
            for (int c = 0; c < ACC / OUT_COLS; ++c) {
                if (!owns(c * OUT_COLS / 32)) continue;  // another piece of a split tile stores it
#pragma unroll
                for (int j = 0; j < CPR; ++j)
                    *reinterpret_cast<float4*>(stage + chunk_off(lane, j)) =
                        make_float4(acc[OUT_COLS * c + 4 * j], acc[OUT_COLS * c + 4 * j + 1],
                                    acc[OUT_COLS * c + 4 * j + 2], acc[OUT_COLS * c + 4 * j + 3]);
                __syncwarp();
                const int gcol = col0 + OUT_COLS * c + static_cast<int>(4 * q);  // this lane's 4 columns
                const bool full4 = gcol + 3 < p.N;
                float4 bb = make_float4(0.f, 0.f, 0.f, 0.f);
                if (p.bias) {
                    if (full4) {
                        bb = __ldg(reinterpret_cast<const float4*>(p.bias + gcol));
                    } else {
                        if (gcol + 0 < p.N) bb.x = __ldg(p.bias + gcol + 0);
                        if (gcol + 1 < p.N) bb.y = __ldg(p.bias + gcol + 1);
                        if (gcol + 2 < p.N) bb.z = __ldg(p.bias + gcol + 2);
                    }
                }
#pragma unroll
                for (int pass = 0; pass < 32 / RPP; ++pass) {
                    const uint32_t rr = pass * RPP + lane / CPR;
                    const float4 v = *reinterpret_cast<const float4*>(stage + chunk_off(rr, q));
                    const int grow = row0 + static_cast<int>(rr);
                    if (grow >= p.M) continue;
                    float* dst = p.c + static_cast<long long>(grow) * p.ldc + gcol;
                    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (beta != 0.0f) {
                        const float* src_old = p.c_old + static_cast<long long>(grow) * p.ldc + gcol;
                        if (full4) {
                            o = *reinterpret_cast<const float4*>(src_old);
                        } else {
                            if (gcol + 0 < p.N) o.x = src_old[0];
                            if (gcol + 1 < p.N) o.y = src_old[1];
                            if (gcol + 2 < p.N) o.z = src_old[2];
                        }
                        o = make_float4(__fmul_rn(beta, o.x), __fmul_rn(beta, o.y), __fmul_rn(beta, o.z),
                                        __fmul_rn(beta, o.w));
                    }
                    const float4 r = make_float4(__fadd_rn(__fmaf_rn(alpha, v.x, o.x), bb.x),
                                                 __fadd_rn(__fmaf_rn(alpha, v.y, o.y), bb.y),
                                                 __fadd_rn(__fmaf_rn(alpha, v.z, o.z), bb.z),
                                                 __fadd_rn(__fmaf_rn(alpha, v.w, o.w), bb.w));
                    if (full4) {
                        *reinterpret_cast<float4*>(dst) = r;
                    } else {
                        if (gcol + 0 < p.N) dst[0] = r.x;
                        if (gcol + 1 < p.N) dst[1] = r.y;
                        if (gcol + 2 < p.N) dst[2] = r.z;
                    }
                }
                __syncwarp();  // staging buffer free for the next block
            }
        }
    }

    tc_fence_before();
    cluster_sync();  // no CTA leaves while its peer may still use its TMEM or barriers
    tc_fence_after();
    if (warp == WARP_MMA) tmem_dealloc_pair(tmem_base, TMEM_COLS);
}

}  // namespace emu
