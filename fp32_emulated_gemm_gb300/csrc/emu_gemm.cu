// emu_gemm.cu -- host side of libemu_gemm.so: argument checks, TMA tensor
// maps, launch of the sm_103a kernels, and the C ABI declared in
// include/emu_gemm.h.
//
// The method (blog "Unlocking Tensor Core performance for machine-learning
// interatomic potentials", "How Tensor Core FP32 bridges the hardware gap",
// Fig. 1, Fig. 2, Eq. 1) runs entirely in the kernels of emu_kernel.cuh; this
// file only marshals arguments.  There is no CPU fallback: without a suitable
// GPU every entry point returns an error.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <atomic>
#include <cmath>
#include <mutex>

#include "../../include/emu_gemm.h"
#include "emu_kernel.cuh"

namespace emu {
namespace {

constexpr unsigned long long kDefaultWaitBudgetNs = 2000000000ull;  // 2 s per wait

// EMU_LOG=1 prints each launch's plan (tiles, split, grid) to stderr.
bool log_enabled() {
    static const bool on = [] {
        const char* s = std::getenv("EMU_LOG");
        return s && s[0] && s[0] != '0';
    }();
    return on;
}


struct DeviceInfo {
    bool ready = false;
    int cc_major = 0, cc_minor = 0, sm_count = 0;
    bool attrs_set = false;
    int max_clusters[2] = {0, 0};  // co-resident CTA pairs per mode (all pipeline shapes)
};

// Split-K workspace: partial tiles plus per-tile arrival counters, owned by
// the library, one per (device, stream) so that calls on different streams
// never share it.  Grown on demand, kept until emu_shutdown() or the end of
// the process.  `epoch` numbers the launches that use its counters.
struct Workspace {
    int device = -1;
    cudaStream_t stream = nullptr;
    float* partials = nullptr;
    size_t partial_floats = 0;
    unsigned long long* counters = nullptr;
    size_t num_counters = 0;
    unsigned long long epoch = 0;
    void* packed = nullptr;   // op(B) split ahead of a product (automatic pre-split)
    size_t packed_bytes = 0;
};
constexpr int kMaxWorkspaces = 64;   // (device, stream) pairs with a workspace at once
Workspace g_ws[kMaxWorkspaces];

// Test hook (emu_debug_fail_allocations): the next n device allocations the
// library attempts fail as if the allocator were out of memory.
std::atomic<int> g_fail_allocs{0};

cudaError_t lib_malloc_async(void** ptr, size_t bytes, cudaStream_t stream) {
    int n = g_fail_allocs.load();
    while (n > 0) {
        if (g_fail_allocs.compare_exchange_weak(n, n - 1)) return cudaErrorMemoryAllocation;
    }
    return cudaMallocAsync(ptr, bytes, stream);
}

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
DeviceInfo g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

template <int MODE, int PIPE, bool STAGED = false>
cudaError_t set_smem_attr() {
    return cudaFuncSetAttribute(emu_gemm_kernel<MODE, PIPE, STAGED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                smem_bytes<MODE, PIPE>());
}

// the emulated modes (tensor cores); EMU_MODE_FP32 is the native one
bool emulated_mode(emu_mode_t mode) {
    return mode == EMU_MODE_BF16X9 || mode == EMU_MODE_TF32X3 || mode == EMU_MODE_TF32X1 ||
           mode == EMU_MODE_BF16X6;
}
bool valid_mode(emu_mode_t mode) { return emulated_mode(mode) || mode == EMU_MODE_FP32; }

const char* mode_name(emu_mode_t mode) {
    switch (mode) {
        case EMU_MODE_BF16X9: return "bf16x9";
        case EMU_MODE_TF32X3: return "tf32x3";
        case EMU_MODE_TF32X1: return "tf32x1";
        case EMU_MODE_BF16X6: return "bf16x6";
        case EMU_MODE_FP32: return "fp32";
    }
    return "?";
}

emu_status_t device_info(DeviceInfo** out) {
    int dev = 0;
    const cudaError_t ge = cudaGetDevice(&dev);
    if (ge != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        if (log_enabled()) std::fprintf(stderr, "[emu] cudaGetDevice: %s (device %d)\n", cudaGetErrorName(ge), dev);
        return EMU_STATUS_LAUNCH_FAILED;
    }
    // Bind the device's primary context to this host thread: a thread that has
    // not made a runtime call yet (e.g. an autograd worker) has none current,
    // and encoding a TMA tensor map needs one.
    const cudaError_t se = cudaSetDevice(dev);
    if (se != cudaSuccess) {
        cudaGetLastError();
        if (log_enabled()) std::fprintf(stderr, "[emu] cudaSetDevice: %s\n", cudaGetErrorName(se));
        return EMU_STATUS_LAUNCH_FAILED;
    }
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceInfo& d = g_dev[dev];
    if (!d.ready) {
        if (cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return EMU_STATUS_LAUNCH_FAILED;
        }
        d.ready = true;
    }
    if (d.cc_major != 10 || d.cc_minor != 3) return EMU_STATUS_ARCH_MISMATCH;
    if (!g_encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) {
            cudaGetLastError();
            return EMU_STATUS_LAUNCH_FAILED;
        }
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    if (!d.attrs_set) {
        if (set_smem_attr<MODE_BF16X9, PIPE_SHORT_K>() != cudaSuccess ||
            set_smem_attr<MODE_BF16X9, PIPE_LONG_K>() != cudaSuccess ||
            set_smem_attr<MODE_BF16X6, PIPE_SHORT_K>() != cudaSuccess ||
            set_smem_attr<MODE_BF16X6, PIPE_LONG_K>() != cudaSuccess ||
            set_smem_attr<MODE_TF32X3, PIPE_SHORT_K>() != cudaSuccess ||
            set_smem_attr<MODE_TF32X1, PIPE_SHORT_K>() != cudaSuccess ||
            set_smem_attr<MODE_BF16X9, PIPE_SHORT_K_PACKED>() != cudaSuccess ||
            set_smem_attr<MODE_BF16X9, PIPE_LONG_K_PACKED>() != cudaSuccess ||
            set_smem_attr<MODE_BF16X6, PIPE_SHORT_K_PACKED>() != cudaSuccess ||
            set_smem_attr<MODE_BF16X6, PIPE_LONG_K_PACKED>() != cudaSuccess ||
            set_smem_attr<MODE_TF32X3, PIPE_SHORT_K_PACKED>() != cudaSuccess ||
            set_smem_attr<MODE_TF32X1, PIPE_SHORT_K_PACKED>() != cudaSuccess ||
            set_smem_attr<MODE_BF16X9, PIPE_SHORT_K, true>() != cudaSuccess ||
            set_smem_attr<MODE_BF16X9, PIPE_LONG_K, true>() != cudaSuccess ||
            set_smem_attr<MODE_BF16X9, PIPE_SHORT_K_PACKED, true>() != cudaSuccess ||
            set_smem_attr<MODE_BF16X9, PIPE_LONG_K_PACKED, true>() != cudaSuccess ||
            set_smem_attr<MODE_TF32X3, PIPE_SHORT_K, true>() != cudaSuccess ||
            set_smem_attr<MODE_TF32X3, PIPE_SHORT_K_PACKED, true>() != cudaSuccess) {
            cudaGetLastError();
            return EMU_STATUS_LAUNCH_FAILED;
        }
        // how many CTA pairs can be resident at once (the persistent grid);
        // every shape uses one CTA per SM, so the smallest count serves all
        for (int m = 0; m < 2; ++m) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(2 * (d.sm_count / 2), 1, 1);
            cfg.blockDim = dim3(NUM_THREADS, 1, 1);
            cfg.dynamicSmemBytes = m == 0 ? smem_bytes<MODE_BF16X9, PIPE_SHORT_K>()
                                          : smem_bytes<MODE_TF32X3, PIPE_SHORT_K>();
            int n = 0;
            const cudaError_t e = m == 0
                ? cudaOccupancyMaxActiveClusters(&n, emu_gemm_kernel<MODE_BF16X9, PIPE_SHORT_K>, &cfg)
                : cudaOccupancyMaxActiveClusters(&n, emu_gemm_kernel<MODE_TF32X3, PIPE_SHORT_K>, &cfg);
            if (e != cudaSuccess || n <= 0) {
                cudaGetLastError();
                n = d.sm_count / 2;
            }
            d.max_clusters[m] = n;
        }
        d.attrs_set = true;
    }
    *out = &d;
    return EMU_STATUS_SUCCESS;
}

// FP32 2-D tensor map over a row-major matrix with `outer` rows of `inner`
// elements (leading dimension ld), box {box_inner, box_outer}, 128-byte
// swizzle, zero fill outside the matrix.
bool encode_f32_2d(CUtensorMap* map, const float* base, uint64_t inner, uint64_t outer, uint64_t ld,
                   uint32_t box_inner, uint32_t box_outer) {
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {ld * sizeof(float)};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides,
                                box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS && log_enabled())
        std::fprintf(stderr, "[emu] tensor map encode failed (%d): base %p dims %llu x %llu ld %llu box %u x %u\n",
                     (int)r, (const void*)base, (unsigned long long)inner, (unsigned long long)outer,
                     (unsigned long long)ld, box_inner, box_outer);
    return r == CUDA_SUCCESS;
}

// op(X) tile map for tiles of `rows` rows (128 for op(A), TN / 2 for op(B)):
// K-major operands (rows of K) load one {32 k, rows} box; MN-major operands
// (rows of MN) load rows / 32 boxes of {32 mn, 32 k}.
bool encode_operand(CUtensorMap* map, const float* X, bool mn_major, int64_t MN, int64_t K, int64_t ld,
                    uint32_t rows) {
    // TMA needs every extent >= 1; a zero extent never reaches here.
    if (!mn_major) return encode_f32_2d(map, X, (uint64_t)K, (uint64_t)MN, (uint64_t)ld, BK, rows);
    return encode_f32_2d(map, X, (uint64_t)MN, (uint64_t)K, (uint64_t)ld, 32, BK);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Packed op(B) (emu_pack_b): the components of op(B)^T, one plane per
// component, each `rows` rows of Kp = K rounded up to 32 elements, zero past
// K: BF16 words for the BF16 modes, FP32 words (TF32 values) for the TF32
// modes.  A stage's box of a plane lands in shared memory in the kernel's
// component layout (64-byte BF16 rows with the 64-byte swizzle, 128-byte TF32
// rows with the 128-byte swizzle).
int ncomp_of(emu_mode_t mode) { return mode == EMU_MODE_TF32X3 ? 2 : mode == EMU_MODE_TF32X1 ? 1 : 3; }
int64_t elem_bytes_of(emu_mode_t mode) { return mode == EMU_MODE_TF32X3 || mode == EMU_MODE_TF32X1 ? 4 : 2; }
__host__ __device__ inline int64_t packed_kp(int64_t K) { return (K + BK - 1) / BK * BK; }
int64_t packed_bytes(emu_mode_t mode, int64_t rows, int64_t K) {
    return ncomp_of(mode) * rows * packed_kp(K) * elem_bytes_of(mode);
}

bool encode_packed(CUtensorMap* map, const void* packed, emu_mode_t mode, int64_t rows, int64_t K) {
    const int64_t es = elem_bytes_of(mode), kp = packed_kp(K);
    const cuuint64_t dims[3] = {(cuuint64_t)kp, (cuuint64_t)rows, (cuuint64_t)ncomp_of(mode)};
    const cuuint64_t strides[2] = {(cuuint64_t)(kp * es), (cuuint64_t)(rows * kp * es)};
    const cuuint32_t box[3] = {BK, (cuuint32_t)(TILE_M / 2), 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = g_encode(map, es == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3,
                                const_cast<void*>(packed), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                es == 2 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS && log_enabled())
        std::fprintf(stderr, "[emu] packed tensor map encode failed (%d): rows %lld K %lld\n", (int)r,
                     (long long)rows, (long long)K);
    return r == CUDA_SUCCESS;
}

// One thread per (row of op(B)^T, 8 consecutive k): the kernel's own split
// of those 8 values, written to every plane.
template <int MODE>
__global__ void pack_kernel(int64_t rows, int64_t K, const float* B, int64_t ldb, int b_k_major, void* packed) {
    using C = Cfg<MODE>;
    const int64_t kp = packed_kp(K), groups = kp / 8, total = rows * groups;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t n = i / groups, k0 = (i % groups) * 8;
        float x[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int64_t k = k0 + j;
            x[j] = k < K ? (b_k_major ? B[n * ldb + k] : B[k * ldb + n]) : 0.0f;
        }
        const int64_t plane = rows * kp;  // elements per plane
        if constexpr (!C::TF32) {
            uint4 s0, s1, s2;
            split_bf16x9_8(x, s0, s1, s2);
            uint16_t* out = reinterpret_cast<uint16_t*>(packed) + n * kp + k0;
            *reinterpret_cast<uint4*>(out) = s0;
            *reinterpret_cast<uint4*>(out + plane) = s1;
            *reinterpret_cast<uint4*>(out + 2 * plane) = s2;
        } else {
            uint32_t h[8], l[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if constexpr (C::NCOMP == 2) split_tf32x3_1(x[j], h[j], l[j]);
                else h[j] = tf32_rn_bits(__float_as_uint(x[j]));
            }
            uint32_t* out = reinterpret_cast<uint32_t*>(packed) + n * kp + k0;
            *reinterpret_cast<uint4*>(out) = make_uint4(h[0], h[1], h[2], h[3]);
            *reinterpret_cast<uint4*>(out + 4) = make_uint4(h[4], h[5], h[6], h[7]);
            if constexpr (C::NCOMP == 2) {
                *reinterpret_cast<uint4*>(out + plane) = make_uint4(l[0], l[1], l[2], l[3]);
                *reinterpret_cast<uint4*>(out + plane + 4) = make_uint4(l[4], l[5], l[6], l[7]);
            }
        }
    }
}

// ---------------------------------------------------------- native FP32 ----
// C = alpha op(A) op(B) + beta C_old + bias on the CUDA cores: each output is
// one chain acc = fmaf(a_k, b_k, acc) over k = 0, 1, ..., K-1 from acc = +0,
// then C = fmaf(alpha, acc, beta * C_old) (beta == 0: C_old not read), plus
// the bias when there is one.  A block of 16 x 16 threads computes a 16R x 16R
// tile of C, R x R outputs per thread (rows R ty + i, columns R tx + j), from
// k-slices of depth KT = 64 / R staged in shared memory (the smaller the
// tile, the longer the slice: fewer load round trips per chain).  The chains
// cannot be split along k, so small outputs take a smaller R to occupy the SMs.
constexpr int NAT_MAX_GRID_Y = 65535;
template <int R>
__global__ void __launch_bounds__(256) native_sgemm_kernel(int M, int N, int K, float alpha, const float* A,
                                                           long long lda, int a_mn, const float* B, long long ldb,
                                                           int b_mn, float beta, float* C, long long ldc,
                                                           const float* bias) {
    constexpr int T = 16 * R, LD = T + 4;  // +4: fewer bank conflicts, rows stay 16-byte aligned
    constexpr int KT = 64 / R;             // slice depth
    constexpr int NQ = KT * T / 256;       // elements of each operand's slice per thread (4)
    __shared__ __align__(16) float As[KT][LD];
    __shared__ __align__(16) float Bs[KT][LD];
    const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
    const int m0 = blockIdx.x * T, n0 = blockIdx.y * T;
    float acc[R][R];
#pragma unroll
    for (int i = 0; i < R; ++i)
#pragma unroll
        for (int j = 0; j < R; ++j) acc[i][j] = 0.0f;
    // each slice is KT x T elements, NQ per thread: element e = threadIdx.x + 256 q
    // is (k, r) = (e / T, e % T) for an MN-major source and (e % KT, e / KT)
    // for a K-major one, so that neighbouring threads read neighbouring
    // addresses.  The next slice is fetched into registers while the current
    // one is used.
    float ra_[NQ], rb_[NQ];
    auto fetch = [&](int k0) {
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            const int e = threadIdx.x + 256 * q;
            const int ka = a_mn ? e / T : e % KT, ra = a_mn ? e % T : e / KT;
            const int gm = m0 + ra, gka = k0 + ka;
            ra_[q] = (gm < M && gka < K) ? A[a_mn ? (long long)gka * lda + gm : (long long)gm * lda + gka] : 0.0f;
            const int kb = b_mn ? e / T : e % KT, cb = b_mn ? e % T : e / KT;
            const int gn = n0 + cb, gkb = k0 + kb;
            rb_[q] = (gn < N && gkb < K) ? B[b_mn ? (long long)gkb * ldb + gn : (long long)gn * ldb + gkb] : 0.0f;
        }
    };
    auto step = [&](int k) {
        float av[R], bv[R];
        if constexpr (R == 4) {
            const float4 a = *reinterpret_cast<const float4*>(&As[k][4 * ty]);
            const float4 b = *reinterpret_cast<const float4*>(&Bs[k][4 * tx]);
            av[0] = a.x; av[1] = a.y; av[2] = a.z; av[3] = a.w;
            bv[0] = b.x; bv[1] = b.y; bv[2] = b.z; bv[3] = b.w;
        } else if constexpr (R == 2) {
            const float2 a = *reinterpret_cast<const float2*>(&As[k][2 * ty]);
            const float2 b = *reinterpret_cast<const float2*>(&Bs[k][2 * tx]);
            av[0] = a.x; av[1] = a.y;
            bv[0] = b.x; bv[1] = b.y;
        } else {
            av[0] = As[k][ty];
            bv[0] = Bs[k][tx];
        }
#pragma unroll
        for (int i = 0; i < R; ++i)
#pragma unroll
            for (int j = 0; j < R; ++j) acc[i][j] = __fmaf_rn(av[i], bv[j], acc[i][j]);
    };
    if (K > 0) fetch(0);
    for (int k0 = 0; k0 < K; k0 += KT) {
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            const int e = threadIdx.x + 256 * q;
            As[a_mn ? e / T : e % KT][a_mn ? e % T : e / KT] = ra_[q];
            Bs[b_mn ? e / T : e % KT][b_mn ? e % T : e / KT] = rb_[q];
        }
        __syncthreads();
        if (k0 + KT < K) fetch(k0 + KT);
        if (K - k0 >= KT) {
#pragma unroll
            for (int k = 0; k < KT; ++k) step(k);
        } else {
            for (int k = 0; k < K - k0; ++k) step(k);  // only k < K enters the chains
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < R; ++i) {
        const int gm = m0 + R * ty + i;
        if (gm >= M) continue;
#pragma unroll
        for (int j = 0; j < R; ++j) {
            const int gn = n0 + R * tx + j;
            if (gn >= N) continue;
            float* c = C + (long long)gm * ldc + gn;
            const float bc = beta != 0.0f ? __fmul_rn(beta, *c) : 0.0f;
            float v = __fmaf_rn(alpha, acc[i][j], bc);
            if (bias) v = __fadd_rn(v, bias[gn]);
            *c = v;
        }
    }
}

// The largest R whose grid still gives every SM a block.
int native_r(int64_t M, int64_t N, int sm_count) {
    for (int R = 4; R > 1; R /= 2) {
        const int64_t t = 16 * R, blocks = ((M + t - 1) / t) * ((N + t - 1) / t);
        if (blocks >= sm_count && (N + t - 1) / t <= NAT_MAX_GRID_Y) return R;
    }
    return 1;
}

cudaError_t launch_native(int64_t M, int64_t N, int64_t K, float alpha, const float* A, int64_t lda, bool a_mn,
                          const float* B, int64_t ldb, bool b_mn, float beta, float* C, int64_t ldc,
                          const float* bias, int sm_count, cudaStream_t stream) {
    int R = native_r(M, N, sm_count);
    while (R < 4 && (N + 16 * R - 1) / (16 * R) > NAT_MAX_GRID_Y) R *= 2;
    const int64_t t = 16 * R, gx = (M + t - 1) / t, gy = (N + t - 1) / t;
    if (gy > NAT_MAX_GRID_Y || gx > INT32_MAX) return cudaErrorInvalidConfiguration;
    const dim3 grid((unsigned)gx, (unsigned)gy, 1);
    cudaGetLastError();
    switch (R) {
        case 4: native_sgemm_kernel<4><<<grid, 256, 0, stream>>>((int)M, (int)N, (int)K, alpha, A, lda, a_mn, B, ldb,
                                                                 b_mn, beta, C, ldc, bias); break;
        case 2: native_sgemm_kernel<2><<<grid, 256, 0, stream>>>((int)M, (int)N, (int)K, alpha, A, lda, a_mn, B, ldb,
                                                                 b_mn, beta, C, ldc, bias); break;
        default: native_sgemm_kernel<1><<<grid, 256, 0, stream>>>((int)M, (int)N, (int)K, alpha, A, lda, a_mn, B,
                                                                  ldb, b_mn, beta, C, ldc, bias);
    }
    return cudaGetLastError();
}

std::atomic<int> g_strategy{EMU_STRATEGY_EAGER};

// Predicted GPU times in microseconds on GB300, fitted to measured kernel
// times (CUDA graphs of back-to-back calls, 66 shapes from 64^3 to 2048^3,
// rms error about 6% emulated and 14% native).  Emulated: a fixed start-up,
// the plan's pipeline stages (waves x (k-stages + stores)) at the mode's
// stage time, and for split tiles a reduction that grows with the pieces per
// tile.  Native: a fixed cost plus, per k of the chains, a latency term that
// depends on the micro-tile and a throughput term that grows with the FMAs
// each SM carries.
struct EmuTimeModel { double fixed, stage, split_fixed, split_per_piece; };
EmuTimeModel emu_time_model(emu_mode_t mode) {
    switch (mode) {
        case EMU_MODE_BF16X9: return {3.8, 1.262, 2.64, 0.51};
        case EMU_MODE_TF32X3: return {3.9, 1.572, 2.96, 0.44};
        // the comparators were not fitted: BF16x9's start-up and reduction,
        // stage times estimated from their share of the MMA work
        case EMU_MODE_BF16X6: return {3.8, 1.0, 2.64, 0.51};
        default: return {3.8, 0.8, 2.64, 0.51};  // TF32x1
    }
}
constexpr double kNatFixedUs = 1.46, kNatPerFmaPerSmUs = 1.105e-5;
// per k of the chain, by micro-tile size R = 1, 2, 4
double nat_per_k_us(int R) { return R == 1 ? 0.0172 : R == 2 ? 0.0254 : 0.0292; }

__global__ void scale_kernel(int64_t M, int64_t N, float beta, float* C, int64_t ldc, const float* bias) {
    const int64_t total = M * N;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / N, c = i % N;
        float* e = C + r * ldc + c;
        const float v = beta != 0.0f ? __fmul_rn(beta, *e) : 0.0f;
        *e = __fadd_rn(v, bias ? bias[c] : 0.0f);
    }
}

emu_status_t check_error_flag(bool clear) {
    unsigned int flag = 0;
    if (cudaMemcpyFromSymbol(&flag, g_error_flag, sizeof(flag)) != cudaSuccess) {
        cudaGetLastError();
        return EMU_STATUS_LAUNCH_FAILED;
    }
    if (flag && clear) {
        const unsigned int zero = 0;
        cudaMemcpyToSymbol(g_error_flag, &zero, sizeof(zero));
    }
    return flag ? EMU_STATUS_DEVICE_TIMEOUT : EMU_STATUS_SUCCESS;
}

// The slot of (device, stream) in the workspace table, taken on first use;
// nullptr when all kMaxWorkspaces slots hold other pairs.  Caller holds g_mutex.
Workspace* workspace_slot(int dev, cudaStream_t stream) {
    for (auto& c : g_ws)
        if (c.device == dev && c.stream == stream) return &c;
    for (auto& c : g_ws)
        if (c.device < 0) { c.device = dev; c.stream = stream; return &c; }
    return nullptr;
}

// The workspace for (current device, stream) with at least `floats` partial
// floats and `counters` arrival counters, and a new epoch for the launch
// about to use it.  Allocation happens only when the cached one is too
// small; new counters are zeroed on the stream (epoch 0, which no launch
// uses).
emu_status_t workspace_for(int dev, cudaStream_t stream, size_t floats, size_t counters, Workspace** out,
                           unsigned long long* epoch) {
    std::lock_guard<std::mutex> lock(g_mutex);
    Workspace* w = workspace_slot(dev, stream);
    if (!w) return EMU_STATUS_ALLOC_FAILED;
    if (w->partial_floats < floats) {
        if (w->partials && cudaFreeAsync(w->partials, stream) != cudaSuccess) cudaGetLastError();
        w->partials = nullptr;
        w->partial_floats = 0;
        if (lib_malloc_async(reinterpret_cast<void**>(&w->partials), floats * sizeof(float), stream) != cudaSuccess) {
            cudaGetLastError();
            return EMU_STATUS_ALLOC_FAILED;
        }
        w->partial_floats = floats;
    }
    if (w->num_counters < counters) {
        if (w->counters && cudaFreeAsync(w->counters, stream) != cudaSuccess) cudaGetLastError();
        w->counters = nullptr;
        w->num_counters = 0;
        const size_t bytes = counters * sizeof(unsigned long long);
        if (lib_malloc_async(reinterpret_cast<void**>(&w->counters), bytes, stream) != cudaSuccess ||
            cudaMemsetAsync(w->counters, 0, bytes, stream) != cudaSuccess) {
            cudaGetLastError();
            return EMU_STATUS_ALLOC_FAILED;
        }
        w->num_counters = counters;
    }
    *epoch = ++w->epoch;
    *out = w;
    return EMU_STATUS_SUCCESS;
}

// A buffer for an automatically pre-split op(B), per (device, stream), grown
// on demand and kept.
emu_status_t packed_buffer_for(int dev, cudaStream_t stream, size_t bytes, void** out) {
    std::lock_guard<std::mutex> lock(g_mutex);
    Workspace* w = workspace_slot(dev, stream);
    if (!w) return EMU_STATUS_ALLOC_FAILED;
    if (w->packed_bytes < bytes) {
        if (w->packed && cudaFreeAsync(w->packed, stream) != cudaSuccess) cudaGetLastError();
        w->packed = nullptr;
        w->packed_bytes = 0;
        if (lib_malloc_async(&w->packed, bytes, stream) != cudaSuccess) {
            cudaGetLastError();
            return EMU_STATUS_ALLOC_FAILED;
        }
        w->packed_bytes = bytes;
    }
    *out = w->packed;
    return EMU_STATUS_SUCCESS;
}

// Automatic pre-split of op(B): for the TF32 modes the split is costly enough
// that splitting op(B) once per product, ahead of it, and loading its
// components pays as soon as several tile rows share them (measured 1.2-1.6x
// on the PET and wide-layer shapes); for the BF16 modes it measured no gain.
// EMU_AUTOPACK=0 turns it off.
constexpr int kAutoPackMinTileRows = 4;
constexpr size_t kAutoPackMaxBytes = size_t(1) << 30;

// The launch plan: pipeline shape, tiles, and how tiles become work units.
struct Plan {
    int pipe;       // PIPE_SHORT_K or PIPE_LONG_K
    int tn;         // pair tile width
    int tiles_m, tiles_n, num_tiles, k_stages;
    int tiles_a, split_a, split_b;  // see Params
    int num_units;
    int chain;      // 1: chained plan (see emu_kernel.cuh); tiles_a = all tiles, whole
    int clusters;   // CTA pairs launched
    long long slots;  // workspace partial tiles (0: no split tile)
    double cost;      // predicted time in pipeline stages (see below)
    long long chain_bound[kMaxChainPairs + 1];  // chained plans: the pairs' stage runs
};

// Long k-loops per work unit favour three component stages; short ones the
// wider output staging (see PipeCfg).
constexpr int kLongKMinStages = 16;

// Costs in units of one pipeline stage (measured on GB300): every work unit
// pays its k-stages plus about 3 stages of output stores, which the two TMEM
// accumulators cannot hide; split tiles add the reduce-scatter (publishing
// (S-1)/S of a partial tile and reading the owned parts back), about 1.5
// stages.  Units run in waves over the resident CTA pairs.
constexpr double kStoreStages = 3.0, kReduceStages = 1.5;

int env_int(const char* name, int dflt) {
    const char* v = std::getenv(name);
    return v ? std::atoi(v) : dflt;
}

// Chained plans (T >= pairs tiles of KS stages; the U = T KS stages taken
// tile by tile, pair c runs [bound[c], bound[c + 1])).  What a pair's run
// costs, in pipeline stages: its stages, plus, at each step from one unit to
// the next, the part of the first unit's output phase (128 KB of stores per
// CTA, or its published running sum) that the next unit's first two stages
// do not hide.  Measured on GB300 with globaltimer stamps of the PET-small
// forward pass (pairs of 8-11 stages; the end of each pair against a pair
// that runs one whole tile): head -> whole tile 1.1 stages, head -> tail
// 1.6, whole tile -> tail 4 (the short tails that follow a whole tile give
// the tensor cores too little work to cover the tile's output phase, and
// their starting-sum loads only go out after it), whole tile -> whole tile
// about 2.  Every run covers at least one tile end or start (a run strictly
// inside one tile would cut it twice).
constexpr double kChainHeadToTile = 1.1, kChainHeadToTail = 1.6, kChainTileToTile = 2.0, kChainTileToTail = 4.0;
constexpr int kChainSlack = 2;  // each bound within this many stages of the even cut c U / pairs
static_assert(kChainSlack <= 127, "bounds travel to the kernel as signed bytes (Params::chain_delta)");
double chain_run_cost(long long s, long long e, int KS) {
    if (e <= s) return -1.0;
    const long long t0 = s / KS, t1 = (e - 1) / KS;
    const long long units = t1 - t0 + 1, lo = s - t0 * KS, hi = e - t1 * KS;
    if (units == 1 && lo > 0 && hi < KS) return -1.0;
    double c = (double)(e - s);
    if (units == 1) return c;
    const bool head = lo > 0, tail = hi < KS;
    if (units == 2) return c + (head ? (tail ? kChainHeadToTail : kChainHeadToTile) : (tail ? kChainTileToTail : kChainTileToTile));
    return c + (head ? kChainHeadToTile : kChainTileToTile) + kChainTileToTile * (double)(units - 3) +
           (tail ? kChainTileToTail : kChainTileToTile);
}

struct ChainPlan {
    double cost;
    int units, cuts;
    long long bound[kMaxChainPairs + 1];
};

// The bounds that minimise the slowest pair's cost (then the total), each
// within kChainSlack stages of the even cut: a bottleneck shortest path over
// the candidate bounds, O(pairs (2 kChainSlack + 1)^2).  False when no valid
// set exists.
bool chain_bounds_optimised(long long U, int KS, int pairs, ChainPlan* out) {
    constexpr int W = 2 * kChainSlack + 1;
    long long cand[kMaxChainPairs + 1][W];
    int ncand[kMaxChainPairs + 1];
    double best_max[kMaxChainPairs + 1][W], best_sum[kMaxChainPairs + 1][W];
    int prev[kMaxChainPairs + 1][W];
    for (int c = 0; c <= pairs; ++c) {
        ncand[c] = 0;
        if (c == 0 || c == pairs) { cand[c][0] = c == 0 ? 0 : U; ncand[c] = 1; continue; }
        const long long even = (long long)c * U / pairs;
        for (int d = -kChainSlack; d <= kChainSlack; ++d) {
            const long long v = even + d;
            if (v >= 1 && v <= U - 1) cand[c][ncand[c]++] = v;
        }
    }
    best_max[0][0] = 0.0; best_sum[0][0] = 0.0; prev[0][0] = -1;
    for (int c = 1; c <= pairs; ++c) {
        for (int i = 0; i < ncand[c]; ++i) {
            best_max[c][i] = -1.0;
            for (int j = 0; j < ncand[c - 1]; ++j) {
                if (best_max[c - 1][j] < 0.0) continue;
                const double rc = chain_run_cost(cand[c - 1][j], cand[c][i], KS);
                if (rc < 0.0) continue;
                const double mx = best_max[c - 1][j] > rc ? best_max[c - 1][j] : rc;
                const double sm = best_sum[c - 1][j] + rc;
                if (best_max[c][i] < 0.0 || mx < best_max[c][i] - 1e-9 ||
                    (mx < best_max[c][i] + 1e-9 && sm < best_sum[c][i] - 1e-9)) {
                    best_max[c][i] = mx; best_sum[c][i] = sm; prev[c][i] = j;
                }
            }
        }
    }
    if (best_max[pairs][0] < 0.0) return false;
    out->cost = best_max[pairs][0];
    for (int c = pairs, i = 0; c >= 0; --c) {
        out->bound[c] = cand[c][i];
        if (c > 0) i = prev[c][i];
    }
    return true;
}

// The even cuts c U / pairs, without optimisation (a diagnostic choice).
bool chain_bounds_even(long long U, int KS, int pairs, ChainPlan* out) {
    out->cost = 0.0;
    for (int c = 0; c <= pairs; ++c) out->bound[c] = (long long)c * U / pairs;
    for (int c = 0; c < pairs; ++c) {
        const double rc = chain_run_cost(out->bound[c], out->bound[c + 1], KS);
        if (rc < 0.0) return false;
        out->cost = rc > out->cost ? rc : out->cost;
    }
    return true;
}

bool chain_plan(long long T, int KS, int pairs, bool even_cuts, ChainPlan* out) {
    if (pairs < 1 || pairs > kMaxChainPairs || T < pairs) return false;
    const long long U = T * KS;
    if (!(even_cuts ? chain_bounds_even(U, KS, pairs, out) : chain_bounds_optimised(U, KS, pairs, out)))
        return false;
    out->units = 0; out->cuts = 0;
    for (int c = 0; c < pairs; ++c) {
        out->units += (int)((out->bound[c + 1] - 1) / KS - out->bound[c] / KS + 1);
        if (c > 0 && out->bound[c] % KS != 0) ++out->cuts;
    }
    return true;
}

// Candidate plans (a split tile's S pieces wait for one another, so they
// must run in the same wave of units: S is at most the number of pairs, and
// at most 32, the 32-column chunks of a CTA's half-tile):
//   uniform: every tile in S pieces; with more than one wave the pairs in
//     use are a multiple of S, so that waves hold whole tiles;
//   hybrid: W full waves of whole tiles on all pairs, then the remaining
//     tiles (fewer than the pairs) in S pieces, one more wave at most;
//   chained: at least as many tiles as pairs, every pair one run of stages
//     (chain_plan), a tile cut at a run boundary finished by the pair whose
//     run ends there.
// EMU_SPLIT_K (uniform S), EMU_SPLIT_TAIL (hybrid with that S for the
// remaining tiles, where a hybrid plan exists), EMU_CHAIN (0: never chained;
// 1: chained wherever it is possible; 2: the same with the even cuts
// c U / pairs instead of the optimised bounds) and EMU_PIPE (0 short-k,
// 1 long-k) override the choice, for diagnostics and tuning.
Plan make_plan(int64_t M, int64_t N, int64_t K, int pairs) {
    Plan plan{};
    plan.tn = 256;
    plan.tiles_m = (int)((M + TILE_M - 1) / TILE_M);
    plan.tiles_n = (int)((N + plan.tn - 1) / plan.tn);
    plan.num_tiles = plan.tiles_m * plan.tiles_n;
    plan.k_stages = (int)((K + BK - 1) / BK);
    const long long T = plan.num_tiles;
    const int KS = plan.k_stages;
    auto set_uniform = [&](int S) {
        plan.tiles_a = (int)T; plan.split_a = S; plan.split_b = 1;
        const long long units = T * S;
        const long long used = units <= pairs || S == 1 ? pairs : pairs / S * S;
        plan.clusters = (int)(units < used ? units : used);
    };
    auto cost_uniform = [&](int S) {
        const long long units = T * S;
        const long long used = units <= pairs || S == 1 ? pairs : pairs / S * S;
        const long long waves = (units + used - 1) / used;
        return (double)waves * ((KS + S - 1) / S + kStoreStages) + (S > 1 ? kReduceStages : 0.0);
    };
    const int force_split = env_int("EMU_SPLIT_K", 0);
    const int force_tail = env_int("EMU_SPLIT_TAIL", 0);
    const int s_max = KS < 32 ? KS : 32;
    const long long W0 = T / pairs, tail0 = T - W0 * pairs;
    const bool tail_forced = force_split < 1 && force_tail >= 2 && W0 >= 1 && tail0 >= 1 && force_tail <= s_max &&
                             tail0 * force_tail <= pairs;
    if (tail_forced) {
        const int S = force_tail;
        plan.tiles_a = (int)(W0 * pairs); plan.split_a = 1; plan.split_b = S;
        plan.clusters = pairs;
        plan.cost = (double)W0 * (KS + kStoreStages) + ((KS + S - 1) / S + kStoreStages) + kReduceStages;
    } else if (force_split >= 1) {
        int S = force_split < s_max ? force_split : s_max;
        S = S < pairs ? S : pairs;
        set_uniform(S);
        plan.cost = cost_uniform(S);
    } else {
        double best = -1.0;
        for (int S = 1; S <= s_max && S <= pairs; ++S) {
            if (S > 1 && KS / S < 2) break;
            const double c = cost_uniform(S);
            if (best < 0 || c < best - 1e-9) { best = c; set_uniform(S); }
        }
        const long long W = T / pairs, tail = T - W * pairs;
        if (W >= 1 && tail >= 1) {
            for (int S = 2; S <= s_max && tail * S <= pairs; ++S) {
                if (KS / S < 2) break;
                const double c = (double)W * (KS + kStoreStages) + ((KS + S - 1) / S + kStoreStages) + kReduceStages;
                if (c < best - 1e-9) {
                    best = c;
                    plan.tiles_a = (int)(W * pairs); plan.split_a = 1; plan.split_b = S;
                    plan.clusters = pairs;
                }
            }
        }
        plan.cost = best;
    }
    plan.num_units = plan.tiles_a * plan.split_a + (plan.num_tiles - plan.tiles_a) * plan.split_b;
    plan.slots = (plan.split_a > 1 ? (long long)plan.tiles_a * plan.split_a : 0) +
                 (plan.split_b > 1 ? (long long)(plan.num_tiles - plan.tiles_a) * plan.split_b : 0);
    const int force_chain = env_int("EMU_CHAIN", -1);
    if (force_split < 1 && !tail_forced && force_chain != 0 && T >= pairs && T > 1) {
        // without a cut tile a chained plan splits the work as whole-tile
        // waves do, so it is taken only when forced
        ChainPlan c;
        if (chain_plan(T, KS, pairs, force_chain == 2, &c) &&
            (force_chain >= 1 || (c.cuts > 0 && c.cost < plan.cost - 1e-9))) {
            plan.tiles_a = (int)T; plan.split_a = 1; plan.split_b = 1;
            plan.chain = 1;
            plan.clusters = pairs;
            plan.num_units = c.units;
            plan.slots = c.cuts > 0 ? pairs - 1 : 0;
            plan.cost = c.cost;
            for (int i = 0; i <= pairs; ++i) plan.chain_bound[i] = c.bound[i];
        }
    }
    const int per_unit = (KS + plan.split_a - 1) / plan.split_a;
    const int force_pipe = env_int("EMU_PIPE", -1);
    plan.pipe = force_pipe == PIPE_SHORT_K || force_pipe == PIPE_LONG_K ? force_pipe
              : per_unit >= kLongKMinStages ? PIPE_LONG_K : PIPE_SHORT_K;
    return plan;
}

// The mode a product runs in: the requested one, except that the performant
// strategy runs an emulated product in native FP32 when that is predicted
// faster.  `pairs`: the device's co-resident CTA pairs; `sm_count`: its SMs.
emu_mode_t dispatch_mode(emu_mode_t mode, int64_t M, int64_t N, int64_t K, int pairs, int sm_count) {
    if (mode == EMU_MODE_FP32 || g_strategy.load(std::memory_order_relaxed) != EMU_STRATEGY_PERFORMANT) return mode;
    const Plan plan = make_plan(M, N, K, pairs);
    const int S = plan.split_a > plan.split_b ? plan.split_a : plan.split_b;
    const EmuTimeModel em = emu_time_model(mode);
    const double emu_us = em.fixed + em.stage * (plan.cost - (S > 1 ? kReduceStages : 0.0)) +
                          (S > 1 ? em.split_fixed + em.split_per_piece * S : 0.0);
    const int R = native_r(M, N, sm_count);
    const double t = 16.0 * R, blocks = std::ceil((double)M / t) * std::ceil((double)N / t);
    const double fma_per_sm_per_k = blocks / sm_count * 256.0 * R * R;
    const double nat_us = kNatFixedUs + (double)K * (nat_per_k_us(R) + kNatPerFmaPerSmUs * fma_per_sm_per_k);
    return nat_us < emu_us ? EMU_MODE_FP32 : mode;
}

unsigned long long wait_budget_ns() {
    static unsigned long long v = [] {
        const char* s = std::getenv("EMU_WAIT_BUDGET_NS");
        unsigned long long x = s ? std::strtoull(s, nullptr, 10) : 0ull;
        return x ? x : kDefaultWaitBudgetNs;
    }();
    return v;
}

template <int MODE, int PIPE, bool STAGED = false>
cudaError_t launch_one(cudaLaunchConfig_t cfg, const Params& p) {
    cfg.dynamicSmemBytes = smem_bytes<MODE, PIPE>();
    return cudaLaunchKernelEx(&cfg, emu_gemm_kernel<MODE, PIPE, STAGED>, p);
}

// Uniform plans whose tiles are split into this many pieces or more use the
// kernel's staged reduction (BF16x9 and TF32x3; the comparators keep the
// register one).
constexpr int kStagedMinPieces = 12;

// The launch's own status (cudaLaunchKernelEx), so that an error left by an
// unrelated earlier runtime call on this host thread is not reported as ours.
// Programmatic dependent launch (EMU_PDL=0 turns it off): the kernel may be
// scheduled while the previous kernel in the stream finishes; it runs its
// set-up and then waits for that kernel before touching global memory.
bool pdl_enabled() {
    static const bool v = env_int("EMU_PDL", 1) != 0;
    return v;
}

cudaError_t launch_gemm(emu_mode_t mode, int pipe, const Params& p, int clusters, cudaStream_t stream) {
    // only uniform plans: in a hybrid plan the split tail is a small part of
    // the work, and the whole tiles run measurably slower in the staged build
    const bool staged = p.split_a >= kStagedMinPieces;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * clusters, 1, 1);
    cfg.blockDim = dim3(NUM_THREADS, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (pdl_enabled()) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    const bool long_k = pipe == PIPE_LONG_K || pipe == PIPE_LONG_K_PACKED, packed = pipe_packed(pipe);
    cudaError_t e;
    switch (mode) {
        case EMU_MODE_TF32X3:
            if (staged)
                e = packed ? launch_one<MODE_TF32X3, PIPE_SHORT_K_PACKED, true>(cfg, p)
                           : launch_one<MODE_TF32X3, PIPE_SHORT_K, true>(cfg, p);
            else
                e = packed ? launch_one<MODE_TF32X3, PIPE_SHORT_K_PACKED>(cfg, p) : launch_one<MODE_TF32X3, PIPE_SHORT_K>(cfg, p);
            break;
        case EMU_MODE_TF32X1:
            e = packed ? launch_one<MODE_TF32X1, PIPE_SHORT_K_PACKED>(cfg, p) : launch_one<MODE_TF32X1, PIPE_SHORT_K>(cfg, p);
            break;
        case EMU_MODE_BF16X6:
            e = packed ? (long_k ? launch_one<MODE_BF16X6, PIPE_LONG_K_PACKED>(cfg, p)
                                 : launch_one<MODE_BF16X6, PIPE_SHORT_K_PACKED>(cfg, p))
                       : (long_k ? launch_one<MODE_BF16X6, PIPE_LONG_K>(cfg, p) : launch_one<MODE_BF16X6, PIPE_SHORT_K>(cfg, p));
            break;
        default:
            if (staged)
                e = packed ? (long_k ? launch_one<MODE_BF16X9, PIPE_LONG_K_PACKED, true>(cfg, p)
                                     : launch_one<MODE_BF16X9, PIPE_SHORT_K_PACKED, true>(cfg, p))
                           : (long_k ? launch_one<MODE_BF16X9, PIPE_LONG_K, true>(cfg, p)
                                     : launch_one<MODE_BF16X9, PIPE_SHORT_K, true>(cfg, p));
            else
                e = packed ? (long_k ? launch_one<MODE_BF16X9, PIPE_LONG_K_PACKED>(cfg, p)
                                     : launch_one<MODE_BF16X9, PIPE_SHORT_K_PACKED>(cfg, p))
                           : (long_k ? launch_one<MODE_BF16X9, PIPE_LONG_K>(cfg, p)
                                     : launch_one<MODE_BF16X9, PIPE_SHORT_K>(cfg, p));
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        if (log_enabled()) std::fprintf(stderr, "[emu] launch failed: %s\n", cudaGetErrorName(e));
    }
    return e;
}

// Core: C = alpha * op(A) op(B) + beta * C_old + bias, with C_old == C.
// packed_b != nullptr: op(B) comes packed (emu_pack_b); B and ldb are unused.
// One launch of the pack kernel on `stream` (the caller checked the arguments).
cudaError_t launch_pack(emu_mode_t mode, int64_t N, int64_t K, const float* B, int64_t ldb, bool k_major,
                        void* packed, int sm_count, cudaStream_t stream) {
    const int64_t items = N * (packed_kp(K) / 8);
    const int threads = 256;
    const int64_t blocks64 = (items + threads - 1) / threads;
    const int blocks = (int)(blocks64 < sm_count * 16 ? blocks64 : sm_count * 16);
    cudaGetLastError();
    switch (mode) {
        case EMU_MODE_TF32X3: pack_kernel<MODE_TF32X3><<<blocks, threads, 0, stream>>>(N, K, B, ldb, k_major, packed); break;
        case EMU_MODE_TF32X1: pack_kernel<MODE_TF32X1><<<blocks, threads, 0, stream>>>(N, K, B, ldb, k_major, packed); break;
        default: pack_kernel<MODE_BF16X9><<<blocks, threads, 0, stream>>>(N, K, B, ldb, k_major, packed);  // BF16x6 too
    }
    return cudaGetLastError();
}

emu_status_t run_gemm(emu_mode_t mode, bool a_mn, bool b_mn, int64_t M, int64_t N, int64_t K, float alpha,
                      const float* A, int64_t lda, const float* B, int64_t ldb, float beta, float* C,
                      int64_t ldc, const float* bias, cudaStream_t stream, const void* packed_b = nullptr) {
    if (!valid_mode(mode)) return EMU_STATUS_INVALID_VALUE;
    if (M < 0 || N < 0 || K < 0) return EMU_STATUS_INVALID_VALUE;
    if (M > INT32_MAX - 256 || N > INT32_MAX - 256 || K > INT32_MAX - 256) return EMU_STATUS_NOT_SUPPORTED;
    if (M == 0 || N == 0) return EMU_STATUS_SUCCESS;
    const int64_t a_rows = a_mn ? K : M, a_cols = a_mn ? M : K;
    const int64_t b_rows = b_mn ? K : N, b_cols = b_mn ? N : K;
    (void)a_rows; (void)b_rows;
    if (ldc < N || !C) return EMU_STATUS_INVALID_VALUE;
    const bool gemm = K > 0 && alpha != 0.0f;
    if (gemm && packed_b) {
        if (!A || lda < a_cols) return EMU_STATUS_INVALID_VALUE;
        if (!aligned16(A) || !aligned16(packed_b) || (lda & 3)) return EMU_STATUS_NOT_SUPPORTED;
    } else if (gemm) {
        if (!A || !B || lda < a_cols || ldb < b_cols) return EMU_STATUS_INVALID_VALUE;
        if (!aligned16(A) || !aligned16(B) || (lda & 3) || (ldb & 3)) return EMU_STATUS_NOT_SUPPORTED;
    }
    if (!aligned16(C) || (ldc & 3)) return EMU_STATUS_NOT_SUPPORTED;
    if (bias && !aligned16(bias)) return EMU_STATUS_NOT_SUPPORTED;

    DeviceInfo* dev = nullptr;
    emu_status_t st = device_info(&dev);
    if (st != EMU_STATUS_SUCCESS) return st;

    if (!gemm) {
        const int64_t total = M * N;
        const int threads = 256;
        const int64_t blocks64 = (total + threads - 1) / threads;
        const int blocks = (int)(blocks64 < dev->sm_count * 8 ? blocks64 : dev->sm_count * 8);
        cudaGetLastError();  // only this launch's status below
        scale_kernel<<<blocks, threads, 0, stream>>>(M, N, beta, C, ldc, bias);
        return cudaGetLastError() == cudaSuccess ? EMU_STATUS_SUCCESS : EMU_STATUS_LAUNCH_FAILED;
    }

    const int pairs = dev->max_clusters[mode == EMU_MODE_TF32X3 ? 1 : 0];
    if (!packed_b) mode = dispatch_mode(mode, M, N, K, pairs, dev->sm_count);
    if (mode == EMU_MODE_FP32) {
        if (N > 64LL * NAT_MAX_GRID_Y) return EMU_STATUS_NOT_SUPPORTED;
        if (log_enabled())
            std::fprintf(stderr, "[emu] fp32 M=%lld N=%lld K=%lld a_mn=%d b_mn=%d (native)\n", (long long)M,
                         (long long)N, (long long)K, (int)a_mn, (int)b_mn);
        return launch_native(M, N, K, alpha, A, lda, a_mn, B, ldb, b_mn, beta, C, ldc, bias, dev->sm_count, stream) == cudaSuccess
                   ? EMU_STATUS_SUCCESS : EMU_STATUS_LAUNCH_FAILED;
    }
    Plan plan = make_plan(M, N, K, pairs);
    int devid = 0;
    cudaGetDevice(&devid);
    // Everything that can fail -- the library's buffers, the tensor maps --
    // comes before the first launch, so that a call that returns an error
    // has enqueued nothing.
    static const bool autopack = env_int("EMU_AUTOPACK", 1) != 0;
    void* autopack_buf = nullptr;
    if (!packed_b && autopack && (mode == EMU_MODE_TF32X3 || mode == EMU_MODE_TF32X1) &&
        plan.tiles_m >= kAutoPackMinTileRows && (size_t)packed_bytes(mode, N, K) <= kAutoPackMaxBytes) {
        st = packed_buffer_for(devid, stream, (size_t)packed_bytes(mode, N, K), &autopack_buf);
        if (st != EMU_STATUS_SUCCESS) return st;
    }
    const void* b_packed = packed_b ? packed_b : autopack_buf;
    if (b_packed) plan.pipe = plan.pipe == PIPE_LONG_K ? PIPE_LONG_K_PACKED : PIPE_SHORT_K_PACKED;
    Params p{};
    if (!encode_operand(&p.tmA, A, a_mn, M, K, lda, HALF) ||
        !(b_packed ? encode_packed(&p.tmB, b_packed, mode, N, K)
                   : encode_operand(&p.tmB, B, b_mn, N, K, ldb, (uint32_t)plan.tn / 2)))
        return EMU_STATUS_LAUNCH_FAILED;
    p.M = (int)M; p.N = (int)N; p.K = (int)K;
    p.a_mn_major = a_mn; p.b_mn_major = b_packed ? 0 : b_mn;
    p.tiles_m = plan.tiles_m;
    p.tiles_n = plan.tiles_n;
    p.num_tiles = plan.num_tiles;
    p.k_stages = plan.k_stages;
    p.tiles_a = plan.tiles_a; p.split_a = plan.split_a; p.split_b = plan.split_b;
    p.num_units = plan.num_units;
    p.chain = plan.chain;
    if (plan.chain) {
        const long long U = (long long)plan.num_tiles * plan.k_stages;
        p.chain_q = U / plan.clusters;
        p.chain_r = (int)(U % plan.clusters);
        for (int i = 0; i <= plan.clusters; ++i)
            p.chain_delta[i] = (signed char)(plan.chain_bound[i] - (long long)i * U / plan.clusters);
    }
    p.alpha = alpha; p.beta = beta;
    p.c_old = C; p.c = C; p.ldc = ldc;
    p.bias = bias;
    p.wait_budget_ns = wait_budget_ns();
    if (plan.slots > 0) {
        Workspace* w = nullptr;
        const size_t floats = (size_t)plan.slots * TILE_M * plan.tn;
        st = workspace_for(devid, stream, floats, (size_t)p.num_tiles * 2, &w, &p.epoch);
        if (st != EMU_STATUS_SUCCESS) return st;
        p.workspace = w->partials;
        p.counters = w->counters;
    }
    if (autopack_buf && launch_pack(mode, N, K, B, ldb, !b_mn, autopack_buf, dev->sm_count, stream) != cudaSuccess)
        return EMU_STATUS_LAUNCH_FAILED;
    const int clusters = plan.clusters;
    if (log_enabled())
        std::fprintf(stderr, "[emu] %s M=%lld N=%lld K=%lld a_mn=%d b_mn=%d pipe=%d tile=256x%d tiles=%dx%d "
                             "k_stages=%d units=%d (%d tiles x %d, then x %d) pairs=%d (max %d)\n",
                     mode_name(mode), (long long)M, (long long)N, (long long)K, (int)a_mn, (int)b_mn, plan.pipe,
                     plan.tn, p.tiles_m, p.tiles_n, p.k_stages, p.num_units, p.tiles_a, p.split_a, p.split_b,
                     clusters, pairs);
    return launch_gemm(mode, plan.pipe, p, clusters, stream) == cudaSuccess ? EMU_STATUS_SUCCESS
                                                                             : EMU_STATUS_LAUNCH_FAILED;
}

// ----------------------------------------------------------- split dump ----
// One 128-row operand tile through the kernel's split.
template <int MODE, int ROWS>
__global__ void __launch_bounds__(256, 1) split_dump_kernel(const __grid_constant__ CUtensorMap tm, int R, int Kc,
                                                            int mn_major, void* out) {
    using C = Cfg<MODE>;
    constexpr uint32_t F32_BYTES = ROWS * BK * 4, COMP = ROWS * C::ROW_BYTES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* f32 = smem;
    uint8_t* comp = smem + F32_BYTES;
    uint64_t* bar = reinterpret_cast<uint64_t*>(comp + C::NCOMP * COMP);
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        mbar_arrive_expect_tx(bar, F32_BYTES);
        if (!mn_major) tma_load_2d(f32, &tm, bar, 0, 0);
        else for (int j = 0; j < ROWS / 32; ++j) tma_load_2d(f32 + j * 4096, &tm, bar, 32 * j, 0);
    }
    volatile int no_abort = 0;
    if (!mbar_wait_warp(bar, 0, &no_abort, 1000000000ull, 5)) return;
    split_operand<MODE, 256, ROWS>(f32, comp, mn_major != 0, threadIdx.x);
    __syncthreads();
    for (int i = threadIdx.x; i < R * Kc; i += blockDim.x) {
        const uint32_t r = i / Kc, k = i % Kc;
        for (int c = 0; c < C::NCOMP; ++c) {
            const uint8_t* tile = comp + c * COMP;
            if constexpr (MODE == MODE_BF16X9) {
                const uint16_t v = *reinterpret_cast<const uint16_t*>(tile + off_bf16_chunk(r, k >> 3) + (k & 7u) * 2);
                reinterpret_cast<uint16_t*>(out)[(size_t)c * R * Kc + i] = v;
            } else {
                const uint32_t v = *reinterpret_cast<const uint32_t*>(tile + off_f32_chunk(r, k >> 2) + (k & 3u) * 4);
                reinterpret_cast<uint32_t*>(out)[(size_t)c * R * Kc + i] = v;
            }
        }
    }
}

// Self-test of the bounded waits: one warp waits on a barrier that nothing
// arrives on, with the caller's budget, through the same routine the GEMM
// kernel's split and epilogue warps use.  The wait gives up, records the
// timeout in the device error word and the kernel returns normally.
__global__ void wait_timeout_selftest_kernel(unsigned long long budget_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncwarp();
    mbar_wait_warp(&bar, 0, &abort_flag, budget_ns, 7);
}

// Self-test of the split-K counters after a timeout: for one launch epoch,
// every counter gets one arrival (as if one piece of every split tile had
// published), then thread 0 waits for a second arrival that never comes, as
// a split piece whose partner pieces are lost would; its wait gives up after
// the budget.  The counts it leaves behind belong to that epoch.
__global__ void split_timeout_selftest_kernel(unsigned long long* counters, int n, unsigned long long epoch,
                                              unsigned long long budget_ns) {
    __shared__ int abort_flag;
    if (threadIdx.x == 0) abort_flag = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += blockDim.x) epoch_arrive(&counters[i], epoch);
    __syncthreads();
    if (threadIdx.x == 0) wait_epoch_count(&counters[0], epoch, 2u, &abort_flag, budget_ns, 8);
}

}  // namespace
}  // namespace emu

using namespace emu;

extern "C" {

emu_status_t emu_sgemm(emu_mode_t mode, emu_op_t transA, emu_op_t transB, int64_t M, int64_t N, int64_t K,
                       float alpha, const float* A, int64_t lda, const float* B, int64_t ldb, float beta,
                       float* C, int64_t ldc, emu_stream_t stream) {
    if ((transA != EMU_OP_N && transA != EMU_OP_T) || (transB != EMU_OP_N && transB != EMU_OP_T))
        return EMU_STATUS_INVALID_VALUE;
    // op(A) is K-major in memory when A is stored M x K; op(B) when B is N x K.
    return run_gemm(mode, transA == EMU_OP_T, transB == EMU_OP_N, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
                    nullptr, reinterpret_cast<cudaStream_t>(stream));
}

emu_status_t emu_linear_fwd(emu_mode_t mode, int64_t M, int64_t N, int64_t K, const float* X, const float* W,
                            const float* bias, float* Y, emu_stream_t stream) {
    // Y = X W^T + b: op(A) = X (K-major), op(B) = W^T (W is N x K, K-major)
    return run_gemm(mode, false, false, M, N, K, 1.0f, X, K, W, K, 0.0f, Y, N, bias,
                    reinterpret_cast<cudaStream_t>(stream));
}

emu_status_t emu_linear_bwd_input(emu_mode_t mode, int64_t M, int64_t N, int64_t K, const float* dY,
                                  const float* W, float* dX, emu_stream_t stream) {
    // dX[M,K] = dY[M,N] W[N,K]: GEMM with output width K and contraction N;
    // op(B) = W is MN-major (rows are the contraction index)
    return run_gemm(mode, false, true, M, K, N, 1.0f, dY, N, W, K, 0.0f, dX, K, nullptr,
                    reinterpret_cast<cudaStream_t>(stream));
}

emu_status_t emu_linear_bwd_weight(emu_mode_t mode, int64_t M, int64_t N, int64_t K, const float* dY,
                                   const float* X, float beta, float* dW, emu_stream_t stream) {
    // dW[N,K] = dY^T X: output rows N, output columns K, contraction M; both
    // operands are MN-major (their rows are the contraction index)
    return run_gemm(mode, true, true, N, K, M, 1.0f, dY, N, X, K, beta, dW, K, nullptr,
                    reinterpret_cast<cudaStream_t>(stream));
}

int64_t emu_pack_bytes(emu_mode_t mode, int64_t N, int64_t K) {
    if (!emulated_mode(mode) || N < 0 || K < 0) return -1;
    return packed_bytes(mode, N, K);
}

emu_status_t emu_pack_b(emu_mode_t mode, emu_op_t transB, int64_t N, int64_t K, const float* B, int64_t ldb,
                        void* packed, emu_stream_t stream) {
    if (!emulated_mode(mode) || (transB != EMU_OP_N && transB != EMU_OP_T)) return EMU_STATUS_INVALID_VALUE;
    if (N < 0 || K < 0) return EMU_STATUS_INVALID_VALUE;
    if (N > INT32_MAX - 256 || K > INT32_MAX - 256) return EMU_STATUS_NOT_SUPPORTED;
    if (N == 0 || K == 0) return EMU_STATUS_SUCCESS;
    const bool k_major = transB == EMU_OP_T;  // op(B)^T rows are B's rows when B is stored N x K
    if (!B || !packed || ldb < (k_major ? K : N)) return EMU_STATUS_INVALID_VALUE;
    if (!aligned16(packed)) return EMU_STATUS_NOT_SUPPORTED;
    DeviceInfo* dev = nullptr;
    emu_status_t st = device_info(&dev);
    if (st != EMU_STATUS_SUCCESS) return st;
    return launch_pack(mode, N, K, B, ldb, k_major, packed, dev->sm_count, reinterpret_cast<cudaStream_t>(stream)) ==
                   cudaSuccess ? EMU_STATUS_SUCCESS : EMU_STATUS_LAUNCH_FAILED;
}

emu_status_t emu_sgemm_packed_b(emu_mode_t mode, emu_op_t transA, int64_t M, int64_t N, int64_t K, float alpha,
                                const float* A, int64_t lda, const void* packed_b, float beta, float* C,
                                int64_t ldc, emu_stream_t stream) {
    if (!emulated_mode(mode) || (transA != EMU_OP_N && transA != EMU_OP_T)) return EMU_STATUS_INVALID_VALUE;
    if (!packed_b && K > 0 && alpha != 0.0f) return EMU_STATUS_INVALID_VALUE;
    return run_gemm(mode, transA == EMU_OP_T, false, M, N, K, alpha, A, lda, nullptr, 0, beta, C, ldc, nullptr,
                    reinterpret_cast<cudaStream_t>(stream), packed_b);
}

emu_status_t emu_linear_fwd_packed(emu_mode_t mode, int64_t M, int64_t N, int64_t K, const float* X,
                                   const void* W_packed, const float* bias, float* Y, emu_stream_t stream) {
    if (!emulated_mode(mode) || (!W_packed && K > 0)) return EMU_STATUS_INVALID_VALUE;
    return run_gemm(mode, false, false, M, N, K, 1.0f, X, K, nullptr, 0, 0.0f, Y, N, bias,
                    reinterpret_cast<cudaStream_t>(stream), W_packed);
}

emu_status_t emu_linear_bwd_input_packed(emu_mode_t mode, int64_t M, int64_t N, int64_t K, const float* dY,
                                         const void* Wt_packed, float* dX, emu_stream_t stream) {
    if (!emulated_mode(mode) || (!Wt_packed && N > 0)) return EMU_STATUS_INVALID_VALUE;
    return run_gemm(mode, false, false, M, K, N, 1.0f, dY, N, nullptr, 0, 0.0f, dX, K, nullptr,
                    reinterpret_cast<cudaStream_t>(stream), Wt_packed);
}

const char* emu_status_string(emu_status_t s) {
    switch (s) {
        case EMU_STATUS_SUCCESS: return "EMU_STATUS_SUCCESS";
        case EMU_STATUS_INVALID_VALUE: return "EMU_STATUS_INVALID_VALUE";
        case EMU_STATUS_NOT_SUPPORTED: return "EMU_STATUS_NOT_SUPPORTED";
        case EMU_STATUS_ARCH_MISMATCH: return "EMU_STATUS_ARCH_MISMATCH";
        case EMU_STATUS_ALLOC_FAILED: return "EMU_STATUS_ALLOC_FAILED";
        case EMU_STATUS_LAUNCH_FAILED: return "EMU_STATUS_LAUNCH_FAILED";
        case EMU_STATUS_DEVICE_TIMEOUT: return "EMU_STATUS_DEVICE_TIMEOUT";
    }
    return "EMU_STATUS_UNKNOWN";
}

emu_status_t emu_stream_check(emu_stream_t stream) {
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return EMU_STATUS_LAUNCH_FAILED;
    }
    return check_error_flag(true);
}

emu_status_t emu_split_dump(emu_mode_t mode, int64_t R, int64_t Kc, const float* X, int64_t ldx, int mn_major,
                            void* out, emu_stream_t stream) {
    if (mode != EMU_MODE_BF16X9 && mode != EMU_MODE_TF32X3) return EMU_STATUS_INVALID_VALUE;
    if (R <= 0 || R > HALF || Kc <= 0 || Kc > BK || !X || !out) return EMU_STATUS_INVALID_VALUE;
    if (ldx < (mn_major ? R : Kc)) return EMU_STATUS_INVALID_VALUE;
    if (!aligned16(X) || (ldx & 3)) return EMU_STATUS_NOT_SUPPORTED;
    DeviceInfo* dev = nullptr;
    emu_status_t st = device_info(&dev);
    if (st != EMU_STATUS_SUCCESS) return st;
    CUtensorMap tm;
    if (!encode_operand(&tm, X, mn_major != 0, R, Kc, ldx, (uint32_t)HALF)) return EMU_STATUS_LAUNCH_FAILED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int R32 = (int)R, K32 = (int)Kc;
    // shared memory: FP32 tile, the components, the barrier, alignment slack
    const uint32_t rows = HALF;
    const uint32_t bytes = mode == EMU_MODE_BF16X9
        ? 1024 + rows * BK * 4 + 3 * rows * Cfg<MODE_BF16X9>::ROW_BYTES + 64
        : 1024 + rows * BK * 4 + 2 * rows * Cfg<MODE_TF32X3>::ROW_BYTES + 64;
    auto run = [&](auto kernel) {
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        cudaGetLastError();
        kernel<<<1, 256, bytes, s>>>(tm, R32, K32, mn_major, out);
    };
    if (mode == EMU_MODE_BF16X9) run(split_dump_kernel<MODE_BF16X9, HALF>);
    else run(split_dump_kernel<MODE_TF32X3, HALF>);
    return cudaGetLastError() == cudaSuccess ? EMU_STATUS_SUCCESS : EMU_STATUS_LAUNCH_FAILED;
}

emu_status_t emu_selftest_wait_timeout(uint64_t budget_ns, emu_stream_t stream) {
    if (budget_ns == 0 || budget_ns > 10000000000ull) return EMU_STATUS_INVALID_VALUE;
    DeviceInfo* dev = nullptr;
    emu_status_t st = device_info(&dev);
    if (st != EMU_STATUS_SUCCESS) return st;
    cudaGetLastError();
    wait_timeout_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(budget_ns);
    return cudaGetLastError() == cudaSuccess ? EMU_STATUS_SUCCESS : EMU_STATUS_LAUNCH_FAILED;
}

emu_status_t emu_selftest_split_timeout(uint64_t budget_ns, int64_t tiles, emu_stream_t stream) {
    if (budget_ns == 0 || budget_ns > 10000000000ull || tiles < 1 || tiles > (int64_t(1) << 24))
        return EMU_STATUS_INVALID_VALUE;
    DeviceInfo* dev = nullptr;
    emu_status_t st = device_info(&dev);
    if (st != EMU_STATUS_SUCCESS) return st;
    int devid = 0;
    cudaGetDevice(&devid);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    Workspace* w = nullptr;
    unsigned long long epoch = 0;
    st = workspace_for(devid, s, 0, (size_t)tiles * 2, &w, &epoch);
    if (st != EMU_STATUS_SUCCESS) return st;
    cudaGetLastError();
    split_timeout_selftest_kernel<<<1, 256, 0, s>>>(w->counters, (int)(tiles * 2), epoch, budget_ns);
    return cudaGetLastError() == cudaSuccess ? EMU_STATUS_SUCCESS : EMU_STATUS_LAUNCH_FAILED;
}

emu_status_t emu_shutdown(void) {
    std::lock_guard<std::mutex> lock(g_mutex);
    int current = 0;
    const bool have_current = cudaGetDevice(&current) == cudaSuccess;
    emu_status_t result = EMU_STATUS_SUCCESS;
    for (auto& w : g_ws) {
        if (w.device < 0) continue;
        if (cudaSetDevice(w.device) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
            cudaGetLastError();
            result = EMU_STATUS_LAUNCH_FAILED;
        }
        // after the device synchronisation nothing uses these buffers
        if (w.partials && cudaFree(w.partials) != cudaSuccess) { cudaGetLastError(); result = EMU_STATUS_LAUNCH_FAILED; }
        if (w.counters && cudaFree(w.counters) != cudaSuccess) { cudaGetLastError(); result = EMU_STATUS_LAUNCH_FAILED; }
        if (w.packed && cudaFree(w.packed) != cudaSuccess) { cudaGetLastError(); result = EMU_STATUS_LAUNCH_FAILED; }
        w = Workspace{};
    }
    if (have_current && cudaSetDevice(current) != cudaSuccess) cudaGetLastError();
    return result;
}

emu_status_t emu_debug_fail_allocations(int n) {
    if (n < 0) return EMU_STATUS_INVALID_VALUE;
    g_fail_allocs.store(n);
    return EMU_STATUS_SUCCESS;
}

emu_status_t emu_plan_query(int64_t M, int64_t N, int64_t K, int pairs, int64_t* out, int n) {
    if (M <= 0 || N <= 0 || K <= 0 || pairs < 1 || !out || n < EMU_PLAN_FIELDS) return EMU_STATUS_INVALID_VALUE;
    if (M > INT32_MAX - 256 || N > INT32_MAX - 256 || K > INT32_MAX - 256) return EMU_STATUS_NOT_SUPPORTED;
    const Plan p = make_plan(M, N, K, pairs);
    const int64_t v[EMU_PLAN_FIELDS] = {p.pipe, p.tn, p.tiles_m, p.tiles_n, p.k_stages, p.tiles_a,
                                        p.split_a, p.split_b, p.num_units, p.clusters, p.slots,
                                        (int64_t)(p.cost * 100.0 + 0.5), p.chain};
    for (int i = 0; i < EMU_PLAN_FIELDS; ++i) out[i] = v[i];
    return EMU_STATUS_SUCCESS;
}

emu_status_t emu_plan_bounds(int64_t M, int64_t N, int64_t K, int pairs, int64_t* out, int n) {
    if (M <= 0 || N <= 0 || K <= 0 || pairs < 1 || !out || n < 1) return EMU_STATUS_INVALID_VALUE;
    if (M > INT32_MAX - 256 || N > INT32_MAX - 256 || K > INT32_MAX - 256) return EMU_STATUS_NOT_SUPPORTED;
    const Plan p = make_plan(M, N, K, pairs);
    if (!p.chain) return EMU_STATUS_NOT_SUPPORTED;
    if (n < p.clusters + 1) return EMU_STATUS_INVALID_VALUE;
    for (int i = 0; i <= p.clusters; ++i) out[i] = p.chain_bound[i];
    return EMU_STATUS_SUCCESS;
}

emu_status_t emu_set_strategy(emu_strategy_t strategy) {
    if (strategy != EMU_STRATEGY_EAGER && strategy != EMU_STRATEGY_PERFORMANT) return EMU_STATUS_INVALID_VALUE;
    g_strategy.store(strategy, std::memory_order_relaxed);
    return EMU_STATUS_SUCCESS;
}

emu_strategy_t emu_get_strategy(void) { return static_cast<emu_strategy_t>(g_strategy.load(std::memory_order_relaxed)); }

emu_status_t emu_dispatch_query(emu_mode_t mode, int64_t M, int64_t N, int64_t K, int pairs, emu_mode_t* out) {
    if (!valid_mode(mode) || M <= 0 || N <= 0 || K <= 0 || pairs < 1 || !out) return EMU_STATUS_INVALID_VALUE;
    if (M > INT32_MAX - 256 || N > INT32_MAX - 256 || K > INT32_MAX - 256) return EMU_STATUS_NOT_SUPPORTED;
    *out = dispatch_mode(mode, M, N, K, pairs, 2 * pairs);
    return EMU_STATUS_SUCCESS;
}

int emu_version(void) { return 200; }

}  // extern "C"

// ---------------------------------------------------------------------------
// emu_sgemm_noalloc: the same GEMM for callers that cannot allocate device
// memory (see include/emu_gemm.h).  Its split-K scratch is a file-scope
// device array instead of a cudaMallocAsync'd workspace; everything else
// (checks, plan, kernel) is what emu_sgemm does.
// ---------------------------------------------------------------------------
namespace emu {

// 64 MiB, held by every device that loads this library until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

// Device address of g_noalloc_scratch for the current device, looked up once
// per device (cudaGetSymbolAddress, not an allocation).  In host code the
// array's name is only a stand-in for the symbol; kernels must get this
// address, never the name's host-side value.
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kMaxDevices] = {};
unsigned long long g_noalloc_epoch[kMaxDevices] = {};

emu_status_t noalloc_scratch(void** out, unsigned long long* epoch) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return EMU_STATUS_LAUNCH_FAILED;
    }
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_ptr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) {
            cudaGetLastError();
            return EMU_STATUS_LAUNCH_FAILED;
        }
        g_noalloc_ptr[dev] = ptr;
    }
    *out = g_noalloc_ptr[dev];
    *epoch = ++g_noalloc_epoch[dev];
    return EMU_STATUS_SUCCESS;
}

emu_status_t run_gemm_noalloc(emu_mode_t mode, bool a_mn, bool b_mn, int64_t M, int64_t N, int64_t K,
                              float alpha, const float* A, int64_t lda, const float* B, int64_t ldb, float beta,
                              float* C, int64_t ldc, cudaStream_t stream) {
    if (!valid_mode(mode)) return EMU_STATUS_INVALID_VALUE;
    if (M < 0 || N < 0 || K < 0) return EMU_STATUS_INVALID_VALUE;
    if (M > INT32_MAX - 256 || N > INT32_MAX - 256 || K > INT32_MAX - 256) return EMU_STATUS_NOT_SUPPORTED;
    if (M == 0 || N == 0) return EMU_STATUS_SUCCESS;
    const int64_t a_cols = a_mn ? M : K, b_cols = b_mn ? N : K;
    if (ldc < N || !C) return EMU_STATUS_INVALID_VALUE;
    const bool gemm = K > 0 && alpha != 0.0f;
    if (gemm) {
        if (!A || !B || lda < a_cols || ldb < b_cols) return EMU_STATUS_INVALID_VALUE;
        if (!aligned16(A) || !aligned16(B) || (lda & 3) || (ldb & 3)) return EMU_STATUS_NOT_SUPPORTED;
    }
    if (!aligned16(C) || (ldc & 3)) return EMU_STATUS_NOT_SUPPORTED;

    DeviceInfo* dev = nullptr;
    emu_status_t st = device_info(&dev);
    if (st != EMU_STATUS_SUCCESS) return st;
    void* scratch = nullptr;
    unsigned long long epoch = 0;
    st = noalloc_scratch(&scratch, &epoch);
    if (st != EMU_STATUS_SUCCESS) return st;

    if (!gemm) {
        const int64_t total = M * N;
        const int threads = 256;
        const int64_t blocks64 = (total + threads - 1) / threads;
        const int blocks = (int)(blocks64 < dev->sm_count * 8 ? blocks64 : dev->sm_count * 8);
        cudaGetLastError();
        scale_kernel<<<blocks, threads, 0, stream>>>(M, N, beta, C, ldc, nullptr);
        return cudaGetLastError() == cudaSuccess ? EMU_STATUS_SUCCESS : EMU_STATUS_LAUNCH_FAILED;
    }

    const int pairs = dev->max_clusters[mode == EMU_MODE_TF32X3 ? 1 : 0];
    if (dispatch_mode(mode, M, N, K, pairs, dev->sm_count) == EMU_MODE_FP32) {
        if (N > 64LL * NAT_MAX_GRID_Y) return EMU_STATUS_NOT_SUPPORTED;
        return launch_native(M, N, K, alpha, A, lda, a_mn, B, ldb, b_mn, beta, C, ldc, nullptr, dev->sm_count, stream) == cudaSuccess
                   ? EMU_STATUS_SUCCESS : EMU_STATUS_LAUNCH_FAILED;
    }
    const Plan plan = make_plan(M, N, K, pairs);
    Params p{};
    if (!encode_operand(&p.tmA, A, a_mn, M, K, lda, HALF) ||
        !encode_operand(&p.tmB, B, b_mn, N, K, ldb, (uint32_t)plan.tn / 2))
        return EMU_STATUS_LAUNCH_FAILED;
    p.M = (int)M; p.N = (int)N; p.K = (int)K;
    p.a_mn_major = a_mn; p.b_mn_major = b_mn;
    p.tiles_m = plan.tiles_m;
    p.tiles_n = plan.tiles_n;
    p.num_tiles = plan.num_tiles;
    p.k_stages = plan.k_stages;
    p.tiles_a = plan.tiles_a; p.split_a = plan.split_a; p.split_b = plan.split_b;
    p.num_units = plan.num_units;
    p.chain = plan.chain;
    if (plan.chain) {
        const long long U = (long long)plan.num_tiles * plan.k_stages;
        p.chain_q = U / plan.clusters;
        p.chain_r = (int)(U % plan.clusters);
        for (int i = 0; i <= plan.clusters; ++i)
            p.chain_delta[i] = (signed char)(plan.chain_bound[i] - (long long)i * U / plan.clusters);
    }
    p.alpha = alpha; p.beta = beta;
    p.c_old = C; p.c = C; p.ldc = ldc;
    p.bias = nullptr;
    p.wait_budget_ns = wait_budget_ns();
    if (plan.slots > 0) {
        // partial tiles first, then the counters
        const size_t partial_bytes = (size_t)plan.slots * TILE_M * plan.tn * sizeof(float);
        const size_t counter_off = (partial_bytes + 255) & ~size_t(255);
        const size_t counter_bytes = (size_t)p.num_tiles * 2 * sizeof(unsigned long long);
        if (counter_off + counter_bytes > kNoAllocScratchBytes) return EMU_STATUS_NOT_SUPPORTED;
        p.workspace = reinterpret_cast<float*>(scratch);
        p.counters = reinterpret_cast<unsigned long long*>(reinterpret_cast<unsigned char*>(scratch) + counter_off);
        p.epoch = epoch;
        // the array keeps the previous call's contents: the counters must start at zero
        if (cudaMemsetAsync(p.counters, 0, counter_bytes, stream) != cudaSuccess) {
            cudaGetLastError();
            return EMU_STATUS_LAUNCH_FAILED;
        }
    }
    const int clusters = plan.clusters;
    return launch_gemm(mode, plan.pipe, p, clusters, stream) == cudaSuccess ? EMU_STATUS_SUCCESS
                                                                             : EMU_STATUS_LAUNCH_FAILED;
}

}  // namespace
}  // namespace emu

extern "C" emu_status_t emu_sgemm_noalloc(emu_mode_t mode, emu_op_t transA, emu_op_t transB, int64_t M,
                                          int64_t N, int64_t K, float alpha, const float* A, int64_t lda,
                                          const float* B, int64_t ldb, float beta, float* C, int64_t ldc,
                                          emu_stream_t stream) {
    using namespace emu;
    if ((transA != EMU_OP_N && transA != EMU_OP_T) || (transB != EMU_OP_N && transB != EMU_OP_T))
        return EMU_STATUS_INVALID_VALUE;
    return run_gemm_noalloc(mode, transA == EMU_OP_T, transB == EMU_OP_N, M, N, K, alpha, A, lda, B, ldb, beta, C,
                            ldc, reinterpret_cast<cudaStream_t>(stream));
}
