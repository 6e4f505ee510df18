// ptx.cuh -- thin inline-PTX wrappers for sm_103a: mbarrier, TMA
// (cp.async.bulk.tensor), tcgen05 (TMEM allocation, MMA, commit, loads) and
// proxy fences.  Every wait is bounded: it gives up after a time budget,
// records the reason in a device-global flag and returns false, so that no
// kernel of this library can hang a GPU.
#pragma once

#include <cstdint>
#include <cuda.h>

namespace emu {

// Device-global error word, read and cleared by emu_stream_check().
// Bit 0: a wait timed out.  Bits 8..15: the role that timed out (for logs).
// (The library is a single translation unit, so the definition lives here.)
__device__ unsigned int g_error_flag = 0;

enum : unsigned { ERR_TIMEOUT = 1u };

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------------------- mbarrier ----
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
                 ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Arrive on the barrier at the same shared-memory offset in CTA `rank` of
// this cluster.  What such an arrival publishes (components in the arriving
// CTA's own shared memory, made visible to the tensor cores by a proxy fence;
// TMEM reads finished with tcgen05.wait::ld) needs only CTA-scope release
// ordering.  A cluster-scope release waits for the SM's outstanding memory
// traffic and measured 1-2 thousand cycles per arrival on this kernel.
__device__ __forceinline__ void mbar_arrive_cluster(uint64_t* bar, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(bar)), "r"(rank));
    asm volatile("mbarrier.arrive.release.cta.shared::cluster.b64 _, [%0];" ::"r"(remote) : "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t num_clusters_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}
// Programmatic dependent launch.  launch_dependents lets the next kernel in
// the stream (if it was launched with programmatic serialisation) be
// scheduled before this grid completes; wait blocks until every grid this
// one depends on has completed and its memory operations are visible.
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// All threads of both CTAs of the pair.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Cluster barrier without release ordering on the arrive side: enough where
// the only cross-CTA fact to publish is barrier initialisation, which
// fence.mbarrier_init orders by itself.
__device__ __forceinline__ void cluster_sync_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Wait for the phase of `bar` with the given parity to complete.  Returns
// false, without waiting further, when *abort is set by another warp or when
// the time budget runs out (then it sets the device error flag and *abort).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          uint64_t budget_ns, unsigned role) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 15u) == 0) {
            if (*abort) return false;
            if (globaltimer_ns() - t0 > budget_ns) {
                atomicOr(&g_error_flag, ERR_TIMEOUT | (role << 8));
                *abort = 1;
                return false;
            }
        }
    }
}

// Split-K arrival counters.  A counter is one 64-bit word: the epoch of the
// launch that last arrived on it (bits 8..63) and how many pieces of that
// launch have arrived (bits 0..7).  Every launch that uses a workspace gets a
// new epoch from the host, so a count left by an earlier launch (one that
// gave up on a wait before every piece arrived, say) belongs to another epoch
// and never counts toward this launch's total; the counters need no reset
// between launches.
__device__ __forceinline__ unsigned long long epoch_word(unsigned long long epoch, unsigned count) {
    return (epoch << 8) | count;
}

// Arrive once on `ctr` for `epoch` (relaxed: the caller's __threadfence and
// barrier order the data it publishes before this).
__device__ __forceinline__ void epoch_arrive(unsigned long long* ctr, unsigned long long epoch) {
    unsigned long long cur = *reinterpret_cast<volatile unsigned long long*>(ctr);
    for (;;) {
        const unsigned long long want = (cur >> 8) == epoch ? cur + 1 : epoch_word(epoch, 1);
        const unsigned long long prev = atomicCAS(ctr, cur, want);
        if (prev == cur) return;
        cur = prev;
    }
}

// Single-thread wait until `target` pieces of `epoch` have arrived on `ctr`
// (acquire at GPU scope, so that the writes the other CTAs released before
// arriving are visible), bounded like the barrier waits.
__device__ __forceinline__ bool wait_epoch_count(const unsigned long long* ctr, unsigned long long epoch,
                                                 unsigned target, volatile int* abort, uint64_t budget_ns,
                                                 unsigned role) {
    uint64_t t0 = 0;
    for (uint32_t i = 0;; ++i) {
        unsigned long long v;
        asm volatile("ld.acquire.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(ctr) : "memory");
        if ((v >> 8) == epoch && (v & 0xFFu) >= target) return true;
        if ((i & 7u) == 7u) {
            if (*abort) return false;
            const uint64_t now = globaltimer_ns();
            if (t0 == 0) {
                t0 = now;
            } else if (now - t0 > budget_ns) {
                atomicOr(&g_error_flag, ERR_TIMEOUT | (role << 8));
                *abort = 1;
                return false;
            }
        }
        __nanosleep(64);
    }
}

// Warp-collective: whether this launch's `target` arrivals are on `ctr`
// now.  Every lane reads the counter with acquire semantics, so that its own
// later loads see what the arriving CTAs released; no lane waits.
__device__ __forceinline__ bool warp_published(const unsigned long long* ctr, unsigned long long epoch,
                                               unsigned target) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(ctr) : "memory");
    return __all_sync(0xFFFFFFFFu, (v >> 8) == epoch && (v & 0xFFu) >= target);
}

// Warp-collective wait for `target` arrivals of `epoch` on `ctr`: every lane
// polls with acquire semantics until all see them; lane 0 keeps the time
// budget like the other waits.  False after a timeout or an abort.
__device__ __forceinline__ bool warp_wait_epoch(const unsigned long long* ctr, unsigned long long epoch,
                                                unsigned target, volatile int* abort, uint64_t budget_ns,
                                                unsigned role) {
    const uint32_t lane = threadIdx.x & 31u;
    uint64_t t0 = 0;
    for (uint32_t i = 0;; ++i) {
        if (warp_published(ctr, epoch, target)) return true;
        if ((i & 7u) == 7u) {
            int give_up = 0;
            if (lane == 0) {
                const uint64_t now = globaltimer_ns();
                if (*abort) {
                    give_up = 1;
                } else if (t0 == 0) {
                    t0 = now;
                } else if (now - t0 > budget_ns) {
                    atomicOr(&g_error_flag, ERR_TIMEOUT | (role << 8));
                    *abort = 1;
                    give_up = 1;
                }
            }
            if (__shfl_sync(0xFFFFFFFFu, give_up, 0)) return false;
        }
        __nanosleep(64);
    }
}

// Warp-collective form: every lane polls, and the warp stops together, so
// that the .sync.aligned instructions that follow see a converged warp.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity, volatile int* abort,
                                               uint64_t budget_ns, unsigned role) {
    const uint32_t lane = threadIdx.x & 31u;
    uint64_t t0 = 0;
    for (uint32_t i = 0;; ++i) {
        const bool done = mbar_try_wait(bar, parity);
        if (__all_sync(0xFFFFFFFFu, done)) return true;
        if ((i & 15u) == 15u) {
            int give_up = 0;
            if (lane == 0) {
                const uint64_t now = globaltimer_ns();
                if (*abort) {
                    give_up = 1;
                } else if (t0 == 0) {
                    t0 = now;
                } else if (now - t0 > budget_ns) {
                    atomicOr(&g_error_flag, ERR_TIMEOUT | (role << 8));
                    *abort = 1;
                    give_up = 1;
                }
            }
            if (__shfl_sync(0xFFFFFFFFu, give_up, 0)) return false;
        }
    }
}

// ------------------------------------------------------------------ TMA ----
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2-D tiled load of one box into shared memory; completion is signalled on
// `bar` as transaction bytes.  x is the inner (contiguous) coordinate.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int32_t x, int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];"
        ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)),
          "r"(x), "r"(y)
        : "memory");
}

// Prefetch one 2-D / 3-D box into L2 (no shared memory, no completion).
// Global memory is coherent at L2, so a prefetch cannot make a later load
// see stale data: it may be issued before the grids this one depends on
// have finished writing.
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* map, int32_t x, int32_t y) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];"
                 ::"l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y) : "memory");
}
__device__ __forceinline__ void tma_prefetch_l2_3d(const CUtensorMap* map, int32_t x, int32_t y, int32_t z) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];"
                 ::"l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z) : "memory");
}

// 3-D tiled load of one box (x inner, then y, then z).
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int32_t x, int32_t y, int32_t z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];"
        ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)),
          "r"(x), "r"(y), "r"(z)
        : "memory");
}

// Order this thread's generic-proxy shared-memory writes before later
// async-proxy reads (tensor-core operand fetches).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// -------------------------------------------------------------- tcgen05 ----
// Pair (cta_group::2) forms: one warp of EACH CTA of the pair executes
// alloc / relinquish / dealloc; MMAs and commits come from the leader CTA.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(smem_u32(dst_smem)), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void mma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                              uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma_tf32_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                              uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::tf32 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive once on the barrier at this offset in every CTA of `cta_mask` when
// all pair MMAs issued so far by this thread have completed.
__device__ __forceinline__ void mma_commit_pair_multicast(uint64_t* bar, uint16_t cta_mask) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
                 ::"r"(smem_u32(bar)), "h"(cta_mask) : "memory");
}
__device__ __forceinline__ void mma_commit_pair(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(smem_u32(bar)) : "memory");
}
// Per-warpgroup register budgets.  The CTA launches 512 threads with 128
// registers each (65,536); the two warpgroups of producer, MMA and split
// warps give up 56 each and the two epilogue warpgroups take 56 more each:
// 2 x 128 x 72 + 2 x 128 x 184 = 65,536, so the increase never waits.
__device__ __forceinline__ void setmaxnreg_dec72() { asm volatile("setmaxnreg.dec.sync.aligned.u32 72;" ::: "memory"); }
__device__ __forceinline__ void setmaxnreg_inc184() { asm volatile("setmaxnreg.inc.sync.aligned.u32 184;" ::: "memory"); }
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 lanes x 16 columns of 32-bit TMEM cells: thread t gets lane (base + t),
// columns [col, col + 16).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32"
        " {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 16-byte asynchronous copy from global memory (L2, not L1) to shared
// memory (the LDGSTS path: generic proxy, no registers held while in flight),
// and waiting for all of this thread's outstanding copies.
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;"
                 :: "r"(smem_u32(smem_dst)), "l"(__cvta_generic_to_global(gsrc)) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major operand tile in the canonical
// swizzled layout: rows of `row_bytes` (32, 64 or 128), 8-row groups packed
// back to back (stride 8 * row_bytes), tile base aligned to the swizzle span.
// Fields: start address >> 4 [0,14); leading byte offset >> 4 [16,30) (not
// used by swizzled K-major layouts, set to 1); stride byte offset >> 4
// [32,46); version 1 [46,48); base offset 0; swizzle mode [61,64):
// 2 = 128-byte, 4 = 64-byte, 6 = 32-byte.
__device__ __forceinline__ uint64_t sdesc_kmajor(uint32_t saddr, uint32_t row_bytes) {
    const uint32_t layout = row_bytes == 128 ? 2u : (row_bytes == 64 ? 4u : 6u);
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>(1u) << 16;
    d |= static_cast<uint64_t>(((8u * row_bytes) >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    d |= static_cast<uint64_t>(layout) << 61;
    return d;
}

// Instruction descriptor for kind::f16 / kind::tf32: D format F32 [4,6) = 1;
// A and B format [7,10) / [10,13): 1 = BF16, 2 = TF32; both K-major (bits 15,
// 16 = 0); N >> 3 at [17,23); M >> 4 at [24,29).
__host__ __device__ constexpr uint32_t make_idesc(uint32_t ab_format, uint32_t M, uint32_t N) {
    return (1u << 4) | (ab_format << 7) | (ab_format << 10) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

}  // namespace emu
