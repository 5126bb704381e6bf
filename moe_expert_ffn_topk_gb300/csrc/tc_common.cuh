// tcgen05 / TMA / mbarrier wrappers shared by the tensor-core kernels (inline PTX for sm_103a).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace moe {
namespace tc {

constexpr uint64_t kWaitTimeoutNs = 2000000000ull;  // every mbarrier wait gives up after 2 s

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// Non-blocking test of the phase with the given parity (true once it has completed).
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// Bounded wait for the phase of `bar` with the given parity to complete. Returns false when
// the CTA gave up (this thread timed out, or another role already aborted).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int32_t* hdr, volatile int* abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > kWaitTimeoutNs) {
            record_error(hdr, MOE_ERR_TIMEOUT);
            *abort_flag = 1;
            return false;
        }
    }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, int w,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], [%6];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Predicated global stores with no memory clobber: epilogue loops stay branch-free and the
// compiler may move independent loads across them.
__device__ __forceinline__ void st_global_u8_if(bool pred, void* ptr, uint8_t v) {
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %0, 0;\n\t@p st.global.u8 [%1], %2;\n\t}" ::"r"((int)pred), "l"(ptr),
                 "h"((uint16_t)v));
}
// predicated 32-byte global store (sm_100 family); 32-byte aligned address
__device__ __forceinline__ void st_global_v8_if(bool pred, void* ptr, const uint32_t* v) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %0, 0;\n\t@p st.global.v8.b32 [%1], {%2, %3, %4, %5, %6, %7, %8, %9};\n\t}" ::"r"(
            (int)pred),
        "l"(ptr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]));
}
__device__ __forceinline__ void st_global_u16_if(bool pred, void* ptr, uint16_t v) {
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %0, 0;\n\t@p st.global.u16 [%1], %2;\n\t}" ::"r"((int)pred), "l"(ptr),
                 "h"(v));
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc)
        : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor: start >> 4 (bits 0-13), leading byte offset >> 4 (16-29),
// stride byte offset >> 4 (32-45), descriptor version 1 (46-47), base offset 0, swizzle
// mode in bits 61-63 (2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((addr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// K-major operand tile with 128-byte swizzle (rows of 64 bf16, 8-row groups 1024 bytes apart):
// the descriptor of the kk-th 16-element K slice. The slice stays inside a swizzle row, so the
// leading byte offset is unused.
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t tile, int kk) { return smem_desc(tile + kk * 32, 16, 1024); }

__device__ __forceinline__ void tmem_alloc(uint32_t holder_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(holder_smem), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// ---- CTA pairs (cluster of two; tcgen05 ops of such a kernel all take .cta_group::2) ----

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
__device__ __forceinline__ uint32_t cluster_count_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}

// Address, in the shared::cluster window, of the variable at the same offset in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

// Arrive on an mbarrier given by its shared::cluster address (this CTA's or the peer's).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// All threads of both CTAs; orders earlier shared-memory and barrier operations cluster-wide.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// TMA loads into this CTA's shared memory that complete on an mbarrier of either CTA of the
// pair (given by its shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map, int x, int y, int z, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void tma_load_4d_pair(uint32_t dst, const CUtensorMap* map, int x, int y, int z, int w,
                                                 uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], [%6];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar)
        : "memory");
}

// Pair MMA: D (128 lanes of each CTA's tensor memory) += A (128 rows from each CTA) x B (N/2
// columns from each CTA); issued by one thread of the even CTA.
__device__ __forceinline__ void tc2_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc)
        : "memory");
}

// Arrive once on the mbarrier at this offset in every CTA of `mask` when the pair MMAs issued
// so far by this thread have completed.
__device__ __forceinline__ void tc2_commit_mc(uint32_t bar, uint16_t mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
        "h"(mask)
        : "memory");
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t holder_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(holder_smem), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Generic-proxy writes to shared memory become visible to the async proxy (TMA, tcgen05.mma).
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Bounded poll used when draining: true if the phase completed within the limit.
__device__ __forceinline__ bool mbar_drain(uint32_t bar, uint32_t parity, int32_t* hdr) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > kWaitTimeoutNs) {
            record_error(hdr, MOE_ERR_TIMEOUT);
            return false;
        }
    }
    return true;
}

// ---------------------------------------------------------------------------------------
// Counters between the tiles of one cooperative launch (every CTA resident): a producer tile
// fences its stores and increments a counter; a dependent tile polls it with acquire loads.
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ int ld_acquire_gpu(const int32_t* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// A 32-bit load through the coherent path (data another CTA of the same launch wrote).
__device__ __forceinline__ uint32_t ld_relaxed_gpu(const void* p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Polls until *c >= target (acquire loads, __nanosleep between), at most kWaitTimeoutNs; on
// time-out (or when another role of the CTA already gave up) records MOE_ERR_TIMEOUT once, sets
// the CTA's abort flag and returns false.
__device__ __forceinline__ bool wait_count(const int32_t* c, int target, int32_t* hdr, volatile int* abort_flag) {
    const uint64_t t0 = globaltimer_ns();
    while (ld_acquire_gpu(c) < target) {
        if (*abort_flag || globaltimer_ns() - t0 > kWaitTimeoutNs) {
            if (!*abort_flag) record_error(hdr, MOE_ERR_TIMEOUT);
            *abort_flag = 1;
            return false;
        }
        __nanosleep(64);
    }
    return true;
}

// Named barrier kBar over 128 threads (four warps), and the same barrier ANDing a predicate: the
// warps that share it leave their loop together.
template <int kBar>
__device__ __forceinline__ void bar_sync128() {
    asm volatile("bar.sync %0, 128;" ::"n"(kBar) : "memory");
}
template <int kBar>
__device__ __forceinline__ bool bar_all128(bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.b32 p, %1, 0;\n\tbar.red.and.pred q, %2, 128, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((int)pred), "n"(kBar)
        : "memory");
    return r != 0;
}

// ---------------------------------------------------------------------------------------
// Re-quantisation jobs of a fused integer launch. A's per-row scale needs whole rows, so the
// route tile's last L1 tile pushes kQuantJobs jobs of kQuantRows rows; the epilogue warps of any
// CTA pop and run them while they would otherwise wait (for their next accumulator, or for an L2
// tile's rows). Pops never wait: a slot that is reserved but not yet written, or taken by
// another CTA first, is left for the next try. Counters live in the workspace, zeroed per launch.
// ---------------------------------------------------------------------------------------
constexpr int kQuantRows = 128 / kQuantJobs;  // rows of A per job

struct QuantQueue {
    int32_t* dep;        // per route tile: finished L1 tiles, then finished jobs
    int32_t* jobs_done;  // jobs finished in the whole launch
    int32_t* head;       // next slot to pop
    int32_t* tail;       // next slot to reserve
    int32_t* slots;      // job + 1 per slot (0: not yet written)
    int n_jobs;          // kQuantJobs x the route tiles that hold rows

    // one thread, after its acquire of the route tile's count: the tile's jobs become visible
    __device__ __forceinline__ void push(int g) const {
        const int s = atomicAdd(tail, kQuantJobs);
        for (int c = 0; c < kQuantJobs; ++c)
            asm volatile("st.release.gpu.global.s32 [%0], %1;" ::"l"(slots + s + c), "r"(g * kQuantJobs + c + 1)
                         : "memory");
    }
    // one thread: a job (its acquire covers the job's rows of A), or -1 when none is written yet;
    // a slot lost to another CTA moves on to the next (a bounded number of times: many CTAs pop at
    // once when a round of L1 tiles ends). `drained` (the caller's, initially false) remembers that
    // every job was taken, so later calls cost no load.
    __device__ __forceinline__ int try_pop(bool& drained) const {
        if (drained) return -1;
        int h = (int)ld_relaxed_gpu(head);
        for (int tries = 0; tries < 64; ++tries) {
            drained = h >= n_jobs;
            if (drained) return -1;
            const int v = ld_acquire_gpu(slots + h);
            if (v == 0) return -1;
            const int old = atomicCAS(head, h, h + 1);
            if (old == h) return v - 1;
            h = old;  // taken: the head has moved on
        }
        return -1;
    }
};

// The four epilogue warps (128 threads sharing named barrier kBar; the leader is thread 0 of the
// first) run one job: kQuantRows / 4 rows per warp, then every thread fences its stores (for the L2 tiles' TMA
// and loads), the warps meet and the leader counts the job for its route tile and the launch.
// (not inlined: the epilogue keeps its registers for its own tiles, the job gets its own)
template <int kBar, int kRegVec>
__device__ __noinline__ void run_quant_job(const QuantQueue& qq, const Plan& p, int job, int q, int lane, bool leader) {
    const int g = job / kQuantJobs;
    const int r0 = g * 128 + (job % kQuantJobs) * kQuantRows;
    for (int r = q; r < kQuantRows; r += 4) quant_a_row<true, kRegVec>(p, r0 + r, lane);
    asm volatile("fence.proxy.async.global;" ::: "memory");
    __threadfence();
    bar_sync128<kBar>();
    if (leader) {
        __threadfence();
        atomicAdd(qq.dep + g, 1);
        atomicAdd(qq.jobs_done, 1);
    }
}

// The four epilogue warps wait until ready() (evaluated by the leader alone) holds, running jobs
// meanwhile; with kOneJob they stop after one job, or at once when none is available (the caller
// then waits in the usual way: a job started late would hold up the MMA that waits for the
// epilogue). The leader's decision reaches the others through `word` (shared memory) between
// two barriers, so all four leave together. At most kWaitTimeoutNs from the first try (a job in
// progress finishes first); on time-out records MOE_ERR_TIMEOUT, sets the abort flag and returns
// false. Loads after a true return are ordered after the leader's acquire in ready(). `drained`
// is the leader's QuantQueue::try_pop flag.
template <int kBar, int kRegVec, bool kOneJob, class Ready>
__device__ __forceinline__ bool idle_with_jobs(const QuantQueue& qq, const Plan& p, volatile int* word,
                                               volatile int* abort_flag, bool* drained, int q, int lane,
                                               Ready ready) {
    const bool leader = q == 0 && lane == 0;
    const uint64_t t0 = leader ? globaltimer_ns() : 0;
    for (;;) {
        if (leader) {
            int v = -1;  // -1 ready (kOneJob: or no job), >= 0 a job, -2 nothing to do yet, -3 give up
            if (!ready()) {
                v = qq.try_pop(*drained);
                if (v < 0 && kOneJob) v = -1;
                if (v < 0 && !kOneJob) {
                    v = -2;
                    if (*abort_flag || globaltimer_ns() - t0 > kWaitTimeoutNs) {
                        if (!*abort_flag) record_error(p.hdr, MOE_ERR_TIMEOUT);
                        *abort_flag = 1;
                        v = -3;
                    }
                }
            }
            *word = v;
        }
        bar_sync128<kBar>();
        const int v = *word;
        bar_sync128<kBar>();  // every thread has read it before the leader writes the next
        if (v == -1) return true;
        if (v == -3) return false;
        if (v == -2) {
            __nanosleep(256);
            continue;
        }
        run_quant_job<kBar, kRegVec>(qq, p, v, q, lane, leader);
        if (kOneJob) return true;
    }
}

}  // namespace tc



// Host helpers (tc_host.cu).
bool tc_make_map_2d(CUtensorMap* map, CUtensorMapDataType dtype, int elem_bytes, const void* ptr, uint64_t inner,
                    uint64_t outer, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle);
bool tc_encode_available();
int tc_num_sms();
// Packed e2m1 tensor [outer, inner_elems] (two codes per byte): TMA expands every 8-byte group of
// 16 codes into a 16-byte slot of the 128-byte-swizzled shared tile (the 4-bit operand layout of
// kind::mxf8f6f4); the transaction byte count is the packed size.
// Rank-1..5 tiled map: dims and box in elements (innermost first), strides in bytes of dims 1..rank-1.
bool tc_make_map_nd(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* ptr, const uint64_t* dims,
                    const uint64_t* strides_bytes, const uint32_t* box, CUtensorMapSwizzle swizzle);
bool tc_make_map_2d_packed4(CUtensorMap* map, const void* ptr, uint64_t inner_elems, uint64_t outer,
                            uint32_t box_inner, uint32_t box_outer);

}  // namespace moe
