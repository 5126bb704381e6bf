// Tensor-core grouped GEMM stages for bf16 operands on sm_103a: tcgen05.mma with fp32
// accumulators in tensor memory, operands staged in shared memory by TMA, a 4-stage mbarrier
// ring between the loader and the MMA issuer, and two TMEM accumulators so the epilogue of
// one tile overlaps the main loop of the next.
//
// Work decomposition (one persistent CTA per SM, static round-robin over tiles):
//   tile = (expert e, 128-row block m of e's padded pool rows, column block n)
//   tiles are ordered expert-major, then n, then m, so the CTAs in flight share a few
//   weight column blocks of one expert in L2 while the expert's rows stay resident.
//
// L1 (Ascend mega_moe page, "Linear1 Projection" + "SwiGLU Activation"): the B tile of a stage
// is the gate column block [n*128, n*128+128) and the up column block [I+n*128, ...) of
// W1[e] (two TMA boxes each), so one 128x256 accumulator holds the gate and up values of the
// same 128 outputs and SwiGLU runs in the epilogue: A = SiLU(gate) * up -> bf16.
// L2 ("Linear2 Projection" + the gate weight of "Token Combine"): 128x256 accumulator over
// H columns; the epilogue multiplies row p by G[row_src[p]] in fp32 and stores bf16 to the
// combine row of (token, slot).
//
// L1, L2 and the combine in one launch (the DeepGEMM page's single kernel with dependency
// counters, §5): the fused instantiation runs every L1 tile, then every L2 tile, over one
// static round-robin order, so each CTA finishes its L1 tiles before it starts on L2, and then
// every warp combines tokens. An L2 tile needs the A rows of its 128-row route tile from all
// I/128 L1 tiles of that route tile: the L1 epilogue publishes each finished tile with a release
// increment of the route tile's counter, and the L2 producer waits (bounded) until the count is
// complete before its TMA reads A. A token's combine needs its routed rows from every L2 column
// block: each L2 epilogue thread publishes its row with an increment of the token's counter,
// and the combining warp waits (bounded) for (its unmasked slots) x (column blocks). CTAs whose
// L2 tiles end early combine while others are still in L2. The launch is cooperative, so every
// CTA is resident and every wait is on work that earlier positions of the order hold.
//
// Warp roles (192 threads): warp 0 = TMA producer, warp 1 = TMEM allocator + MMA issuer,
// warps 2-5 = epilogue (warp w reads TMEM lanes 32*(w%4) .. 32*(w%4)+31).
// Every mbarrier wait is bounded (2 s); on time-out the CTA records MOE_ERR_TIMEOUT, drains
// what it has in flight (again bounded), frees its tensor memory and exits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "tc_common.cuh"

namespace moe {

namespace {

using namespace tc;

constexpr int kBM = 128;                       // rows per tile (MMA M)
constexpr int kBN = 256;                       // accumulator columns per tile (MMA N)
constexpr int kBK = 64;                        // K per stage: 64 bf16 = one 128-byte swizzle row
constexpr int kStages = 4;
constexpr int kABytes = kBM * kBK * 2;         // 16 KB
constexpr int kBBoxBytes = kBK * 64 * 2;       // one 64(K) x 64(N) box, 8 KB
constexpr int kBBytes = 4 * kBBoxBytes;        // 32 KB
constexpr int kStageBytes = kABytes + kBBytes; // 48 KB
constexpr int kThreads = 192;
constexpr int kTmemCols = 512;                 // two 256-column fp32 accumulators
constexpr int kMaxExperts = 1024;

// Instruction descriptor of tcgen05.mma.kind::f16: D fp32 (bits 4-5 = 1), A bf16 (bits 7-9 =
// 1), B bf16 (bits 10-12 = 1), A K-major (bit 15 = 0), B MN-major (bit 16 = 1), N >> 3 in
// bits 17-22, M >> 4 in bits 24-28.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (0u << 15) | (1u << 16) |
                            ((uint32_t)(kBN >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);

struct TcArgs {
    Plan p;
    const float* topk_weights;  // L2 only
    int n_tiles;                // column blocks per expert
    int k_blocks;               // K / 64
    int k_rows;                 // rows of one expert's weight in its 2-D view (L1: H, L2: I)
    int b_one_box;              // B map brings a stage's four 64-column blocks in one copy
    // fused launch: the L2 stage's figures, the per-route-tile count of finished L1 tiles, and
    // (when y is given) the per-token count of finished combine rows and the output
    int n_tiles2, k_blocks2, k_rows2, b_one_box2;
    int32_t* l1_done;
    int32_t* token_done;
    uint16_t* y;
};

constexpr int kL2 = 0, kL1 = 1, kFusedL1L2 = 2;  // what one launch runs

// Count of the finished L1 tiles of a route tile, read with acquire semantics at GPU scope.
__device__ __forceinline__ int ld_acquire_gpu(const int32_t* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// A tile: 128 rows x 64 K, K-major, 128-byte swizzle (the TMA box layout). 8-row groups are
// 1024 bytes apart; the K extent of one MMA (16 elements, 32 bytes) stays inside a swizzle
// row, so the leading byte offset is unused.
__device__ __forceinline__ uint64_t a_desc(uint32_t tile, int kk) { return kmajor_desc(tile, kk); }

// B tile: four 64(K) x 64(N) boxes, N contiguous (MN-major), 128-byte swizzle. The 64-column
// groups are one box (8 KB) apart (leading byte offset); groups of 8 K rows are 1024 bytes
// apart (stride byte offset). One MMA consumes 16 K rows = 2048 bytes of every box.
__device__ __forceinline__ uint64_t b_desc(uint32_t tile, int kk) {
    return smem_desc(tile + kk * 2048, kBBoxBytes, 1024);
}

struct Tile {
    int e, m, n, row0;
};

// Tiles are ordered expert-major: expert e owns tiles [tile_off[e] * n_tiles, tile_off[e+1] * n_tiles).
__device__ __forceinline__ Tile decode_tile(int t, const int* tile_off, int E, int n_tiles) {
    int lo = 0, hi = E - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (tile_off[mid] * n_tiles <= t) lo = mid; else hi = mid - 1;
    }
    Tile tl;
    tl.e = lo;
    const int mt = tile_off[lo + 1] - tile_off[lo];
    const int local = t - tile_off[lo] * n_tiles;
    tl.n = local / mt;
    tl.m = local % mt;
    tl.row0 = (tile_off[lo] + tl.m) * kBM;
    return tl;
}

template <int kKind>  // kL1, kL2 or kFusedL1L2
__global__ void __launch_bounds__(kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ CUtensorMap tmB2, TcArgs args) {
    constexpr bool kFused = kKind == kFusedL1L2;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (base - raw);
    const uint32_t bar0 = base + kStages * kStageBytes;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (kStages + s); };
    auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * kStages + a); };
    auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * kStages + 2 + a); };
    const uint32_t drain_bar = bar0 + 8u * (2 * kStages + 4);
    uint8_t* misc = smem + kStages * kStageBytes + 8 * (2 * kStages + 5);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(misc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 4);
    int* epi_done = reinterpret_cast<int*>(misc + 8);  // fused: epilogue warps done with L1 tiles
    int* tile_off = reinterpret_cast<int*>(misc + 16);

    const Plan& p = args.p;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i <= p.E; i += kThreads) tile_off[i] = p.tile_off[i];
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), 4);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        *epi_done = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_holder)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (warp == 0 && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB)) : "memory");
        if (kFused) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA2)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB2)) : "memory");
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    // tiles [0, total1) are the launch's first stage (L1 when fused), [total1, total) the L2 ones
    const int total1 = tile_off[p.E] * args.n_tiles;
    const int total = kFused ? total1 + tile_off[p.E] * args.n_tiles2 : total1;
    auto is_l1 = [&](int t) { return kKind == kL1 || (kFused && t < total1); };
    auto tile_of = [&](int t) {
        return kFused && t >= total1 ? decode_tile(t - total1, tile_off, p.E, args.n_tiles2)
                                     : decode_tile(t, tile_off, p.E, args.n_tiles);
    };
    auto k_blocks_of = [&](int t) { return kFused && t >= total1 ? args.k_blocks2 : args.k_blocks; };

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer ----------------
            int it = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const bool l1 = is_l1(t), second = kFused && !l1;
                const Tile tl = tile_of(t);
                const CUtensorMap* mA = second ? &tmA2 : &tmA;
                const CUtensorMap* mB = second ? &tmB2 : &tmB;
                const int wrow = tl.e * (second ? args.k_rows2 : args.k_rows);
                const int one_box = second ? args.b_one_box2 : args.b_one_box;
                const int KB = k_blocks_of(t);
                if (second) {
                    // every L1 tile of this route tile has published its A rows
                    const int32_t* done = args.l1_done + tile_off[tl.e] + tl.m;
                    const uint64_t t0 = globaltimer_ns();
                    while (ld_acquire_gpu(done) < args.n_tiles) {
                        if (*abort_flag) {
                            ok = false;
                            break;
                        }
                        if (globaltimer_ns() - t0 > kWaitTimeoutNs) {
                            record_error(p.hdr, MOE_ERR_TIMEOUT);
                            *abort_flag = 1;
                            ok = false;
                            break;
                        }
                        __nanosleep(64);
                    }
                    if (!ok) break;
                    // those rows were written through the generic proxy; the TMA reads them
                    asm volatile("fence.proxy.async.global;" ::: "memory");
                }
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    const int s = it % kStages;
                    const uint32_t ph = (uint32_t)(it / kStages) & 1u;
                    if (!mbar_wait(empty_bar(s), ph ^ 1u, p.hdr, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = base + s * kStageBytes, sb = sa + kABytes;
                    mbar_arrive_expect_tx(full_bar(s), kStageBytes);
                    tma_load_2d(sa, mA, kb * kBK, tl.row0, full_bar(s));
                    const int y = wrow + kb * kBK;
                    if (one_box) {
                        // [64 columns][K row][column block](L1: [gate, up]) in one copy
                        if (l1)
                            tma_load_4d(sb, mB, 0, y, 2 * tl.n, 0, full_bar(s));
                        else
                            tma_load_3d(sb, mB, 0, y, 4 * tl.n, full_bar(s));
                    } else if (l1) {
                        const int g0 = tl.n * 128, u0 = p.I + tl.n * 128;
                        tma_load_2d(sb, mB, g0, y, full_bar(s));
                        tma_load_2d(sb + kBBoxBytes, mB, g0 + 64, y, full_bar(s));
                        tma_load_2d(sb + 2 * kBBoxBytes, mB, u0, y, full_bar(s));
                        tma_load_2d(sb + 3 * kBBoxBytes, mB, u0 + 64, y, full_bar(s));
                    } else {
#pragma unroll
                        for (int j = 0; j < 4; ++j) tma_load_2d(sb + j * kBBoxBytes, mB, tl.n * kBN + j * 64, y, full_bar(s));
                    }
                }
            }
            // drain: wait until every load issued into a stage has landed (bounded)
            for (int j = it - kStages < 0 ? 0 : it - kStages; j < it; ++j) {
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait(full_bar(j % kStages), (uint32_t)(j / kStages) & 1u)) {
                    if (globaltimer_ns() - t0 > kWaitTimeoutNs) {
                        record_error(p.hdr, MOE_ERR_TIMEOUT);
                        break;
                    }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            // This thread feeds the tensor pipe, so its per-stage work is kept short: a
            // non-blocking test of the stage first, and descriptors advanced by adding to their
            // address field (start >> 4: +2 per 32 bytes of A's K, +128 per 2 KB of B's K rows,
            // + stage offset >> 4), measured ~1.5 % faster on L2 than rebuilding them per MMA.
            const uint64_t ad0 = a_desc(base, 0), bd0 = b_desc(base + kABytes, 0);
            int it = 0, tc = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++tc) {
                const int a = tc & 1;
                if (!mbar_wait(tempty_bar(a), ((uint32_t)(tc >> 1) & 1u) ^ 1u, p.hdr, abort_flag)) break;
                tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)(a * kBN);
                const int KB = k_blocks_of(t);
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    const int s = it % kStages;
                    const uint32_t par = (uint32_t)(it / kStages) & 1u;
                    if (!mbar_test(full_bar(s), par) && !mbar_wait(full_bar(s), par, p.hdr, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t off = (uint64_t)((s * kStageBytes) >> 4);
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        tc_mma(d, ad0 + off + 2 * kk, bd0 + off + 128 * kk, kIdesc, (kb | kk) != 0);
                    tc_commit(empty_bar(s));  // frees the stage once these MMAs have read it
                }
                if (ok) tc_commit(tfull_bar(a));
            }
            // drain: every MMA issued so far has completed before tensor memory is freed
            tc_commit(drain_bar);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(drain_bar, 0)) {
                if (globaltimer_ns() - t0 > kWaitTimeoutNs) {
                    record_error(p.hdr, MOE_ERR_TIMEOUT);
                    break;
                }
            }
        }
    } else {
        // ---------------- epilogue (warps 2..5) ----------------
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        int tc = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x, ++tc) {
            const int a = tc & 1;
            const bool l1 = is_l1(t);
            const Tile tl = tile_of(t);
            const int64_t row = tl.row0 + q * 32 + lane;
            // L2: the row's combine slot and gate weight, read while the tile's MMAs still run
            int src = -1;
            float gw = 0.0f;
            if (!l1) {
                src = debug_row(p.hdr, __ldg(p.pool_src + row), (int64_t)p.T * p.K);
                gw = src >= 0 ? __ldg(args.topk_weights + src) : 0.0f;
            }
            // every lane waits; the warp goes on only if all of them saw the phase complete
            const bool ok = mbar_wait(tfull_bar(a), (uint32_t)(tc >> 1) & 1u, p.hdr, abort_flag);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc_fence_after();
            const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(a * kBN);
            if (l1) {
                uint16_t* out = reinterpret_cast<uint16_t*>(p.a_pool) + row * p.I + tl.n * 128;
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    uint32_t g[32], u[32];
                    tmem_ld32(tbase + c * 32, g);
                    tmem_ld32(tbase + 128 + c * 32, u);
                    tmem_ld_wait();
                    uint32_t packed[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float a0 = swiglu1(__uint_as_float(g[2 * j]), __uint_as_float(u[2 * j]), p.act_clamp);
                        const float a1 = swiglu1(__uint_as_float(g[2 * j + 1]), __uint_as_float(u[2 * j + 1]), p.act_clamp);
                        packed[j] = (uint32_t)float_to_bf16_bits(a0) | ((uint32_t)float_to_bf16_bits(a1) << 16);
                    }
                    st_global_v8_if(true, out + c * 32, packed);
                    st_global_v8_if(true, out + c * 32 + 16, packed + 8);
                }
                if (kFused) {
                    // publish the tile: each warp fences its own stores; the last of the four
                    // warps to finish counts the tile for its route tile (no warp waits here)
                    __threadfence();
                    __syncwarp();
                    if (lane == 0 && (atomicAdd(epi_done, 1) & 3) == 3) {
                        __threadfence();
                        atomicAdd(args.l1_done + tile_off[tl.e] + tl.m, 1);
                    }
                }
            } else {
                uint16_t* out = p.comb + (int64_t)(src >= 0 ? src : 0) * p.H + tl.n * kBN;
#pragma unroll 1
                for (int c = 0; c < kBN / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld32(tbase + c * 32, r);
                    tmem_ld_wait();
                    uint32_t packed[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float y0 = __fmul_rn(gw, __uint_as_float(r[2 * j]));
                        const float y1 = __fmul_rn(gw, __uint_as_float(r[2 * j + 1]));
                        packed[j] = (uint32_t)float_to_bf16_bits(y0) | ((uint32_t)float_to_bf16_bits(y1) << 16);
                    }
                    st_global_v8_if(src >= 0, out + c * 32, packed);
                    st_global_v8_if(src >= 0, out + c * 32 + 16, packed + 8);
                }
                if (kFused && args.y != nullptr && src >= 0) {  // publish this combine row's columns
                    __threadfence();
                    atomicAdd(args.token_done + src / p.K, 1);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty_bar(a));
        }
    }

    if constexpr (kFused) {
        if (args.y != nullptr) {
            // ---------------- combine (S6), every warp ----------------
            // y[t] = bf16( sum over the unmasked slots k of comb[t*K + k] ), fp32 in slot order (as
            // the combine kernel); the rows were written by other CTAs, so they are read through
            // L2 once the token's count is complete
            __syncwarp();
            constexpr int kWarps = kThreads / 32;
            const int K = p.K, row_vecs = p.H / 8;
            const uint4* comb = reinterpret_cast<const uint4*>(p.comb);
            uint4* y = reinterpret_cast<uint4*>(args.y);
            for (int t = blockIdx.x * kWarps + warp; t < p.T && !*abort_flag; t += gridDim.x * kWarps) {
                const int sr = lane < K ? __ldg(p.slot_row + (int64_t)t * K + lane) : -1;
                const unsigned valid = __ballot_sync(0xffffffffu, sr >= 0);
                const int target = __popc(valid) * args.n_tiles2;
                int ok = 1;
                if (lane == 0) {
                    const uint64_t t0 = globaltimer_ns();
                    while (ld_acquire_gpu(args.token_done + t) < target) {
                        if (*abort_flag) {
                            ok = 0;
                            break;
                        }
                        if (globaltimer_ns() - t0 > kWaitTimeoutNs) {
                            record_error(p.hdr, MOE_ERR_TIMEOUT);
                            *abort_flag = 1;
                            ok = 0;
                            break;
                        }
                        __nanosleep(128);
                    }
                }
                if (!__shfl_sync(0xffffffffu, ok, 0)) break;
                // four vectors per lane in flight: every slot's load is issued before the adds
                constexpr int kV = 4;
                for (int v0 = lane; v0 < row_vecs; v0 += 32 * kV) {
                    float acc[kV][8];
#pragma unroll
                    for (int u = 0; u < kV; ++u)
#pragma unroll
                        for (int j = 0; j < 8; ++j) acc[u][j] = 0.0f;
                    for (int k = 0; k < K; ++k) {
                        if (!((valid >> k) & 1u)) continue;  // masked route: contributes nothing
                        const uint4* row = comb + ((int64_t)t * K + k) * row_vecs;
                        uint4 c[kV];
#pragma unroll
                        for (int u = 0; u < kV; ++u) c[u] = v0 + 32 * u < row_vecs ? __ldcg(row + v0 + 32 * u) : make_uint4(0, 0, 0, 0);
#pragma unroll
                        for (int u = 0; u < kV; ++u) {
                            const uint32_t w[4] = {c[u].x, c[u].y, c[u].z, c[u].w};
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                acc[u][2 * j] = __fadd_rn(acc[u][2 * j], __uint_as_float(w[j] << 16));
                                acc[u][2 * j + 1] = __fadd_rn(acc[u][2 * j + 1], __uint_as_float(w[j] & 0xffff0000u));
                            }
                        }
                    }
#pragma unroll
                    for (int u = 0; u < kV; ++u) {
                        if (v0 + 32 * u >= row_vecs) break;
                        uint32_t o[4];
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            o[j] = (uint32_t)float_to_bf16_bits(acc[u][2 * j]) |
                                   ((uint32_t)float_to_bf16_bits(acc[u][2 * j + 1]) << 16);
                        y[(int64_t)t * row_vecs + v0 + 32 * u] = make_uint4(o[0], o[1], o[2], o[3]);
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTmemCols)
                     : "memory");
    }
}

// ---------------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------------

// 2-D bf16 tensor [outer, inner] (row-major), boxes of box_outer x 64 elements, 128-byte swizzle.
bool make_map(CUtensorMap* map, const void* ptr, uint64_t inner, uint64_t outer, uint32_t box_outer) {
    return tc_make_map_2d(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ptr, inner, outer, 64, box_outer,
                          CU_TENSOR_MAP_SWIZZLE_128B);
}

constexpr size_t smem_bytes() {
    return 1024 + (size_t)kStages * kStageBytes + 8 * (2 * kStages + 5) + 16 + 4 * (kMaxExperts + 1);
}

template <int kKind>
cudaError_t set_smem_attr() {
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(tc_gemm_kernel<kKind>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)smem_bytes());
    });
    return attr_err;
}

template <int kKind>
cudaError_t launch_tc(const Plan& p, const CUtensorMap& a, const CUtensorMap& b, TcArgs args, cudaStream_t s) {
    const cudaError_t attr_err = set_smem_attr<kKind>();
    if (attr_err != cudaSuccess) return attr_err;
    const int64_t max_tiles = (p.pool_rows / kBM) * args.n_tiles;
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(max_tiles, tc_num_sms()));
    tc_gemm_kernel<kKind><<<grid, kThreads, smem_bytes(), s>>>(a, b, a, b, args);
    return cudaGetLastError();
}

}  // namespace

bool tc_supported(const Plan& p, int stage) {
    if (p.mode != MOE_A16W16 || p.E > kMaxExperts || !tc_encode_available()) return false;
    if (stage == 1) return p.I % 128 == 0;
    return p.H % kBN == 0;
}

// B (weights, N contiguous) as [64 columns][K row][64-column block] (+ [gate, up] for L1), so one
// box brings a stage's four 8 KB blocks in the MMA's layout: the dimensions are listed in the
// order the box is written, so their strides do not increase. Falls back to 2-D boxes (four
// copies a stage) when the driver's encoder does not take such a map.
bool make_b_map(CUtensorMap* map, const void* w, uint64_t n_cols, uint64_t rows, uint64_t half_cols, bool l1,
                int* one_box) {
    const uint64_t pitch = n_cols * 2;
    bool ok;
    if (l1) {
        const uint64_t dims[4] = {64, rows, half_cols / 64, 2};
        const uint64_t strides[3] = {pitch, 128, half_cols * 2};
        const uint32_t box[4] = {64, (uint32_t)kBK, 2, 2};
        ok = tc_make_map_nd(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, w, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
    } else {
        const uint64_t dims[3] = {64, rows, n_cols / 64};
        const uint64_t strides[2] = {pitch, 128};
        const uint32_t box[3] = {64, (uint32_t)kBK, 4};
        ok = tc_make_map_nd(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, w, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
    }
    *one_box = ok ? 1 : 0;
    return ok || make_map(map, w, n_cols, rows, kBK);
}

cudaError_t launch_l1_tc(const Plan& p, const void* w1, const void*, cudaStream_t s) {
    CUtensorMap a, b;
    int one_box = 0;
    if (!make_map(&a, p.x_pool, (uint64_t)p.H, (uint64_t)p.pool_rows, kBM)) return cudaErrorInvalidValue;
    if (!make_b_map(&b, w1, (uint64_t)2 * p.I, (uint64_t)p.E * p.H, (uint64_t)p.I, true, &one_box))
        return cudaErrorInvalidValue;
    TcArgs args{p, nullptr, p.I / 128, p.H / kBK, p.H, one_box, 0, 0, 0, 0, nullptr, nullptr, nullptr};
    return launch_tc<kL1>(p, a, b, args, s);
}

cudaError_t launch_l2_tc(const Plan& p, const void* w2, const void*, const float* topk_weights, cudaStream_t s) {
    CUtensorMap a, b;
    int one_box = 0;
    if (!make_map(&a, p.a_pool, (uint64_t)p.I, (uint64_t)p.pool_rows, kBM)) return cudaErrorInvalidValue;
    if (!make_b_map(&b, w2, (uint64_t)p.H, (uint64_t)p.E * p.I, (uint64_t)p.H, false, &one_box))
        return cudaErrorInvalidValue;
    TcArgs args{p, topk_weights, p.H / kBN, p.I / kBK, p.I, one_box, 0, 0, 0, 0, nullptr, nullptr, nullptr};
    return launch_tc<kL2>(p, a, b, args, s);
}

cudaError_t launch_ffn_fused_tc(const Plan& p, const void* w1, const void* w2, const float* topk_weights,
                                uint16_t* y, cudaStream_t s) {
    CUtensorMap a1, b1, a2, b2;
    int one_box1 = 0, one_box2 = 0;
    if (!make_map(&a1, p.x_pool, (uint64_t)p.H, (uint64_t)p.pool_rows, kBM) ||
        !make_b_map(&b1, w1, (uint64_t)2 * p.I, (uint64_t)p.E * p.H, (uint64_t)p.I, true, &one_box1) ||
        !make_map(&a2, p.a_pool, (uint64_t)p.I, (uint64_t)p.pool_rows, kBM) ||
        !make_b_map(&b2, w2, (uint64_t)p.H, (uint64_t)p.E * p.I, (uint64_t)p.H, false, &one_box2))
        return cudaErrorInvalidValue;
    // the counters (one per 128-row route tile, then one per token) start at zero every launch
    const int64_t route_tiles = p.pool_rows / kBM;
    cudaError_t e = cudaMemsetAsync(p.ffn_counters, 0, sizeof(int32_t) * (size_t)(route_tiles + p.T), s);
    if (e != cudaSuccess) return e;
    if ((e = set_smem_attr<kFusedL1L2>()) != cudaSuccess) return e;
    TcArgs args{p,          topk_weights, p.I / 128,        p.H / kBK, p.H, one_box1, p.H / kBN, p.I / kBK, p.I,
                one_box2,   p.ffn_counters, p.ffn_counters + route_tiles, y};
    // every CTA resident at once (cooperative launch): an L2 tile waits only for L1 tiles that
    // earlier positions of the same round-robin order hold, all of them running
    int per_sm = 0;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, tc_gemm_kernel<kFusedL1L2>, kThreads,
                                                           smem_bytes())) != cudaSuccess)
        return e;
    const int64_t max_tiles = route_tiles * (p.I / 128 + p.H / kBN);
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(max_tiles, (int64_t)tc_num_sms() * std::max(per_sm, 1)));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem_bytes();
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, tc_gemm_kernel<kFusedL1L2>, a1, b1, a2, b2, args);
}

}  // namespace moe
