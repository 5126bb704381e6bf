// INT8 grouped GEMM on the tensor cores with exact int32 results (Ascend mega_moe page, A8W8-INT
// use case: C = Q_e . W1^int8 and D = A^int8 . W2^int8 in int32, then (C * s^W) * s^X in fp32).
//
// sm_103a has no integer tcgen05.mma kind, so the integers travel as f16 (kind::f16, fp32
// accumulation in TMEM), which is exact as long as every partial sum stays below 2^24:
// - the token codes are split as q = 16*hi + lo with hi = floor(q/16) in [-8, 7] and
//   lo = q mod 16 in [0, 15] (the identity of the page's A8W4-INT MSD scheme); the dispatch
//   stage (x) and the row quantiser (A) store them as two f16 planes;
// - the weights stay int8 in HBM; TMA brings them into a staging ring (64-byte swizzle) and four
//   converter warps expand them to f16 (q ^ 0x80 placed under the exponent of 1024 gives
//   1152 + q exactly; one f16 subtraction removes the 1152), in the 128-byte-swizzled K-major
//   layout of the MMA;
// - one tile is 128 weight rows x the n tokens of one route tile rounded up to 16 (n16 <= 128);
//   its B tile holds the tokens' hi rows, then their lo rows (N = 2 * n16), so |partial sum| <=
//   15 * 128 * K < 2^24 for K <= 8704, and the epilogue rebuilds the exact accumulator as
//   16 * D_hi + D_lo in int32 before the fp32 dequantisation. An expert's last route tile is
//   usually partial (on average half of it is padding), and its MMAs cover only n16 tokens: full
//   tiles take the 128-row token box, partial ones n16 / 16 boxes of 16 rows per plane.
// Weight-major orientation as in the block-scaled kernel: M = weight rows; L1 tiles carry the
// gate block and the up block of the same 128 outputs (two accumulators sharing B), L2 tiles two
// 128-row blocks of hidden columns.
//
// Warp roles (352 threads): warp 0 TMA of raw weights, warp 1 TMEM allocation + MMA issue,
// warps 2-5 epilogue, warps 6-9 weight converters, warp 10 TMA of the token tiles.
// Every wait is bounded; on time-out the CTA records MOE_ERR_TIMEOUT, drains and exits.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "tc_common.cuh"

namespace moe {

namespace {

using namespace tc;

constexpr int kWR = 128;        // weight rows per block (MMA M)
constexpr int kTok = 128;       // tokens per tile (one route tile)
constexpr int kBK = 64;         // K per stage: 64 f16 = one 128-byte swizzle row
constexpr int kThreads = 352;
constexpr int kMaxExperts = 1024;
constexpr int kABytes = 2 * kWR * 128;   // two f16 weight blocks
constexpr int kTokBytes = 2 * kTok * 128;  // hi rows, then lo rows
constexpr int kRawBytes = 2 * kWR * kBK;   // two int8 weight blocks
constexpr int kTokBox = 16;  // token rows per TMA box of a partial tile

// Shared-memory layout. Int8 weights: TMA fills a ring of raw int8 tiles that the converter warps
// expand into a ring of f16 tiles. Prepared weights (exact f16 codes written once by
// moe_prepare_weights): TMA fills the f16 ring directly, which takes the raw ring's space as a
// third stage, and the converter warps stay idle.
template <bool kPrep>
struct Layout {
    static constexpr int kRawStages = kPrep ? 0 : 3, kHfStages = kPrep ? 3 : 2, kTokStages = 3;
    static constexpr int kHfOff = 0;
    static constexpr int kTokOff = kHfOff + kHfStages * kABytes;
    static constexpr int kRawOff = kTokOff + kTokStages * kTokBytes;
    static constexpr int kBarOff = kRawOff + kRawStages * kRawBytes;
    static constexpr int kNumBars = 2 * (kRawStages + kHfStages + kTokStages) + 2 + 1;
    static constexpr int kMiscOff = kBarOff + 8 * kNumBars;
    static constexpr int kTileOffOff = kMiscOff + 16;
    static constexpr int kCountsOff = kTileOffOff + 4 * (kMaxExperts + 1);
    static constexpr int kTabOff = kCountsOff + 4 * kMaxExperts;  // L2 epilogue: per warp [slot, gate, s^A] x 128 rows
    static constexpr size_t kSmem = 1024 + (size_t)kTabOff + 4 * 3 * 4 * kTok;
    static_assert(kSmem <= 232448, "shared memory");
};
// largest K with every partial sum below 2^24: |lo * w| <= 15 * 128
constexpr int kMaxK = 8704;

// kind::f16 instruction descriptor: D fp32 (bits 4-5 = 1), A and B f16 (formats 0), both
// K-major, N = 2 * n16 (>> 3 in bits 17-22, set per tile), M = 128 (>> 4 in bits 24-28).
constexpr uint32_t kIdescM = (1u << 4) | ((uint32_t)(kWR >> 4) << 24);
__device__ __forceinline__ uint32_t idesc_n(int n) { return kIdescM | ((uint32_t)(n >> 3) << 17); }

// Tokens of a route tile rounded up to 16 (the B rows of each plane that its MMAs use).
__device__ __forceinline__ int tile_n16(const int* counts, int e, int m) {
    const int n = min(kTok, counts[e] - m * kTok);
    return min(kTok, (n + 15) & ~15);
}

struct I8Args {
    Plan p;
    const float* w_scale;       // fp32 per output channel [E*n_out]
    const float* topk_weights;  // L2
    int n_slabs, k_blocks, n_out;
    // the fused launch (L1 then L2 in one launch): the fields above describe its L1, these its L2
    const float* w_scale2;
    int n_slabs2, k_blocks2;
    int32_t* ctr;  // the workspace's counters: per route tile, then the re-quantisation job queue
};

constexpr int kL2 = 0, kL1 = 1, kFusedL1L2 = 2;  // what one launch runs
constexpr int kEpiBar = 1;                       // named barrier of the 4 epilogue warps
constexpr int kQuantRegVec = 12;  // fused launch: rows of A up to 1536 elements re-quantised from registers

struct Tile {
    int e, s, m, row0;
};

__device__ __forceinline__ Tile decode(int t, const int* tile_off, int E, int n_slabs) {
    int lo = 0, hi = E - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (tile_off[mid] * n_slabs <= t) lo = mid; else hi = mid - 1;
    }
    Tile tl;
    tl.e = lo;
    const int mt = tile_off[lo + 1] - tile_off[lo];
    const int local = t - tile_off[lo] * n_slabs;
    tl.s = local / mt;
    tl.m = local % mt;
    tl.row0 = (tile_off[lo] + tl.m) * kTok;
    return tl;
}

// 4 int8 codes (one 32-bit word) -> 2 f16x2 words, exactly: u = q ^ 0x80 = q + 128 placed as
// the mantissa of f16 1024 gives 1152 + q; subtracting 1152 leaves q.
__device__ __forceinline__ void int8x4_to_f16(uint32_t w, uint32_t& lo, uint32_t& hi) {
    const uint32_t u = w ^ 0x80808080u;
    const uint32_t a = __byte_perm(u, 0x64646464u, 0x5140);  // bytes u0, 0x64, u1, 0x64
    const uint32_t b = __byte_perm(u, 0x64646464u, 0x7362);  // bytes u2, 0x64, u3, 0x64
    const __half2 off = __half2half2(__ushort_as_half((unsigned short)0x6480));  // 1152
    const __half2 ra = __hsub2(*reinterpret_cast<const __half2*>(&a), off);
    const __half2 rb = __hsub2(*reinterpret_cast<const __half2*>(&b), off);
    lo = *reinterpret_cast<const uint32_t*>(&ra);
    hi = *reinterpret_cast<const uint32_t*>(&rb);
}

// Weight row r's 64 int8 codes from the raw tile (64-byte rows, 64-byte swizzle: chunk index
// ^= address bits 7-8), as four 16-byte chunks in K order. The converters load every chunk of
// their rows before the first store: the compiler cannot tell the raw and f16 tiles apart, so a
// load placed after a store would wait for it.
__device__ __forceinline__ void load_row(const uint8_t* raw_tile, int r, uint4 (&c)[4]) {
    const uint8_t* row = raw_tile + r * 64;
    const int x = (r >> 1) & 3;
#pragma unroll
    for (int q = 0; q < 4; ++q) c[q] = *reinterpret_cast<const uint4*>(row + ((q ^ x) << 4));
}

// Expand them into f16 row r of a 128-byte-swizzled K-major tile.
__device__ __forceinline__ void store_row(const uint4 (&c)[4], uint8_t* tile, int r) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {  // 16 codes -> two 16-byte chunks of 8 f16
        uint32_t o[8];
        int8x4_to_f16(c[q].x, o[0], o[1]);
        int8x4_to_f16(c[q].y, o[2], o[3]);
        int8x4_to_f16(c[q].z, o[4], o[5]);
        int8x4_to_f16(c[q].w, o[6], o[7]);
        const int ch0 = 2 * q, ch1 = 2 * q + 1;
        *reinterpret_cast<uint4*>(tile + r * 128 + ((ch0 ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
        *reinterpret_cast<uint4*>(tile + r * 128 + ((ch1 ^ (r & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
    }
}

__device__ __forceinline__ int exact_int(uint32_t hi_bits, uint32_t lo_bits) {
    return 16 * __float2int_rn(__uint_as_float(hi_bits)) + __float2int_rn(__uint_as_float(lo_bits));
}

template <int kKind, bool kPrep>
__global__ void __launch_bounds__(kThreads, 1)
    tc_int8_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                   const __grid_constant__ CUtensorMap tmX16, const __grid_constant__ CUtensorMap tmW2,
                   const __grid_constant__ CUtensorMap tmX2, const __grid_constant__ CUtensorMap tmX16_2,
                   I8Args args) {
    constexpr bool kFused = kKind == kFusedL1L2;
    using L = Layout<kPrep>;
    constexpr int kRawStages = L::kRawStages, kHfStages = L::kHfStages, kTokStages = L::kTokStages;
    constexpr int kHfOff = L::kHfOff, kTokOff = L::kTokOff, kRawOff = L::kRawOff, kBarOff = L::kBarOff;
    constexpr int kMiscOff = L::kMiscOff, kTileOffOff = L::kTileOffOff, kCountsOff = L::kCountsOff;
    constexpr int kTabOff = L::kTabOff;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = smem_u32(smem_raw);
    const uint32_t base = (raw_base + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (base - raw_base);
    const uint32_t bars = base + kBarOff;
    auto raw_full = [&](int i) { return bars + 8u * i; };
    auto raw_empty = [&](int i) { return bars + 8u * (kRawStages + i); };
    auto hf_full = [&](int i) { return bars + 8u * (2 * kRawStages + i); };
    auto hf_empty = [&](int i) { return bars + 8u * (2 * kRawStages + kHfStages + i); };
    constexpr int kTokBar = 2 * (kRawStages + kHfStages);
    auto tok_full = [&](int i) { return bars + 8u * (kTokBar + i); };
    auto tok_empty = [&](int i) { return bars + 8u * (kTokBar + kTokStages + i); };
    const uint32_t acc_full = bars + 8u * (kTokBar + 2 * kTokStages);
    const uint32_t acc_empty = acc_full + 8u;
    const uint32_t drain_bar = acc_full + 16u;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + kMiscOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kMiscOff + 4);
    volatile int* job_word = reinterpret_cast<volatile int*>(smem + kMiscOff + 8);  // fused: the epilogue leader's decision
    int* tile_off = reinterpret_cast<int*>(smem + kTileOffOff);
    int* counts = reinterpret_cast<int*>(smem + kCountsOff);

    const Plan& p = args.p;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i <= p.E; i += kThreads) tile_off[i] = p.tile_off[i];
    for (int i = threadIdx.x; i < p.E; i += kThreads) counts[i] = p.counts[i];
    if (threadIdx.x == 0) {
        for (int i = 0; i < kRawStages; ++i) {
            mbar_init(raw_full(i), 1);
            mbar_init(raw_empty(i), 128);
        }
        for (int i = 0; i < kHfStages; ++i) {
            mbar_init(hf_full(i), kPrep ? 1 : 128);  // the weight TMA (arrive + bytes), or the 128 converter threads
            mbar_init(hf_empty(i), 1);
        }
        for (int i = 0; i < kTokStages; ++i) {
            mbar_init(tok_full(i), 1);   // the token TMA (arrive + bytes)
            mbar_init(tok_empty(i), 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, 4);
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_holder), 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    // tiles [0, total1) are the launch's first stage (L1 when fused), [total1, total) the L2 ones;
    // every L1 tile precedes every L2 tile in the round-robin order
    const int n_route = tile_off[p.E];
    const int total1 = n_route * args.n_slabs;
    const int total = kFused ? total1 + n_route * args.n_slabs2 : total1;
    const int I = p.I, H = p.H;
    auto is_l1 = [&](int t) { return kKind == kL1 || (kFused && t < total1); };
    auto second = [&](int t) { return kFused && t >= total1; };  // an L2 tile of the fused launch
    auto tile_of = [&](int t) {
        return second(t) ? decode(t - total1, tile_off, p.E, args.n_slabs2) : decode(t, tile_off, p.E, args.n_slabs);
    };
    auto kb_of = [&](int t) { return second(t) ? args.k_blocks2 : args.k_blocks; };
    auto wrow = [&](const Tile& tl, int blk, bool l1) {
        if (l1) return tl.e * 2 * I + (blk ? I : 0) + tl.s * kWR;
        return tl.e * H + tl.s * 2 * kWR + blk * kWR;
    };
    // fused launch: per route tile the count of its finished L1 tiles, then of its finished
    // re-quantisation jobs (an L2 tile waits for dep_target); then the job queue
    const int route_tiles = (int)(p.pool_rows / kTok);
    const QuantQueue qq{args.ctr, args.ctr + route_tiles, args.ctr + route_tiles + 1, args.ctr + route_tiles + 2,
                        args.ctr + route_tiles + 3, kQuantJobs * n_route};
    const int dep_target = args.n_slabs + kQuantJobs;

    if (warp == 0) {
        if constexpr (kPrep) {
            if (lane == 0) {
                // ---------------- f16 weight TMA straight into the MMA's ring ----------------
                int it = 0;
                bool ok = true;
                for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                    const Tile tl = tile_of(t);
                    const bool l1 = is_l1(t);
                    const int w0 = wrow(tl, 0, l1), w1 = wrow(tl, 1, l1), KB = kb_of(t);
                    const CUtensorMap* mW = second(t) ? &tmW2 : &tmW;
                    for (int kb = 0; kb < KB; ++kb, ++it) {
                        const int b = it % kHfStages;
                        if (!mbar_wait(hf_empty(b), ((uint32_t)(it / kHfStages) & 1u) ^ 1u, p.hdr, abort_flag)) {
                            ok = false;
                            break;
                        }
                        const uint32_t dst = base + kHfOff + b * kABytes;
                        mbar_arrive_expect_tx(hf_full(b), kABytes);
                        tma_load_2d(dst, mW, kb * kBK, w0, hf_full(b));
                        tma_load_2d(dst + kWR * 128, mW, kb * kBK, w1, hf_full(b));
                    }
                }
                for (int j = it - kHfStages < 0 ? 0 : it - kHfStages; j < it; ++j)
                    mbar_drain(hf_full(j % kHfStages), (uint32_t)(j / kHfStages) & 1u, p.hdr);
            }
        } else if (lane == 0) {
            // ---------------- raw weight TMA ----------------
            int it = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const Tile tl = tile_of(t);
                const bool l1 = is_l1(t);
                const int w0 = wrow(tl, 0, l1), w1 = wrow(tl, 1, l1), KB = kb_of(t);
                const CUtensorMap* mW = second(t) ? &tmW2 : &tmW;
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    const int r = it % kRawStages;
                    if (!mbar_wait(raw_empty(r), ((uint32_t)(it / kRawStages) & 1u) ^ 1u, p.hdr, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t dst = base + kRawOff + r * kRawBytes;
                    mbar_arrive_expect_tx(raw_full(r), kRawBytes);
                    tma_load_2d(dst, mW, kb * kBK, w0, raw_full(r));
                    tma_load_2d(dst + kWR * kBK, mW, kb * kBK, w1, raw_full(r));
                }
            }
            for (int j = it - kRawStages < 0 ? 0 : it - kRawStages; j < it; ++j)
                mbar_drain(raw_full(j % kRawStages), (uint32_t)(j / kRawStages) & 1u, p.hdr);
        }
    } else if (warp == 10) {
        // ---------------- token TMA: hi plane rows, then lo plane rows ----------------
        if (lane == 0) {
            int it = 0;
            bool ok = true, all_q = false;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const Tile tl = tile_of(t);
                const int KB = kb_of(t);
                const CUtensorMap* mX = second(t) ? &tmX2 : &tmX;
                const CUtensorMap* mX16 = second(t) ? &tmX16_2 : &tmX16;
                if (second(t) && !all_q) {
                    // the route tile's rows are re-quantised (bounded wait); once every job of the
                    // launch is finished, no later L2 tile needs a check
                    all_q = ld_acquire_gpu(qq.jobs_done) >= qq.n_jobs;
                    if (!all_q && !wait_count(qq.dep + tile_off[tl.e] + tl.m, dep_target, p.hdr, abort_flag))
                        break;
                    // the planes were written through the generic proxy; the TMA reads them
                    asm volatile("fence.proxy.async.global;" ::: "memory");
                }
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    const int b = it % kTokStages;
                    if (!mbar_wait(tok_empty(b), ((uint32_t)(it / kTokStages) & 1u) ^ 1u, p.hdr, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t dst = base + kTokOff + b * kTokBytes;
                    const int n16 = tile_n16(counts, tl.e, tl.m);
                    mbar_arrive_expect_tx(tok_full(b), (uint32_t)(2 * n16 * 128));
                    if (n16 == kTok) {
                        // one copy per plane: each TMA instruction costs the issuing thread ~75 cycles
                        for (int pl = 0; pl < 2; ++pl)
                            tma_load_2d(dst + pl * kTok * 128, mX, kb * kBK, (int)(pl * p.pool_rows) + tl.row0,
                                        tok_full(b));
                    } else {
                        // hi rows [0, n16), lo rows [n16, 2 n16): one contiguous B operand of N = 2 n16
                        for (int pl = 0; pl < 2; ++pl)
                            for (int j = 0; j < n16; j += kTokBox)
                                tma_load_2d(dst + (pl * n16 + j) * 128, mX16, kb * kBK,
                                            (int)(pl * p.pool_rows) + tl.row0 + j, tok_full(b));
                    }
                }
            }
            for (int j = it - kTokStages < 0 ? 0 : it - kTokStages; j < it; ++j)
                mbar_drain(tok_full(j % kTokStages), (uint32_t)(j / kTokStages) & 1u, p.hdr);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        // This thread feeds the tensor pipe, so its per-stage work is kept short: a non-blocking
        // test of each barrier before the bounded wait, ring positions kept as counters, and
        // descriptors advanced by adding to their address field (start >> 4: +2 per 16 K of a
        // K-major tile, + the stage's offset >> 4).
        if (lane == 0) {
            const uint64_t ad0 = kmajor_desc(base + kHfOff, 0), bd0 = kmajor_desc(base + kTokOff, 0);
            int b = 0, tb = 0, tc = 0;
            uint32_t hph = 0, tph = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++tc) {
                if (!mbar_wait(acc_empty, ((uint32_t)tc & 1u) ^ 1u, p.hdr, abort_flag)) break;
                tc_fence_after();
                const Tile tl = tile_of(t);
                const uint32_t idesc = idesc_n(2 * tile_n16(counts, tl.e, tl.m));
                const int KB = kb_of(t);
                for (int kb = 0; kb < KB; ++kb) {
                    if (!(mbar_test(hf_full(b), hph) || mbar_wait(hf_full(b), hph, p.hdr, abort_flag)) ||
                        !(mbar_test(tok_full(tb), tph) || mbar_wait(tok_full(tb), tph, p.hdr, abort_flag))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = ad0 + (uint64_t)((b * kABytes) >> 4);
                    const uint64_t bd = bd0 + (uint64_t)((tb * kTokBytes) >> 4);
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk) {
                        tc_mma(tmem_base, ad + 2 * kk, bd + 2 * kk, idesc, (kb | kk) != 0);
                        tc_mma(tmem_base + 256, ad + ((kWR * 128) >> 4) + 2 * kk, bd + 2 * kk, idesc, (kb | kk) != 0);
                    }
                    tc_commit(hf_empty(b));
                    tc_commit(tok_empty(tb));
                    if (++b == kHfStages) b = 0, hph ^= 1u;
                    if (++tb == kTokStages) tb = 0, tph ^= 1u;
                }
                if (ok) tc_commit(acc_full);
            }
            tc_commit(drain_bar);
            mbar_drain(drain_bar, 0, p.hdr);
        }
    } else if (warp >= 6) {
        if constexpr (!kPrep) {
            // ---------------- weight converters ----------------
            const int c = threadIdx.x - 192;  // row of each 128-row weight block
            int it = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const int KB = kb_of(t);
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    const int r = it % kRawStages, b = it % kHfStages;
                    bool w_ok = mbar_wait(raw_full(r), (uint32_t)(it / kRawStages) & 1u, p.hdr, abort_flag);
                    w_ok = w_ok && mbar_wait(hf_empty(b), ((uint32_t)(it / kHfStages) & 1u) ^ 1u, p.hdr, abort_flag);
                    if (!__all_sync(0xffffffffu, w_ok)) {
                        ok = false;
                        break;
                    }
                    const uint8_t* rw = smem + kRawOff + r * kRawBytes;
                    uint8_t* dst = smem + kHfOff + b * kABytes;
                    uint4 r0[4], r1[4];
                    load_row(rw, c, r0);
                    load_row(rw + kWR * kBK, c, r1);
                    store_row(r0, dst, c);
                    store_row(r1, dst + kWR * 128, c);
                    fence_proxy_async_smem();
                    mbar_arrive(raw_empty(r));
                    mbar_arrive(hf_full(b));
                }
            }
        }
    } else if (warp >= 2 && warp < 6) {
        // ---------------- epilogue (warps 2..5) ----------------
        // The per-row values (token scales, L2 slots and gate weights) and the per-channel weight
        // scales are read before the accumulator wait, while the tile's MMAs still run: the
        // accumulator is single-buffered, so the epilogue adds directly to the tile time.
        const int q = warp & 3;
        int* w_src = reinterpret_cast<int*>(smem + kTabOff) + q * 3 * kTok;
        float* w_g = reinterpret_cast<float*>(w_src + kTok);
        float* w_sa = w_g + kTok;
        int tc = 0;
        const bool leader = q == 0 && lane == 0;
        bool all_q = false;  // (the leader's) fused launch: every job of the launch seen finished
        bool drained = false;  // (the leader's) fused launch: every job of the launch taken
        for (int t = blockIdx.x; t < total; t += gridDim.x, ++tc) {
            const Tile tl = tile_of(t);
            const bool l1 = is_l1(t);
            const int n_valid = min(kTok, counts[tl.e] - tl.m * kTok);
            const int n16 = min(kTok, (n_valid + 15) & ~15);  // lo plane columns start here
            float sx_l[kTok / 32];
            float sg = 0.0f, su = 0.0f, s2[2] = {0.0f, 0.0f};
            bool dep_ok = true;
            if (second(t)) {
                // s^A of the route tile's rows comes from its re-quantisation in this launch (jobs
                // run meanwhile); the loads below follow the leader's acquire through the barrier
                const int32_t* dep = qq.dep + tile_off[tl.e] + tl.m;
                dep_ok = idle_with_jobs<kEpiBar, kQuantRegVec, false>(qq, p, job_word, abort_flag, &drained, q, lane, [&] {
                    if (!all_q) all_q = ld_acquire_gpu(qq.jobs_done) >= qq.n_jobs;
                    return all_q || ld_acquire_gpu(dep) >= dep_target;
                });
            }
            if (l1) {
                const int j = tl.s * kWR + q * 32 + lane;
                const float* s1 = args.w_scale + (int64_t)tl.e * 2 * I;
                sg = __ldg(s1 + j);
                su = __ldg(s1 + I + j);
#pragma unroll
                for (int ci = 0; ci < kTok / 32; ++ci)
                    sx_l[ci] = __ldg(reinterpret_cast<const float*>(p.x_pool_scale) + tl.row0 + 32 * ci + lane);
            } else {
                const float* ws2 = second(t) ? args.w_scale2 : args.w_scale;
#pragma unroll
                for (int blk = 0; blk < 2; ++blk)
                    s2[blk] = __ldg(ws2 + (int64_t)tl.e * H + tl.s * 2 * kWR + blk * kWR + q * 32 + lane);
                int src[kTok / 32];
#pragma unroll
                for (int ci = 0; ci < kTok / 32; ++ci) {
                    const int n = 32 * ci + lane;
                    src[ci] = n < n_valid ? debug_row(p.hdr, __ldg(p.pool_src + tl.row0 + n), (int64_t)p.T * p.K) : -1;
                    const float* sa = reinterpret_cast<const float*>(p.a_pool_scale) + tl.row0 + n;
                    sx_l[ci] = second(t) ? __uint_as_float(ld_relaxed_gpu(sa)) : __ldg(sa);
                }
#pragma unroll
                for (int ci = 0; ci < kTok / 32; ++ci) {
                    const float g = src[ci] >= 0 ? __ldg(args.topk_weights + src[ci]) : 0.0f;
                    w_src[32 * ci + lane] = src[ci];
                    w_g[32 * ci + lane] = g;
                    w_sa[32 * ci + lane] = sx_l[ci];
                }
                __syncwarp();
            }
            if (kFused && dep_ok)  // a re-quantisation job while this tile's MMAs run, if there is one
                dep_ok = idle_with_jobs<kEpiBar, kQuantRegVec, true>(qq, p, job_word, abort_flag, &drained, q, lane,
                                                                     [&] { return mbar_test(acc_full, (uint32_t)tc & 1u); });
            const bool w_ok = dep_ok && mbar_wait(acc_full, (uint32_t)tc & 1u, p.hdr, abort_flag);
            if (!bar_all128<kEpiBar>(w_ok)) break;  // one decision for the four warps (they share kEpiBar)
            tc_fence_after();
            const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16);
            if (l1) {
                // C = 16 D_hi + D_lo; H = (C * s^W1) * s^X; A = SiLU(H_gate) * H_up for the tile's
                // 32-token chunks up to n16 (the padding rows' values are never read back as results)
                const int j = tl.s * kWR + q * 32 + lane;
#pragma unroll
                for (int ci = 0; ci < kTok / 32; ++ci) {
                    const int c0 = 32 * ci;
                    if (c0 >= n16) break;  // uniform across the warp
                    uint32_t hi[32], lo[32];
                    float hg[32];
                    tmem_ld32(tb + c0, hi);
                    tmem_ld32(tb + n16 + c0, lo);
                    tmem_ld_wait();
#pragma unroll
                    for (int tt = 0; tt < 32; ++tt) hg[tt] = __int2float_rn(exact_int(hi[tt], lo[tt]));
                    tmem_ld32(tb + 256 + c0, hi);
                    tmem_ld32(tb + 256 + n16 + c0, lo);
                    tmem_ld_wait();
#pragma unroll
                    for (int tt = 0; tt < 32; ++tt) {
                        const float sx = __shfl_sync(0xffffffffu, sx_l[ci], tt);
                        const float Hg = __fmul_rn(__fmul_rn(hg[tt], sg), sx);
                        const float Hu = __fmul_rn(__fmul_rn(__int2float_rn(exact_int(hi[tt], lo[tt])), su), sx);
                        p.a_f32[(int64_t)(tl.row0 + c0 + tt) * I + j] = swiglu1(Hg, Hu, p.act_clamp);
                    }
                }
            } else {
                // D = 16 D_hi + D_lo; Y = (D * s^W2) * s^A; c = bf16(G * Y) to the combine row.
                // Branch-free: the slot, gate and s^A of token tt are broadcast reads of the table.
#pragma unroll
                for (int ci = 0; ci < kTok / 32; ++ci) {
                    const int c0 = 32 * ci;
                    if (c0 >= n_valid) break;  // uniform across the warp
#pragma unroll
                    for (int blk = 0; blk < 2; ++blk) {
                        const int h = tl.s * 2 * kWR + blk * kWR + q * 32 + lane;
                        uint32_t hi[32], lo[32];
                        tmem_ld32(tb + blk * 256 + c0, hi);
                        tmem_ld32(tb + blk * 256 + n16 + c0, lo);
                        tmem_ld_wait();
#pragma unroll
                        for (int tt = 0; tt < 32; ++tt) {  // slot < 0 past the routed rows
                            const int src = w_src[c0 + tt];
                            const float y = __fmul_rn(__fmul_rn(__int2float_rn(exact_int(hi[tt], lo[tt])), s2[blk]), w_sa[c0 + tt]);
                            st_global_u16_if(src >= 0, p.comb + (int64_t)src * H + h, float_to_bf16_bits(__fmul_rn(w_g[c0 + tt], y)));
                        }
                    }
                }
                __syncwarp();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty);
            if (kFused && l1) {
                // The accumulator is free for the next tile. Publish this tile's rows of A: every
                // thread fences its own stores, the four warps meet, the leader counts the tile for
                // its route tile; the route tile's last L1 tile queues its re-quantisation jobs
                // (whole rows of A are needed), which any CTA's epilogue then runs.
                const int g = tile_off[tl.e] + tl.m;
                __threadfence();
                bar_sync128<kEpiBar>();
                if (leader) {
                    __threadfence();
                    if (atomicAdd(qq.dep + g, 1) == args.n_slabs - 1) {
                        __threadfence();
                        qq.push(g);
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, 512);
}

template <int kKind, bool kPrep>
cudaError_t set_int8_smem_attr() {
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(tc_int8_kernel<kKind, kPrep>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)Layout<kPrep>::kSmem);
    });
    return attr_err;
}

// Weights of one stage (int8 bytes in 64-byte-swizzled boxes of 128 rows x 64 K, or prepared f16
// codes in 128-byte-swizzled ones) and its token operand: the f16 planes (x for L1, A for L2) in
// 128-row boxes and 16-row boxes for a route tile's ragged end.
template <bool kPrep>
bool make_int8_maps(const Plan& p, const void* w, bool l1, CUtensorMap* tmW, CUtensorMap* tmX, CUtensorMap* tmX16) {
    const int n_out = l1 ? 2 * p.I : p.H;
    const int kin = l1 ? p.H : p.I;
    const bool w_ok = kPrep ? tc_make_map_2d(tmW, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, w, (uint64_t)kin,
                                             (uint64_t)p.E * n_out, kBK, kWR, CU_TENSOR_MAP_SWIZZLE_128B)
                            : tc_make_map_2d(tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, w, (uint64_t)kin,
                                             (uint64_t)p.E * n_out, kBK, kWR, CU_TENSOR_MAP_SWIZZLE_64B);
    const void* planes = l1 ? (const void*)p.x_planes : (const void*)p.a_planes;
    return w_ok &&
           tc_make_map_2d(tmX, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, planes, (uint64_t)kin, 2 * (uint64_t)p.pool_rows, kBK,
                          kTok, CU_TENSOR_MAP_SWIZZLE_128B) &&
           tc_make_map_2d(tmX16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, planes, (uint64_t)kin, 2 * (uint64_t)p.pool_rows,
                          kBK, kTokBox, CU_TENSOR_MAP_SWIZZLE_128B);
}

template <bool kIsL1, bool kPrep>
cudaError_t launch_int8(const Plan& p, const void* w, const void* w_scale, const float* topk_weights, cudaStream_t s) {
    using L = Layout<kPrep>;
    constexpr int kKind = kIsL1 ? kL1 : kL2;
    const cudaError_t attr_err = set_int8_smem_attr<kKind, kPrep>();
    if (attr_err != cudaSuccess) return attr_err;
    CUtensorMap tmW, tmX, tmX16;
    if (!make_int8_maps<kPrep>(p, w, kIsL1, &tmW, &tmX, &tmX16)) return cudaErrorInvalidValue;
    I8Args args{};
    args.p = p;
    args.w_scale = static_cast<const float*>(w_scale);
    args.topk_weights = topk_weights;
    args.n_slabs = kIsL1 ? p.I / kWR : p.H / (2 * kWR);
    args.k_blocks = (kIsL1 ? p.H : p.I) / kBK;
    args.n_out = kIsL1 ? 2 * p.I : p.H;
    const int64_t max_tiles = (p.pool_rows / kTok) * args.n_slabs;
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(max_tiles, tc_num_sms()));
    tc_int8_kernel<kKind, kPrep><<<grid, kThreads, L::kSmem, s>>>(tmW, tmX, tmX16, tmW, tmX, tmX16, args);
    return cudaGetLastError();
}

// L1 then L2 in one cooperative launch: every CTA is resident, so an L2 tile waits (bounded) only
// on L1 tiles and re-quantisations that earlier positions of the same round-robin order hold
template <bool kPrep>
cudaError_t launch_int8_fused(const Plan& p, const void* w1, const void* w1_scale, const void* w2,
                              const void* w2_scale, const float* topk_weights, cudaStream_t s) {
    using L = Layout<kPrep>;
    cudaError_t e = set_int8_smem_attr<kFusedL1L2, kPrep>();
    if (e != cudaSuccess) return e;
    CUtensorMap tmW1, tmX1, tmX16_1, tmW2, tmX2, tmX16_2;
    if (!make_int8_maps<kPrep>(p, w1, true, &tmW1, &tmX1, &tmX16_1) ||
        !make_int8_maps<kPrep>(p, w2, false, &tmW2, &tmX2, &tmX16_2))
        return cudaErrorInvalidValue;
    const int64_t route_tiles = p.pool_rows / kTok;
    // the counters (one per route tile, then the job queue's) start at zero every launch
    if ((e = cudaMemsetAsync(p.ffn_counters, 0, sizeof(int32_t) * (size_t)fused_int_counters(route_tiles), s)) !=
        cudaSuccess)
        return e;
    I8Args args{};
    args.p = p;
    args.w_scale = static_cast<const float*>(w1_scale);
    args.topk_weights = topk_weights;
    args.n_slabs = p.I / kWR;
    args.k_blocks = p.H / kBK;
    args.n_out = 2 * p.I;
    args.w_scale2 = static_cast<const float*>(w2_scale);
    args.n_slabs2 = p.H / (2 * kWR);
    args.k_blocks2 = p.I / kBK;
    args.ctr = p.ffn_counters;
    int per_sm = 0;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, tc_int8_kernel<kFusedL1L2, kPrep>, kThreads,
                                                           L::kSmem)) != cudaSuccess)
        return e;
    if (per_sm < 1) return cudaErrorCooperativeLaunchTooLarge;
    const int64_t max_tiles = route_tiles * (args.n_slabs + args.n_slabs2);
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(max_tiles, (int64_t)tc_num_sms() * per_sm));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = L::kSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, tc_int8_kernel<kFusedL1L2, kPrep>, tmW1, tmX1, tmX16_1, tmW2, tmX2, tmX16_2, args);
}

// One-time preparation of int8 weights for the f16 tensor-core GEMM: every code q becomes the f16
// value q (exact), 16 codes per thread and step.
__global__ void prepare_int8_kernel(const uint4* __restrict__ w, uint4* __restrict__ out, int64_t n16) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n16; i += (int64_t)gridDim.x * blockDim.x) {
        const uint4 c = __ldg(w + i);
        uint32_t o[8];
        int8x4_to_f16(c.x, o[0], o[1]);
        int8x4_to_f16(c.y, o[2], o[3]);
        int8x4_to_f16(c.z, o[4], o[5]);
        int8x4_to_f16(c.w, o[6], o[7]);
        out[2 * i] = make_uint4(o[0], o[1], o[2], o[3]);
        out[2 * i + 1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
}

}  // namespace

bool int8_tc_supported(const Plan& p, int stage) {
    if (p.mode != MOE_A8W8_INT8 || p.E > kMaxExperts || !tc_encode_available()) return false;
    if (stage == 1) return p.I % kWR == 0 && p.H % kBK == 0 && p.H <= kMaxK;
    return p.H % (2 * kWR) == 0 && p.I % kBK == 0 && p.I <= kMaxK;
}

cudaError_t launch_l1_int8_tc(const Plan& p, const void* w1, const void* w1_scale, bool prepared, cudaStream_t s) {
    return prepared ? launch_int8<true, true>(p, w1, w1_scale, nullptr, s)
                    : launch_int8<true, false>(p, w1, w1_scale, nullptr, s);
}

cudaError_t launch_l2_int8_tc(const Plan& p, const void* w2, const void* w2_scale, const float* topk_weights,
                              bool prepared, cudaStream_t s) {
    return prepared ? launch_int8<false, true>(p, w2, w2_scale, topk_weights, s)
                    : launch_int8<false, false>(p, w2, w2_scale, topk_weights, s);
}

cudaError_t launch_ffn_fused_int8(const Plan& p, const void* w1, const void* w1_scale, const void* w2,
                                  const void* w2_scale, const float* topk_weights, bool prepared, cudaStream_t s) {
    return prepared ? launch_int8_fused<true>(p, w1, w1_scale, w2, w2_scale, topk_weights, s)
                    : launch_int8_fused<false>(p, w1, w1_scale, w2, w2_scale, topk_weights, s);
}

cudaError_t launch_prepare_int8(const void* w, void* out, int64_t n, cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    const int64_t n16 = n / 16;  // the caller guarantees n % 16 == 0 (K is a multiple of 128)
    const int grid = (int)std::min<int64_t>((n16 + 255) / 256, (int64_t)tc_num_sms() * 8);
    prepare_int8_kernel<<<grid, 256, 0, s>>>(static_cast<const uint4*>(w), static_cast<uint4*>(out), n16);
    return cudaGetLastError();
}

}  // namespace moe
