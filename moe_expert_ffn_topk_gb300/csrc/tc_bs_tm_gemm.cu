// Token-major block-scaled grouped GEMM for the FP8 modes at prefill sizes (A8W8-FP8: e4m3
// weights, A8W4: e2m1 weights; e4m3 tokens), on tcgen05.mma kind::mxf8f6f4.block_scale with
// one UE8M0 scale per 32 elements of K applied by the tensor core (the Ascend mega_moe page,
// A8W8-FP use case: the MX dequantisation happens within the matrix multiply; DeepGEMM page,
// section 4, step 5: block-scaled MMA with UE8M0 scale factors in tensor memory).
//
// Tile: M = 128 pool rows (one 128-row route tile of an expert) x N weight rows, K = 128 per
// stage (MMAs of K = 32):
// - L1: the 128 gate rows and the 128 up rows of outputs [128s, 128s + 128) (one 4-D TMA box),
//   so a thread of the epilogue holds its token's gate and up values of the same outputs and
//   applies SwiGLU (Ascend page, "SwiGLU Activation") and the MX FP8 re-quantisation of A (one
//   exponent per 32 outputs) without any exchange between threads;
// - L2: N = 224 hidden columns when H is a multiple of 224 (else 256); the epilogue scales the
//   token's row by G and writes its bf16 combine row (Ascend page, "Token Combine").
// Why this shape: these GEMMs are bound by how fast TMA fills shared memory (about 55-68 bytes
// per clock per SM measured on this GPU with 192 KB in flight). Per 128-K stage a tile takes
// 16 KB of tokens and 32 KB of weights (e2m1 occupies a byte per code in the MMA's 4-bit
// layout) for 128 x 256 x 128 MACs: 24 KB per 128^3, where 128 weight rows x 128 tokens take
// 32 KB. With N = 256 the accumulator is single-buffered (two 256-column accumulators fill the
// 512 TMEM columns and leave none for the scale factors): eight epilogue warps, two per lane
// quarter, each drain half of its columns and release it as soon as they are in registers.
// N = 224 (L2) fits two accumulators and the scale ring (2 * 224 + 64 = 512 columns), so the
// epilogue of a tile overlaps the main loop of the next.
//
// TMEM: accumulator(s) from column 0; scale factors in a ring of 16-column slots after them, one
// per stage. Layout the MMA reads (measured on this GPU, M = 128): the scale word of A
// row r (a token) in lane r, column slot + r/32; the scale word of B row n (a weight row) in
// lane 32*q + n%32 of every lane quarter q, column slot + 4 + n/32; byte k of a word is the
// scale of K group k of the stage.
//
// Scale words (4 UE8M0 bytes per row and 128-element K atom; fp32 per atom for the FP8xFP4
// tokens) come by TMA too, in blocks of 4 atoms (16 bytes of every row) two blocks ahead of their
// use, into a 4-deep ring: scattered 4-byte loads of them by the scale warps slowed the operand
// TMA down by a quarter (measured). The scale warps only move them from shared to tensor memory.
//
// Warp roles (448 threads): 0 TMA producer, 1 TMEM allocation + MMA issuer, 2-5 and 10-13
// epilogue (warp w owns TMEM lanes 32*(w%4) .. +31, i.e. those token rows; warps 2-5 take the
// first half of the columns, 10-13 the second), 6-9 scale writers. Every wait is bounded; on
// time-out the CTA records MOE_ERR_TIMEOUT, drains and exits.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "tc_common.cuh"

namespace moe {

namespace {

using namespace tc;

constexpr int kTM = 128;          // token rows per tile (MMA M)
constexpr int kAtomK = 128;       // K per stage: one 128-byte swizzle atom of e4m3 / expanded e2m1
constexpr int kStages = 4;
constexpr int kThreads = 448;
constexpr int kMaxExperts = 1024;
constexpr int kTokBytes = kTM * 128;   // 16 KB
constexpr int kSfColsPerStage = 16;    // SFA 4 columns, SFB N/32 columns
constexpr int kSfBlk = 4;              // K atoms per scale block (16 bytes of a row)
constexpr int kSfBufs = 4;             // scale ring depth: blocks issued two ahead of their use
constexpr int kSfTBytes = kTM * 16;    // token scale words of a block: [128 rows][4 atoms]

template <int kWN>  // weight rows per tile (MMA N): 256, or 224 with two accumulators
struct TmCfg {
    static constexpr int kAccs = 2 * kWN + kStages * kSfColsPerStage <= 512 ? 2 : 1;
    static constexpr int kSfCol0 = kAccs * kWN;
    static constexpr int kWBytes = kWN * 128;  // in shared memory
    static constexpr int kStageBytes = kTokBytes + kWBytes;
    static constexpr int kSfWBytes = kWN * 16;  // weight scale words of a block: [N rows][4 atoms]
    static constexpr int kSfOff = kStages * kStageBytes;
    static constexpr int kBarOff = kSfOff + kSfBufs * (kSfWBytes + kSfTBytes);
    // full, empty, acc full/empty x2, drain, scale full/empty
    static constexpr int kNumBars = 2 * kStages + 4 + 1 + 2 * kSfBufs;
    static constexpr int kMiscOff = kBarOff + 8 * kNumBars;
    static constexpr int kTileOffOff = kMiscOff + 16;
    static constexpr int kCountsOff = kTileOffOff + 4 * (kMaxExperts + 1);
    static constexpr size_t kSmem = 1024 + (size_t)kCountsOff + 4 * kMaxExperts;
    static_assert(kSmem <= 232448, "shared memory");
    static_assert(kSfCol0 + kStages * kSfColsPerStage <= 512, "tensor memory");
    static_assert(kWN % 32 == 0 && kWN <= 256 && 4 + kWN / 32 <= kSfColsPerStage, "tile");
};

struct TmArgs {
    Plan p;
    const uint8_t* w_scale;     // UE8M0 [E*n_out][kin/32]
    const float* topk_weights;  // L2
    int n_slabs, k_blocks, n_out, kin;
};

struct Tile {
    int e, s, m, row0, n_valid;
};

// Tiles are ordered expert-major, then weight slab, then route tile, so the CTAs in flight
// share one expert's slabs in L2 while its token rows stay resident.
__device__ __forceinline__ Tile decode_tile(int t, const int* tile_off, const int* counts, int E, int n_slabs) {
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
    tl.row0 = (tile_off[lo] + tl.m) * kTM;
    tl.n_valid = min(kTM, counts[lo] - tl.m * kTM);
    return tl;
}

// kind::mxf8f6f4.block_scale instruction descriptor: B scale id (bits 4-5), A type (7-9: the
// tokens, e4m3 = 0, e5m2 = 1), B type (10-12: e4m3 = 0, e5m2 = 1, e2m1 = 5), both K-major,
// N >> 3 (17-22), UE8M0 scales (bit 23), M >> 4 (24-28), A scale id (29-30).
__device__ __forceinline__ uint32_t tm_idesc(uint32_t afmt, uint32_t bfmt, int n, int sf_id) {
    return ((uint32_t)sf_id << 4) | (afmt << 7) | (bfmt << 10) | ((uint32_t)(n >> 3) << 17) | (1u << 23) |
           ((uint32_t)(kTM >> 4) << 24) | ((uint32_t)sf_id << 29);
}

__device__ __forceinline__ void tm_mma(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t sfa,
                                       uint32_t sfb, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
        ::"r"(d), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
        : "memory");
}

// 16 consecutive columns of the warp's 32 lanes, one 32-bit word per lane and column
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
        "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}

// two floats -> two e4m3 (or e5m2) codes (RN, saturating), the first in the low byte
template <bool kE5>
__device__ __forceinline__ uint32_t fp8x2(float lo, float hi) {
    uint16_t pair;
    if constexpr (kE5) asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(pair) : "f"(hi), "f"(lo));
    else asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(pair) : "f"(hi), "f"(lo));
    return pair;
}

template <int MODE, bool kL1, int kWN>
__global__ void __launch_bounds__(kThreads, 1)
    tc_bs_tm_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                    const __grid_constant__ CUtensorMap tmSW, const __grid_constant__ CUtensorMap tmSX, TmArgs args) {
    using Cfg = TmCfg<kWN>;
    constexpr bool kFp4 = MODE == MOE_A8W4_FP8_FP4;
    constexpr bool kE5 = MODE == MOE_A8W8_FP8_E5M2;  // e5m2 tokens, weights and A
    constexpr uint32_t kAfmt = kE5 ? 1u : 0u;
    constexpr uint32_t kBfmt = kFp4 ? 5u : kAfmt;
    constexpr uint32_t kWTx = kFp4 ? kWN * kAtomK / 2 : kWN * kAtomK;  // TMA counts the packed global bytes
    constexpr int kStageBytes = Cfg::kStageBytes, kSfOff = Cfg::kSfOff, kSfWBytes = Cfg::kSfWBytes;
    constexpr int kSfCol0 = Cfg::kSfCol0, kAccs = Cfg::kAccs;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = smem_u32(smem_raw);
    const uint32_t base = (raw_base + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (base - raw_base);
    const uint32_t bars = base + Cfg::kBarOff;
    auto full_bar = [&](int s) { return bars + 8u * s; };
    auto empty_bar = [&](int s) { return bars + 8u * (kStages + s); };
    auto acc_full = [&](int a) { return bars + 8u * (2 * kStages + a); };
    auto acc_empty = [&](int a) { return bars + 8u * (2 * kStages + 2 + a); };
    const uint32_t drain_bar = bars + 8u * (2 * kStages + 4);
    auto sf_full = [&](int b) { return bars + 8u * (2 * kStages + 5 + b); };
    auto sf_empty = [&](int b) { return bars + 8u * (2 * kStages + 5 + kSfBufs + b); };
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + Cfg::kMiscOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::kMiscOff + 4);
    int* tile_off = reinterpret_cast<int*>(smem + Cfg::kTileOffOff);
    int* counts = reinterpret_cast<int*>(smem + Cfg::kCountsOff);

    const Plan& p = args.p;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i <= p.E; i += kThreads) tile_off[i] = p.tile_off[i];
    for (int i = threadIdx.x; i < p.E; i += kThreads) counts[i] = p.counts[i];
    if (threadIdx.x == 32) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full_bar(s), 1 + 4);  // TMA (arrive + bytes) + the 4 scale-writer warps
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(acc_full(a), 1);
            mbar_init(acc_empty(a), 8);  // the 8 epilogue warps
        }
        mbar_init(drain_bar, 1);
        for (int b = 0; b < kSfBufs; ++b) {
            mbar_init(sf_full(b), 1);   // the producer (arrive + bytes)
            mbar_init(sf_empty(b), 4);  // the 4 scale-writer warps
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0 && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmW)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmX)) : "memory");
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_holder), 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    const int total = tile_off[p.E] * args.n_slabs;
    const int KB = args.k_blocks;
    const int I = p.I, H = p.H;
    auto tile_of = [&](int t) { return decode_tile(t, tile_off, counts, p.E, args.n_slabs); };
    // global weight row of row n (0..255) of the tile's B operand
    auto wrow = [&](const Tile& tl, int n) {
        if (kL1) return tl.e * args.n_out + (n >= 128 ? I : 0) + tl.s * 128 + (n & 127);
        return tl.e * args.n_out + tl.s * kWN + n;
    };

    if (warp == 0) {
        // ---------------- TMA producer: 128 token rows, 256 weight rows per stage ----------------
        if (lane == 0) {
            const int n_sfb = (KB + kSfBlk - 1) / kSfBlk;  // scale blocks per tile
            // scale blocks in the order they are used: (tile, block), counted by sj
            int st_t = blockIdx.x, st_b = 0, sj = 0;
            Tile st_tl = tile_of(st_t < total ? st_t : 0);  // decoded once per tile
            bool ok = true;
            auto issue_scales = [&]() {  // the next scale block, if any
                if (st_t >= total || !ok) return;
                const int buf = sj % kSfBufs;
                if (!mbar_wait(sf_empty(buf), ((uint32_t)(sj / kSfBufs) & 1u) ^ 1u, p.hdr, abort_flag)) {
                    ok = false;
                    return;
                }
                const Tile& tl = st_tl;
                const uint32_t dw = base + kSfOff + buf * (kSfWBytes + kSfTBytes), dt = dw + kSfWBytes;
                mbar_arrive_expect_tx(sf_full(buf), (uint32_t)(kSfWBytes + kSfTBytes));
                const int xw = st_b * kSfBlk * 4;  // byte offset of the block within a row's scales
                if constexpr (kL1)
                    tma_load_4d(dw, &tmSW, xw, tl.s * 128, 0, tl.e, sf_full(buf));
                else
                    tma_load_2d(dw, &tmSW, xw, wrow(tl, 0), sf_full(buf));
                tma_load_2d(dt, &tmSX, kL1 && kFp4 ? st_b * kSfBlk : xw, tl.row0, sf_full(buf));
                ++sj;
                if (++st_b == n_sfb) {
                    st_b = 0;
                    st_t += gridDim.x;
                    if (st_t < total) st_tl = tile_of(st_t);
                }
            };
            issue_scales();
            issue_scales();
            int it = 0;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const Tile tl = tile_of(t);
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    const int s = it % kStages;
                    if (!ok || !mbar_wait(empty_bar(s), ((uint32_t)(it / kStages) & 1u) ^ 1u, p.hdr, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = base + s * kStageBytes, sb = sa + kTokBytes;
                    mbar_arrive_expect_tx(full_bar(s), (uint32_t)kTokBytes + kWTx);
                    const int x = kb * kAtomK;
                    tma_load_2d(sa, &tmX, x, tl.row0, full_bar(s));
                    if constexpr (kL1)
                        tma_load_4d(sb, &tmW, x, tl.s * 128, 0, tl.e, full_bar(s));
                    else
                        tma_load_2d(sb, &tmW, x, wrow(tl, 0), full_bar(s));
                    // after the stage's operands, which the MMA waits for first: the scale
                    // block two ahead of the one this stage starts
                    if (kb % kSfBlk == 0) issue_scales();
                }
            }
            // drain: every copy issued has landed (bounded)
            for (int j = it - kStages < 0 ? 0 : it - kStages; j < it; ++j)
                mbar_drain(full_bar(j % kStages), (uint32_t)(j / kStages) & 1u, p.hdr);
            for (int j = sj - kSfBufs < 0 ? 0 : sj - kSfBufs; j < sj; ++j)
                mbar_drain(sf_full(j % kSfBufs), (uint32_t)(j / kSfBufs) & 1u, p.hdr);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        // (per-stage work kept short: a non-blocking test of the stage before the bounded wait,
        // the stage position kept as a counter, descriptors advanced by adding to their address
        // field: start >> 4, +2 per 32 K of a K-major atom, + the stage's offset >> 4)
        if (lane == 0) {
            const uint64_t ad0 = kmajor_desc(base, 0), bd0 = kmajor_desc(base + kTokBytes, 0);
            uint32_t idesc[kAtomK / 32];
#pragma unroll
            for (int kk = 0; kk < kAtomK / 32; ++kk) idesc[kk] = tm_idesc(kAfmt, kBfmt, kWN, kk);
            int s = 0, tc = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++tc) {
                const int a = tc % kAccs;
                if (!mbar_wait(acc_empty(a), ((uint32_t)(tc / kAccs) & 1u) ^ 1u, p.hdr, abort_flag)) break;
                tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)(a * kWN);
                for (int kb = 0; kb < KB; ++kb) {
                    if (!(mbar_test(full_bar(s), ph) || mbar_wait(full_bar(s), ph, p.hdr, abort_flag))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t so = (uint64_t)((s * kStageBytes) >> 4);
                    const uint32_t sf = tmem_base + kSfCol0 + s * kSfColsPerStage;
#pragma unroll
                    for (int kk = 0; kk < kAtomK / 32; ++kk)
                        tm_mma(d, ad0 + so + 2 * kk, bd0 + so + 2 * kk, idesc[kk], sf, sf + 4, (kb | kk) != 0);
                    tc_commit(empty_bar(s));
                    if (++s == kStages) s = 0, ph ^= 1u;
                }
                if (ok) tc_commit(acc_full(a));
            }
            tc_commit(drain_bar);
            mbar_drain(drain_bar, 0, p.hdr);
        }
    } else if (warp >= 6 && warp < 10) {
        // ---------------- scale writers ----------------
        // Lane l of warp q writes TMEM lane 32q + l: the A word of token row r = 32q + l and the
        // B words of weight rows 32c + l (c < N/32), all read from the scale block in shared
        // memory ([row][4 atoms] words; 4-way bank conflicts at most).
        const int q = warp & 3;
        const int r = 32 * q + lane;
        int it = 0, sj = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
            const Tile tl = tile_of(t);
            const bool tok_valid = r < tl.n_valid;
            for (int kb = 0; kb < KB && ok; kb += kSfBlk) {
                const int buf = sj % kSfBufs;
                const bool f_ok = mbar_wait(sf_full(buf), (uint32_t)(sj / kSfBufs) & 1u, p.hdr, abort_flag);
                if (!__all_sync(0xffffffffu, f_ok)) {
                    ok = false;
                    break;
                }
                const uint32_t* sw = reinterpret_cast<const uint32_t*>(smem + kSfOff + buf * (kSfWBytes + kSfTBytes));
                const uint32_t* sx = sw + kSfWBytes / 4;
                for (int i = 0; i < kSfBlk && kb + i < KB; ++i, ++it) {
                    const int s = it % kStages;
                    const bool w_ok = mbar_wait(empty_bar(s), ((uint32_t)(it / kStages) & 1u) ^ 1u, p.hdr, abort_flag);
                    if (!__all_sync(0xffffffffu, w_ok)) {
                        ok = false;
                        break;
                    }
                    uint32_t ta = sx[r * kSfBlk + i];
                    if constexpr (kL1 && kFp4) ta = ((ta >> 23) & 0xffu) * 0x01010101u;  // power-of-two fp32 scale
                    if (!tok_valid) ta = 0x7f7f7f7fu;  // 1.0 for the padding rows
                    // slot columns: 0-3 the A word (the MMA reads column q of lane quarter q), then
                    // the B words of weight rows 32c + lane (c < N/32), the rest unused
                    uint32_t v[16];
#pragma unroll
                    for (int c = 0; c < 4; ++c) v[c] = ta;
#pragma unroll
                    for (int c = 0; c < 12; ++c) v[4 + c] = c < kWN / 32 ? sw[(32 * c + lane) * kSfBlk + i] : 0x7f7f7f7fu;
                    tmem_st16(tmem_base + ((uint32_t)(32 * q) << 16) + kSfCol0 + s * kSfColsPerStage, v);
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(full_bar(s));
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(sf_empty(buf));
                ++sj;
            }
        }
    } else {
        // ---------------- epilogue (warps 2..5, 10..13): thread = token row ----------------
        const int q = warp & 3;
        const int half = warp >= 10;  // which half of the tile's columns this warp drains
        const int r = 32 * q + lane;
        int tc = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x, ++tc) {
            const int a = tc % kAccs;
            const uint32_t tb = tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(a * kWN);
            const Tile tl = tile_of(t);
            const bool valid = r < tl.n_valid;
            const int64_t row = tl.row0 + r;
            // L2: this row's combine slot and gate weight, read while the tile's MMAs run
            int src = -1;
            float gw = 0.0f;
            if constexpr (!kL1) {
                src = valid ? debug_row(p.hdr, __ldg(p.pool_src + row), (int64_t)p.T * p.K) : -1;
                gw = src >= 0 ? __ldg(args.topk_weights + src) : 0.0f;
            }
            const bool w_ok = mbar_wait(acc_full(a), (uint32_t)(tc / kAccs) & 1u, p.hdr, abort_flag);
            if (!__all_sync(0xffffffffu, w_ok)) break;
            tc_fence_after();
            auto release = [&]() {  // this warp's columns of the accumulator are in registers
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(acc_empty(a));
            };
            if constexpr (kL1) {
                // A = SiLU(gate) * up for outputs 128s + 32c .. +31 (c = 2 half, 2 half + 1), then MX
                // FP8: one UE8M0 exponent per 32 outputs of the token, 32 codes in one 32-byte store
#pragma unroll 1
                for (int c = 2 * half; c < 2 * half + 2; ++c) {
                    uint32_t g[32], u[32];
                    tmem_ld32(tb + 32 * c, g);
                    tmem_ld32(tb + 128 + 32 * c, u);
                    tmem_ld_wait();
                    if (c == 2 * half + 1) release();
                    float av[32];
                    float amax = 0.0f;
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj) {
                        av[jj] = swiglu1(__uint_as_float(g[jj]), __uint_as_float(u[jj]), p.act_clamp);
                        amax = fmaxf(amax, fabsf(av[jj]));
                    }
                    const int ex = mx_exponent_fp8<kE5>(amax);
                    const float inv = exp2_neg_int(ex);
                    uint32_t w[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        w[k] = fp8x2<kE5>(av[4 * k] * inv, av[4 * k + 1] * inv) |
                               (fp8x2<kE5>(av[4 * k + 2] * inv, av[4 * k + 3] * inv) << 16);
                    const int j0 = tl.s * 128 + 32 * c;
                    st_global_v8_if(valid, p.a_pool + row * I + j0, w);
                    st_global_u8_if(valid, p.a_pool_scale + row * (I / 32) + (j0 >> 5), (uint8_t)(ex + 127));
                }
            } else {
                // c = bf16(G * y) for this warp's half of the tile's hidden columns: packed into
                // registers first, so the accumulator is released before the stores (a thread's
                // bytes go to its own combine row in 32-byte stores; with 32 rows per warp store
                // instruction the stores are the slow part)
                constexpr int kChunks = kWN / 32, kMine = (kChunks + 1) / 2;
                const int c0 = half * kMine, nc = half ? kChunks - kMine : kMine;
                uint32_t w[16 * kMine];
#pragma unroll
                for (int i = 0; i < kMine; ++i) {
                    if (i < nc) {
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {  // 16 columns per load keeps the registers in bounds
                            uint32_t y[16];
                            tmem_ld16(tb + 32 * (c0 + i) + 16 * hh, y);
                            tmem_ld_wait();
#pragma unroll
                            for (int k = 0; k < 8; ++k)
                                w[16 * i + 8 * hh + k] =
                                    (uint32_t)float_to_bf16_bits(__fmul_rn(gw, __uint_as_float(y[2 * k]))) |
                                    ((uint32_t)float_to_bf16_bits(__fmul_rn(gw, __uint_as_float(y[2 * k + 1]))) << 16);
                        }
                    }
                }
                release();
                uint16_t* dst = p.comb + (int64_t)(src >= 0 ? src : 0) * H + tl.s * kWN + 32 * c0;
#pragma unroll
                for (int k = 0; k < 2 * kMine; ++k)
                    if (k < 2 * nc) st_global_v8_if(src >= 0, dst + 16 * k, w + 8 * k);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, 512);
}

template <int MODE, bool kL1, int kWN>
cudaError_t launch_tm(const Plan& p, const void* w, const void* w_scale, const float* topk_weights, cudaStream_t s) {
    using Cfg = TmCfg<kWN>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(tc_bs_tm_kernel<MODE, kL1, kWN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)Cfg::kSmem);
    });
    if (attr_err != cudaSuccess) return attr_err;
    const int n_out = kL1 ? 2 * p.I : p.H;
    const int kin = kL1 ? p.H : p.I;
    constexpr bool kFp4 = MODE == MOE_A8W4_FP8_FP4;
    const CUtensorMapDataType wtype = kFp4 ? CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    const uint64_t pitch = kFp4 ? (uint64_t)kin / 2 : (uint64_t)kin;  // bytes per weight row
    CUtensorMap tmW, tmX;
    bool ok_w;
    if (kL1) {
        // [K][row within the gate or up half][half][expert]: one box holds a tile's 128 gate and 128 up rows
        const uint64_t dims[4] = {(uint64_t)kin, (uint64_t)p.I, 2, (uint64_t)p.E};
        const uint64_t strides[3] = {pitch, pitch * p.I, pitch * 2 * p.I};
        const uint32_t box[4] = {kAtomK, 128, 2, 1};
        ok_w = tc_make_map_nd(&tmW, wtype, 4, w, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
    } else {
        const uint64_t dims[2] = {(uint64_t)kin, (uint64_t)p.E * n_out};
        const uint64_t strides[1] = {pitch};
        const uint32_t box[2] = {kAtomK, kWN};
        ok_w = tc_make_map_nd(&tmW, wtype, 2, w, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
    }
    if (!ok_w) return cudaErrorInvalidValue;
    if (!tc_make_map_2d(&tmX, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, kL1 ? (const void*)p.x_pool : (const void*)p.a_pool,
                        (uint64_t)kin, (uint64_t)p.pool_rows, kAtomK, kTM, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    // scale words, 16 bytes (4 K atoms) of every row per copy, unswizzled
    CUtensorMap tmSW, tmSX;
    const uint64_t sp = (uint64_t)kin / 32;  // scale bytes per weight row
    if (kL1) {
        const uint64_t dims[4] = {sp, (uint64_t)p.I, 2, (uint64_t)p.E};
        const uint64_t strides[3] = {sp, sp * p.I, sp * 2 * p.I};
        const uint32_t box[4] = {16, 128, 2, 1};
        ok_w = tc_make_map_nd(&tmSW, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, w_scale, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
    } else {
        const uint64_t dims[2] = {sp, (uint64_t)p.E * n_out};
        const uint64_t strides[1] = {sp};
        const uint32_t box[2] = {16, kWN};
        ok_w = tc_make_map_nd(&tmSW, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, w_scale, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
    }
    if (!ok_w) return cudaErrorInvalidValue;
    bool ok_x;
    if (kL1 && kFp4) {  // fp32 per 128 elements of a token row
        const uint64_t dims[2] = {(uint64_t)kin / 128, (uint64_t)p.pool_rows};
        const uint64_t strides[1] = {(uint64_t)kin / 128 * 4};
        const uint32_t box[2] = {4, kTM};
        ok_x = tc_make_map_nd(&tmSX, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, p.x_pool_scale, dims, strides, box,
                              CU_TENSOR_MAP_SWIZZLE_NONE);
    } else {  // UE8M0 per 32 elements
        const uint64_t dims[2] = {sp, (uint64_t)p.pool_rows};
        const uint64_t strides[1] = {sp};
        const uint32_t box[2] = {16, kTM};
        ok_x = tc_make_map_nd(&tmSX, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, kL1 ? (const void*)p.x_pool_scale : (const void*)p.a_pool_scale,
                              dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
    }
    if (!ok_x) return cudaErrorInvalidValue;
    TmArgs args{p, static_cast<const uint8_t*>(w_scale), topk_weights, kL1 ? p.I / 128 : p.H / kWN, kin / kAtomK, n_out,
                kin};
    const int64_t max_tiles = std::max<int64_t>(1, (p.pool_rows / kTM) * args.n_slabs);
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(max_tiles, tc_num_sms()));
    tc_bs_tm_kernel<MODE, kL1, kWN><<<grid, kThreads, Cfg::kSmem, s>>>(tmW, tmX, tmSW, tmSX, args);
    return cudaGetLastError();
}

}  // namespace

bool bs_tm_supported(const Plan& p, int stage) {
    if ((p.mode != MOE_A8W8_FP8 && p.mode != MOE_A8W8_FP8_E5M2 && p.mode != MOE_A8W4_FP8_FP4) ||
        p.E > kMaxExperts || !tc_encode_available())
        return false;
    // scale rows by TMA: their byte pitch (K / 32; K / 32 for the fp32 per-128 token scales
    // too) must be a multiple of 16
    if (stage == 1) return p.I % 128 == 0 && p.H % 512 == 0;
    return (p.H % 224 == 0 || p.H % 256 == 0) && p.I % 512 == 0;
}

cudaError_t launch_l1_bs_tm(const Plan& p, const void* w1, const void* w1_scale, cudaStream_t s) {
    if (p.mode == MOE_A8W4_FP8_FP4) return launch_tm<MOE_A8W4_FP8_FP4, true, 256>(p, w1, w1_scale, nullptr, s);
    if (p.mode == MOE_A8W8_FP8) return launch_tm<MOE_A8W8_FP8, true, 256>(p, w1, w1_scale, nullptr, s);
    if (p.mode == MOE_A8W8_FP8_E5M2) return launch_tm<MOE_A8W8_FP8_E5M2, true, 256>(p, w1, w1_scale, nullptr, s);
    return cudaErrorNotSupported;
}

cudaError_t launch_l2_bs_tm(const Plan& p, const void* w2, const void* w2_scale, const float* topk_weights,
                            cudaStream_t s) {
    // N = 224 keeps two accumulators in TMEM (the epilogue overlaps the next tile)
    const bool n224 = p.H % 224 == 0;
    if (p.mode == MOE_A8W4_FP8_FP4)
        return n224 ? launch_tm<MOE_A8W4_FP8_FP4, false, 224>(p, w2, w2_scale, topk_weights, s)
                    : launch_tm<MOE_A8W4_FP8_FP4, false, 256>(p, w2, w2_scale, topk_weights, s);
    if (p.mode == MOE_A8W8_FP8)
        return n224 ? launch_tm<MOE_A8W8_FP8, false, 224>(p, w2, w2_scale, topk_weights, s)
                    : launch_tm<MOE_A8W8_FP8, false, 256>(p, w2, w2_scale, topk_weights, s);
    if (p.mode == MOE_A8W8_FP8_E5M2)
        return n224 ? launch_tm<MOE_A8W8_FP8_E5M2, false, 224>(p, w2, w2_scale, topk_weights, s)
                    : launch_tm<MOE_A8W8_FP8_E5M2, false, 256>(p, w2, w2_scale, topk_weights, s);
    return cudaErrorNotSupported;
}

}  // namespace moe
