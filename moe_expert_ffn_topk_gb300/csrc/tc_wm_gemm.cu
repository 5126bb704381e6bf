// Weight-major tensor-core grouped GEMM with in-kernel weight dequantisation. The INT8 mode runs
// on it (sm_103a has no integer tcgen05.mma kind); the FP8 modes use the block-scaled kernel in
// tc_bs_gemm.cu, and the FP8 / e2m1 converter branches below are kept as the template's other
// instances of the same pipeline.
//
// Orientation: the MMA's M dimension runs over 128 weight rows and its N dimension over the
// tokens routed to one expert (N = 16..128 per tile, or 256 for INT8, see below), so the same
// kernel serves decode (a handful of tokens per expert: the weights stream through once) and
// prefill (hundreds of tokens per tile). Each tile carries two 128-row weight blocks that share
// the token operand: L1 = the gate rows and the up rows of the same 128 outputs of A (Ascend
// mega_moe page, "SwiGLU Activation": the gate half and the up half of H), so one thread holds
// gate and up of the same (output, token) pair; L2 = two adjacent 128-row blocks of hidden
// columns.
//
// Operands on the tensor cores are bf16 (tcgen05.mma kind::f16, fp32 accumulation in TMEM):
// - tokens: the dispatch stage (and for L2 the L1 epilogue / INT8 row quantiser) already wrote
//   them dequantised to bf16; x~ = e4m3 code * power-of-two scale is exact in bf16. TMA loads
//   them straight into the 128-byte-swizzled K-major tile.
// - weights stay in HBM in their compact storage format (e2m1, e4m3 or int8); TMA brings the
//   raw bytes into a staging ring (32- or 64-byte swizzled) and four converter warps expand
//   them, with their UE8M0 block scale, to bf16 in the 128-byte-swizzled layout (exact as well). This keeps the HBM stream at 0.5 or
//   1 byte per weight, which is what decode is bound by.
// INT8: every product q_x * q_w is an integer, and the fp32 accumulator is exact while the
// partial sums stay below 2^24. The token codes are split as q = 16*hi + lo with
// hi = floor(q/16) in [-8, 7] and lo = q mod 16 in [0, 15] (the identity of the page's A8W4-INT
// "MSD" scheme), stored as two bf16 planes; the B tile holds 128 tokens' hi rows then their lo
// rows (N = 256), every partial sum is bounded by 15 * 127 * K < 2^24 for K <= 8800, and the
// epilogue rebuilds the exact int32 accumulator as 16 * D_hi + D_lo before the page's fp32
// dequantisation (C * s^W) * s^X.
//
// Warp roles (352 threads): warp 0 TMA of raw weights, warp 1 TMEM allocation + MMA issue,
// warps 2-5 epilogue, warps 6-9 weight converters, warp 10 TMA of the token tiles.
// Every wait is bounded; on time-out the CTA records MOE_ERR_TIMEOUT, drains and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "tc_common.cuh"

namespace moe {

namespace {

using namespace tc;

constexpr int kWR = 128;        // weight rows per block (MMA M)
constexpr int kTokTile = 128;   // tokens per tile (one route tile)
constexpr int kBK = 64;         // K per stage
constexpr int kTokBox = 16;     // token rows per TMA box
constexpr int kThreads = 352;
constexpr int kMaxExperts = 1024;
constexpr int kABytes = 2 * kWR * 128;  // two 128-row bf16 weight blocks per stage

// Three rings per CTA: raw weight codes (TMA), the weights converted to bf16 (converter warps)
// and the bf16 token tiles (TMA). The token ring is separate so its loads run ahead of the
// converters by its own depth.
template <int MODE>
struct WmCfg;
template <>
struct WmCfg<MOE_A8W8_INT8> {
    static constexpr int kWRaw = 64, kBRows = 256, kAccCols = 256, kBufs = 1;
    static constexpr int kRawStages = 3, kBfStages = 2, kTokStages = 3;
};

template <int MODE>
struct WmLayout {
    using C = WmCfg<MODE>;
    static constexpr int kBfBytes = kABytes;                // two bf16 weight blocks
    static constexpr int kTokBytes = C::kBRows * 128;       // bf16 token tile (INT8: hi + lo rows)
    static constexpr int kRawBytes = 2 * kWR * C::kWRaw;
    static constexpr int kBfOff = 0;
    static constexpr int kTokOff = kBfOff + C::kBfStages * kBfBytes;
    static constexpr int kRawOff = kTokOff + C::kTokStages * kTokBytes;
    static constexpr int kBarOff = kRawOff + C::kRawStages * kRawBytes;
    static constexpr int kNumBars = 2 * C::kRawStages + 2 * C::kBfStages + 2 * C::kTokStages + 4 + 1;
    static constexpr int kMiscOff = kBarOff + 8 * kNumBars;     // tmem holder, abort flag
    static constexpr int kTileOff = kMiscOff + 16;              // int[E+1]
    static constexpr int kCountsOff = kTileOff + 4 * (kMaxExperts + 1);
    static constexpr int kBytes = kCountsOff + 4 * kMaxExperts;
    static constexpr size_t kSmem = 1024 + (size_t)kBytes;
};

// kind::f16 instruction descriptor: D fp32, A and B bf16, both K-major, M = 128; N added per tile.
constexpr uint32_t kIdescBase = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kWR >> 4) << 24);

struct WmArgs {
    Plan p;
    const uint8_t* w_scale;     // UE8M0 [E*n_out][kin/32] (FP8 modes) or fp32 [E*n_out] (INT8)
    const float* topk_weights;  // L2
    int n_slabs;                // tiles per (expert, token tile)
    int k_blocks;               // kin / 64
    int n_out;                  // weight rows per expert (L1: 2I, L2: H)
    int kin;                    // K
};

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
    tl.row0 = (tile_off[lo] + tl.m) * kTokTile;
    return tl;
}

// Token columns the MMA covers for a tile: the valid tokens rounded up to 16 (the MMA's N
// granularity for M = 128), or the fixed 128 hi + 128 lo rows of the INT8 split.
template <int MODE>
__device__ __forceinline__ int tile_n(int n_valid) {
    if constexpr (MODE == MOE_A8W8_INT8) return 256;
    else return (n_valid + 15) & ~15;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    return (uint32_t)float_to_bf16_bits(lo) | ((uint32_t)float_to_bf16_bits(hi) << 16);
}

__device__ __forceinline__ void store_chunk(uint8_t* tile, int r, int ch, uint32_t a, uint32_t b, uint32_t c,
                                            uint32_t d) {
    *reinterpret_cast<uint4*>(tile + r * 128 + ((ch ^ (r & 7)) << 4)) = make_uint4(a, b, c, d);
}

// 8 e2m1 codes (one 32-bit word, element 2j in the low nibble of byte j) times a power-of-two
// scale, as 4 bf16x2 words. e2m1 -> f16 is exact, the fp32 product is exact, and so is the
// rounding to bf16.
__device__ __forceinline__ void e2m1x8_to_bf16(uint32_t w, float sc, uint32_t (&o)[4]) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const __half2_raw h = __nv_cvt_fp4x2_to_halfraw2((__nv_fp4x2_storage_t)((w >> (8 * j)) & 0xffu), __NV_E2M1);
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h));
        o[j] = pack_bf16x2(f.x * sc, f.y * sc);
    }
}

// 8 e4m3 codes (two 32-bit words) times a power-of-two scale, as 4 bf16x2 words (exact).
__device__ __forceinline__ void e4m3x8_to_bf16(uint32_t w0, uint32_t w1, float sc, uint32_t (&o)[4]) {
    const uint32_t ww[2] = {w0, w1};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t pair = (ww[j >> 1] >> (16 * (j & 1))) & 0xffffu;
        const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)pair, __NV_E4M3);
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h));
        o[j] = pack_bf16x2(f.x * sc, f.y * sc);
    }
}

// 8 int8 codes (two 32-bit words) as 4 bf16x2 words (exact).
__device__ __forceinline__ void int8x8_to_bf16(uint32_t w0, uint32_t w1, uint32_t (&o)[4]) {
    const uint32_t ww[2] = {w0, w1};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t pair = ww[j >> 1] >> (16 * (j & 1));
        o[j] = pack_bf16x2((float)(int8_t)(pair & 0xffu), (float)(int8_t)((pair >> 8) & 0xffu));
    }
}

// Expand weight row r's K block (64 elements) from the raw tile, which TMA wrote with the
// 32-byte (e2m1: 32-byte rows) or 64-byte (one-byte codes: 64-byte rows) swizzle, into the
// 128-byte-swizzled bf16 row r of a K-major MMA tile. Reads and writes are 16-byte accesses
// and, with the swizzles, free of bank conflicts across a warp.
template <int MODE>
__device__ __forceinline__ void convert_row(const uint8_t* raw_tile, uint32_t scales2, uint8_t* tile, int r) {
    const float s0 = ue8m0_to_float((uint8_t)(scales2 & 0xffu));
    const float s1 = ue8m0_to_float((uint8_t)((scales2 >> 8) & 0xffu));
    if constexpr (MODE == MOE_A8W4_FP8_FP4) {
        const uint8_t* row = raw_tile + r * 32;
        const int x = (r >> 2) & 1;  // 32-byte swizzle: chunk ^= address bit 7
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const uint4 c = *reinterpret_cast<const uint4*>(row + ((q ^ x) << 4));
            const float sc = q == 0 ? s0 : s1;
            const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                uint32_t o[4];
                e2m1x8_to_bf16(w[k], sc, o);
                store_chunk(tile, r, q * 4 + k, o[0], o[1], o[2], o[3]);
            }
        }
    } else {
        const uint8_t* row = raw_tile + r * 64;
        const int x = (r >> 1) & 3;  // 64-byte swizzle: chunk ^= address bits 7-8
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint4 c = *reinterpret_cast<const uint4*>(row + ((q ^ x) << 4));
            uint32_t o[4], o2[4];
            if constexpr (MODE == MOE_A8W8_FP8) {
                const float sc = q < 2 ? s0 : s1;
                e4m3x8_to_bf16(c.x, c.y, sc, o);
                e4m3x8_to_bf16(c.z, c.w, sc, o2);
            } else {
                int8x8_to_bf16(c.x, c.y, o);
                int8x8_to_bf16(c.z, c.w, o2);
            }
            store_chunk(tile, r, 2 * q, o[0], o[1], o[2], o[3]);
            store_chunk(tile, r, 2 * q + 1, o2[0], o2[1], o2[2], o2[3]);
        }
    }
}

template <int MODE, bool kL1>
__global__ void __launch_bounds__(kThreads, 1)
    tc_wm_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX, WmArgs args) {
    using C = WmCfg<MODE>;
    using L = WmLayout<MODE>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = smem_u32(smem_raw);
    const uint32_t base = (raw_base + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (base - raw_base);
    const uint32_t bars = base + L::kBarOff;
    auto raw_full = [&](int i) { return bars + 8u * i; };
    auto raw_empty = [&](int i) { return bars + 8u * (C::kRawStages + i); };
    auto bf_full = [&](int i) { return bars + 8u * (2 * C::kRawStages + i); };
    auto bf_empty = [&](int i) { return bars + 8u * (2 * C::kRawStages + C::kBfStages + i); };
    constexpr int kTokBar = 2 * C::kRawStages + 2 * C::kBfStages;
    auto tok_full = [&](int i) { return bars + 8u * (kTokBar + i); };
    auto tok_empty = [&](int i) { return bars + 8u * (kTokBar + C::kTokStages + i); };
    constexpr int kAccBar = kTokBar + 2 * C::kTokStages;
    auto acc_full = [&](int i) { return bars + 8u * (kAccBar + i); };
    auto acc_empty = [&](int i) { return bars + 8u * (kAccBar + 2 + i); };
    const uint32_t drain_bar = bars + 8u * (kAccBar + 4);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);
    int* tile_off = reinterpret_cast<int*>(smem + L::kTileOff);
    int* counts = reinterpret_cast<int*>(smem + L::kCountsOff);

    const Plan& p = args.p;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i <= p.E; i += kThreads) tile_off[i] = p.tile_off[i];
    for (int i = threadIdx.x; i < p.E; i += kThreads) counts[i] = p.counts[i];
    if (threadIdx.x == 0) {
        for (int i = 0; i < C::kRawStages; ++i) {
            mbar_init(raw_full(i), 1);
            mbar_init(raw_empty(i), 128);
        }
        for (int i = 0; i < C::kBfStages; ++i) {
            mbar_init(bf_full(i), 128);      // the 128 converter threads
            mbar_init(bf_empty(i), 1);
        }
        for (int i = 0; i < C::kTokStages; ++i) {
            mbar_init(tok_full(i), 1);       // the token TMA (arrive + bytes)
            mbar_init(tok_empty(i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(acc_full(i), 1);
            mbar_init(acc_empty(i), 4);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_holder), 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    const int total = tile_off[p.E] * args.n_slabs;
    const int KB = args.k_blocks;
    const int I = p.I, H = p.H;

    if (warp == 0) {
        // ---------------- raw weight TMA ----------------
        if (lane == 0) {
            int it = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const Tile tl = decode(t, tile_off, p.E, args.n_slabs);
                const int w0 = tl.e * args.n_out + (kL1 ? tl.s * kWR : tl.s * 2 * kWR);
                const int w1 = kL1 ? w0 + I : w0 + kWR;
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    const int r = it % C::kRawStages;
                    if (!mbar_wait(raw_empty(r), ((uint32_t)(it / C::kRawStages) & 1u) ^ 1u, p.hdr, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t dst = base + L::kRawOff + r * L::kRawBytes;
                    mbar_arrive_expect_tx(raw_full(r), L::kRawBytes);
                    tma_load_2d(dst, &tmW, kb * C::kWRaw, w0, raw_full(r));
                    tma_load_2d(dst + kWR * C::kWRaw, &tmW, kb * C::kWRaw, w1, raw_full(r));
                }
            }
            for (int j = it - C::kRawStages < 0 ? 0 : it - C::kRawStages; j < it; ++j)
                mbar_drain(raw_full(j % C::kRawStages), (uint32_t)(j / C::kRawStages) & 1u, p.hdr);
        }
    } else if (warp == 10) {
        // ---------------- token TMA (bf16, swizzled) ----------------
        if (lane == 0) {
            int it = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const Tile tl = decode(t, tile_off, p.E, args.n_slabs);
                const int n_valid = min(kTokTile, counts[tl.e] - tl.m * kTokTile);
                const int n = tile_n<MODE>(n_valid);
                const int boxes = (MODE == MOE_A8W8_INT8 ? kTokTile : n) / kTokBox;
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    const int b = it % C::kTokStages;
                    if (!mbar_wait(tok_empty(b), ((uint32_t)(it / C::kTokStages) & 1u) ^ 1u, p.hdr, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t dst = base + L::kTokOff + b * L::kTokBytes;
                    const int planes = MODE == MOE_A8W8_INT8 ? 2 : 1;
                    mbar_arrive_expect_tx(tok_full(b), (uint32_t)(planes * boxes * kTokBox * 128));
                    for (int pl = 0; pl < planes; ++pl)
                        for (int i = 0; i < boxes; ++i)
                            tma_load_2d(dst + (pl * kTokTile + i * kTokBox) * 128, &tmX, kb * kBK,
                                        (int)(pl * p.pool_rows) + tl.row0 + i * kTokBox, tok_full(b));
                }
            }
            for (int j = it - C::kTokStages < 0 ? 0 : it - C::kTokStages; j < it; ++j)
                mbar_drain(tok_full(j % C::kTokStages), (uint32_t)(j / C::kTokStages) & 1u, p.hdr);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            int it = 0, tc = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++tc) {
                const int a = tc % C::kBufs;
                if (!mbar_wait(acc_empty(a), ((uint32_t)(tc / C::kBufs) & 1u) ^ 1u, p.hdr, abort_flag)) break;
                tc_fence_after();
                const Tile tl = decode(t, tile_off, p.E, args.n_slabs);
                const int n = tile_n<MODE>(min(kTokTile, counts[tl.e] - tl.m * kTokTile));
                const uint32_t idesc = kIdescBase | ((uint32_t)(n >> 3) << 17);
                const uint32_t d0 = tmem_base + (uint32_t)(a * 2 * C::kAccCols);
                const uint32_t d1 = d0 + C::kAccCols;
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    const int b = it % C::kBfStages, tb = it % C::kTokStages;
                    if (!mbar_wait(bf_full(b), (uint32_t)(it / C::kBfStages) & 1u, p.hdr, abort_flag) ||
                        !mbar_wait(tok_full(tb), (uint32_t)(it / C::kTokStages) & 1u, p.hdr, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa0 = base + L::kBfOff + b * L::kBfBytes;
                    const uint32_t sa1 = sa0 + kWR * 128;
                    const uint32_t sb = base + L::kTokOff + tb * L::kTokBytes;
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk) {
                        const uint64_t bd = kmajor_desc(sb, kk);
                        tc_mma(d0, kmajor_desc(sa0, kk), bd, idesc, (kb | kk) != 0);
                        tc_mma(d1, kmajor_desc(sa1, kk), bd, idesc, (kb | kk) != 0);
                    }
                    tc_commit(bf_empty(b));
                    tc_commit(tok_empty(tb));
                }
                if (ok) tc_commit(acc_full(a));
            }
            tc_commit(drain_bar);
            mbar_drain(drain_bar, 0, p.hdr);
        }
    } else if (warp >= 6) {
        // ---------------- weight converters ----------------
        const int c = threadIdx.x - 192;  // row of each 128-row weight block
        const int spr = args.kin / 32;    // scale bytes per weight row (a multiple of 4)
        int it = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
            const Tile tl = decode(t, tile_off, p.E, args.n_slabs);
            const int64_t g0 = (int64_t)tl.e * args.n_out + (kL1 ? tl.s * kWR : tl.s * 2 * kWR) + c;
            const int64_t g1 = kL1 ? g0 + I : g0 + kWR;
            // the scales of 8 k-blocks (16 bytes per row) are loaded one group ahead of use
            uint32_t cur0[4] = {}, cur1[4] = {}, nxt0[4] = {}, nxt1[4] = {};
            auto load_group = [&](int grp, uint32_t (&d0)[4], uint32_t (&d1)[4]) {
                if constexpr (MODE != MOE_A8W8_INT8) {
                    const uint32_t* r0 = reinterpret_cast<const uint32_t*>(args.w_scale + g0 * spr);
                    const uint32_t* r1 = reinterpret_cast<const uint32_t*>(args.w_scale + g1 * spr);
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        const int word = grp * 4 + w;
                        d0[w] = word < spr / 4 ? __ldg(r0 + word) : 0u;
                        d1[w] = word < spr / 4 ? __ldg(r1 + word) : 0u;
                    }
                }
            };
            load_group(0, cur0, cur1);
            load_group(1, nxt0, nxt1);
            for (int kb = 0; kb < KB; ++kb, ++it) {
                const int r = it % C::kRawStages, b = it % C::kBfStages;
                if (kb > 0 && (kb & 7) == 0) {
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        cur0[w] = nxt0[w];
                        cur1[w] = nxt1[w];
                    }
                    load_group((kb >> 3) + 1, nxt0, nxt1);
                }
                const int sel = (kb & 7) >> 1, sh = 16 * (kb & 1);
                uint32_t s0 = 0, s1 = 0;
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    if (w == sel) {
                        s0 = (cur0[w] >> sh) & 0xffffu;
                        s1 = (cur1[w] >> sh) & 0xffffu;
                    }
                }
                bool w_ok = mbar_wait(raw_full(r), (uint32_t)(it / C::kRawStages) & 1u, p.hdr, abort_flag);
                w_ok = w_ok && mbar_wait(bf_empty(b), ((uint32_t)(it / C::kBfStages) & 1u) ^ 1u, p.hdr, abort_flag);
                if (!__all_sync(0xffffffffu, w_ok)) {
                    ok = false;
                    break;
                }
                const uint8_t* rw = smem + L::kRawOff + r * L::kRawBytes;
                uint8_t* dst = smem + L::kBfOff + b * L::kBfBytes;
                convert_row<MODE>(rw, s0, dst, c);
                convert_row<MODE>(rw + kWR * C::kWRaw, s1, dst + kWR * 128, c);
                fence_proxy_async_smem();
                mbar_arrive(raw_empty(r));
                mbar_arrive(bf_full(b));
            }
        }
    } else {
        // ---------------- epilogue (warps 2..5) ----------------
        const int q = warp & 3;
        int tc = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x, ++tc) {
            const int a = tc % C::kBufs;
            const bool w_ok = mbar_wait(acc_full(a), (uint32_t)(tc / C::kBufs) & 1u, p.hdr, abort_flag);
            if (!__all_sync(0xffffffffu, w_ok)) break;
            tc_fence_after();
            const Tile tl = decode(t, tile_off, p.E, args.n_slabs);
            const int n_valid = min(kTokTile, counts[tl.e] - tl.m * kTokTile);
            const int n = tile_n<MODE>(n_valid);
            const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(a * 2 * C::kAccCols);
            if constexpr (kL1 && MODE != MOE_A8W8_INT8) {
                const int j = tl.s * kWR + q * 32 + lane;
                for (int c0 = 0; c0 < n; c0 += 32) {
                    uint32_t g[32], u[32];
                    tmem_ld32(tb + c0, g);
                    tmem_ld32(tb + C::kAccCols + c0, u);
                    tmem_ld_wait();
#pragma unroll
                    for (int tt = 0; tt < 32; ++tt) {
                        if (c0 + tt >= n) break;  // uniform across the warp
                        const float av = silu(__uint_as_float(g[tt])) * __uint_as_float(u[tt]);
                        float amax = fabsf(av);
#pragma unroll
                        for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
                        const int ex = mx_exponent_e4m3(amax);
                        const uint8_t code = float_to_e4m3_satfinite(av * exp2_neg_int(ex));
                        const int64_t row = tl.row0 + c0 + tt;
                        p.a_pool[row * I + j] = code;
                        p.a_bf16[row * I + j] =
                            float_to_bf16_bits(e4m3_to_float(code) * ue8m0_to_float((uint8_t)(ex + 127)));
                        if (lane == 0) p.a_pool_scale[row * (I / 32) + (tl.s * kWR + q * 32) / 32] = (uint8_t)(ex + 127);
                    }
                }
            } else if constexpr (kL1) {
                // INT8: C = 16 * D_hi + D_lo, H = (C * s^W1) * s^X, A = SiLU(H_gate) * H_up in fp32
                const int j = tl.s * kWR + q * 32 + lane;
                const float* s1 = reinterpret_cast<const float*>(args.w_scale) + (int64_t)tl.e * 2 * I;
                const float sg = s1[j], su = s1[I + j];
                for (int c0 = 0; c0 < kTokTile; c0 += 32) {
                    const float sx_l = reinterpret_cast<const float*>(p.x_pool_scale)[tl.row0 + c0 + lane];
                    uint32_t hi[32], lo[32];
                    float hg[32];
                    tmem_ld32(tb + c0, hi);
                    tmem_ld32(tb + kTokTile + c0, lo);
                    tmem_ld_wait();
#pragma unroll
                    for (int tt = 0; tt < 32; ++tt) {
                        const int cg = 16 * __float2int_rn(__uint_as_float(hi[tt])) + __float2int_rn(__uint_as_float(lo[tt]));
                        hg[tt] = __int2float_rn(cg);
                    }
                    tmem_ld32(tb + C::kAccCols + c0, hi);
                    tmem_ld32(tb + C::kAccCols + kTokTile + c0, lo);
                    tmem_ld_wait();
#pragma unroll
                    for (int tt = 0; tt < 32; ++tt) {
                        const float sx = __shfl_sync(0xffffffffu, sx_l, tt);
                        const int cu = 16 * __float2int_rn(__uint_as_float(hi[tt])) + __float2int_rn(__uint_as_float(lo[tt]));
                        const float Hg = __fmul_rn(__fmul_rn(hg[tt], sg), sx);
                        const float Hu = __fmul_rn(__fmul_rn(__int2float_rn(cu), su), sx);
                        p.a_f32[(int64_t)(tl.row0 + c0 + tt) * I + j] = silu(Hg) * Hu;
                    }
                }
            } else {
                // L2: c = bf16(G * y) to the combine row of (token, slot)
                for (int c0 = 0; c0 < n_valid; c0 += 32) {
                    const int src_l = c0 + lane < n_valid ? p.pool_src[tl.row0 + c0 + lane] : -1;
                    const float g_l = src_l >= 0 ? args.topk_weights[src_l] : 0.0f;
                    float sa_l = 0.0f;
                    if constexpr (MODE == MOE_A8W8_INT8)
                        sa_l = reinterpret_cast<const float*>(p.a_pool_scale)[tl.row0 + c0 + lane];
#pragma unroll 1
                    for (int blk = 0; blk < 2; ++blk) {
                        const int h = tl.s * 2 * kWR + blk * kWR + q * 32 + lane;
                        uint32_t y[32];
                        float yv[32];
                        if constexpr (MODE == MOE_A8W8_INT8) {
                            uint32_t lo[32];
                            tmem_ld32(tb + blk * C::kAccCols + c0, y);
                            tmem_ld32(tb + blk * C::kAccCols + kTokTile + c0, lo);
                            tmem_ld_wait();
                            const float s2 = reinterpret_cast<const float*>(args.w_scale)[(int64_t)tl.e * H + h];
#pragma unroll
                            for (int tt = 0; tt < 32; ++tt) {
                                const int d = 16 * __float2int_rn(__uint_as_float(y[tt])) + __float2int_rn(__uint_as_float(lo[tt]));
                                yv[tt] = __fmul_rn(__fmul_rn(__int2float_rn(d), s2), __shfl_sync(0xffffffffu, sa_l, tt));
                            }
                        } else {
                            tmem_ld32(tb + blk * C::kAccCols + c0, y);
                            tmem_ld_wait();
#pragma unroll
                            for (int tt = 0; tt < 32; ++tt) yv[tt] = __uint_as_float(y[tt]);
                        }
#pragma unroll
                        for (int tt = 0; tt < 32; ++tt) {
                            if (c0 + tt >= n_valid) break;  // uniform across the warp
                            const int src = __shfl_sync(0xffffffffu, src_l, tt);
                            const float gw = __shfl_sync(0xffffffffu, g_l, tt);
                            if (src >= 0) p.comb[(int64_t)src * H + h] = float_to_bf16_bits(__fmul_rn(gw, yv[tt]));
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty(a));
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, 512);
}

template <int MODE, bool kL1>
cudaError_t launch_wm(const Plan& p, const void* w, const void* w_scale, const float* topk_weights, cudaStream_t s) {
    using C = WmCfg<MODE>;
    using L = WmLayout<MODE>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(tc_wm_kernel<MODE, kL1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)L::kSmem);
    });
    if (attr_err != cudaSuccess) return attr_err;
    const int n_out = kL1 ? 2 * p.I : p.H;
    const int kin = kL1 ? p.H : p.I;
    const int kin_bytes = MODE == MOE_A8W4_FP8_FP4 ? kin / 2 : kin;
    const int planes = MODE == MOE_A8W8_INT8 ? 2 : 1;
    CUtensorMap tmW, tmX;
    if (!tc_make_map_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, w, (uint64_t)kin_bytes, (uint64_t)p.E * n_out,
                        C::kWRaw, kWR, C::kWRaw == 32 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_64B))
        return cudaErrorInvalidValue;
    if (!tc_make_map_2d(&tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, kL1 ? (const void*)p.x_bf16 : (const void*)p.a_bf16,
                        (uint64_t)kin, (uint64_t)planes * p.pool_rows, kBK, kTokBox, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    WmArgs args{p, static_cast<const uint8_t*>(w_scale), topk_weights, kL1 ? p.I / kWR : p.H / (2 * kWR),
                kin / kBK, n_out, kin};
    const int64_t max_tiles = (p.pool_rows / kTokTile) * args.n_slabs;
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(max_tiles, tc_num_sms()));
    tc_wm_kernel<MODE, kL1><<<grid, kThreads, L::kSmem, s>>>(tmW, tmX, args);
    return cudaGetLastError();
}

}  // namespace

bool wm_supported(const Plan& p, int stage) {
    if (p.mode != MOE_A8W8_INT8 || p.E > kMaxExperts || !tc_encode_available()) return false;
    if (stage == 1) return p.I % kWR == 0 && p.H % kBK == 0;
    return p.H % (2 * kWR) == 0 && p.I % kBK == 0;
}

cudaError_t launch_l1_wm(const Plan& p, const void* w1, const void* w1_scale, cudaStream_t s) {
    if (p.mode != MOE_A8W8_INT8) return cudaErrorNotSupported;
    return launch_wm<MOE_A8W8_INT8, true>(p, w1, w1_scale, nullptr, s);
}

cudaError_t launch_l2_wm(const Plan& p, const void* w2, const void* w2_scale, const float* topk_weights, cudaStream_t s) {
    if (p.mode != MOE_A8W8_INT8) return cudaErrorNotSupported;
    return launch_wm<MOE_A8W8_INT8, false>(p, w2, w2_scale, topk_weights, s);
}

}  // namespace moe
