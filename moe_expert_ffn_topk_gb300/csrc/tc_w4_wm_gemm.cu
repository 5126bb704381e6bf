// A8W4-INT grouped GEMM on the tensor cores, weight-major, with exact integer results (Ascend
// mega_moe page, A8W4-INT use case: int8 activations x signed int4 weights, C = Q_e . W1 and
// D = A^int8 . W2 as integers, then (C * s^W) * s^X in fp32).
//
// The operands travel as f16 exactly as in the token-major A8W4-INT kernel (kind::f16, fp32
// accumulation in TMEM): the packed int4 weight n becomes the f16 subnormal (n + 8) * 2^-24 in
// the converter warps (codes of a 32-bit word in the order 0 4 1 5 2 6 3 7, which the token plane
// of the dispatch stage and the row quantiser shares), the tokens are one f16 plane of their int8
// codes, the accumulator holds 2^-24 * sum_k (n_k + 8) q_k exactly while K <= 8704, and
// C = 2^24 * D - 8 * sum_k q_k with the per-token code sums.
//
// What differs is the orientation. Here M = 128 weight rows (the TMEM lanes) and N = the tokens:
// one tile takes up to 256 pool rows of an expert (two route tiles) and rounds its token count
// up to 16, so
// - an expert's weight slab is converted once for up to 256 of its tokens (the token-major tile
//   converts it again for every 128-row route tile), and
// - an expert's last, partial route tile costs MMA work only for its tokens (rounded to 16),
//   where a token-major tile computes all 128 rows.
// L1 tiles carry the gate block and the up block of the same 128 outputs (two accumulators of
// up to 256 columns sharing B), so an epilogue thread holds one output's gate and up values for
// every token and applies SwiGLU (Ascend page, "SwiGLU Activation"); L2 tiles carry two 128-row
// blocks of hidden columns and the epilogue scales each token's values by G and writes its bf16
// combine row (Ascend page, "Token Combine"). The two accumulators fill TMEM: the epilogue of a
// tile does not overlap the next tile's main loop.
//
// Larger tiles mean fewer of them: the kernel is chosen when the experts' weight slabs give at
// least four rounds of tiles on the GPU (w4_wm_preferred); below that the last, partly filled
// round costs more than the conversions saved (measured: 16 experts, 192 tiles on 152 SMs, 130 us
// against 114 us token-major; 64 experts, 768 tiles, step 0.715 against 0.766 ms).
//
// Warp roles (352 threads): warp 0 TMA of packed weights, warp 1 TMEM allocation + MMA issue,
// warps 2-5 epilogue (warp w owns TMEM lanes 32*(w%4) .. +31, i.e. those weight rows), warps 6-9
// converters (thread = one row of each weight block), warp 10 TMA of the token rows.
// Every wait is bounded; on time-out the CTA records MOE_ERR_TIMEOUT, drains and exits.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "tc_common.cuh"

namespace moe {

namespace {

using namespace tc;

constexpr int kWR = 128;         // weight rows per block (MMA M)
constexpr int kRouteRows = 128;  // pool rows of a route tile
constexpr int kTokMax = 256;     // tokens per tile (MMA N at most): two route tiles
constexpr int kTokBox = 16;      // token rows per TMA box of a tile's ragged end
constexpr int kBK = 64;          // K per stage: 64 f16 = one 128-byte swizzle row
constexpr int kThreads = 352;
constexpr int kMaxExperts = 1024;
constexpr int kRawStages = 3, kHfStages = 2, kTokStages = 3;
constexpr int kRawRow = kBK / 2;             // bytes of a packed weight row per stage
constexpr int kABytes = 2 * kWR * 128;       // two f16 weight blocks
constexpr int kTokBytes = kTokMax * 128;     // f16 token rows
constexpr int kRawBytes = 2 * kWR * kRawRow; // two packed weight blocks
constexpr int kHfOff = 0;
constexpr int kTokOff = kHfOff + kHfStages * kABytes;
constexpr int kRawOff = kTokOff + kTokStages * kTokBytes;
constexpr int kBarOff = kRawOff + kRawStages * kRawBytes;
constexpr int kNumBars = 2 * (kRawStages + kHfStages + kTokStages) + 2 + 1;
constexpr int kMiscOff = kBarOff + 8 * kNumBars;
constexpr int kTileOffOff = kMiscOff + 16;
constexpr int kChunkOffOff = kTileOffOff + 4 * (kMaxExperts + 1);
constexpr int kCountsOff = kChunkOffOff + 4 * (kMaxExperts + 1);
constexpr int kTabOff = kCountsOff + 4 * kMaxExperts;  // per epilogue warp [slot, gate, s^A, 8 * sum] x tokens
constexpr size_t kSmem = 1024 + (size_t)kTabOff + 4 * 4 * 4 * kTokMax;
static_assert(kSmem <= 232448, "shared memory");
// largest K with every partial sum of u * q below 2^24 (u <= 15, |q| <= 128)
constexpr int kMaxK = 8704;

// kind::f16 instruction descriptor: D fp32 (bits 4-5 = 1), A and B f16 (formats 0), both
// K-major, N >> 3 in bits 17-22 (the tile's tokens rounded up to 16), M = 128 (>> 4 in bits 24-28).
__device__ __forceinline__ uint32_t idesc_n(int n) {
    return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(kWR >> 4) << 24);
}

struct W4WmArgs {
    Plan p;
    const float* w_scale;       // fp32 per output channel [E * n_out]
    const float* topk_weights;  // L2
    const float* row_scale;     // s^X or s^A per pool row
    const int32_t* row_sums;    // code sums per pool row
    int n_slabs, k_blocks, n_out;
    // the fused launch (L1 then L2 in one launch): the fields above describe its L1, these its L2
    const float* w_scale2;
    const float* row_scale2;
    const int32_t* row_sums2;
    int n_slabs2, k_blocks2;
    int32_t* ctr;  // the workspace's counters: per route tile, then the re-quantisation job queue
};

constexpr int kL2 = 0, kL1 = 1, kFusedL1L2 = 2;  // what one launch runs
constexpr int kEpiBar = 1;                       // named barrier of the 4 epilogue warps
constexpr int kQuantRegVec = 12;  // fused launch: rows of A up to 1536 elements re-quantised from registers

struct Tile {
    int e, s, row0, n_valid, n16;
};

// Tiles are ordered expert-major, then weight slab, then token chunk (up to two route tiles):
// expert e owns [chunk_off[e] * n_slabs, chunk_off[e+1] * n_slabs).
__device__ __forceinline__ Tile decode_tile(int t, const int* tile_off, const int* chunk_off, const int* counts,
                                            int E, int n_slabs) {
    int lo = 0, hi = E - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (chunk_off[mid] * n_slabs <= t) lo = mid; else hi = mid - 1;
    }
    Tile tl;
    tl.e = lo;
    const int nc = chunk_off[lo + 1] - chunk_off[lo];
    const int local = t - chunk_off[lo] * n_slabs;
    tl.s = local / nc;
    const int j = local % nc;
    tl.row0 = (tile_off[lo] + 2 * j) * kRouteRows;
    tl.n_valid = min(kTokMax, counts[lo] - j * kTokMax);
    tl.n16 = (tl.n_valid + 15) & ~15;
    return tl;
}

// 8 int4 codes (one word, code 2j in the low nibble of byte j) -> 4 f16x2 words holding
// u = n + 8 as the subnormal u * 2^-24; word i holds codes i (low half) and i + 4 (high half).
__device__ __forceinline__ void int4x8_to_sub_f16(uint32_t w, uint32_t (&o)[4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t x = w >> (4 * i);
        uint32_t v;
        // (x & 0x000f000f) ^ 0x00080008: the two nibbles, sign bits flipped
        asm("lop3.b32 %0, %1, %2, %3, 0x6a;" : "=r"(v) : "r"(x), "r"(0x000f000fu), "r"(0x00080008u));
        o[i] = v;
    }
}

// Packed row r of a raw block (32 bytes, 32-byte swizzle: the 16-byte chunk index ^= address
// bit 7) -> f16 row r of a 128-byte-swizzled K-major tile.
__device__ __forceinline__ void convert_row(const uint8_t* raw_block, uint8_t* hf_block, int r) {
    const uint8_t* src = raw_block + r * kRawRow;
    const int x = (r >> 2) & 1;
    const uint4 c0 = *reinterpret_cast<const uint4*>(src + ((0 ^ x) << 4));
    const uint4 c1 = *reinterpret_cast<const uint4*>(src + ((1 ^ x) << 4));
    const uint32_t wd[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
    uint8_t* dst = hf_block + r * 128;
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {  // word ch: codes 8ch .. 8ch + 7 -> 16-byte chunk ch
        uint32_t o[4];
        int4x8_to_sub_f16(wd[ch], o);
        *reinterpret_cast<uint4*>(dst + ((ch ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// Exact integer C = 2^24 D - 8 * (code sum of the token), from the accumulator bits; 2^24 D is
// an integer below 2^24 (padding tokens hold anything: unsigned arithmetic keeps their
// discarded values defined).
__device__ __forceinline__ float exact_c(uint32_t bits, int sum8) {
    return __int2float_rn((int)((uint32_t)__float2int_rn(__uint_as_float(bits) * 16777216.0f) - (uint32_t)sum8));
}

template <int kKind>
__global__ void __launch_bounds__(kThreads, 1)
    tc_w4_wm_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                    const __grid_constant__ CUtensorMap tmX16, const __grid_constant__ CUtensorMap tmW2,
                    const __grid_constant__ CUtensorMap tmX2, const __grid_constant__ CUtensorMap tmX16_2,
                    W4WmArgs args) {
    constexpr bool kFused = kKind == kFusedL1L2;
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
    int* chunk_off = reinterpret_cast<int*>(smem + kChunkOffOff);
    int* counts = reinterpret_cast<int*>(smem + kCountsOff);

    const Plan& p = args.p;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i <= p.E; i += kThreads) tile_off[i] = p.tile_off[i];
    for (int i = threadIdx.x; i < p.E; i += kThreads) counts[i] = p.counts[i];
    __syncthreads();
    if (warp == 2) {
        // chunk_off = exclusive prefix sum of ceil(route tiles of e / 2), one warp scan per 32 experts
        int carry = 0;
        for (int b = 0; b < p.E; b += 32) {
            const int e = b + lane;
            int v = e < p.E ? (tile_off[e + 1] - tile_off[e] + 1) >> 1 : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += u;
            }
            if (e < p.E) chunk_off[e + 1] = carry + v;
            carry += __shfl_sync(0xffffffffu, v, 31);
        }
        if (lane == 0) chunk_off[0] = 0;
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < kRawStages; ++i) {
            mbar_init(raw_full(i), 1);
            mbar_init(raw_empty(i), 4);  // one arrival per converter warp
        }
        for (int i = 0; i < kHfStages; ++i) {
            mbar_init(hf_full(i), 4);
            mbar_init(hf_empty(i), 1);
        }
        for (int i = 0; i < kTokStages; ++i) {
            mbar_init(tok_full(i), 1);  // the token TMA (arrive + bytes)
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
    const int total1 = chunk_off[p.E] * args.n_slabs;
    const int total = kFused ? total1 + chunk_off[p.E] * args.n_slabs2 : total1;
    const int I = p.I, H = p.H;
    auto is_l1 = [&](int t) { return kKind == kL1 || (kFused && t < total1); };
    auto second = [&](int t) { return kFused && t >= total1; };  // an L2 tile of the fused launch
    auto tile_of = [&](int t) {
        return second(t) ? decode_tile(t - total1, tile_off, chunk_off, counts, p.E, args.n_slabs2)
                         : decode_tile(t, tile_off, chunk_off, counts, p.E, args.n_slabs);
    };
    auto kb_of = [&](int t) { return second(t) ? args.k_blocks2 : args.k_blocks; };
    // first weight row of block `blk` of the tile (L1: gate rows, then the up rows of the same outputs)
    auto wrow = [&](const Tile& tl, int blk, bool l1) {
        if (l1) return tl.e * 2 * I + (blk ? I : 0) + tl.s * kWR;
        return tl.e * H + tl.s * 2 * kWR + blk * kWR;
    };
    // fused launch: per route tile the count of its finished L1 tiles, then of its finished
    // re-quantisation jobs (an L2 tile waits for dep_target on each route tile of its token chunk);
    // then the job queue
    const int route_tiles = (int)(p.pool_rows / kRouteRows);
    const QuantQueue qq{args.ctr, args.ctr + route_tiles, args.ctr + route_tiles + 1, args.ctr + route_tiles + 2,
                        args.ctr + route_tiles + 3, kQuantJobs * n_route};
    const int dep_target = args.n_slabs + kQuantJobs;
    auto chunk_ready = [&](const Tile& tl) {  // acquire loads
        const int g = tl.row0 / kRouteRows;
        return ld_acquire_gpu(qq.dep + g) >= dep_target &&
               (tl.n_valid <= kRouteRows || ld_acquire_gpu(qq.dep + g + 1) >= dep_target);
    };
    auto wait_chunk = [&](const Tile& tl) {  // bounded
        const int g = tl.row0 / kRouteRows;
        return wait_count(qq.dep + g, dep_target, p.hdr, abort_flag) &&
               (tl.n_valid <= kRouteRows || wait_count(qq.dep + g + 1, dep_target, p.hdr, abort_flag));
    };

    if (warp == 0) {
        // ---------------- packed weight TMA: 2 x 128 rows x 32 bytes per stage ----------------
        if (lane == 0) {
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
                    tma_load_2d(dst, mW, kb * kRawRow, w0, raw_full(r));
                    tma_load_2d(dst + kWR * kRawRow, mW, kb * kRawRow, w1, raw_full(r));
                }
            }
            for (int j = it - kRawStages < 0 ? 0 : it - kRawStages; j < it; ++j)
                mbar_drain(raw_full(j % kRawStages), (uint32_t)(j / kRawStages) & 1u, p.hdr);
        }
    } else if (warp == 10) {
        // ---------------- token TMA: the tile's n16 rows (128-row boxes, then 16-row boxes) ----------------
        if (lane == 0) {
            int it = 0;
            bool ok = true, all_q = false;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const Tile tl = tile_of(t);
                const int KB = kb_of(t);
                const CUtensorMap* mX = second(t) ? &tmX2 : &tmX;
                const CUtensorMap* mX16 = second(t) ? &tmX16_2 : &tmX16;
                if (second(t) && !all_q) {
                    // once every job of the launch is finished, no later L2 tile needs a check
                    all_q = ld_acquire_gpu(qq.jobs_done) >= qq.n_jobs;
                    if (!all_q && !wait_chunk(tl)) break;
                    // the plane was written through the generic proxy; the TMA reads it
                    asm volatile("fence.proxy.async.global;" ::: "memory");
                }
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    const int b = it % kTokStages;
                    if (!mbar_wait(tok_empty(b), ((uint32_t)(it / kTokStages) & 1u) ^ 1u, p.hdr, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t dst = base + kTokOff + b * kTokBytes;
                    mbar_arrive_expect_tx(tok_full(b), (uint32_t)(tl.n16 * 128));
                    int j = 0;
                    for (; j + kRouteRows <= tl.n16; j += kRouteRows)
                        tma_load_2d(dst + j * 128, mX, kb * kBK, tl.row0 + j, tok_full(b));
                    for (; j < tl.n16; j += kTokBox)
                        tma_load_2d(dst + j * 128, mX16, kb * kBK, tl.row0 + j, tok_full(b));
                }
            }
            for (int j = it - kTokStages < 0 ? 0 : it - kTokStages; j < it; ++j)
                mbar_drain(tok_full(j % kTokStages), (uint32_t)(j / kTokStages) & 1u, p.hdr);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        // (per-stage work kept short: a non-blocking test of each barrier before the bounded
        // wait, ring positions kept as counters, descriptors advanced by adding to their address
        // field: start >> 4, +2 per 16 K of a K-major tile, + the stage's offset >> 4)
        if (lane == 0) {
            const uint64_t ad0 = kmajor_desc(base + kHfOff, 0), bd0 = kmajor_desc(base + kTokOff, 0);
            int b = 0, tb = 0, tc = 0;
            uint32_t hph = 0, tph = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++tc) {
                if (!mbar_wait(acc_empty, ((uint32_t)tc & 1u) ^ 1u, p.hdr, abort_flag)) break;
                tc_fence_after();
                const uint32_t idesc = idesc_n(tile_of(t).n16);
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
        // ---------------- converters: row c of each weight block ----------------
        const int c = threadIdx.x - 192;
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
                uint8_t* hf = smem + kHfOff + b * kABytes;
                convert_row(rw, hf, c);
                convert_row(rw + kWR * kRawRow, hf + kWR * 128, c);
                fence_proxy_async_smem();  // each thread's stores -> the MMA's async proxy
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(raw_empty(r));
                    mbar_arrive(hf_full(b));
                }
            }
        }
    } else {
        // ---------------- epilogue (warps 2..5): thread = weight row 32q + lane of each block ----------------
        // The tokens' values go into a table per warp (every entry rewritten each tile: tokens
        // past the tile's own get slot -1), read while the tile's MMAs still run; the token of
        // column tt is then a broadcast read of the table.
        const int q = warp & 3;
        int* w_src = reinterpret_cast<int*>(smem + kTabOff) + q * 4 * kTokMax;
        float* w_g = reinterpret_cast<float*>(w_src + kTokMax);
        float* w_s = w_g + kTokMax;                            // s^X or s^A
        int* w_sum8 = reinterpret_cast<int*>(w_s + kTokMax);   // 8 * code sum
        int tc = 0;
        const bool leader = q == 0 && lane == 0;
        bool all_q = false;  // (the leader's) fused launch: every job of the launch seen finished
        bool drained = false;  // (the leader's) fused launch: every job of the launch taken
        for (int t = blockIdx.x; t < total; t += gridDim.x, ++tc) {
            const Tile tl = tile_of(t);
            const bool l1 = is_l1(t), sec = second(t);
            bool dep_ok = true;
            if (sec) {
                // s^A and the code sums of the chunk's rows come from their re-quantisation in this
                // launch (jobs run meanwhile); the loads below follow the leader's acquire through
                // the barrier
                dep_ok = idle_with_jobs<kEpiBar, kQuantRegVec, false>(qq, p, job_word, abort_flag, &drained, q, lane, [&] {
                    if (!all_q) all_q = ld_acquire_gpu(qq.jobs_done) >= qq.n_jobs;
                    return all_q || chunk_ready(tl);
                });
            }
            const float* row_scale = sec ? args.row_scale2 : args.row_scale;
            const int32_t* row_sums = sec ? args.row_sums2 : args.row_sums;
            {
                // every load of the table in flight at once (rows beyond the tile read row0's
                // values, which are discarded), then the dependent gate loads, then the stores
                constexpr int kC = kTokMax / 32;
                int src[kC];
                uint32_t sv[kC], sm[kC];
#pragma unroll
                for (int i = 0; i < kC; ++i) {
                    const int n = 32 * i + lane;
                    const int64_t row = tl.row0 + (n < tl.n16 ? n : 0);
                    src[i] = (!l1 && n < tl.n_valid) ? __ldg(p.pool_src + row) : -1;
                    sv[i] = sec ? ld_relaxed_gpu(row_scale + row) : __float_as_uint(__ldg(row_scale + row));
                    sm[i] = sec ? ld_relaxed_gpu(row_sums + row) : (uint32_t)__ldg(row_sums + row);
                }
                float g[kC];
#pragma unroll
                for (int i = 0; i < kC; ++i) {
                    src[i] = src[i] >= 0 ? debug_row(p.hdr, src[i], (int64_t)p.T * p.K) : -1;
                    g[i] = src[i] >= 0 ? __ldg(args.topk_weights + src[i]) : 0.0f;
                }
#pragma unroll
                for (int i = 0; i < kC; ++i) {
                    const int n = 32 * i + lane;
                    const bool in = n < tl.n16;  // rows of the tile's route tiles
                    w_src[n] = src[i];
                    w_g[n] = g[i];
                    w_s[n] = in ? __uint_as_float(sv[i]) : 0.0f;
                    w_sum8[n] = in ? (int)(8u * sm[i]) : 0;
                }
            }
            __syncwarp();
            float sw0, sw1;  // per-channel weight scales of this thread's rows in the two blocks
            if (l1) {
                const float* s1 = args.w_scale + (int64_t)tl.e * 2 * I + tl.s * kWR + q * 32 + lane;
                sw0 = __ldg(s1);      // gate
                sw1 = __ldg(s1 + I);  // up
            } else {
                const float* s2 = (sec ? args.w_scale2 : args.w_scale) + (int64_t)tl.e * H + tl.s * 2 * kWR + q * 32 + lane;
                sw0 = __ldg(s2);
                sw1 = __ldg(s2 + kWR);
            }
            if (kFused && dep_ok)  // a re-quantisation job while this tile's MMAs run, if there is one
                dep_ok = idle_with_jobs<kEpiBar, kQuantRegVec, true>(qq, p, job_word, abort_flag, &drained, q, lane,
                                                                     [&] { return mbar_test(acc_full, (uint32_t)tc & 1u); });
            const bool w_ok = dep_ok && mbar_wait(acc_full, (uint32_t)tc & 1u, p.hdr, abort_flag);
            if (!bar_all128<kEpiBar>(w_ok)) break;  // one decision for the four warps (they share kEpiBar)
            tc_fence_after();
            const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16);
            if (l1) {
                // H = (C * s^W1) * s^X; A[token, j] = SiLU(H_gate) * H_up for output j
                const int j = tl.s * kWR + q * 32 + lane;
#pragma unroll 1
                for (int c0 = 0; c0 < tl.n16; c0 += 32) {  // uniform across the warp
                    uint32_t g[32], u[32];
                    tmem_ld32(tb + c0, g);
                    tmem_ld32(tb + 256 + c0, u);
                    tmem_ld_wait();
#pragma unroll
                    for (int tt = 0; tt < 32; ++tt) {
                        const int n = c0 + tt;
                        const float sx = w_s[n];
                        const int s8 = w_sum8[n];
                        const float Hg = __fmul_rn(__fmul_rn(exact_c(g[tt], s8), sw0), sx);
                        const float Hu = __fmul_rn(__fmul_rn(exact_c(u[tt], s8), sw1), sx);
                        if (n < tl.n_valid)  // uniform across the warp
                            p.a_f32[(int64_t)(tl.row0 + n) * I + j] = swiglu1(Hg, Hu, p.act_clamp);
                    }
                }
            } else {
                // Y = (D * s^W2) * s^A; c = bf16(G * Y) to the combine row of the token
#pragma unroll 1
                for (int c0 = 0; c0 < tl.n_valid; c0 += 32) {  // uniform across the warp
#pragma unroll
                    for (int blk = 0; blk < 2; ++blk) {
                        const int h = tl.s * 2 * kWR + blk * kWR + q * 32 + lane;
                        const float sw = blk ? sw1 : sw0;
                        uint32_t d[32];
                        tmem_ld32(tb + blk * 256 + c0, d);
                        tmem_ld_wait();
#pragma unroll
                        for (int tt = 0; tt < 32; ++tt) {  // slot < 0 past the routed rows
                            const int n = c0 + tt;
                            const int src = w_src[n];
                            const float y = __fmul_rn(__fmul_rn(exact_c(d[tt], w_sum8[n]), sw), w_s[n]);
                            st_global_u16_if(src >= 0, p.comb + (int64_t)(src >= 0 ? src : 0) * H + h,
                                             float_to_bf16_bits(__fmul_rn(w_g[n], y)));
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty);
            if (kFused && l1) {
                // The accumulator is free for the next tile. Publish this tile's rows of A (one or
                // two route tiles): every thread fences its own stores, the four warps meet, the
                // leader counts the tile for each route tile; a route tile's last L1 tile queues its
                // re-quantisation jobs (whole rows of A are needed), which any CTA's epilogue runs.
                const int g = tl.row0 / kRouteRows;
                const int n_rt = tl.n_valid > kRouteRows ? 2 : 1;
                __threadfence();
                bar_sync128<kEpiBar>();
                if (leader) {
                    __threadfence();
                    for (int h = 0; h < n_rt; ++h)
                        if (atomicAdd(qq.dep + g + h, 1) == args.n_slabs - 1) {
                            __threadfence();
                            qq.push(g + h);
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

template <int kKind>
cudaError_t set_w4_wm_smem_attr() {
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(tc_w4_wm_kernel<kKind>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
    });
    return attr_err;
}

// packed weights as bytes [E * n_out, kin / 2] in boxes of 128 rows x 32 bytes; the f16 token
// plane (x for L1, A for L2) in 128-row boxes and 16-row boxes for a tile's ragged end
bool make_w4_wm_maps(const Plan& p, const void* w, bool l1, CUtensorMap* tmW, CUtensorMap* tmX, CUtensorMap* tmX16) {
    const int n_out = l1 ? 2 * p.I : p.H;
    const int kin = l1 ? p.H : p.I;
    const uint16_t* planes = l1 ? p.x_planes : p.a_planes;
    return tc_make_map_2d(tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, w, (uint64_t)kin / 2, (uint64_t)p.E * n_out, kRawRow,
                          kWR, CU_TENSOR_MAP_SWIZZLE_32B) &&
           tc_make_map_2d(tmX, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, planes, (uint64_t)kin, (uint64_t)p.pool_rows, kBK,
                          kRouteRows, CU_TENSOR_MAP_SWIZZLE_128B) &&
           tc_make_map_2d(tmX16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, planes, (uint64_t)kin, (uint64_t)p.pool_rows, kBK,
                          kTokBox, CU_TENSOR_MAP_SWIZZLE_128B);
}

// at most (route tiles + experts) / 2 token chunks per weight slab
int64_t max_chunks(const Plan& p) { return (p.pool_rows / kRouteRows + p.E) / 2 + 1; }

template <bool kIsL1>
cudaError_t launch_w4_wm(const Plan& p, const void* w, const void* w_scale, const float* topk_weights,
                         cudaStream_t s) {
    constexpr int kKind = kIsL1 ? kL1 : kL2;
    const cudaError_t attr_err = set_w4_wm_smem_attr<kKind>();
    if (attr_err != cudaSuccess) return attr_err;
    CUtensorMap tmW, tmX, tmX16;
    if (!make_w4_wm_maps(p, w, kIsL1, &tmW, &tmX, &tmX16)) return cudaErrorInvalidValue;
    W4WmArgs args{};
    args.p = p;
    args.w_scale = static_cast<const float*>(w_scale);
    args.topk_weights = topk_weights;
    args.row_scale = reinterpret_cast<const float*>(kIsL1 ? p.x_pool_scale : p.a_pool_scale);
    args.row_sums = kIsL1 ? p.x_sums : p.a_sums;
    args.n_slabs = kIsL1 ? p.I / kWR : p.H / (2 * kWR);
    args.k_blocks = (kIsL1 ? p.H : p.I) / kBK;
    args.n_out = kIsL1 ? 2 * p.I : p.H;
    const int64_t max_tiles = max_chunks(p) * args.n_slabs;
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(max_tiles, tc_num_sms()));
    tc_w4_wm_kernel<kKind><<<grid, kThreads, kSmem, s>>>(tmW, tmX, tmX16, tmW, tmX, tmX16, args);
    return cudaGetLastError();
}

// L1 then L2 in one cooperative launch: every CTA is resident, so an L2 tile waits (bounded) only
// on L1 tiles and re-quantisations that earlier positions of the same round-robin order hold
cudaError_t launch_w4_wm_fused(const Plan& p, const void* w1, const void* w1_scale, const void* w2,
                               const void* w2_scale, const float* topk_weights, cudaStream_t s) {
    cudaError_t e = set_w4_wm_smem_attr<kFusedL1L2>();
    if (e != cudaSuccess) return e;
    CUtensorMap tmW1, tmX1, tmX16_1, tmW2, tmX2, tmX16_2;
    if (!make_w4_wm_maps(p, w1, true, &tmW1, &tmX1, &tmX16_1) || !make_w4_wm_maps(p, w2, false, &tmW2, &tmX2, &tmX16_2))
        return cudaErrorInvalidValue;
    const int64_t route_tiles = p.pool_rows / kRouteRows;
    // the counters (one per route tile, then the job queue's) start at zero every launch
    if ((e = cudaMemsetAsync(p.ffn_counters, 0, sizeof(int32_t) * (size_t)fused_int_counters(route_tiles), s)) !=
        cudaSuccess)
        return e;
    W4WmArgs args{};
    args.p = p;
    args.w_scale = static_cast<const float*>(w1_scale);
    args.topk_weights = topk_weights;
    args.row_scale = reinterpret_cast<const float*>(p.x_pool_scale);
    args.row_sums = p.x_sums;
    args.n_slabs = p.I / kWR;
    args.k_blocks = p.H / kBK;
    args.n_out = 2 * p.I;
    args.w_scale2 = static_cast<const float*>(w2_scale);
    args.row_scale2 = reinterpret_cast<const float*>(p.a_pool_scale);
    args.row_sums2 = p.a_sums;
    args.n_slabs2 = p.H / (2 * kWR);
    args.k_blocks2 = p.I / kBK;
    args.ctr = p.ffn_counters;
    int per_sm = 0;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, tc_w4_wm_kernel<kFusedL1L2>, kThreads, kSmem)) !=
        cudaSuccess)
        return e;
    if (per_sm < 1) return cudaErrorCooperativeLaunchTooLarge;
    const int64_t max_tiles = max_chunks(p) * (args.n_slabs + args.n_slabs2);
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(max_tiles, (int64_t)tc_num_sms() * per_sm));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, tc_w4_wm_kernel<kFusedL1L2>, tmW1, tmX1, tmX16_1, tmW2, tmX2, tmX16_2, args);
}

}  // namespace

// Weight-major tiles pay off when there are enough of them: experts x weight slabs (a lower
// bound on the tiles of the experts that have rows) of at least four rounds on the GPU.
bool w4_wm_preferred(const Plan& p, int stage) {
    const int64_t slabs = stage == 1 ? p.I / kWR : p.H / (2 * kWR);
    return (int64_t)p.E * slabs >= 4 * (int64_t)tc_num_sms();
}

bool w4_wm_supported(const Plan& p, int stage) {
    if (p.mode != MOE_A8W4_INT || p.E > kMaxExperts || !tc_encode_available()) return false;
    if (stage == 1) return p.I % kWR == 0 && p.H % kBK == 0 && p.H <= kMaxK;
    return p.H % (2 * kWR) == 0 && p.I % kBK == 0 && p.I <= kMaxK;
}

cudaError_t launch_l1_w4_wm(const Plan& p, const void* w1, const void* w1_scale, cudaStream_t s) {
    return launch_w4_wm<true>(p, w1, w1_scale, nullptr, s);
}

cudaError_t launch_l2_w4_wm(const Plan& p, const void* w2, const void* w2_scale, const float* topk_weights,
                            cudaStream_t s) {
    return launch_w4_wm<false>(p, w2, w2_scale, topk_weights, s);
}

cudaError_t launch_ffn_fused_w4_wm(const Plan& p, const void* w1, const void* w1_scale, const void* w2,
                                   const void* w2_scale, const float* topk_weights, cudaStream_t s) {
    return launch_w4_wm_fused(p, w1, w1_scale, w2, w2_scale, topk_weights, s);
}

}  // namespace moe
