// Token-major block-scaled grouped GEMM for the FP8 modes at prefill sizes (A8W8-FP8: e4m3
// weights, A8W4: e2m1 weights; e4m3 tokens), on tcgen05.mma kind::mxf8f6f4.block_scale with
// one UE8M0 scale per 32 elements of K applied by the tensor core (the Ascend mega_moe page,
// A8W8-FP use case, "DQ_MX ... implicitly performed inside matmul"; DeepGEMM page, section 4,
// step 5: block-scaled MMA with UE8M0 scale factors in tensor memory).
//
// Tile: M = 128 pool rows (one 128-row route tile of an expert) x N = 256 weight rows, K = 128
// per stage (MMAs of K = 32):
// - L1: the 128 gate rows and the 128 up rows of outputs [128s, 128s + 128) (one 4-D TMA box),
//   so a thread of the epilogue holds its token's gate and up values of the same outputs and
//   applies SwiGLU (Ascend page, "SwiGLU Activation") and the MX FP8 re-quantisation of A (one
//   exponent per 32 outputs) without any exchange between threads;
// - L2: 256 hidden columns; the epilogue scales the token's row by G and writes its bf16
//   combine row (Ascend page, "Token Combine") with 16-byte stores.
// Why this shape: these GEMMs are bound by how fast TMA fills shared memory (about 55-68 bytes
// per clock per SM measured on this GPU with 192 KB in flight). Per 128-K stage a tile takes
// 16 KB of tokens and 32 KB of weights (e2m1 occupies a byte per code in the MMA's 4-bit
// layout) for 128 x 256 x 128 MACs: 24 KB per 128^3, where 128 weight rows x 128 tokens take
// 32 KB. The price is a single-buffered accumulator: two 256-column accumulators fill the
// 512 TMEM columns and leave none for the scale factors. The epilogue releases it as soon as
// its last columns are loaded into registers.
//
// TMEM: accumulator in columns 0-255; scale factors in a ring of 16-column slots from column
// 256, one per stage. Layout the MMA reads (measured on this GPU, M = 128): the scale word of A
// row r (a token) in lane r, column slot + r/32; the scale word of B row n (a weight row) in
// lane 32*q + n%32 of every lane quarter q, column slot + 4 + n/32; byte k of a word is the
// scale of K group k of the stage.
//
// Warp roles (320 threads): 0 TMA producer, 1 TMEM allocation + MMA issuer, 2-5 epilogue (warp
// w owns TMEM lanes 32*(w%4) .. +31, i.e. those token rows), 6-9 scale writers. Every wait is
// bounded; on time-out the CTA records MOE_ERR_TIMEOUT, drains and exits.
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
constexpr int kWN = 256;          // weight rows per tile (MMA N)
constexpr int kAtomK = 128;       // K per stage: one 128-byte swizzle atom of e4m3 / expanded e2m1
constexpr int kStages = 4;
constexpr int kThreads = 320;
constexpr int kMaxExperts = 1024;
constexpr int kTokBytes = kTM * 128;                 // 16 KB
constexpr int kWBytes = kWN * 128;                   // 32 KB in shared memory
constexpr int kStageBytes = kTokBytes + kWBytes;
constexpr int kSfCol0 = 256;
constexpr int kSfColsPerStage = 16;  // SFA 4 columns, SFB 8 columns
constexpr int kNumBars = 2 * kStages + 2 + 1 + 2;  // full, empty, acc full/empty, drain, 2 weight-scale buffers
constexpr int kBarOff = kStages * kStageBytes;
constexpr int kMiscOff = kBarOff + 8 * kNumBars;
constexpr int kTileOffOff = kMiscOff + 16;
constexpr int kCountsOff = kTileOffOff + 4 * (kMaxExperts + 1);
constexpr int kWsfOff = (kCountsOff + 4 * kMaxExperts + 15) & ~15;  // u32 [2][8 groups][8 atoms][32 lanes]
constexpr size_t kSmem = 1024 + (size_t)kWsfOff + 2 * 8 * 8 * 32 * 4;
static_assert(kSmem <= 232448, "shared memory");
static_assert(kSfCol0 + kStages * kSfColsPerStage <= 512, "tensor memory");

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

// kind::mxf8f6f4.block_scale instruction descriptor: B scale id (bits 4-5), A type (7-9: e4m3
// tokens = 0), B type (10-12: e4m3 = 0, e2m1 = 5), both K-major, N >> 3 (17-22), UE8M0 scales
// (bit 23), M >> 4 (24-28), A scale id (29-30).
__device__ __forceinline__ uint32_t tm_idesc(uint32_t bfmt, int sf_id) {
    return ((uint32_t)sf_id << 4) | (0u << 7) | (bfmt << 10) | ((uint32_t)(kWN >> 3) << 17) | (1u << 23) |
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

// predicated 16-byte global store (no memory clobber: independent loads may move across it)
__device__ __forceinline__ void st_global_v4_if(bool pred, void* ptr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %0, 0;\n\t@p st.global.v4.b32 [%1], {%2, %3, %4, %5};\n\t}" ::"r"(
                     (int)pred),
                 "l"(ptr), "r"(a), "r"(b), "r"(c), "r"(d));
}

// two floats -> two e4m3 codes (RN, saturating), the first in the low byte
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    uint16_t pair;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(pair) : "f"(hi), "f"(lo));
    return pair;
}

template <int MODE, bool kL1>
__global__ void __launch_bounds__(kThreads, 1)
    tc_bs_tm_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX, TmArgs args) {
    constexpr bool kFp4 = MODE == MOE_A8W4_FP8_FP4;
    constexpr uint32_t kBfmt = kFp4 ? 5u : 0u;
    constexpr uint32_t kWTx = kFp4 ? kWN * kAtomK / 2 : kWN * kAtomK;  // TMA counts the packed global bytes
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = smem_u32(smem_raw);
    const uint32_t base = (raw_base + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (base - raw_base);
    const uint32_t bars = base + kBarOff;
    auto full_bar = [&](int s) { return bars + 8u * s; };
    auto empty_bar = [&](int s) { return bars + 8u * (kStages + s); };
    const uint32_t acc_full = bars + 8u * (2 * kStages);
    const uint32_t acc_empty = acc_full + 8u;
    const uint32_t drain_bar = acc_full + 16u;
    auto wsf_bar = [&](int b) { return bars + 8u * (2 * kStages + 3 + b); };
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + kMiscOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kMiscOff + 4);
    int* tile_off = reinterpret_cast<int*>(smem + kTileOffOff);
    int* counts = reinterpret_cast<int*>(smem + kCountsOff);
    uint32_t* wsf = reinterpret_cast<uint32_t*>(smem + kWsfOff);

    const Plan& p = args.p;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i <= p.E; i += kThreads) tile_off[i] = p.tile_off[i];
    for (int i = threadIdx.x; i < p.E; i += kThreads) counts[i] = p.counts[i];
    if (threadIdx.x == 32) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full_bar(s), 1 + 4);  // TMA (arrive + bytes) + the 4 scale-writer warps
            mbar_init(empty_bar(s), 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, 4);
        mbar_init(drain_bar, 1);
        for (int b = 0; b < 2; ++b) mbar_init(wsf_bar(b), 4);
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
            int it = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const Tile tl = tile_of(t);
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    const int s = it % kStages;
                    if (!mbar_wait(empty_bar(s), ((uint32_t)(it / kStages) & 1u) ^ 1u, p.hdr, abort_flag)) {
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
                }
            }
            for (int j = it - kStages < 0 ? 0 : it - kStages; j < it; ++j)
                mbar_drain(full_bar(j % kStages), (uint32_t)(j / kStages) & 1u, p.hdr);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            int it = 0, tc = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++tc) {
                if (!mbar_wait(acc_empty, ((uint32_t)tc & 1u) ^ 1u, p.hdr, abort_flag)) break;
                tc_fence_after();
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    const int s = it % kStages;
                    if (!mbar_wait(full_bar(s), (uint32_t)(it / kStages) & 1u, p.hdr, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = base + s * kStageBytes, sb = sa + kTokBytes;
                    const uint32_t sf = tmem_base + kSfCol0 + s * kSfColsPerStage;
#pragma unroll
                    for (int kk = 0; kk < kAtomK / 32; ++kk)
                        tm_mma(tmem_base, kmajor_desc(sa, kk), kmajor_desc(sb, kk), tm_idesc(kBfmt, kk), sf, sf + 4,
                               (kb | kk) != 0);
                    tc_commit(empty_bar(s));
                }
                if (ok) tc_commit(acc_full);
            }
            tc_commit(drain_bar);
            mbar_drain(drain_bar, 0, p.hdr);
        }
    } else if (warp >= 6) {
        // ---------------- scale writers ----------------
        // Lane l of warp q owns token row r = 32q + l (its A scale) and loads the weight rows
        // 32c + l for c = 2q, 2q+1; the B scales are needed in every lane quarter, so each warp
        // publishes its two groups through shared memory (an mbarrier per buffer). Scale words
        // (one per row and 128-element K atom) are read 8 atoms at a time, so a lane's 32 bytes
        // fill one sector, and two blocks ahead of their use; the loaded words are only
        // converted when the block is written out, so the loads stay in flight.
        const int q = warp & 3;
        const int r = 32 * q + lane;
        const int spr = args.kin / 32;
        const int n_words = args.kin / kAtomK;
        const int n_blk = (n_words + 7) >> 3;
        struct Blk {
            uint32_t a[8], w0[8], w1[8];
            bool tok_valid;
        };
        auto load_blk = [&](int t, int blk) {
            Blk w;
            const Tile tl = tile_of(t);
            w.tok_valid = r < tl.n_valid;
            const int64_t row = tl.row0 + r;  // a pool row of the route tile
            const uint32_t* ws0 = reinterpret_cast<const uint32_t*>(args.w_scale + (int64_t)wrow(tl, 64 * q + lane) * spr);
            const uint32_t* ws1 =
                reinterpret_cast<const uint32_t*>(args.w_scale + (int64_t)wrow(tl, 64 * q + 32 + lane) * spr);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int g = min(blk * 8 + i, n_words - 1);  // K atom: elements 128g .. 128g+127
                if constexpr (kL1 && kFp4)
                    w.a[i] = __float_as_uint(__ldg(reinterpret_cast<const float*>(p.x_pool_scale) + row * (H / 128) + g));
                else if constexpr (kL1)
                    w.a[i] = __ldg(reinterpret_cast<const uint32_t*>(p.x_pool_scale + row * (H / 32)) + g);
                else
                    w.a[i] = __ldg(reinterpret_cast<const uint32_t*>(p.a_pool_scale + row * (I / 32)) + g);
                w.w0[i] = __ldg(ws0 + g);
                w.w1[i] = __ldg(ws1 + g);
            }
            return w;
        };
        // token word as the MMA reads it: 4 UE8M0 bytes; 1.0 for the padding rows
        auto tok_word = [&](const Blk& w, uint32_t raw) -> uint32_t {
            if (!w.tok_valid) return 0x7f7f7f7fu;
            if constexpr (kL1 && kFp4) return ((raw >> 23) & 0xffu) * 0x01010101u;  // power-of-two fp32 scale
            return raw;
        };
        auto next_pos = [&](int& t, int& blk) {
            if (++blk == n_blk) {
                blk = 0;
                t += gridDim.x;
            }
        };
        int t0 = blockIdx.x, b0 = 0, t1 = t0, b1 = b0;
        next_pos(t1, b1);
        int t2 = t1, b2 = b1;
        int it = 0, nb = 0;  // stages and blocks done
        bool ok = true;
        // writes out block (t0, b0) from `use` after starting the loads of block (t2, b2) into
        // `fill`; the three buffers rotate by name, so no register holding a load in flight is copied
        auto run_block = [&](const Blk& use, Blk& fill) -> bool {
            if (t0 >= total || !ok) return false;
            next_pos(t2, b2);
            if (t2 < total) fill = load_blk(t2, b2);
            const int buf = nb & 1;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                wsf[((buf * 8 + 2 * q) * 8 + i) * 32 + lane] = use.w0[i];
                wsf[((buf * 8 + 2 * q + 1) * 8 + i) * 32 + lane] = use.w1[i];
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(wsf_bar(buf));
            const bool b_ok = mbar_wait(wsf_bar(buf), (uint32_t)(nb >> 1) & 1u, p.hdr, abort_flag);
            if (!__all_sync(0xffffffffu, b_ok)) return ok = false;
            // working copy of the token words (loaded a block ago), shifted one per stage so the
            // rolled loop below indexes registers statically
            uint32_t ta[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) ta[i] = tok_word(use, use.a[i]);
#pragma unroll 1
            for (int i = 0; i < 8; ++i) {
                const int kb = b0 * 8 + i;
                if (kb >= KB) break;  // uniform across the CTA's scale warps
                const int s = it % kStages;
                const bool w_ok = mbar_wait(empty_bar(s), ((uint32_t)(it / kStages) & 1u) ^ 1u, p.hdr, abort_flag);
                if (!__all_sync(0xffffffffu, w_ok)) return ok = false;
                // slot columns: 0-3 the A word (the MMA reads column q of lane quarter q), 4-11
                // the B words of weight rows 32c + lane, 12-15 unused
                uint32_t v[16];
#pragma unroll
                for (int c = 0; c < 4; ++c) v[c] = ta[0];
#pragma unroll
                for (int c = 0; c < 8; ++c) v[4 + c] = wsf[((buf * 8 + c) * 8 + i) * 32 + lane];
#pragma unroll
                for (int c = 12; c < 16; ++c) v[c] = 0x7f7f7f7fu;
                tmem_st16(tmem_base + ((uint32_t)(32 * q) << 16) + kSfCol0 + s * kSfColsPerStage, v);
#pragma unroll
                for (int j = 0; j < 7; ++j) ta[j] = ta[j + 1];
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(full_bar(s));
                ++it;
            }
            t0 = t1;
            b0 = b1;
            t1 = t2;
            b1 = b2;
            ++nb;
            return true;
        };
        Blk A{}, B{}, C{};
        if (t0 < total) A = load_blk(t0, b0);
        if (t1 < total) B = load_blk(t1, b1);
        while (run_block(A, C) && run_block(B, A) && run_block(C, B)) {
        }
    } else {
        // ---------------- epilogue (warps 2..5): thread = token row ----------------
        const int q = warp & 3;
        const int r = 32 * q + lane;
        const uint32_t tb = tmem_base + ((uint32_t)(32 * q) << 16);
        int tc = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x, ++tc) {
            const Tile tl = tile_of(t);
            const bool valid = r < tl.n_valid;
            const int64_t row = tl.row0 + r;
            // L2: this row's combine slot and gate weight, read while the tile's MMAs run
            int src = -1;
            float gw = 0.0f;
            if constexpr (!kL1) {
                src = valid ? __ldg(p.pool_src + row) : -1;
                gw = src >= 0 ? __ldg(args.topk_weights + src) : 0.0f;
            }
            const bool w_ok = mbar_wait(acc_full, (uint32_t)tc & 1u, p.hdr, abort_flag);
            if (!__all_sync(0xffffffffu, w_ok)) break;
            tc_fence_after();
            auto release = [&]() {  // every column of the accumulator is in registers
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(acc_empty);
            };
            if constexpr (kL1) {
                // A = SiLU(gate) * up for outputs 128s + 32c .. +31, then MX FP8: one UE8M0
                // exponent per 32 outputs of the token, 32 codes as two 16-byte stores
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    uint32_t g[32], u[32];
                    tmem_ld32(tb + 32 * c, g);
                    tmem_ld32(tb + 128 + 32 * c, u);
                    tmem_ld_wait();
                    if (c == 3) release();
                    float av[32];
                    float amax = 0.0f;
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj) {
                        av[jj] = silu(__uint_as_float(g[jj])) * __uint_as_float(u[jj]);
                        amax = fmaxf(amax, fabsf(av[jj]));
                    }
                    const int ex = mx_exponent_e4m3(amax);
                    const float inv = exp2_neg_int(ex);
                    uint32_t w[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        w[k] = e4m3x2(av[4 * k] * inv, av[4 * k + 1] * inv) |
                               (e4m3x2(av[4 * k + 2] * inv, av[4 * k + 3] * inv) << 16);
                    const int j0 = tl.s * 128 + 32 * c;
                    uint8_t* dst = p.a_pool + row * I + j0;
                    st_global_v4_if(valid, dst, w[0], w[1], w[2], w[3]);
                    st_global_v4_if(valid, dst + 16, w[4], w[5], w[6], w[7]);
                    st_global_u8_if(valid, p.a_pool_scale + row * (I / 32) + (j0 >> 5), (uint8_t)(ex + 127));
                }
            } else {
                // c = bf16(G * y) for hidden columns 256s + 32c .. +31: 64 bytes of the combine row
#pragma unroll 1
                for (int c = 0; c < 8; ++c) {
                    uint32_t y[32];
                    tmem_ld32(tb + 32 * c, y);
                    tmem_ld_wait();
                    if (c == 7) release();
                    uint32_t w[16];
#pragma unroll
                    for (int k = 0; k < 16; ++k)
                        w[k] = (uint32_t)float_to_bf16_bits(__fmul_rn(gw, __uint_as_float(y[2 * k]))) |
                               ((uint32_t)float_to_bf16_bits(__fmul_rn(gw, __uint_as_float(y[2 * k + 1]))) << 16);
                    uint16_t* dst = p.comb + (int64_t)(src >= 0 ? src : 0) * H + tl.s * kWN + 32 * c;
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        st_global_v4_if(src >= 0, dst + 8 * k, w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, 512);
}

template <int MODE, bool kL1>
cudaError_t launch_tm(const Plan& p, const void* w, const void* w_scale, const float* topk_weights, cudaStream_t s) {
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(tc_bs_tm_kernel<MODE, kL1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
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
    TmArgs args{p, static_cast<const uint8_t*>(w_scale), topk_weights, kL1 ? p.I / 128 : p.H / kWN, kin / kAtomK, n_out,
                kin};
    const int64_t max_tiles = std::max<int64_t>(1, (p.pool_rows / kTM) * args.n_slabs);
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(max_tiles, tc_num_sms()));
    tc_bs_tm_kernel<MODE, kL1><<<grid, kThreads, kSmem, s>>>(tmW, tmX, args);
    return cudaGetLastError();
}

}  // namespace

bool bs_tm_supported(const Plan& p, int stage) {
    if ((p.mode != MOE_A8W8_FP8 && p.mode != MOE_A8W4_FP8_FP4) || p.E > kMaxExperts || !tc_encode_available())
        return false;
    if (stage == 1) return p.I % 128 == 0 && p.H % kAtomK == 0;
    return p.H % kWN == 0 && p.I % kAtomK == 0;
}

cudaError_t launch_l1_bs_tm(const Plan& p, const void* w1, const void* w1_scale, cudaStream_t s) {
    if (p.mode == MOE_A8W4_FP8_FP4) return launch_tm<MOE_A8W4_FP8_FP4, true>(p, w1, w1_scale, nullptr, s);
    if (p.mode == MOE_A8W8_FP8) return launch_tm<MOE_A8W8_FP8, true>(p, w1, w1_scale, nullptr, s);
    return cudaErrorNotSupported;
}

cudaError_t launch_l2_bs_tm(const Plan& p, const void* w2, const void* w2_scale, const float* topk_weights,
                            cudaStream_t s) {
    if (p.mode == MOE_A8W4_FP8_FP4) return launch_tm<MOE_A8W4_FP8_FP4, false>(p, w2, w2_scale, topk_weights, s);
    if (p.mode == MOE_A8W8_FP8) return launch_tm<MOE_A8W8_FP8, false>(p, w2, w2_scale, topk_weights, s);
    return cudaErrorNotSupported;
}

}  // namespace moe
