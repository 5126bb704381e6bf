// Block-scaled grouped GEMM for the FP8 modes at prefill sizes on CTA pairs (A8W8-FP8: e4m3 or
// e5m2 weights; FP8 x FP4: e2m1 weights; FP8 tokens), on tcgen05.mma.cta_group::2.kind::
// mxf8f6f4.block_scale: one UE8M0 scale per 32 elements of K applied to each operand by the
// tensor cores (the Ascend mega_moe page, A8W8-FP use case: the MX dequantisation happens within
// the matrix multiply; DeepGEMM page §4 step 5: L1 on 2-CTA block-scaled MMAs).
//
// Weight-major pair tiles: M = 256 weight rows, 128 in each CTA of a cluster of two; N = up to
// 192 tokens of one expert (rounded up to 16), each CTA staging half of them; K = 128 per stage.
// Per SM and stage that is 16 KB of weights (e2m1 takes a byte per code in the MMA's operand
// layout) and 12 KB of tokens for 128 x 192 x 128 MACs: 18.7 KB per 128^3 against 24 KB for the
// single-CTA token-major tile (128 tokens x 256 weight rows), and shared-memory fill by TMA is what
// bounds that tile; six stages keep 168 KB in flight per SM (the fill rate is the bytes in flight
// over a load latency of 1.5-2.5 us). Tokens are the N side, so an expert's last tile is padded to 16
// tokens, not to 128 rows.
// - L1: the pair's 256 rows are the gate and up rows of 128 outputs; CTA c holds the 64 gate and 64
//   up rows of outputs [128 s + 64 c, +64), so its epilogue pairs lane r (gate) with lane r + 64
//   (up) through shared memory, applies SwiGLU (Ascend page, "SwiGLU Activation") and the MX FP8
//   re-quantisation of A (one exponent per 32 outputs).
// - L2: 256 hidden columns per pair tile; the epilogue scales token n's value by its gate weight
//   and stores the bf16 combine row element of (token, slot).
//
// Scale factors (measured on this GPU with a probe kept out of the product): each CTA's half of the
// pair MMA reads the scale of its A row r (a weight row) from its own tensor memory, lane r,
// column slot + r/32, and the scale of B column n (a token) from its own tensor memory too, lane
// 32q + n%32 of the lane quarter q of the output row, column slot + 4 + n/32, for every n of the
// tile: both CTAs hold the token scales of all N columns. Weight and token scale words come by
// TMA in blocks of 4 K atoms (16 bytes of every row) two blocks ahead of their use; four warps per
// CTA move them into tensor memory.
//
// Synchronisation (as in the bf16 pair kernel):
//   full[s]   (even CTA): both CTAs' TMA loads of stage s complete on it (the even CTA's producer
//             arrives with both CTAs' byte count) and the four scale-writer warps of each CTA arrive
//             on it when the stage's scale words are in tensor memory (the odd CTA's without a
//             release fence, see mbar_arrive_cluster_relaxed);
//   empty[s]  (each CTA): the MMA commit arrives on both CTAs' barriers;
//   acc_full[a] (each CTA): commit to both; acc_empty[a] (even CTA): the four epilogue warps of
//             both CTAs.
// Warp roles (320 threads per CTA): 0 TMA producer, 1 tensor-memory allocation (both) + MMA issue
// (even CTA), 2-5 epilogue, 6-9 scale writers. Every wait is bounded; on time-out the CTA records
// MOE_ERR_TIMEOUT and leaves its loops; both CTAs meet at a cluster barrier before tensor memory is
// freed.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "tc_common.cuh"

namespace moe {

namespace {

using namespace tc;

constexpr int kHM = 128;      // weight rows per CTA (the pair MMA has M = 256)
constexpr int kHalf = 64;     // L1: a CTA's gate rows, then its up rows
constexpr int kNT = 192;      // tokens per tile at most (MMA N)
constexpr int kHT = kNT / 2;  // token rows staged per CTA
constexpr int kAtomK = 128;   // K per stage: one 128-byte swizzle atom
constexpr int kStages = 6;
constexpr int kThreads = 320;
constexpr int kMaxExperts = 1024;
constexpr int kABytes = kHM * 128;           // 16 KB
constexpr int kBBytes = kHT * 128;           // 14 KB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kTokBox = 16;                  // token rows per TMA box of a partial tile
constexpr int kSfBlk = 4;                    // K atoms per scale block (16 bytes of a row)
constexpr int kSfBufs = 4;
constexpr int kSfWBytes = kHM * 16;          // weight scale words of a block: [128 rows][4 atoms]
constexpr int kSfTBytes = kNT * 16;          // token scale words of a block: [kNT rows][4 atoms]
constexpr int kSfCol0 = 2 * kNT;             // two 192-column accumulators, then the scale ring
constexpr int kSfColsPerStage = 16;          // A word in columns 0-3, token words in 4..9
constexpr int kEpiBar = 1;                   // named barrier of the 4 epilogue warps
constexpr int kSfOff = kStages * kStageBytes;
constexpr int kBarOff = kSfOff + kSfBufs * (kSfWBytes + kSfTBytes);
constexpr int kNumBars = 2 * kStages + 4 + 1 + 2 * kSfBufs;
constexpr int kXbufOff = kBarOff + 8 * kNumBars;  // L1: 2 x 16 tokens x 64 outputs fp32; L2: slot/gate tables
constexpr int kXbufBytes = 4 * 2 * kNT * 4 > 2 * 16 * kHalf * 4 ? 4 * 2 * kNT * 4 : 2 * 16 * kHalf * 4;
constexpr int kMiscOff = kXbufOff + kXbufBytes;
constexpr int kTileOffOff = kMiscOff + 16;
constexpr int kSubOffOff = kTileOffOff + 4 * (kMaxExperts + 1);
constexpr int kCountsOff = kSubOffOff + 4 * (kMaxExperts + 1);
constexpr size_t kSmem = 1024 + (size_t)kCountsOff + 4 * kMaxExperts;
static_assert(kSmem <= 232448, "shared memory");
static_assert(kSfCol0 + kStages * kSfColsPerStage <= 512, "tensor memory");
static_assert(4 + (kNT + 31) / 32 <= kSfColsPerStage, "scale slot");

struct PairBsArgs {
    Plan p;
    const float* topk_weights;  // L2
    int n_slabs;                // pair slabs per expert: L1 I / 128, L2 H / 256
    int k_blocks;               // K / 128
    int kin;
};

struct Tile {
    int e, s, row0, n_valid;
};

// Tiles are ordered expert-major, then weight slab, then token sub-tile, so consecutive clusters
// read the same weight slab (from L2 after the first) while its tokens change.
__device__ __forceinline__ Tile decode(int t, const int* sub_off, const int* tile_off, const int* counts, int E,
                                       int n_slabs) {
    int lo = 0, hi = E - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (sub_off[mid] * n_slabs <= t) lo = mid; else hi = mid - 1;
    }
    Tile tl;
    tl.e = lo;
    const int ns = sub_off[lo + 1] - sub_off[lo];
    const int local = t - sub_off[lo] * n_slabs;
    tl.s = local / ns;
    const int j = local % ns;
    tl.row0 = tile_off[lo] * 128 + j * kNT;
    tl.n_valid = min(kNT, counts[lo] - j * kNT);
    return tl;
}

// kind::mxf8f6f4.block_scale instruction descriptor: B scale id (bits 4-5), A type (7-9: the
// weights, e4m3 0, e5m2 1, e2m1 5), B type (10-12: the tokens), both K-major, N >> 3 (17-22), UE8M0
// scales (bit 23), M >> 4 (24-28: M = 256), A scale id (29-30).
__device__ __forceinline__ uint32_t pair_idesc(uint32_t afmt, uint32_t bfmt, int n, int sf_id) {
    return ((uint32_t)sf_id << 4) | (afmt << 7) | (bfmt << 10) | ((uint32_t)(n >> 3) << 17) | (1u << 23) |
           ((uint32_t)(256 >> 4) << 24) | ((uint32_t)sf_id << 29);
}

__device__ __forceinline__ void tc2_mma_bs(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t sfa,
                                           uint32_t sfb, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
        ::"r"(d), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
        "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}

// Arrive on the even CTA's barrier (given by its shared::cluster address) without a release fence.
// The scale writers use it after tcgen05.wait::st, which already blocks until their tensor-memory
// writes are complete, so no ordering is left for a fence to provide; a cluster-scope release fence
// per stage and warp stalled the writers (~2000 cycles a stage, measured) and with them the MMA.
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync %0, 128;" ::"n"(kEpiBar) : "memory"); }
// The same barrier, ANDing `pred` over the four epilogue warps: they leave the tile loop together.
__device__ __forceinline__ bool epi_all(bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.b32 p, %1, 0;\n\tbar.red.and.pred q, %2, 128, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((int)pred), "n"(kEpiBar)
        : "memory");
    return r != 0;
}

// token rows a CTA stages for a tile of n tokens (N = n rounded up to 16, half of it per CTA): the
// whole 112-row box for a full tile, else 16-row boxes
__device__ __forceinline__ int staged_rows(int n_valid) {
    const int half = ((n_valid + 15) & ~15) >> 1;
    return n_valid == kNT ? kHT : (half + kTokBox - 1) / kTokBox * kTokBox;
}

template <int MODE, bool kL1>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    tc_bs_pair_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                      const __grid_constant__ CUtensorMap tmX16, const __grid_constant__ CUtensorMap tmSW,
                      const __grid_constant__ CUtensorMap tmSX, PairBsArgs args) {
    constexpr bool kFp4 = MODE == MOE_A8W4_FP8_FP4;
    constexpr bool kE5 = MODE == MOE_A8W8_FP8_E5M2;
    constexpr uint32_t kBfmt = kE5 ? 1u : 0u;         // tokens (and A of L2)
    constexpr uint32_t kAfmt = kFp4 ? 5u : kBfmt;     // weights
    constexpr uint32_t kATx = kFp4 ? kHM * kAtomK / 2 : kHM * kAtomK;  // TMA counts the packed global bytes
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = smem_u32(smem_raw);
    const uint32_t base = (raw_base + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (base - raw_base);
    const uint32_t bars = base + kBarOff;
    auto full_bar = [&](int s) { return bars + 8u * s; };
    auto empty_bar = [&](int s) { return bars + 8u * (kStages + s); };
    auto acc_full = [&](int a) { return bars + 8u * (2 * kStages + a); };
    auto acc_empty = [&](int a) { return bars + 8u * (2 * kStages + 2 + a); };
    const uint32_t drain_bar = bars + 8u * (2 * kStages + 4);
    auto sf_full = [&](int b) { return bars + 8u * (2 * kStages + 5 + b); };
    auto sf_empty = [&](int b) { return bars + 8u * (2 * kStages + 5 + kSfBufs + b); };
    float* xbuf = reinterpret_cast<float*>(smem + kXbufOff);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + kMiscOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kMiscOff + 4);
    int* tile_off = reinterpret_cast<int*>(smem + kTileOffOff);
    int* sub_off = reinterpret_cast<int*>(smem + kSubOffOff);
    int* counts = reinterpret_cast<int*>(smem + kCountsOff);

    const Plan& p = args.p;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool even = rank == 0;
    const int cluster = (int)cluster_id_x(), clusters = (int)cluster_count_x();
    for (int i = threadIdx.x; i <= p.E; i += kThreads) tile_off[i] = p.tile_off[i];
    for (int i = threadIdx.x; i < p.E; i += kThreads) counts[i] = p.counts[i];
    if (warp == 0) {
        // sub-tiles of kNT tokens per expert, exclusive prefix over the experts
        int carry = 0;
        for (int b = 0; b < p.E; b += 32) {
            const int e = b + lane;
            const int v = e < p.E ? (p.counts[e] + kNT - 1) / kNT : 0;
            int x = v;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, x, d);
                if (lane >= d) x += y;
            }
            if (e < p.E) sub_off[e] = carry + x - v;
            carry += __shfl_sync(0xffffffffu, x, 31);
        }
        if (lane == 0) sub_off[p.E] = carry;
    }
    if (threadIdx.x == 32) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full_bar(s), 1 + 8);  // even producer (arrive + both CTAs' bytes) + 4 scale warps per CTA
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(acc_full(a), 1);
            mbar_init(acc_empty(a), 8);  // four epilogue warps in each CTA
        }
        mbar_init(drain_bar, 1);
        for (int b = 0; b < kSfBufs; ++b) {
            mbar_init(sf_full(b), 1);   // this CTA's producer (arrive + bytes)
            mbar_init(sf_empty(b), 4);  // this CTA's scale writers
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) tmem_alloc_pair(smem_u32(tmem_holder), 512);  // one warp of each CTA, together
    if (warp == 0 && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmW)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmX)) : "memory");
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // both CTAs' barriers are initialised before either signals the other's
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    const int total = sub_off[p.E] * args.n_slabs;
    const int KB = args.k_blocks;
    const int I = p.I, H = p.H;
    auto tile_of = [&](int t) { return decode(t, sub_off, tile_off, counts, p.E, args.n_slabs); };
    // first weight row of this CTA in the 2-D view of the weights (L2), or its 64-row block (L1)
    auto wblock = [&](const Tile& tl) { return kL1 ? 2 * tl.s + (int)rank : tl.e * H + tl.s * 256 + (int)rank * kHM; };

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer (each CTA: its weight rows, its half of the tokens) ----------------
            const int n_sfb = (KB + kSfBlk - 1) / kSfBlk;
            int st_t = cluster, st_b = 0, sj = 0;
            Tile st_tl = tile_of(st_t < total ? st_t : 0);
            bool ok = true;
            auto issue_scales = [&]() {  // the next scale block of this CTA, if any
                if (st_t >= total || !ok) return;
                const int buf = sj % kSfBufs;
                if (!mbar_wait(sf_empty(buf), ((uint32_t)(sj / kSfBufs) & 1u) ^ 1u, p.hdr, abort_flag)) {
                    ok = false;
                    return;
                }
                const uint32_t dw = base + kSfOff + buf * (kSfWBytes + kSfTBytes), dt = dw + kSfWBytes;
                mbar_arrive_expect_tx(sf_full(buf), (uint32_t)(kSfWBytes + kSfTBytes));
                const int xw = st_b * kSfBlk * 4;  // byte offset of the block within a row's scales
                if constexpr (kL1)
                    tma_load_4d(dw, &tmSW, xw, wblock(st_tl) * kHalf, 0, st_tl.e, sf_full(buf));
                else
                    tma_load_2d(dw, &tmSW, xw, wblock(st_tl), sf_full(buf));
                // the token scales of all the tile's columns (each CTA's half of the MMA reads them all)
                tma_load_2d(dt, &tmSX, kL1 && kFp4 ? st_b * kSfBlk : xw, st_tl.row0, sf_full(buf));
                ++sj;
                if (++st_b == n_sfb) {
                    st_b = 0;
                    st_t += clusters;
                    if (st_t < total) st_tl = tile_of(st_t);
                }
            };
            issue_scales();
            issue_scales();
            int it = 0;
            for (int t = cluster; t < total && ok; t += clusters) {
                const Tile tl = tile_of(t);
                const int half = ((tl.n_valid + 15) & ~15) >> 1;  // tokens per CTA
                const int rows = staged_rows(tl.n_valid);
                const int trow = tl.row0 + (int)rank * half;
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    const int s = it % kStages;
                    if (!ok || !mbar_wait(empty_bar(s), ((uint32_t)(it / kStages) & 1u) ^ 1u, p.hdr, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = base + s * kStageBytes, sb = sa + kABytes;
                    const uint32_t fb = mapa_shared(full_bar(s), 0);
                    if (even) mbar_arrive_expect_tx(full_bar(s), 2u * (kATx + (uint32_t)rows * 128u));
                    const int x = kb * kAtomK;
                    if constexpr (kL1)
                        tma_load_4d_pair(sa, &tmW, x, wblock(tl) * kHalf, 0, tl.e, fb);
                    else
                        tma_load_2d_pair(sa, &tmW, x, wblock(tl), fb);
                    if (rows == kHT)
                        tma_load_2d_pair(sb, &tmX, x, trow, fb);
                    else
                        for (int j = 0; j < rows; j += kTokBox) tma_load_2d_pair(sb + j * 128, &tmX16, x, trow + j, fb);
                    // after the stage's operands, which the MMA waits for first: the scale block
                    // two ahead of the one this stage starts
                    if (kb % kSfBlk == 0) issue_scales();
                }
            }
            // drain (bounded): the even CTA's stages (both halves' bytes land there), each CTA's scale blocks
            if (even)
                for (int j = it - kStages < 0 ? 0 : it - kStages; j < it; ++j)
                    if (!mbar_drain(full_bar(j % kStages), (uint32_t)(j / kStages) & 1u, p.hdr)) break;
            for (int j = sj - kSfBufs < 0 ? 0 : sj - kSfBufs; j < sj; ++j)
                mbar_drain(sf_full(j % kSfBufs), (uint32_t)(j / kSfBufs) & 1u, p.hdr);
        }
    } else if (warp == 1) {
        if (lane == 0 && even) {
            // ---------------- MMA issuer (even CTA) ----------------
            const uint64_t ad0 = kmajor_desc(base, 0), bd0 = kmajor_desc(base + kABytes, 0);
            int s = 0, tc = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int t = cluster; t < total && ok; t += clusters, ++tc) {
                const int a = tc & 1;
                if (!mbar_wait(acc_empty(a), ((uint32_t)(tc >> 1) & 1u) ^ 1u, p.hdr, abort_flag)) break;
                tc_fence_after();
                const Tile tl = tile_of(t);
                const int n = (tl.n_valid + 15) & ~15;
                uint32_t idesc[kAtomK / 32];
#pragma unroll
                for (int kk = 0; kk < kAtomK / 32; ++kk) idesc[kk] = pair_idesc(kAfmt, kBfmt, n, kk);
                const uint32_t d = tmem_base + (uint32_t)(a * kNT);
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
                        tc2_mma_bs(d, ad0 + so + 2 * kk, bd0 + so + 2 * kk, idesc[kk], sf, sf + 4, (kb | kk) != 0);
                    tc2_commit_mc(empty_bar(s), 0x3);  // both CTAs may refill stage s
                    if (++s == kStages) s = 0, ph ^= 1u;
                }
                if (ok) tc2_commit_mc(acc_full(a), 0x3);
            }
            // drain: every MMA issued so far has completed before tensor memory is freed
            tc2_commit_mc(drain_bar, 0x1);
            mbar_drain(drain_bar, 0, p.hdr);
        }
    } else if (warp >= 6) {
        // ---------------- scale writers (each CTA) ----------------
        // Lane l of warp q writes tensor-memory lane 32q + l of this CTA: the A word of weight row
        // r = 32q + l (columns 0-3 of the slot; the MMA reads column q in lane quarter q) and the
        // words of tokens 32c + l, c < 7 (columns 4 + c), every token of the tile in both CTAs.
        const int q = warp & 3;
        const int r = 32 * q + lane;
        int it = 0, sj = 0;
        bool ok = true;
        for (int t = cluster; t < total && ok; t += clusters) {
            const Tile tl = tile_of(t);
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
                    uint32_t v[16];
                    const uint32_t wa = sw[r * kSfBlk + i];
#pragma unroll
                    for (int c = 0; c < 4; ++c) v[c] = wa;
#pragma unroll
                    for (int c = 0; c < 12; ++c) {
                        const int n = 32 * c + lane;
                        uint32_t tw = 0x7f7f7f7fu;  // 1.0 for the padding tokens
                        if (c < kNT / 32 && n < tl.n_valid) {
                            tw = sx[n * kSfBlk + i];
                            if constexpr (kL1 && kFp4) tw = ((tw >> 23) & 0xffu) * 0x01010101u;  // power-of-two fp32 scale
                        }
                        v[4 + c] = tw;
                    }
                    tmem_st16(tmem_base + ((uint32_t)(32 * q) << 16) + kSfCol0 + s * kSfColsPerStage, v);
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        if (even) mbar_arrive(full_bar(s));
                        else mbar_arrive_cluster_relaxed(mapa_shared(full_bar(s), 0));
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(sf_empty(buf));
                ++sj;
            }
        }
    } else {
        // ---------------- epilogue (warps 2..5, each CTA) ----------------
        const int q = warp & 3;
        int tc = 0;
        for (int t = cluster; t < total; t += clusters, ++tc) {
            const int a = tc & 1;
            const Tile tl = tile_of(t);
            const int n = (tl.n_valid + 15) & ~15;
            if constexpr (!kL1) {
                // the tokens' combine slots and gate weights as a per-warp table, read while the
                // tile's MMAs run (broadcast reads below, no dependency chain through the stores)
                int* w_src = reinterpret_cast<int*>(xbuf) + q * 2 * kNT;
                float* w_g = reinterpret_cast<float*>(w_src + kNT);
#pragma unroll
                for (int ci = 0; ci < kNT / 32; ++ci) {
                    const int nn = 32 * ci + lane;
                    const int src = nn < tl.n_valid ? debug_row(p.hdr, __ldg(p.pool_src + tl.row0 + nn), (int64_t)p.T * p.K) : -1;
                    w_src[nn] = src;
                    w_g[nn] = src >= 0 ? __ldg(args.topk_weights + src) : 0.0f;
                }
                __syncwarp();
            }
            const bool w_ok = mbar_wait(acc_full(a), (uint32_t)(tc >> 1) & 1u, p.hdr, abort_flag);
            if (!epi_all(w_ok)) break;  // one decision for the four warps (they share epi_sync)
            tc_fence_after();
            const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(a * kNT);
            if constexpr (kL1) {
                // lanes 0-63 hold the gate rows and lanes 64-127 the up rows of this CTA's 64 outputs.
                // Of each 32-token chunk the gate warps finish tokens 0-15 and the up warps tokens
                // 16-31; each hands its partner the other half through xbuf.
                const bool gate = q < 2;
                const int jl = 32 * (q & 1) + lane;  // output within this CTA's 64
                const int j = tl.s * 128 + (int)rank * kHalf + jl;
                float* xg = xbuf;               // [16 tokens][64 outputs]: gate values of tokens 16-31
                float* xu = xbuf + 16 * kHalf;  // [16 tokens][64 outputs]: up values of tokens 0-15
                for (int c0 = 0; c0 < n; c0 += 32) {
                    uint32_t v[32];
                    tmem_ld32(tb + c0, v);
                    tmem_ld_wait();
                    if (gate) {
#pragma unroll
                        for (int tt = 0; tt < 16; ++tt) xg[tt * kHalf + jl] = __uint_as_float(v[16 + tt]);
                    } else {
#pragma unroll
                        for (int tt = 0; tt < 16; ++tt) xu[tt * kHalf + jl] = __uint_as_float(v[tt]);
                    }
                    epi_sync();
                    // n is a multiple of 16: a warp's 16 tokens are all below n or all above
                    if (gate || c0 + 16 < n) {
                        const int64_t row0 = tl.row0 + c0 + (gate ? 0 : 16);
                        const int nv = tl.n_valid - (c0 + (gate ? 0 : 16));  // routed tokens among these 16
                        uint32_t my_sc = 0;  // lane tt keeps the UE8M0 byte of token tt
#pragma unroll
                        for (int tt = 0; tt < 16; ++tt) {
                            const float gv = gate ? __uint_as_float(v[tt]) : xg[tt * kHalf + jl];
                            const float uv = gate ? xu[tt * kHalf + jl] : __uint_as_float(v[16 + tt]);
                            const float av = swiglu1(gv, uv, p.act_clamp);
                            const float amax = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(av))));
                            const int ex = mx_exponent_fp8<kE5>(amax);
                            st_global_u8_if(tt < nv, p.a_pool + (row0 + tt) * I + j,
                                            float_to_fp8_satfinite<kE5>(av * exp2_neg_int(ex)));
                            my_sc = lane == tt ? (uint32_t)(ex + 127) : my_sc;
                        }
                        st_global_u8_if(lane < 16 && lane < nv, p.a_pool_scale + (row0 + lane) * (I / 32) + (j >> 5),
                                        (uint8_t)my_sc);
                    }
                    epi_sync();
                }
            } else {
                const int h = tl.s * 256 + (int)rank * kHM + q * 32 + lane;
                const int* w_src = reinterpret_cast<const int*>(xbuf) + q * 2 * kNT;
                const float* w_g = reinterpret_cast<const float*>(w_src + kNT);
                for (int c0 = 0; c0 < tl.n_valid; c0 += 32) {
                    uint32_t y[32];
                    tmem_ld32(tb + c0, y);
                    tmem_ld_wait();
#pragma unroll
                    for (int tt = 0; tt < 32; ++tt) {  // slot < 0 past the routed tokens
                        const int src = w_src[min(c0 + tt, kNT - 1)];
                        st_global_u16_if(src >= 0 && c0 + tt < tl.n_valid, p.comb + (int64_t)(src >= 0 ? src : 0) * H + h,
                                         float_to_bf16_bits(__fmul_rn(w_g[min(c0 + tt, kNT - 1)], __uint_as_float(y[tt]))));
                    }
                }
                __syncwarp();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(mapa_shared(acc_empty(a), 0));
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();  // no CTA frees tensor memory or exits while its pair still uses it
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem_base, 512);
}

// Clusters of the kernel that can be resident at once (a pair needs two free SMs of one GPC).
template <int MODE, bool kL1>
int resident_clusters() {
    static std::once_flag once;
    static int n = 0;
    std::call_once(once, [] {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * std::max(1, tc_num_sms() / 2));
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = kSmem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, tc_bs_pair_kernel<MODE, kL1>, &cfg) != cudaSuccess || n < 1) {
            (void)cudaGetLastError();
            n = std::max(1, tc_num_sms() / 2);
        }
    });
    return n;
}

template <int MODE, bool kL1>
cudaError_t launch_bs_pair_t(const Plan& p, const void* w, const void* w_scale, const float* topk_weights,
                             cudaStream_t s) {
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(tc_bs_pair_kernel<MODE, kL1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)kSmem);
    });
    if (attr_err != cudaSuccess) return attr_err;
    const int n_out = kL1 ? 2 * p.I : p.H;
    const int kin = kL1 ? p.H : p.I;
    constexpr bool kFp4 = MODE == MOE_A8W4_FP8_FP4;
    const CUtensorMapDataType wtype = kFp4 ? CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    const uint64_t pitch = kFp4 ? (uint64_t)kin / 2 : (uint64_t)kin;  // bytes per weight row
    CUtensorMap tmW, tmX, tmX16, tmSW, tmSX;
    bool ok;
    const uint64_t sp = (uint64_t)kin / 32;  // scale bytes per weight row
    if (kL1) {
        // [K][row within the gate or up half][half][expert]: one box holds a CTA's 64 gate and 64 up rows
        const uint64_t dims[4] = {(uint64_t)kin, (uint64_t)p.I, 2, (uint64_t)p.E};
        const uint64_t strides[3] = {pitch, pitch * p.I, pitch * 2 * p.I};
        const uint32_t box[4] = {kAtomK, kHalf, 2, 1};
        ok = tc_make_map_nd(&tmW, wtype, 4, w, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
        const uint64_t sdims[4] = {sp, (uint64_t)p.I, 2, (uint64_t)p.E};
        const uint64_t sstrides[3] = {sp, sp * p.I, sp * 2 * p.I};
        const uint32_t sbox[4] = {16, kHalf, 2, 1};
        ok = ok && tc_make_map_nd(&tmSW, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, w_scale, sdims, sstrides, sbox,
                                  CU_TENSOR_MAP_SWIZZLE_NONE);
    } else {
        const uint64_t dims[2] = {(uint64_t)kin, (uint64_t)p.E * n_out};
        const uint64_t strides[1] = {pitch};
        const uint32_t box[2] = {kAtomK, kHM};
        ok = tc_make_map_nd(&tmW, wtype, 2, w, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
        const uint64_t sdims[2] = {sp, (uint64_t)p.E * n_out};
        const uint64_t sstrides[1] = {sp};
        const uint32_t sbox[2] = {16, kHM};
        ok = ok && tc_make_map_nd(&tmSW, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, w_scale, sdims, sstrides, sbox,
                                  CU_TENSOR_MAP_SWIZZLE_NONE);
    }
    const void* xs = kL1 ? (const void*)p.x_pool : (const void*)p.a_pool;
    ok = ok && tc_make_map_2d(&tmX, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, xs, (uint64_t)kin, (uint64_t)p.pool_rows, kAtomK,
                              kHT, CU_TENSOR_MAP_SWIZZLE_128B);
    ok = ok && tc_make_map_2d(&tmX16, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, xs, (uint64_t)kin, (uint64_t)p.pool_rows,
                              kAtomK, kTokBox, CU_TENSOR_MAP_SWIZZLE_128B);
    if (kL1 && kFp4) {  // fp32 per 128 elements of a token row
        const uint64_t dims[2] = {(uint64_t)kin / 128, (uint64_t)p.pool_rows};
        const uint64_t strides[1] = {(uint64_t)kin / 128 * 4};
        const uint32_t box[2] = {4, kNT};
        ok = ok && tc_make_map_nd(&tmSX, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, p.x_pool_scale, dims, strides, box,
                                  CU_TENSOR_MAP_SWIZZLE_NONE);
    } else {  // UE8M0 per 32 elements
        const uint64_t dims[2] = {sp, (uint64_t)p.pool_rows};
        const uint64_t strides[1] = {sp};
        const uint32_t box[2] = {16, kNT};
        ok = ok && tc_make_map_nd(&tmSX, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                                  kL1 ? (const void*)p.x_pool_scale : (const void*)p.a_pool_scale, dims, strides, box,
                                  CU_TENSOR_MAP_SWIZZLE_NONE);
    }
    if (!ok) return cudaErrorInvalidValue;
    PairBsArgs args{p, topk_weights, kL1 ? p.I / 128 : p.H / 256, kin / kAtomK, kin};
    // at most one tile per kNT routed rows plus one per expert, per slab
    const int64_t max_tiles = ((int64_t)p.T * p.K / kNT + p.E + 1) * args.n_slabs;
    const int clusters = (int)std::max<int64_t>(1, std::min<int64_t>(max_tiles, resident_clusters<MODE, kL1>()));
    tc_bs_pair_kernel<MODE, kL1><<<2 * clusters, kThreads, kSmem, s>>>(tmW, tmX, tmX16, tmSW, tmSX, args);
    return cudaGetLastError();
}

}  // namespace

bool bs_pair_supported(const Plan& p, int stage) {
    if ((p.mode != MOE_A8W8_FP8 && p.mode != MOE_A8W8_FP8_E5M2 && p.mode != MOE_A8W4_FP8_FP4) ||
        p.E > kMaxExperts || !tc_encode_available() || tc_num_sms() < 2)
        return false;
    // scale rows by TMA: their byte pitch (K / 32, and K / 32 for the fp32 per-128 token scales) must be
    // a multiple of 16
    if (stage == 1) return p.I % 128 == 0 && p.H % 512 == 0;
    return p.H % 256 == 0 && p.I % 512 == 0;
}

cudaError_t launch_l1_bs_pair(const Plan& p, const void* w1, const void* w1_scale, cudaStream_t s) {
    if (p.mode == MOE_A8W4_FP8_FP4) return launch_bs_pair_t<MOE_A8W4_FP8_FP4, true>(p, w1, w1_scale, nullptr, s);
    if (p.mode == MOE_A8W8_FP8) return launch_bs_pair_t<MOE_A8W8_FP8, true>(p, w1, w1_scale, nullptr, s);
    if (p.mode == MOE_A8W8_FP8_E5M2) return launch_bs_pair_t<MOE_A8W8_FP8_E5M2, true>(p, w1, w1_scale, nullptr, s);
    return cudaErrorNotSupported;
}

cudaError_t launch_l2_bs_pair(const Plan& p, const void* w2, const void* w2_scale, const float* topk_weights,
                              cudaStream_t s) {
    if (p.mode == MOE_A8W4_FP8_FP4) return launch_bs_pair_t<MOE_A8W4_FP8_FP4, false>(p, w2, w2_scale, topk_weights, s);
    if (p.mode == MOE_A8W8_FP8) return launch_bs_pair_t<MOE_A8W8_FP8, false>(p, w2, w2_scale, topk_weights, s);
    if (p.mode == MOE_A8W8_FP8_E5M2) return launch_bs_pair_t<MOE_A8W8_FP8_E5M2, false>(p, w2, w2_scale, topk_weights, s);
    return cudaErrorNotSupported;
}

}  // namespace moe
