// Block-scaled weight-major tensor-core grouped GEMM for the FP8 modes (A8W8-FP8: e4m3 weights,
// A8W4: e2m1 weights; e4m3 tokens in both), on tcgen05.mma kind::mxf8f6f4.block_scale: the
// tensor core consumes the stored codes and applies one UE8M0 scale per 32 elements of K to
// each operand, so nothing is dequantised in software (the Ascend mega_moe page, A8W8-FP use
// case: the MX dequantisation happens within the matrix multiply; DeepGEMM page §4 step 5:
// block-scaled MMA with UE8M0 scale factors in tensor memory).
//
// Tiles (M = 128 weight rows, N = tokens, K = 128 or 256 per stage, MMAs of K = 32):
// - L1: the 128 rows are 64 gate rows and the 64 up rows of the same 64 outputs of A, so the
//   epilogue pairs lane r (gate) with lane r + 64 (up) through a small shared buffer and applies
//   SwiGLU (Ascend page, "SwiGLU Activation") and the MX FP8 re-quantisation of A.
// - L2: 128 rows of hidden columns.
// - tokens: a sub-tile of kNT rows of one expert: kNT = 128 with K = 128 stages for
//   prefill-sized experts; kNT = 16 with K = 256 stages for decode-sized ones, where the weights
//   stream from HBM and each load should cover whole 128-byte lines. The sub-tiles of every
//   expert are counted in-kernel from the routed-row counts.
// Accumulators are double-buffered in tensor memory, so the epilogue of a tile overlaps the
// main loop of the next.
//
// Operand staging: weights by TMA with 128-byte swizzle (e2m1 through the 16U4_ALIGN16B element
// type, which expands each packed 8-byte group of 16 codes into a 16-byte slot: the 4-bit
// operand layout of kind::mxf8f6f4; its transaction count is the packed size), one copy per K
// atom for all 128 rows (L1: a 4-D box [K][64 rows][gate, up][expert]); tokens by one TMA copy
// per K atom of the sub-tile's kNT pool rows (e4m3 codes; rows past the sub-tile feed no MMA
// column); scales by four "scale warps" that write the stage's UE8M0 bytes into tensor memory
// with one tcgen05.st per K atom. Each TMA instruction costs the producer about 75 cycles to
// issue (measured), so a stage is moved in as few copies as the layout allows. Layout the MMA reads (measured on this GPU):
// the scale of A row r is in TMEM lane r, column base + r/32, byte = the K group (a_sf_id); the
// scale of B row n is in lane 32*q + n%32 of every lane quarter q, column base + n/32, byte =
// b_sf_id; one 32-bit word holds a row's 4 scales of a stage.
//
// Warp roles (320 threads): 0 TMA producer, 1 TMEM allocation + MMA issuer, 2-5 epilogue,
// 6-9 scale writers. Every wait is bounded; on time-out the CTA records MOE_ERR_TIMEOUT, drains
// and exits.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "tc_common.cuh"

namespace moe {

namespace {

using namespace tc;

constexpr int kWR = 128;          // weight rows per tile (MMA M)
constexpr int kHalf = 64;         // L1: gate rows, then up rows
constexpr int kAtomK = 128;       // K of one 128-byte swizzle atom (a stage holds kAtoms of them)
constexpr int kThreads = 320;
constexpr int kMaxExperts = 1024;
constexpr int kABytes = kWR * 128;
constexpr int kSfCol0 = 256;      // first TMEM column of the scale ring
constexpr int kSfColsPerStage = 16;  // per K atom: SFA 4 columns, SFB up to 4 columns
constexpr int kEpiBar = 1;        // named barrier of the 4 epilogue warps

template <int kNT, int kStages, int kAtoms>
struct BsCfg {
    static constexpr int kBBytes = kNT * 128;                          // one K atom of tokens
    static constexpr int kStageBytes = kAtoms * (kABytes + kBBytes);   // [A atoms][B atoms]
    static constexpr int kBarOff = kStages * kStageBytes;
    static constexpr int kNumBars = 2 * kStages + 4 + 1 + 2;  // + two token-scale buffers
    static constexpr int kXbufOff = kBarOff + 8 * kNumBars;           // 2 x 16 tokens x 64 outputs (fp32)
    static constexpr int kMiscOff = kXbufOff + 32 * kHalf * 4;
    static constexpr int kTileOffOff = kMiscOff + 16;                 // int[E+1] 128-row tiles per expert
    static constexpr int kSubOffOff = kTileOffOff + 4 * (kMaxExperts + 1);   // int[E+1] kNT sub-tiles
    static constexpr int kCountsOff = kSubOffOff + 4 * (kMaxExperts + 1);    // int[E]
    static constexpr int kTokWords = kNT < 32 ? 1 : kNT / 32;                 // token scale words per lane
    static constexpr int kTokSfOff = (kCountsOff + 4 * kMaxExperts + 15) & ~15;  // u32[2][kTokWords][8][32]
    static constexpr size_t kSmem = 1024 + (size_t)kTokSfOff + 2 * kTokWords * 8 * 32 * 4;
    static_assert(kSmem <= 232448, "shared memory");
    static_assert(2 * kNT <= kSfCol0 && kSfCol0 + kStages * kSfColsPerStage <= 512, "tensor memory");
    static_assert(kAtoms == 1 || kAtoms == 2, "atoms per stage");
};

struct BsArgs {
    Plan p;
    const uint8_t* w_scale;     // UE8M0 [E*n_out][kin/32]
    const float* topk_weights;  // L2
    int n_slabs, k_blocks, n_out, kin;  // k_blocks = stages per tile; the last may hold one atom
    // the fused launch (L1 then L2 in one launch): the fields above describe its L1, these its L2
    const uint8_t* w_scale2;
    int n_slabs2, k_blocks2, n_out2, kin2;
    int32_t* l1_done;           // finished L1 tiles per 128-row route tile (zeroed before the launch)
    int32_t* l1_total;          // finished L1 tiles of the whole launch (zeroed before the launch)
};

constexpr int kL2 = 0, kL1 = 1, kFusedL1L2 = 2;  // what one launch runs

struct Tile {
    int e, s, row0, n_valid;
};

// Tiles are ordered expert-major, then weight slab, then token sub-tile.
template <int kNT>
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

// Instruction descriptor of kind::mxf8f6f4.block_scale: B scale-factor id (bits 4-5), A and B
// element types (7-9, 10-12: e4m3 = 0, e5m2 = 1, e2m1 = 5), both K-major, N >> 3 (17-22), scale
// type UE8M0 (bit 23), M >> 4 (24-28), A scale-factor id (29-30).
__device__ __forceinline__ uint32_t bs_idesc(uint32_t afmt, uint32_t bfmt, int n, int sf_id) {
    return ((uint32_t)sf_id << 4) | (afmt << 7) | (bfmt << 10) | ((uint32_t)(n >> 3) << 17) | (1u << 23) |
           ((uint32_t)(kWR >> 4) << 24) | ((uint32_t)sf_id << 29);
}

__device__ __forceinline__ void tc_mma_bs(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t sfa,
                                          uint32_t sfb, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
        ::"r"(d), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
        : "memory");
}

// 8 consecutive columns of the warp's 32 lanes, one 32-bit word per lane and column
__device__ __forceinline__ void tmem_st8(uint32_t taddr, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t a4,
                                         uint32_t a5, uint32_t a6, uint32_t a7) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr), "r"(a0),
                 "r"(a1), "r"(a2), "r"(a3), "r"(a4), "r"(a5), "r"(a6), "r"(a7)
                 : "memory");
}
__device__ __forceinline__ void epi_sync() { bar_sync128<kEpiBar>(); }
// The same barrier, ANDing `pred` over the four epilogue warps: they leave the tile loop together,
// since a warp that left alone would keep the others waiting at the next epi_sync.
__device__ __forceinline__ bool epi_all(bool pred) { return bar_all128<kEpiBar>(pred); }

template <int MODE, int kKind, int kNT, int kStages, int kAtoms>
__global__ void __launch_bounds__(kThreads, 1)
    tc_bs_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                 const __grid_constant__ CUtensorMap tmW2, const __grid_constant__ CUtensorMap tmX2, BsArgs args) {
    using Cfg = BsCfg<kNT, kStages, kAtoms>;
    constexpr bool kFused = kKind == kFusedL1L2;
    constexpr int kBK = kAtoms * kAtomK;  // K per stage
    constexpr bool kFp4 = MODE == MOE_A8W4_FP8_FP4;
    constexpr bool kE5 = MODE == MOE_A8W8_FP8_E5M2;  // e5m2 weights, tokens and A
    constexpr uint32_t kBfmt = kE5 ? 1u : 0u;
    constexpr uint32_t kAfmt = kFp4 ? 5u : kBfmt;
    constexpr uint32_t kABoxTx = kFp4 ? kHalf * kAtomK / 2 : kHalf * kAtomK;  // TMA counts the packed global bytes
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
    auto tok_bar = [&](int b) { return bars + 8u * (2 * kStages + 5 + b); };
    float* xbuf = reinterpret_cast<float*>(smem + Cfg::kXbufOff);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + Cfg::kMiscOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::kMiscOff + 4);
    int* tile_off = reinterpret_cast<int*>(smem + Cfg::kTileOffOff);
    int* sub_off = reinterpret_cast<int*>(smem + Cfg::kSubOffOff);
    int* counts = reinterpret_cast<int*>(smem + Cfg::kCountsOff);

    const Plan& p = args.p;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
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
            mbar_init(full_bar(s), 1 + 4);  // TMA (arrive + bytes) + the 4 scale-writer warps
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(acc_full(a), 1);
            mbar_init(acc_empty(a), 4);
        }
        mbar_init(drain_bar, 1);
        for (int b = 0; b < 2; ++b) mbar_init(tok_bar(b), 4);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_holder), 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    // tiles [0, total1) are the launch's first stage (L1 when fused), [total1, total) the L2 ones
    const int total1 = sub_off[p.E] * args.n_slabs;
    const int total = kFused ? total1 + sub_off[p.E] * args.n_slabs2 : total1;
    const int I = p.I, H = p.H;
    auto is_l1 = [&](int t) { return kKind == kL1 || (kFused && t < total1); };
    auto second = [&](int t) { return kFused && t >= total1; };  // an L2 tile of the fused launch
    auto tile_of = [&](int t) {
        return second(t) ? decode<kNT>(t - total1, sub_off, tile_off, counts, p.E, args.n_slabs2)
                         : decode<kNT>(t, sub_off, tile_off, counts, p.E, args.n_slabs);
    };
    auto kin_of = [&](int t) { return second(t) ? args.kin2 : args.kin; };
    auto kb_of = [&](int t) { return second(t) ? args.k_blocks2 : args.k_blocks; };
    auto atoms_of = [&](int kb, int kin) { return min(kAtoms, (kin - kb * kBK) / kAtomK); };
    // first global weight row of each 64-row half of the tile
    auto wrow = [&](const Tile& tl, int half, bool l1, int n_out) {
        if (l1) return tl.e * n_out + (half ? I : 0) + tl.s * kHalf;
        return tl.e * n_out + tl.s * kWR + half * kHalf;
    };
    auto nout_of = [&](int t) { return second(t) ? args.n_out2 : args.n_out; };
    // fused launch: the route-tile counter an L2 tile of sub-tile row row0 waits on, and its target
    // (every L1 weight slab of every sub-tile of that route tile)
    auto dep_of = [&](const Tile& tl, int* target) {
        const int m = (tl.row0 - tile_off[tl.e] * 128) / 128;
        const int rows = min(128, counts[tl.e] - m * 128);
        *target = (rows + kNT - 1) / kNT * args.n_slabs;
        return args.l1_done + tile_off[tl.e] + m;
    };

    if (warp == 0) {
        // ---------------- TMA producer: weights (two 64-row boxes) and tokens ----------------
        if (lane == 0) {
            int it = 0;
            bool ok = true, all_l1 = false;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const Tile tl = tile_of(t);
                const bool l1 = is_l1(t), sec = second(t);
                const int KB = kb_of(t), kin = kin_of(t);
                const CUtensorMap* mW = sec ? &tmW2 : &tmW;
                const CUtensorMap* mX = sec ? &tmX2 : &tmX;
                if (sec && !all_l1) {
                    // every L1 tile of this route tile has published its A rows (bounded wait);
                    // once every L1 tile of the launch has, no later L2 tile needs a check
                    all_l1 = ld_acquire_gpu(args.l1_total) >= total1;
                    int target;
                    const int32_t* done = dep_of(tl, &target);
                    const uint64_t t0 = globaltimer_ns();
                    while (!all_l1 && ld_acquire_gpu(done) < target) {
                        if (*abort_flag || globaltimer_ns() - t0 > kWaitTimeoutNs) {
                            if (!*abort_flag) record_error(p.hdr, MOE_ERR_TIMEOUT);
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
                    if (!mbar_wait(empty_bar(s), ((uint32_t)(it / kStages) & 1u) ^ 1u, p.hdr, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = base + s * Cfg::kStageBytes, sb = sa + kAtoms * kABytes;
                    const int na = atoms_of(kb, kin);
                    mbar_arrive_expect_tx(full_bar(s), (uint32_t)na * (2 * kABoxTx + (uint32_t)Cfg::kBBytes));
                    for (int at = 0; at < na; ++at) {
                        const int x = kb * kBK + at * kAtomK;
                        if (l1)
                            tma_load_4d(sa + at * kABytes, mW, x, tl.s * kHalf, 0, tl.e, full_bar(s));
                        else
                            tma_load_2d(sa + at * kABytes, mW, x, wrow(tl, 0, false, nout_of(t)), full_bar(s));
                        tma_load_2d(sb + at * Cfg::kBBytes, mX, x, tl.row0, full_bar(s));
                    }
                }
            }
            for (int j = it - kStages < 0 ? 0 : it - kStages; j < it; ++j)
                mbar_drain(full_bar(j % kStages), (uint32_t)(j / kStages) & 1u, p.hdr);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        // At decode sizes this thread sets the pace (eight MMAs of N = 16 per 32 KB stage), so
        // its per-stage work is kept short: a non-blocking test of the stage before the bounded
        // wait, the stage position kept as a counter, the tile's four instruction descriptors
        // made once, and the operand descriptors advanced by adding to their address field
        // (start >> 4: +2 per 32 K of a K-major atom, + the atom's and the stage's offset >> 4).
        if (lane == 0) {
            const uint64_t ad0 = kmajor_desc(base, 0), bd0 = kmajor_desc(base + kAtoms * kABytes, 0);
            int s = 0, tc = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++tc) {
                const int a = tc & 1;
                if (!mbar_wait(acc_empty(a), ((uint32_t)(tc >> 1) & 1u) ^ 1u, p.hdr, abort_flag)) break;
                tc_fence_after();
                const Tile tl = tile_of(t);
                const int n = (tl.n_valid + 15) & ~15;
                const int KB = kb_of(t), kin = kin_of(t);
                const uint32_t d = tmem_base + (uint32_t)(a * kNT);
                uint32_t idesc[kAtomK / 32];
#pragma unroll
                for (int kk = 0; kk < kAtomK / 32; ++kk) idesc[kk] = bs_idesc(kAfmt, kBfmt, n, kk);
                for (int kb = 0; kb < KB; ++kb) {
                    if (!(mbar_test(full_bar(s), ph) || mbar_wait(full_bar(s), ph, p.hdr, abort_flag))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t so = (uint64_t)((s * Cfg::kStageBytes) >> 4);
                    const uint32_t sf = tmem_base + kSfCol0 + s * kSfColsPerStage;
                    const int na = atoms_of(kb, kin);
                    for (int at = 0; at < na; ++at) {
                        const uint64_t ad = ad0 + so + (uint64_t)((at * kABytes) >> 4);
                        const uint64_t bd = bd0 + so + (uint64_t)((at * Cfg::kBBytes) >> 4);
#pragma unroll
                        for (int kk = 0; kk < kAtomK / 32; ++kk)
                            tc_mma_bs(d, ad + 2 * kk, bd + 2 * kk, idesc[kk], sf + 8 * at, sf + 8 * at + 4,
                                      (kb | at | kk) != 0);
                    }
                    tc_commit(empty_bar(s));
                    if (++s == kStages) s = 0, ph ^= 1u;
                }
                if (ok) tc_commit(acc_full(a));
            }
            tc_commit(drain_bar);
            mbar_drain(drain_bar, 0, p.hdr);
        }
    } else if (warp >= 6) {
        // ---------------- scale writers ----------------
        // Each lane owns weight row r = 32q + lane of the tile and, for the token rows, the group
        // c = q: rows 32c + lane. The scale words (one per row and 128-element K atom) are read 8
        // atoms at a time, so the 32 bytes a lane reads fill one sector, and two blocks ahead of
        // their use, which covers the load latency of a busy memory system. Token words are
        // needed by all four warps (the MMA reads them in every lane quarter): each warp
        // publishes its group through shared memory, guarded by an mbarrier per buffer.
        const int q = warp & 3;  // lane quarter this warp writes
        const int r = 32 * q + lane;  // weight row within the tile
        auto n_blk_of = [&](int t) { return (kin_of(t) / kAtomK + 7) >> 3; };  // 8-word blocks per row
        constexpr int kTokWords = Cfg::kTokWords;
        constexpr int kStagesPerBlk = 8 / kAtoms;
        const int cq = q % kTokWords;  // token group this warp loads
        uint32_t* tok_sf = reinterpret_cast<uint32_t*>(smem + Cfg::kTokSfOff);
        // Raw words only: nothing computed from a load happens before the block is used, so
        // the loads stay in flight (addresses are clamped into the tensors instead of predicated).
        // Fused launch: the token words of an L2 tile are A's scales, written by L1 tiles of this
        // launch; they are loaded ahead only when the tile's L1 tiles are already counted, else
        // the block is marked lazy and loaded when it is written out (never waiting ahead of work
        // this CTA still owes).
        struct Blk {
            uint32_t a[8], b[8];
            bool tok_valid, lazy;
        };
        bool all_l1 = false;  // fused launch: every L1 tile of the launch seen finished
        auto tok_ptr = [&](int t, const Tile& tl, int g) -> const uint32_t* {
            const int n = 32 * cq + lane;
            const int64_t row = tl.row0 + min(n, kNT - 1);  // a pool row of the sub-tile
            if (is_l1(t)) {
                if constexpr (kFp4) return reinterpret_cast<const uint32_t*>(p.x_pool_scale) + row * (H / 128) + g;
                return reinterpret_cast<const uint32_t*>(p.x_pool_scale + row * (H / 32)) + g;
            }
            return reinterpret_cast<const uint32_t*>(p.a_pool_scale + row * (I / 32)) + g;
        };
        auto load_blk = [&](int t, int blk) {
            Blk w;
            const Tile tl = tile_of(t);
            const bool l1 = is_l1(t);
            const int kin = kin_of(t), n_words = kin / kAtomK;
            const int wr = wrow(tl, r >= kHalf, l1, nout_of(t)) + (r & (kHalf - 1));
            const uint32_t* ws = reinterpret_cast<const uint32_t*>((second(t) ? args.w_scale2 : args.w_scale) +
                                                                   (int64_t)wr * (kin / 32));
            w.tok_valid = 32 * cq + lane < tl.n_valid;
            w.lazy = false;
            if (second(t) && !all_l1) {  // warp-uniform decisions: each lane loads after its own acquire
                all_l1 = __all_sync(0xffffffffu, ld_acquire_gpu(args.l1_total) >= total1);
                int target;
                w.lazy = !all_l1 && !__all_sync(0xffffffffu, ld_acquire_gpu(dep_of(tl, &target)) >= target);
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int g = min(blk * 8 + i, n_words - 1);  // K atom: elements 128g .. 128g+127
                w.a[i] = __ldg(ws + g);
                if (second(t))
                    w.b[i] = w.lazy ? 0u : ld_relaxed_gpu(tok_ptr(t, tl, g));
                else if (is_l1(t) && kFp4)
                    w.b[i] = __float_as_uint(__ldg(reinterpret_cast<const float*>(tok_ptr(t, tl, g))));
                else
                    w.b[i] = __ldg(tok_ptr(t, tl, g));
            }
            return w;
        };
        // token word as the MMA reads it: 4 UE8M0 bytes; 1.0 for the padding tokens
        auto tok_word = [&](const Blk& w, uint32_t raw, bool l1) -> uint32_t {
            if (!w.tok_valid) return 0x7f7f7f7fu;
            if (kFp4 && l1) return ((raw >> 23) & 0xffu) * 0x01010101u;  // power-of-two fp32 scale
            return raw;
        };
        // (tile, block) positions in the producer's order: t0 is being written out, t1 and t2 are
        // in flight
        auto next_pos = [&](int& t, int& blk) {
            if (++blk == n_blk_of(t)) {
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
            const bool l1 = is_l1(t0);
            const int KB = kb_of(t0);
            uint32_t ub[8];  // the block's token words (a lazy block loads them now)
#pragma unroll
            for (int i = 0; i < 8; ++i) ub[i] = use.b[i];
            if (use.lazy) {
                // every block before this one is written out: wait (bounded) for the tile's L1 tiles
                const Tile tl = tile_of(t0);
                int target;
                const int32_t* done = dep_of(tl, &target);
                const uint64_t w0 = globaltimer_ns();
                bool d_ok = true;
                while (ld_acquire_gpu(done) < target) {
                    if (*abort_flag || globaltimer_ns() - w0 > kWaitTimeoutNs) {
                        if (!*abort_flag) record_error(p.hdr, MOE_ERR_TIMEOUT);
                        *abort_flag = 1;
                        d_ok = false;
                        break;
                    }
                    __nanosleep(64);
                }
                if (!__all_sync(0xffffffffu, d_ok)) return ok = false;
                const int n_words = kin_of(t0) / kAtomK;
#pragma unroll
                for (int i = 0; i < 8; ++i) ub[i] = ld_relaxed_gpu(tok_ptr(t0, tl, min(b0 * 8 + i, n_words - 1)));
            }
            if constexpr (kTokWords > 1) {
#pragma unroll
                for (int i = 0; i < 8; ++i) tok_sf[((buf * kTokWords + cq) * 8 + i) * 32 + lane] = tok_word(use, ub[i], l1);
                __syncwarp();
                if (lane == 0) mbar_arrive(tok_bar(buf));
                const bool t_ok = mbar_wait(tok_bar(buf), (uint32_t)(nb >> 1) & 1u, p.hdr, abort_flag);
                if (!__all_sync(0xffffffffu, t_ok)) return ok = false;
            }
            // working copy of the block (its loads landed a block ago), shifted by one stage's
            // words per stage so the rolled loop below indexes registers statically
            uint32_t wa[8], wb[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                wa[i] = use.a[i];
                wb[i] = tok_word(use, ub[i], l1);
            }
#pragma unroll 1
            for (int j = 0; j < kStagesPerBlk; ++j) {
                const int kb = b0 * kStagesPerBlk + j;
                if (kb >= KB) break;  // uniform across the CTA's scale warps
                const int s = it % kStages;
                const bool w_ok = mbar_wait(empty_bar(s), ((uint32_t)(it / kStages) & 1u) ^ 1u, p.hdr, abort_flag);
                if (!__all_sync(0xffffffffu, w_ok)) return ok = false;
                const uint32_t sf = tmem_base + ((uint32_t)(32 * q) << 16) + kSfCol0 + s * kSfColsPerStage;
                // per K atom 8 columns: the A word in columns 0-3 (the MMA reads column q of lane
                // quarter q), the token words in columns 4.. (unused columns get copies)
#pragma unroll
                for (int at = 0; at < kAtoms; ++at) {
                    const int i = j * kAtoms + at;
                    uint32_t tw[4];
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        if constexpr (kTokWords > 1)
                            tw[c] = tok_sf[((buf * kTokWords + c % kTokWords) * 8 + i) * 32 + lane];
                        else
                            tw[c] = wb[at];
                    }
                    tmem_st8(sf + 8 * at, wa[at], wa[at], wa[at], wa[at], tw[0], tw[1], tw[2], tw[3]);
                }
#pragma unroll
                for (int i = 0; i + kAtoms < 8; ++i) {
                    wa[i] = wa[i + kAtoms];
                    wb[i] = wb[i + kAtoms];
                }
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
        // ---------------- epilogue (warps 2..5) ----------------
        const int q = warp & 3;
        constexpr int kChunks = (kNT + 31) / 32;  // 32-token chunks of a sub-tile
        int tc = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x, ++tc) {
            const int a = tc & 1;
            const Tile tl = tile_of(t);
            const bool l1 = is_l1(t);
            // L2: destination slot and gate weight of each row, read while the MMAs of this tile
            // still run (two dependent loads that would otherwise sit on the epilogue's path)
            int src_l[kChunks];
            float g_l[kChunks];
            if (!l1) {
#pragma unroll
                for (int ci = 0; ci < kChunks; ++ci) {
                    const int n = 32 * ci + lane;
                    src_l[ci] = n < tl.n_valid ? debug_row(p.hdr, __ldg(p.pool_src + tl.row0 + n), (int64_t)p.T * p.K) : -1;
                }
#pragma unroll
                for (int ci = 0; ci < kChunks; ++ci) g_l[ci] = src_l[ci] >= 0 ? __ldg(args.topk_weights + src_l[ci]) : 0.0f;
            }
            const bool w_ok = mbar_wait(acc_full(a), (uint32_t)(tc >> 1) & 1u, p.hdr, abort_flag);
            if (!epi_all(w_ok)) break;  // one decision for the four warps (they share epi_sync)
            tc_fence_after();
            const int n = (tl.n_valid + 15) & ~15;
            const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(a * kNT);
            if (l1) {
                // lanes 0-63 hold the gate rows and lanes 64-127 the up rows of the same 64 outputs j.
                // Of each 32-token chunk the gate warps finish tokens 0-15 and the up warps tokens
                // 16-31; each hands its partner the other half through xbuf.
                const bool gate = q < 2;
                const int jl = 32 * (q & 1) + lane;  // output within the tile
                const int j = tl.s * kHalf + jl;
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
                        uint32_t my_sc = 0;  // lane tt keeps the UE8M0 byte of token tt
                        // A = SiLU(gate) * up, then MX FP8: one exponent per 32 outputs of a token.
                        // Branch-free, so the 16 tokens' dependency chains overlap.
#pragma unroll
                        for (int tt = 0; tt < 16; ++tt) {
                            const float gv = gate ? __uint_as_float(v[tt]) : xg[tt * kHalf + jl];
                            const float uv = gate ? xu[tt * kHalf + jl] : __uint_as_float(v[16 + tt]);
                            const float av = swiglu1(gv, uv, p.act_clamp);
                            const float amax = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(av))));
                            const int ex = mx_exponent_fp8<kE5>(amax);
                            st_global_u8_if(true, p.a_pool + (row0 + tt) * I + j, float_to_fp8_satfinite<kE5>(av * exp2_neg_int(ex)));
                            my_sc = lane == tt ? (uint32_t)(ex + 127) : my_sc;
                        }
                        st_global_u8_if(lane < 16, p.a_pool_scale + (row0 + lane) * (I / 32) + (j >> 5), (uint8_t)my_sc);
                    }
                    epi_sync();
                }
                if (kFused) {
                    // publish the tile's A rows and scales (an L2 tile's TMA reads the rows, its
                    // scale writers the scales): every thread orders its own stores before the
                    // async proxy's later reads and fences them, the four warps meet, and one thread
                    // fences again and counts the tile for its route tile (no one waits here)
                    asm volatile("fence.proxy.async.global;" ::: "memory");
                    __threadfence();
                    epi_sync();
                    if (q == 0 && lane == 0) {
                        int target;
                        __threadfence();
                        atomicAdd(dep_of(tl, &target), 1);
                        atomicAdd(args.l1_total, 1);
                    }
                }
            } else {
                const int h = tl.s * kWR + q * 32 + lane;
                // the rows' slots and gate weights as a per-warp table (xbuf is free in L2):
                // broadcast reads instead of shuffles, and no dependency chain through the stores
                int* w_src = reinterpret_cast<int*>(xbuf) + q * 2 * kNT;
                float* w_g = reinterpret_cast<float*>(w_src + kNT);
#pragma unroll
                for (int ci = 0; ci < kChunks; ++ci) {
                    if (32 * ci + lane < kNT) {
                        w_src[32 * ci + lane] = src_l[ci];
                        w_g[32 * ci + lane] = g_l[ci];
                    }
                }
                __syncwarp();
#pragma unroll
                for (int ci = 0; ci < kChunks; ++ci) {
                    const int c0 = 32 * ci;
                    if (c0 >= tl.n_valid) break;  // uniform across the warp
                    uint32_t y[32];
                    tmem_ld32(tb + c0, y);
                    tmem_ld_wait();
#pragma unroll
                    for (int tt = 0; tt < 32 && c0 + tt < kNT; ++tt) {  // src < 0 past the routed rows
                        const int src = w_src[c0 + tt];
                        const float gw = w_g[c0 + tt];
                        st_global_u16_if(src >= 0, p.comb + (int64_t)src * H + h,
                                         float_to_bf16_bits(__fmul_rn(gw, __uint_as_float(y[tt]))));
                    }
                }
                __syncwarp();
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

template <int MODE, int kKind, int kNT, int kStages, int kAtoms>
cudaError_t set_bs_smem_attr() {
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(tc_bs_kernel<MODE, kKind, kNT, kStages, kAtoms>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)BsCfg<kNT, kStages, kAtoms>::kSmem);
    });
    return attr_err;
}

// sub-tiles of kNT rows: at most one per routed row, and 128/kNT per 128-row route tile
template <int kNT>
int64_t max_sub_tiles(const Plan& p) {
    return std::max<int64_t>(1, std::min<int64_t>((int64_t)p.T * p.K, (p.pool_rows / 128) * (128 / kNT)));
}

template <int MODE, int kKind, int kNT, int kStages, int kAtoms>
cudaError_t launch_bs_cfg(const Plan& p, const CUtensorMap& tmW, const CUtensorMap& tmX, BsArgs args,
                          cudaStream_t s) {
    using Cfg = BsCfg<kNT, kStages, kAtoms>;
    args.k_blocks = (args.kin + kAtoms * kAtomK - 1) / (kAtoms * kAtomK);
    const cudaError_t attr_err = set_bs_smem_attr<MODE, kKind, kNT, kStages, kAtoms>();
    if (attr_err != cudaSuccess) return attr_err;
    const int64_t max_tiles = max_sub_tiles<kNT>(p) * args.n_slabs;
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(max_tiles, tc_num_sms()));
    tc_bs_kernel<MODE, kKind, kNT, kStages, kAtoms><<<grid, kThreads, Cfg::kSmem, s>>>(tmW, tmX, tmW, tmX, args);
    return cudaGetLastError();
}

// L1 then L2 in one cooperative launch: every CTA is resident, so an L2 tile waits (bounded) only
// for L1 tiles that earlier positions of the same round-robin order hold, all of them running
template <int MODE, int kNT, int kStages, int kAtoms>
cudaError_t launch_bs_fused_cfg(const Plan& p, const CUtensorMap& tmW1, const CUtensorMap& tmX1,
                                const CUtensorMap& tmW2, const CUtensorMap& tmX2, BsArgs args, cudaStream_t s) {
    using Cfg = BsCfg<kNT, kStages, kAtoms>;
    constexpr int kBK = kAtoms * kAtomK;
    args.k_blocks = (args.kin + kBK - 1) / kBK;
    args.k_blocks2 = (args.kin2 + kBK - 1) / kBK;
    cudaError_t e = set_bs_smem_attr<MODE, kFusedL1L2, kNT, kStages, kAtoms>();
    if (e != cudaSuccess) return e;
    // the counters (one per 128-row route tile) start at zero every launch
    // (the launch-wide count follows the route tiles' counts)
    if ((e = cudaMemsetAsync(args.l1_done, 0, sizeof(int32_t) * (size_t)(p.pool_rows / 128 + 1), s)) != cudaSuccess)
        return e;
    int per_sm = 0;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, tc_bs_kernel<MODE, kFusedL1L2, kNT, kStages, kAtoms>,
                                                           kThreads, Cfg::kSmem)) != cudaSuccess)
        return e;
    if (per_sm < 1) return cudaErrorCooperativeLaunchTooLarge;
    const int64_t max_tiles = max_sub_tiles<kNT>(p) * (args.n_slabs + args.n_slabs2);
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(max_tiles, (int64_t)tc_num_sms() * per_sm));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = Cfg::kSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, tc_bs_kernel<MODE, kFusedL1L2, kNT, kStages, kAtoms>, tmW1, tmX1, tmW2, tmX2, args);
}

// W1 as [K][row within the gate or up half][half][expert] (one box holds a tile's 64 gate and 64
// up rows), W2 as [K][expert * H]; e2m1 weights packed two to a byte
template <int MODE>
bool make_w_map(CUtensorMap* m, const Plan& p, const void* w, bool l1) {
    constexpr bool kFp4 = MODE == MOE_A8W4_FP8_FP4;
    const CUtensorMapDataType wtype = kFp4 ? CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    const int kin = l1 ? p.H : p.I;
    const uint64_t pitch = kFp4 ? (uint64_t)kin / 2 : (uint64_t)kin;  // bytes per weight row
    if (l1) {
        const uint64_t dims[4] = {(uint64_t)kin, (uint64_t)p.I, 2, (uint64_t)p.E};
        const uint64_t strides[3] = {pitch, pitch * p.I, pitch * 2 * p.I};
        const uint32_t box[4] = {kAtomK, kHalf, 2, 1};
        return tc_make_map_nd(m, wtype, 4, w, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
    }
    const uint64_t dims[2] = {(uint64_t)kin, (uint64_t)p.E * p.H};
    const uint64_t strides[1] = {pitch};
    const uint32_t box[2] = {kAtomK, kWR};
    return tc_make_map_nd(m, wtype, 2, w, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// token rows (x_pool for L1, a_pool for L2): one copy brings a sub-tile's rows
bool make_x_map(CUtensorMap* m, const Plan& p, bool l1, int rows) {
    return tc_make_map_2d(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, l1 ? (const void*)p.x_pool : (const void*)p.a_pool,
                          (uint64_t)(l1 ? p.H : p.I), (uint64_t)p.pool_rows, kAtomK, (uint32_t)rows,
                          CU_TENSOR_MAP_SWIZZLE_128B);
}

// few routed rows per expert: the weights stream from HBM; 16-token sub-tiles and K = 256 stages
// (whole 128-byte lines of every weight row per load)
bool is_decode(const Plan& p) { return (int64_t)p.T * p.K <= (int64_t)16 * p.E; }

template <int MODE, bool kIsL1>
cudaError_t launch_bs(const Plan& p, const void* w, const void* w_scale, const float* topk_weights, uint32_t flags,
                      cudaStream_t s) {
    const bool weight_major = (flags & MOE_FLAG_WEIGHT_MAJOR) != 0;
    const bool decode = is_decode(p);
    // prefill sizes: token-major tiles, or with MOE_FLAG_PAIR_L1 weight-major tiles on CTA pairs (M = 256
    // weight rows, tokens as N; measured slower: Zipf prefill L1 2.48 against 1.50 ms)
    if (!decode && !weight_major && (flags & MOE_FLAG_PAIR_L1) && bs_pair_supported(p, kIsL1 ? 1 : 2))
        return kIsL1 ? launch_l1_bs_pair(p, w, w_scale, s) : launch_l2_bs_pair(p, w, w_scale, topk_weights, s);
    if (!decode && !weight_major && bs_tm_supported(p, kIsL1 ? 1 : 2))
        return kIsL1 ? launch_l1_bs_tm(p, w, w_scale, s) : launch_l2_bs_tm(p, w, w_scale, topk_weights, s);
    CUtensorMap tmW, tmX;
    if (!make_w_map<MODE>(&tmW, p, w, kIsL1) || !make_x_map(&tmX, p, kIsL1, decode ? 16 : 128))
        return cudaErrorInvalidValue;
    BsArgs args{};
    args.p = p;
    args.w_scale = static_cast<const uint8_t*>(w_scale);
    args.topk_weights = topk_weights;
    args.n_slabs = kIsL1 ? p.I / kHalf : p.H / kWR;
    args.n_out = kIsL1 ? 2 * p.I : p.H;
    args.kin = kIsL1 ? p.H : p.I;
    constexpr int kKind = kIsL1 ? kL1 : kL2;
    if (decode) return launch_bs_cfg<MODE, kKind, 16, 5, 2>(p, tmW, tmX, args, s);
    return launch_bs_cfg<MODE, kKind, 128, 6, 1>(p, tmW, tmX, args, s);
}

template <int MODE>
cudaError_t launch_fused(const Plan& p, const void* w1, const void* w1_scale, const void* w2, const void* w2_scale,
                         const float* topk_weights, cudaStream_t s) {
    const bool decode = is_decode(p);
    CUtensorMap tmW1, tmX1, tmW2, tmX2;
    if (!make_w_map<MODE>(&tmW1, p, w1, true) || !make_x_map(&tmX1, p, true, decode ? 16 : 128) ||
        !make_w_map<MODE>(&tmW2, p, w2, false) || !make_x_map(&tmX2, p, false, decode ? 16 : 128))
        return cudaErrorInvalidValue;
    BsArgs args{};
    args.p = p;
    args.w_scale = static_cast<const uint8_t*>(w1_scale);
    args.topk_weights = topk_weights;
    args.n_slabs = p.I / kHalf;
    args.n_out = 2 * p.I;
    args.kin = p.H;
    args.w_scale2 = static_cast<const uint8_t*>(w2_scale);
    args.n_slabs2 = p.H / kWR;
    args.n_out2 = p.H;
    args.kin2 = p.I;
    args.l1_done = p.ffn_counters;
    args.l1_total = p.ffn_counters + p.pool_rows / 128;
    if (decode) return launch_bs_fused_cfg<MODE, 16, 5, 2>(p, tmW1, tmX1, tmW2, tmX2, args, s);
    return launch_bs_fused_cfg<MODE, 128, 6, 1>(p, tmW1, tmX1, tmW2, tmX2, args, s);
}

}  // namespace

bool bs_supported(const Plan& p, int stage) {
    if ((p.mode != MOE_A8W8_FP8 && p.mode != MOE_A8W8_FP8_E5M2 && p.mode != MOE_A8W4_FP8_FP4) ||
        p.E > kMaxExperts || !tc_encode_available())
        return false;
    if (stage == 1) return p.I % kHalf == 0 && p.H % kAtomK == 0;
    return p.H % kWR == 0 && p.I % kAtomK == 0;
}

cudaError_t launch_l1_bs(const Plan& p, const void* w1, const void* w1_scale, uint32_t flags, cudaStream_t s) {
    if (p.mode == MOE_A8W4_FP8_FP4) return launch_bs<MOE_A8W4_FP8_FP4, true>(p, w1, w1_scale, nullptr, flags, s);
    if (p.mode == MOE_A8W8_FP8) return launch_bs<MOE_A8W8_FP8, true>(p, w1, w1_scale, nullptr, flags, s);
    if (p.mode == MOE_A8W8_FP8_E5M2) return launch_bs<MOE_A8W8_FP8_E5M2, true>(p, w1, w1_scale, nullptr, flags, s);
    return cudaErrorNotSupported;
}

cudaError_t launch_l2_bs(const Plan& p, const void* w2, const void* w2_scale, const float* topk_weights, uint32_t flags,
                         cudaStream_t s) {
    if (p.mode == MOE_A8W4_FP8_FP4) return launch_bs<MOE_A8W4_FP8_FP4, false>(p, w2, w2_scale, topk_weights, flags, s);
    if (p.mode == MOE_A8W8_FP8) return launch_bs<MOE_A8W8_FP8, false>(p, w2, w2_scale, topk_weights, flags, s);
    if (p.mode == MOE_A8W8_FP8_E5M2) return launch_bs<MOE_A8W8_FP8_E5M2, false>(p, w2, w2_scale, topk_weights, flags, s);
    return cudaErrorNotSupported;
}

cudaError_t launch_ffn_fused_bs(const Plan& p, const void* w1, const void* w1_scale, const void* w2,
                                const void* w2_scale, const float* topk_weights, cudaStream_t s) {
    if (p.mode == MOE_A8W4_FP8_FP4) return launch_fused<MOE_A8W4_FP8_FP4>(p, w1, w1_scale, w2, w2_scale, topk_weights, s);
    if (p.mode == MOE_A8W8_FP8) return launch_fused<MOE_A8W8_FP8>(p, w1, w1_scale, w2, w2_scale, topk_weights, s);
    if (p.mode == MOE_A8W8_FP8_E5M2)
        return launch_fused<MOE_A8W8_FP8_E5M2>(p, w1, w1_scale, w2, w2_scale, topk_weights, s);
    return cudaErrorNotSupported;
}

}  // namespace moe
