// Tensor-core grouped GEMM stages for bf16 operands on CTA pairs (sm_103a): a cluster of two
// CTAs on neighbouring SMs runs one tcgen05.mma.cta_group::2 per 16 K, a 256 x 256 product
// whose A rows are split between the two CTAs' shared memory (128 each), whose B columns are
// split the same way (128 each), and whose fp32 accumulator rows land in the tensor memory of
// the CTA that holds them. Per SM this is the single-CTA kernel's 128 x 256 tile of MMA work
// for two thirds of its shared-memory fill (16 KB of A and 16 KB of B per 64 K instead of
// 16 + 32 KB), and the fill, not the tensor pipe, is what bounds the single-CTA kernel.
//
// Same stages and epilogues as the single-CTA kernel (Ascend mega_moe page, "Linear1
// Projection" + "SwiGLU Activation", "Linear2 Projection" + the gate weight of "Token
// Combine"):
//   L1: the even CTA holds the gate column block [n*128, n*128+128) of W1[e], the odd CTA the
//       up block [I+n*128, ...); both CTAs' accumulators then hold gate and up values of the
//       same 128 outputs for their own 128 rows, and SwiGLU runs in each CTA's epilogue.
//   L2: 256 H columns per pair tile, 128 from each CTA; the epilogue scales row p by
//       G[row_src[p]] and stores bf16 to the combine row of (token, slot).
//
// Pair tiles: an expert's 128-row route tiles are taken two at a time, (2j, 2j+1); when the
// expert has an odd number of them the odd CTA's half of its last pair lies outside the expert,
// its MMA rows are computed from whatever rows are there and its epilogue stores nothing.
// Tiles are ordered expert-major, then column block, then row pair; each cluster takes every
// (number of clusters)-th one.
//
// Synchronisation between the two CTAs:
//   full[s]   (even CTA): both CTAs' TMA loads of stage s complete on it; the even CTA's
//             producer arrives with the byte count of both halves.
//   empty[s]  (each CTA): the MMA issuer's commit arrives on both CTAs' barriers once the MMAs
//             that read stage s are done, so each producer refills its own half.
//   tfull[a]  (each CTA): accumulator a is complete (commit to both CTAs).
//   tempty[a] (even CTA): the four epilogue warps of both CTAs have read accumulator a.
// Warp roles (192 threads per CTA): warp 0 = TMA producer (both CTAs), warp 1 = tensor-memory
// allocator (both) and MMA issuer (even CTA only), warps 2-5 = epilogue (both).
// Every wait is bounded (2 s); on time-out the CTA records MOE_ERR_TIMEOUT and leaves its loop;
// both CTAs meet at a cluster barrier before the tensor memory is freed and before exit.
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

constexpr int kPM = 256;                        // rows per pair tile (MMA M)
constexpr int kHM = 128;                        // rows per CTA
constexpr int kPN = 256;                        // accumulator columns (MMA N)
constexpr int kBK = 64;                         // K per stage: one 128-byte swizzle row of bf16
constexpr int kStages = 6;
constexpr int kABytes = kHM * kBK * 2;          // 16 KB
constexpr int kBBoxBytes = kBK * 64 * 2;        // one 64(K) x 64(N) box, 8 KB
constexpr int kBBytes = 2 * kBBoxBytes;         // this CTA's 128 columns of B, 16 KB
constexpr int kStageBytes = kABytes + kBBytes;  // 32 KB
constexpr int kThreads = 192;
constexpr int kTmemCols = 512;                  // two 256-column fp32 accumulators
constexpr int kMaxExperts = 1024;

// Instruction descriptor of tcgen05.mma.kind::f16 (as the single-CTA kernel's, with M = 256):
// D fp32, A and B bf16, A K-major, B MN-major, N >> 3 in bits 17-22, M >> 4 in bits 24-28.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (0u << 15) | (1u << 16) |
                            ((uint32_t)(kPN >> 3) << 17) | ((uint32_t)(kPM >> 4) << 24);

struct PairArgs {
    Plan p;
    const float* topk_weights;  // L2 only
    int n_tiles;                // column blocks per expert (L1: I / 128, L2: H / 256)
    int k_blocks;               // K / 64
    int k_rows;                 // rows of one expert's weight in its 2-D view (L1: H, L2: I)
};

struct PairTile {
    int e, n, row0;    // row0: first pool row of the even CTA's half
    bool odd_valid;    // the odd CTA's 128 rows belong to expert e
};

// Pair tiles are ordered expert-major: expert e owns [pair_off[e] * n_tiles, pair_off[e+1] * n_tiles).
__device__ __forceinline__ PairTile decode_pair(int t, const int* tile_off, const int* pair_off, int E, int n_tiles) {
    int lo = 0, hi = E - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (pair_off[mid] * n_tiles <= t) lo = mid; else hi = mid - 1;
    }
    PairTile tl;
    tl.e = lo;
    const int pt = pair_off[lo + 1] - pair_off[lo];
    const int local = t - pair_off[lo] * n_tiles;
    tl.n = local / pt;
    const int first = tile_off[lo] + 2 * (local % pt);
    tl.row0 = first * kHM;
    tl.odd_valid = first + 1 < tile_off[lo + 1];
    return tl;
}

template <bool kL1>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    tc_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, PairArgs args) {
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
    int* tile_off = reinterpret_cast<int*>(misc + 16);
    int* pair_off = tile_off + (kMaxExperts + 1);

    const Plan& p = args.p;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool even = rank == 0;
    const int cluster = (int)cluster_id_x(), clusters = (int)cluster_count_x();

    for (int i = threadIdx.x; i <= p.E; i += kThreads) tile_off[i] = p.tile_off[i];
    __syncthreads();
    if (warp == 2) {
        // pair_off = exclusive prefix sum of ceil(route tiles of e / 2), one warp scan per 32 experts
        int carry = 0;
        for (int b = 0; b < p.E; b += 32) {
            const int e = b + lane;
            int v = e < p.E ? (tile_off[e + 1] - tile_off[e] + 1) >> 1 : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += u;
            }
            if (e < p.E) pair_off[e + 1] = carry + v;
            carry += __shfl_sync(0xffffffffu, v, 31);
        }
        if (lane == 0) pair_off[0] = 0;
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), 8);  // four epilogue warps in each CTA
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) tmem_alloc_pair(smem_u32(tmem_holder), kTmemCols);  // one warp of each CTA, together
    if (warp == 0 && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB)) : "memory");
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // both CTAs' barriers are initialised before either signals the other's
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    const int total = pair_off[p.E] * args.n_tiles;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer (both CTAs: own rows of A, own half of B) ----------------
            int it = 0;
            bool ok = true;
            for (int t = cluster; t < total && ok; t += clusters) {
                const PairTile tl = decode_pair(t, tile_off, pair_off, p.E, args.n_tiles);
                const int wrow = tl.e * args.k_rows;
                for (int kb = 0; kb < args.k_blocks; ++kb, ++it) {
                    const int s = it % kStages;
                    const uint32_t ph = (uint32_t)(it / kStages) & 1u;
                    if (!mbar_wait(empty_bar(s), ph ^ 1u, p.hdr, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = base + s * kStageBytes, sb = sa + kABytes;
                    const uint32_t fb = mapa_shared(full_bar(s), 0);
                    if (even) mbar_arrive_expect_tx(full_bar(s), 2 * kStageBytes);
                    tma_load_2d_pair(sa, &tmA, kb * kBK, tl.row0 + (int)rank * kHM, fb);
                    const int y = wrow + kb * kBK;
                    if (kL1)
                        tma_load_4d_pair(sb, &tmB, 0, y, 2 * tl.n, (int)rank, fb);  // gate (even) or up (odd)
                    else
                        tma_load_3d_pair(sb, &tmB, 0, y, 4 * tl.n + 2 * (int)rank, fb);
                }
            }
            // drain (even CTA): every stage's loads, both halves, have landed (bounded)
            if (even) {
                for (int j = it - kStages < 0 ? 0 : it - kStages; j < it; ++j)
                    if (!mbar_drain(full_bar(j % kStages), (uint32_t)(j / kStages) & 1u, p.hdr)) break;
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && even) {
            // ---------------- MMA issuer (even CTA) ----------------
            const uint64_t ad0 = kmajor_desc(base, 0);
            const uint64_t bd0 = smem_desc(base + kABytes, kBBoxBytes, 1024);
            int it = 0, tc = 0;
            bool ok = true;
            for (int t = cluster; t < total && ok; t += clusters, ++tc) {
                const int a = tc & 1;
                if (!mbar_wait(tempty_bar(a), ((uint32_t)(tc >> 1) & 1u) ^ 1u, p.hdr, abort_flag)) break;
                tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)(a * kPN);
                for (int kb = 0; kb < args.k_blocks; ++kb, ++it) {
                    const int s = it % kStages;
                    const uint32_t par = (uint32_t)(it / kStages) & 1u;
                    if (!mbar_test(full_bar(s), par) && !mbar_wait(full_bar(s), par, p.hdr, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // descriptors advanced in their address field (>> 4): +2 per 16 K of A
                    // (32 bytes), +128 per 16 K rows of B (2 KB), + the stage offset
                    const uint64_t off = (uint64_t)((s * kStageBytes) >> 4);
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        tc2_mma(d, ad0 + off + 2 * kk, bd0 + off + 128 * kk, kIdesc, (kb | kk) != 0);
                    tc2_commit_mc(empty_bar(s), 0x3);  // both CTAs may refill stage s
                }
                if (ok) tc2_commit_mc(tfull_bar(a), 0x3);
            }
            // drain: every MMA issued so far has completed before tensor memory is freed
            tc2_commit_mc(drain_bar, 0x1);
            mbar_drain(drain_bar, 0, p.hdr);
        }
    } else {
        // ---------------- epilogue (warps 2..5, both CTAs) ----------------
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        int tc = 0;
        for (int t = cluster; t < total; t += clusters, ++tc) {
            const int a = tc & 1;
            const PairTile tl = decode_pair(t, tile_off, pair_off, p.E, args.n_tiles);
            const bool mine = even || tl.odd_valid;  // this CTA's rows belong to the tile's expert
            const int64_t row = tl.row0 + (int)rank * kHM + q * 32 + lane;
            int src = -1;
            float gw = 0.0f;
            if (!kL1 && mine) {
                src = debug_row(p.hdr, __ldg(p.pool_src + row), (int64_t)p.T * p.K);
                gw = src >= 0 ? __ldg(args.topk_weights + src) : 0.0f;
            }
            const bool ok = mbar_wait(tfull_bar(a), (uint32_t)(tc >> 1) & 1u, p.hdr, abort_flag);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc_fence_after();
            const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(a * kPN);
            if (kL1) {
                uint16_t* out = reinterpret_cast<uint16_t*>(p.a_pool) + (mine ? row : 0) * p.I + tl.n * 128;
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
                    st_global_v8_if(mine, out + c * 32, packed);
                    st_global_v8_if(mine, out + c * 32 + 16, packed + 8);
                }
            } else {
                uint16_t* out = p.comb + (int64_t)(src >= 0 ? src : 0) * p.H + tl.n * kPN;
#pragma unroll 1
                for (int c = 0; c < kPN / 32; ++c) {
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
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(mapa_shared(tempty_bar(a), 0));
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();  // no CTA frees tensor memory or exits while its pair still uses it
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem_base, kTmemCols);
}

// ---------------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------------

constexpr size_t pair_smem_bytes() {
    return 1024 + (size_t)kStages * kStageBytes + 8 * (2 * kStages + 5) + 16 + 8 * (kMaxExperts + 1);
}

template <bool kL1>
cudaError_t pair_smem_attr() {
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(tc_pair_kernel<kL1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)pair_smem_bytes());
    });
    return attr_err;
}

// Clusters of this kernel that can be resident at once (a pair needs two free SMs of one GPC,
// so this can be below half the SM count); the persistent grid is sized to it so that no
// cluster waits for another to finish before it starts.
template <bool kL1>
int pair_resident_clusters() {
    static std::once_flag once;
    static int n = 0;
    std::call_once(once, [] {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * std::max(1, tc_num_sms() / 2));
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = pair_smem_bytes();
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, tc_pair_kernel<kL1>, &cfg) != cudaSuccess || n < 1) {
            (void)cudaGetLastError();
            n = std::max(1, tc_num_sms() / 2);  // no figure: one pair per two SMs
        }
    });
    return n;
}

template <bool kL1>
cudaError_t launch_pair(const Plan& p, const CUtensorMap& a, const CUtensorMap& b, PairArgs args, cudaStream_t s) {
    const cudaError_t attr_err = pair_smem_attr<kL1>();
    if (attr_err != cudaSuccess) return attr_err;
    const int resident = pair_resident_clusters<kL1>();
    // at most (route tiles + experts) / 2 row pairs
    const int64_t max_tiles = ((p.pool_rows / kHM + p.E) / 2 + 1) * args.n_tiles;
    const int clusters = (int)std::max<int64_t>(1, std::min<int64_t>(max_tiles, resident));
    tc_pair_kernel<kL1><<<2 * clusters, kThreads, pair_smem_bytes(), s>>>(a, b, args);
    return cudaGetLastError();
}

// A: pool rows [pool_rows, K] bf16, 128 x 64 boxes, 128-byte swizzle.
bool make_a_map(CUtensorMap* map, const void* ptr, uint64_t k, uint64_t rows) {
    return tc_make_map_2d(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ptr, k, rows, 64, kHM, CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace

bool pair_supported(const Plan& p, int stage) {
    if (p.mode != MOE_A16W16 || p.E > kMaxExperts || !tc_encode_available() || tc_num_sms() < 2) return false;
    if (stage == 1) return p.I % 128 == 0;
    return p.H % kPN == 0;
}

// B of one CTA of the pair: [64 columns][K row][two 64-column blocks] in one box (L1: of the
// gate or of the up half of W1, chosen by the last coordinate).
cudaError_t launch_l1_pair(const Plan& p, const void* w1, cudaStream_t s) {
    CUtensorMap a, b;
    if (!make_a_map(&a, p.x_pool, (uint64_t)p.H, (uint64_t)p.pool_rows)) return cudaErrorInvalidValue;
    const uint64_t pitch = (uint64_t)2 * p.I * 2;
    const uint64_t dims[4] = {64, (uint64_t)p.E * p.H, (uint64_t)p.I / 64, 2};
    const uint64_t strides[3] = {pitch, 128, (uint64_t)p.I * 2};
    const uint32_t box[4] = {64, (uint32_t)kBK, 2, 1};
    if (!tc_make_map_nd(&b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, w1, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    PairArgs args{p, nullptr, p.I / 128, p.H / kBK, p.H};
    return launch_pair<true>(p, a, b, args, s);
}

cudaError_t launch_l2_pair(const Plan& p, const void* w2, const float* topk_weights, cudaStream_t s) {
    CUtensorMap a, b;
    if (!make_a_map(&a, p.a_pool, (uint64_t)p.I, (uint64_t)p.pool_rows)) return cudaErrorInvalidValue;
    const uint64_t dims[3] = {64, (uint64_t)p.E * p.I, (uint64_t)p.H / 64};
    const uint64_t strides[2] = {(uint64_t)p.H * 2, 128};
    const uint32_t box[3] = {64, (uint32_t)kBK, 2};
    if (!tc_make_map_nd(&b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, w2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    PairArgs args{p, topk_weights, p.H / kPN, p.I / kBK, p.I};
    return launch_pair<false>(p, a, b, args, s);
}

}  // namespace moe
