// A8W4-INT grouped GEMM on the tensor cores, token-major, with exact integer results (Ascend
// mega_moe page, A8W4-INT use case: int8 activations x signed int4 weights, C = Q_e . W1 and
// D = A^int8 . W2 as integers, then (C * s^W) * s^X in fp32).
//
// sm_103a has no integer tcgen05.mma kind, so the codes travel as f16 (kind::f16, fp32
// accumulation in TMEM) and every partial sum has to stay an exactly representable integer:
// - the weights stay packed int4 in HBM. TMA brings 32 bytes of each of 256 weight rows per
//   stage; the converter warps turn each nibble n into u = n + 8 in [0, 15] and place u in the
//   low mantissa bits of an f16 with a zero exponent field: the subnormal u * 2^-24, exactly, in
//   two ALU operations per pair of codes (a shift, and one lop3 that masks the two nibbles and
//   flips their sign bits). The pair taken from one 32-bit word is (code i, code i + 4), so a
//   group of 8 codes lands in the order 0 4 1 5 2 6 3 7; the dispatch stage and the row
//   quantiser store the token codes in the same order (w4_plane_pos), which leaves every
//   product in the K sum unchanged;
// - the tokens are one f16 plane of the int8 codes q (normal numbers, exact);
// - the accumulator is then 2^-24 * sum_k u_k q_k with |u q| <= 15 * 128, exact while
//   K <= 8704, and C = 2^24 * D - 8 * sum_k q_k: the per-token code sums come from the dispatch
//   stage (x) and the row quantiser (A). The page's MSD scheme reaches the same integer by
//   splitting the activations into two int4 halves with a compensation term 8 * (1^T W) per
//   output channel; on this hardware the offset sits on the weight side instead, with a
//   compensation per token.
//
// Tile: M = 128 pool rows (one route tile of an expert, the TMEM lanes) x N = 256 weight rows,
// K = 64 per stage (four 128 x 256 x 16 MMAs of 128 tensor cycles each; smaller MMAs leave the
// tensor pipe waiting on the single issuing thread):
// - L1: the 128 gate rows and the 128 up rows of outputs [128s, 128s + 128), so an epilogue
//   thread holds its token's gate and up values of the same outputs and applies SwiGLU (Ascend
//   page, "SwiGLU Activation");
// - L2: 256 hidden columns; the epilogue scales the token's row by G and writes its bf16
//   combine row (Ascend page, "Token Combine").
// Two 256-column accumulators fill TMEM, so the epilogue of a tile overlaps the next main loop.
//
// Warp roles (512 threads): warp 0 TMA of raw weights, warp 1 TMEM allocation + MMA issue,
// warp 2 TMA of the token tiles, warp 3 idle, warps 4-7 epilogue (warp w owns TMEM lanes
// 32*(w%4) .. +31, i.e. those token rows), warps 8-15 converters (one weight row per thread).
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

constexpr int kTM = 128;       // token rows per tile (MMA M)
constexpr int kWN = 256;       // weight rows per tile (MMA N)
constexpr int kBK = 64;        // K per stage: 64 f16 = one 128-byte swizzle row
constexpr int kThreads = 512;
constexpr int kConvWarp0 = 8;  // converters: warps 8-15, thread = weight row of the tile
constexpr int kEpiWarp0 = 4;   // epilogue: warps 4-7
constexpr int kMaxExperts = 1024;
constexpr int kHfStages = 4, kTokStages = 3, kRawStages = 3;
constexpr int kHfBytes = kWN * 128;             // f16 weight tile (B operand)
constexpr int kTokBytes = kTM * 128;            // f16 token tile (A operand)
constexpr int kRawRow = kBK / 2;                // bytes of a packed weight row per stage
constexpr int kRawBytes = kWN * kRawRow;
constexpr int kHfOff = 0;
constexpr int kTokOff = kHfOff + kHfStages * kHfBytes;
constexpr int kRawOff = kTokOff + kTokStages * kTokBytes;
constexpr int kBarOff = kRawOff + kRawStages * kRawBytes;
constexpr int kNumBars = 2 * (kHfStages + kTokStages + kRawStages) + 4 + 1;
constexpr int kMiscOff = kBarOff + 8 * kNumBars;
constexpr int kTileOffOff = kMiscOff + 16;
constexpr int kCountsOff = kTileOffOff + 4 * (kMaxExperts + 1);
constexpr size_t kSmem = 1024 + (size_t)kCountsOff + 4 * kMaxExperts;
static_assert(kSmem <= 232448, "shared memory");
// largest K with every partial sum of u * q below 2^24 (u <= 15, |q| <= 128)
constexpr int kMaxK = 8704;
// kind::f16 instruction descriptor: D fp32 (bits 4-5 = 1), A and B f16 (formats 0), both
// K-major, N >> 3 in bits 17-22, M >> 4 in bits 24-28.
constexpr uint32_t kIdesc = (1u << 4) | ((uint32_t)(kWN >> 3) << 17) | ((uint32_t)(kTM >> 4) << 24);

struct W4Args {
    Plan p;
    const float* w_scale;       // fp32 per output channel [E * n_out]
    const float* topk_weights;  // L2
    const uint16_t* planes;     // f16 token codes [pool_rows, kin]
    const float* row_scale;     // s^X or s^A per pool row
    const int32_t* row_sums;    // code sums per pool row
    int n_slabs, k_blocks, n_out;
};

struct Tile {
    int e, s, m, row0, n_valid;
};

// Tiles are ordered expert-major, then weight slab, then route tile (as in the block-scaled
// token-major kernel): the CTAs in flight share one expert's slabs in L2.
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

template <bool kL1>
__global__ void __launch_bounds__(kThreads, 1)
    tc_w4_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX, W4Args args) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = smem_u32(smem_raw);
    const uint32_t base = (raw_base + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (base - raw_base);
    const uint32_t bars = base + kBarOff;
    auto raw_full = [&](int i) { return bars + 8u * i; };
    auto raw_empty = [&](int i) { return bars + 8u * (kRawStages + i); };
    constexpr int kHfBar = 2 * kRawStages;
    auto hf_full = [&](int i) { return bars + 8u * (kHfBar + i); };
    auto hf_empty = [&](int i) { return bars + 8u * (kHfBar + kHfStages + i); };
    constexpr int kTokBar = kHfBar + 2 * kHfStages;
    auto tok_full = [&](int i) { return bars + 8u * (kTokBar + i); };
    auto tok_empty = [&](int i) { return bars + 8u * (kTokBar + kTokStages + i); };
    constexpr int kAccBar = kTokBar + 2 * kTokStages;
    auto acc_full = [&](int a) { return bars + 8u * (kAccBar + a); };
    auto acc_empty = [&](int a) { return bars + 8u * (kAccBar + 2 + a); };
    const uint32_t drain_bar = bars + 8u * (kAccBar + 4);
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + kMiscOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kMiscOff + 4);
    int* tile_off = reinterpret_cast<int*>(smem + kTileOffOff);
    int* counts = reinterpret_cast<int*>(smem + kCountsOff);

    const Plan& p = args.p;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i <= p.E; i += kThreads) tile_off[i] = p.tile_off[i];
    for (int i = threadIdx.x; i < p.E; i += kThreads) counts[i] = p.counts[i];
    if (threadIdx.x == 0) {
        for (int i = 0; i < kRawStages; ++i) {
            mbar_init(raw_full(i), 1);
            mbar_init(raw_empty(i), 8);  // one arrival per converter warp
        }
        for (int i = 0; i < kHfStages; ++i) {
            mbar_init(hf_full(i), 8);
            mbar_init(hf_empty(i), 1);
        }
        for (int i = 0; i < kTokStages; ++i) {
            mbar_init(tok_full(i), 1);
            mbar_init(tok_empty(i), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(acc_full(a), 1);
            mbar_init(acc_empty(a), 4);  // the 4 epilogue warps
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
    auto tile_of = [&](int t) { return decode_tile(t, tile_off, counts, p.E, args.n_slabs); };

    if (warp == 0) {
        // ---------------- raw weight TMA: 256 rows x 32 bytes per stage ----------------
        if (lane == 0) {
            int it = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const Tile tl = tile_of(t);
                const int w0 = kL1 ? tl.e * args.n_out + tl.s * 128 : tl.e * args.n_out + tl.s * kWN;
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    const int r = it % kRawStages;
                    if (!mbar_wait(raw_empty(r), ((uint32_t)(it / kRawStages) & 1u) ^ 1u, p.hdr, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t dst = base + kRawOff + r * kRawBytes;
                    mbar_arrive_expect_tx(raw_full(r), kRawBytes);
                    if (kL1) {  // gate rows, then the up rows of the same outputs
                        tma_load_2d(dst, &tmW, kb * kRawRow, w0, raw_full(r));
                        tma_load_2d(dst + 128 * kRawRow, &tmW, kb * kRawRow, w0 + I, raw_full(r));
                    } else {
                        tma_load_2d(dst, &tmW, kb * kRawRow, w0, raw_full(r));
                    }
                }
            }
            for (int j = it - kRawStages < 0 ? 0 : it - kRawStages; j < it; ++j)
                mbar_drain(raw_full(j % kRawStages), (uint32_t)(j / kRawStages) & 1u, p.hdr);
        }
    } else if (warp == 2) {
        // ---------------- token TMA: 128 rows x 64 f16 per stage ----------------
        if (lane == 0) {
            int it = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const Tile tl = tile_of(t);
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    const int b = it % kTokStages;
                    if (!mbar_wait(tok_empty(b), ((uint32_t)(it / kTokStages) & 1u) ^ 1u, p.hdr, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t dst = base + kTokOff + b * kTokBytes;
                    mbar_arrive_expect_tx(tok_full(b), (uint32_t)kTokBytes);
                    tma_load_2d(dst, &tmX, kb * kBK, tl.row0, tok_full(b));
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
            const uint64_t ad0 = kmajor_desc(base + kTokOff, 0), bd0 = kmajor_desc(base + kHfOff, 0);
            int b = 0, tb = 0, tc = 0;
            uint32_t hph = 0, tph = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++tc) {
                const int a = tc & 1;
                if (!mbar_wait(acc_empty(a), ((uint32_t)(tc >> 1) & 1u) ^ 1u, p.hdr, abort_flag)) break;
                tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)(a * kWN);
                for (int kb = 0; kb < KB; ++kb) {
                    if (!(mbar_test(hf_full(b), hph) || mbar_wait(hf_full(b), hph, p.hdr, abort_flag)) ||
                        !(mbar_test(tok_full(tb), tph) || mbar_wait(tok_full(tb), tph, p.hdr, abort_flag))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = ad0 + (uint64_t)((tb * kTokBytes) >> 4);
                    const uint64_t bd = bd0 + (uint64_t)((b * kHfBytes) >> 4);
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk) tc_mma(d, ad + 2 * kk, bd + 2 * kk, kIdesc, (kb | kk) != 0);
                    tc_commit(hf_empty(b));
                    tc_commit(tok_empty(tb));
                    if (++b == kHfStages) b = 0, hph ^= 1u;
                    if (++tb == kTokStages) tb = 0, tph ^= 1u;
                }
                if (ok) tc_commit(acc_full(a));
            }
            tc_commit(drain_bar);
            mbar_drain(drain_bar, 0, p.hdr);
        }
    } else if (warp >= kConvWarp0) {
        // ---------------- converters: weight row c of the tile ----------------
        const int c = threadIdx.x - 32 * kConvWarp0;
        int it = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
            for (int kb = 0; kb < KB; ++kb, ++it) {
                const int r = it % kRawStages, b = it % kHfStages;
                bool w_ok = mbar_wait(raw_full(r), (uint32_t)(it / kRawStages) & 1u, p.hdr, abort_flag);
                w_ok = w_ok && mbar_wait(hf_empty(b), ((uint32_t)(it / kHfStages) & 1u) ^ 1u, p.hdr, abort_flag);
                if (!__all_sync(0xffffffffu, w_ok)) {
                    ok = false;
                    break;
                }
                // raw row c: 32 bytes, 32-byte swizzle (16-byte chunk index ^= address bit 7)
                const uint8_t* src = smem + kRawOff + r * kRawBytes + c * kRawRow;
                const int x = (c >> 2) & 1;
                const uint4 c0 = *reinterpret_cast<const uint4*>(src + ((0 ^ x) << 4));
                const uint4 c1 = *reinterpret_cast<const uint4*>(src + ((1 ^ x) << 4));
                const uint32_t wd[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
                uint8_t* dst = smem + kHfOff + b * kHfBytes + c * 128;
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {  // word ch: codes 8ch .. 8ch + 7 -> 16-byte chunk ch
                    uint32_t o[4];
                    int4x8_to_sub_f16(wd[ch], o);
                    *reinterpret_cast<uint4*>(dst + ((ch ^ (c & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
                }
                fence_proxy_async_smem();  // each thread's stores -> the MMA's async proxy
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(raw_empty(r));
                    mbar_arrive(hf_full(b));
                }
            }
        }
    } else if (warp >= kEpiWarp0) {
        // ---------------- epilogue (warps 4..7): thread = token row ----------------
        const int q = warp & 3;
        const int r = 32 * q + lane;
        int tc = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x, ++tc) {
            const int a = tc & 1;
            const uint32_t tb = tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(a * kWN);
            const Tile tl = tile_of(t);
            const bool valid = r < tl.n_valid;
            const int64_t row = tl.row0 + r;
            // this row's values, read while the tile's MMAs run
            const float sr = __ldg(args.row_scale + row);
            const int sum8 = (int)(8u * (uint32_t)__ldg(args.row_sums + row));
            int src = -1;
            float gw = 0.0f;
            if constexpr (!kL1) {
                src = valid ? debug_row(p.hdr, __ldg(p.pool_src + row), (int64_t)p.T * p.K) : -1;
                gw = src >= 0 ? __ldg(args.topk_weights + src) : 0.0f;
            }
            const bool w_ok = mbar_wait(acc_full(a), (uint32_t)(tc >> 1) & 1u, p.hdr, abort_flag);
            if (!__all_sync(0xffffffffu, w_ok)) break;
            tc_fence_after();
            auto release = [&]() {  // this warp's lanes of the accumulator are in registers
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(acc_empty(a));
            };
            // exact integer from the accumulator: 2^24 D is an integer below 2^24 (padding rows
            // hold anything; unsigned arithmetic keeps their discarded values defined)
            auto exact = [&](uint32_t bits) {
                const int c = (int)((uint32_t)__float2int_rn(__uint_as_float(bits) * 16777216.0f) - (uint32_t)sum8);
                return __int2float_rn(c);
            };
            if constexpr (kL1) {
                // H = (C * s^W1) * s^X; A = SiLU(H_gate) * H_up for outputs 128s + 16c .. +15
                const float* s1 = args.w_scale + (int64_t)tl.e * 2 * I + tl.s * 128;  // gate; up at + I
                float* arow = p.a_f32 + row * I + tl.s * 128;
#pragma unroll 1
                for (int c = 0; c < 8; ++c) {
                    uint32_t g[16], u[16];
                    tmem_ld16(tb + 16 * c, g);
                    tmem_ld16(tb + 128 + 16 * c, u);
                    tmem_ld_wait();
                    if (c == 7) release();
                    uint32_t out[16];
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {  // the scales: one address across the warp
                        const float Hg = __fmul_rn(__fmul_rn(exact(g[jj]), __ldg(s1 + 16 * c + jj)), sr);
                        const float Hu = __fmul_rn(__fmul_rn(exact(u[jj]), __ldg(s1 + I + 16 * c + jj)), sr);
                        out[jj] = __float_as_uint(swiglu1(Hg, Hu, p.act_clamp));
                    }
                    st_global_v8_if(valid, arow + 16 * c, out);
                    st_global_v8_if(valid, arow + 16 * c + 8, out + 8);
                }
            } else {
                // Y = (D * s^W2) * s^A; c = bf16(G * Y) for hidden columns 256s + 16c .. +15
                const float* s2 = args.w_scale + (int64_t)tl.e * H + tl.s * kWN;
                uint16_t* dst = p.comb + (int64_t)(src >= 0 ? src : 0) * H + tl.s * kWN;
#pragma unroll 1
                for (int c = 0; c < kWN / 16; ++c) {
                    uint32_t d[16];
                    tmem_ld16(tb + 16 * c, d);
                    tmem_ld_wait();
                    if (c == kWN / 16 - 1) release();
                    uint32_t out[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const float y0 = __fmul_rn(__fmul_rn(exact(d[2 * k]), __ldg(s2 + 16 * c + 2 * k)), sr);
                        const float y1 = __fmul_rn(__fmul_rn(exact(d[2 * k + 1]), __ldg(s2 + 16 * c + 2 * k + 1)), sr);
                        out[k] = (uint32_t)float_to_bf16_bits(__fmul_rn(gw, y0)) |
                                 ((uint32_t)float_to_bf16_bits(__fmul_rn(gw, y1)) << 16);
                    }
                    st_global_v8_if(src >= 0, dst + 16 * c, out);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, 512);
}

template <bool kL1>
cudaError_t launch_w4(const Plan& p, const void* w, const void* w_scale, const float* topk_weights, cudaStream_t s) {
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(tc_w4_kernel<kL1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
    });
    if (attr_err != cudaSuccess) return attr_err;
    const int n_out = kL1 ? 2 * p.I : p.H;
    const int kin = kL1 ? p.H : p.I;
    CUtensorMap tmW, tmX;
    // packed weights as bytes [E * n_out, kin / 2]; L1 boxes take 128 rows (gate, then up)
    if (!tc_make_map_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, w, (uint64_t)kin / 2, (uint64_t)p.E * n_out, kRawRow,
                        kL1 ? 128 : kWN, CU_TENSOR_MAP_SWIZZLE_32B))
        return cudaErrorInvalidValue;
    const uint16_t* planes = kL1 ? p.x_planes : p.a_planes;
    if (!tc_make_map_2d(&tmX, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, planes, (uint64_t)kin, (uint64_t)p.pool_rows, kBK, kTM,
                        CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    W4Args args{p,
                static_cast<const float*>(w_scale),
                topk_weights,
                planes,
                reinterpret_cast<const float*>(kL1 ? p.x_pool_scale : p.a_pool_scale),
                kL1 ? p.x_sums : p.a_sums,
                kL1 ? p.I / 128 : p.H / kWN,
                kin / kBK,
                n_out};
    const int64_t max_tiles = (p.pool_rows / kTM) * args.n_slabs;
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(max_tiles, tc_num_sms()));
    tc_w4_kernel<kL1><<<grid, kThreads, kSmem, s>>>(tmW, tmX, args);
    return cudaGetLastError();
}

}  // namespace

bool w4_tc_supported(const Plan& p, int stage) {
    if (p.mode != MOE_A8W4_INT || p.E > kMaxExperts || !tc_encode_available()) return false;
    if (stage == 1) return p.I % 128 == 0 && p.H % kBK == 0 && p.H <= kMaxK;
    return p.H % kWN == 0 && p.I % kBK == 0 && p.I <= kMaxK;
}

cudaError_t launch_l1_w4_tc(const Plan& p, const void* w1, const void* w1_scale, cudaStream_t s) {
    return launch_w4<true>(p, w1, w1_scale, nullptr, s);
}

cudaError_t launch_l2_w4_tc(const Plan& p, const void* w2, const void* w2_scale, const float* topk_weights,
                            cudaStream_t s) {
    return launch_w4<false>(p, w2, w2_scale, topk_weights, s);
}

}  // namespace moe
