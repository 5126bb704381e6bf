// Dense tensor-core rate of the tcgen05 instruction kinds the GEMM stages issue: every CTA keeps
// one A tile (128 rows) and one B tile (256 rows) of 128-byte K-major rows in shared memory and
// one thread issues M = 128, N = 256 MMAs over them back to back into a tensor-memory
// accumulator. No global memory is read, so a launch timed with events measures the tensor pipe
// alone, at the clocks of the moment. The operands hold finite pseudo-random values of the
// kind's element types (toggling bits draw the power that real data draws; zeros would not).
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"
#include "moe_peak.h"
#include "tc_common.cuh"

namespace moe {

namespace {

using namespace tc;

constexpr int kM = 128, kN = 256;
constexpr int kThreads = 128;
constexpr int kABytes = kM * 128, kBBytes = kN * 128;  // one 128-byte swizzle row per operand row
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfCol = 256;  // scale-factor columns after the 256 accumulator columns
constexpr size_t kSmem = 1024 + kABytes + kBBytes + 64;
constexpr int kProbeRecordOffset = 128;  // workspace bytes [128, 144): CTA 0's cycles and nanoseconds

__device__ __forceinline__ uint32_t mix32(uint32_t x) {
    x ^= x >> 16;
    x *= 0x7feb352du;
    x ^= x >> 15;
    x *= 0x846ca68bu;
    x ^= x >> 16;
    return x;
}

// A 32-bit word of finite operand values: bf16 and f16 halves with moderate exponents; e4m3 bytes
// with exponent fields 4..11 (never the NaN code); e2m1 codes are all finite.
template <int KIND>
__device__ __forceinline__ uint32_t operand_word(uint32_t r, bool b_operand) {
    if constexpr (KIND == MOE_PEAK_BF16) {
        const uint32_t lo = ((r & 1u) << 15) | ((120u + ((r >> 1) & 7u)) << 7) | ((r >> 4) & 0x7fu);
        const uint32_t hi = (((r >> 11) & 1u) << 15) | ((120u + ((r >> 12) & 7u)) << 7) | ((r >> 15) & 0x7fu);
        return lo | (hi << 16);
    } else if constexpr (KIND == MOE_PEAK_F16) {
        const uint32_t lo = ((r & 1u) << 15) | ((8u + ((r >> 1) & 7u)) << 10) | ((r >> 4) & 0x3ffu);
        const uint32_t hi = (((r >> 14) & 1u) << 15) | ((8u + ((r >> 15) & 7u)) << 10) | ((r >> 18) & 0x3ffu);
        return lo | (hi << 16);
    } else {
        if (KIND == MOE_PEAK_E4M3_E2M1 && b_operand) return r;  // e2m1 weights
        uint32_t w = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t b = (r >> (8 * i)) & 0xffu;
            w |= ((b & 0x80u) | ((4u + ((b >> 3) & 7u)) << 3) | (b & 7u)) << (8 * i);
        }
        return w;
    }
}

// kind::f16: D fp32 (bits 4-5 = 1), A and B types (7-9, 10-12: f16 0, bf16 1), both K-major,
// N >> 3 (17-22), M >> 4 (24-28). kind::mxf8f6f4.block_scale: B scale id (4-5), A type e4m3 (0),
// B type e4m3 (0) or e2m1 (5), N >> 3, UE8M0 scales (bit 23), M >> 4, A scale id (29-30).
template <int KIND>
__device__ __forceinline__ uint32_t probe_idesc(int sf_id) {
    constexpr uint32_t mn = ((uint32_t)(kN >> 3) << 17) | ((uint32_t)(kM >> 4) << 24);
    if constexpr (KIND == MOE_PEAK_BF16) return (1u << 4) | (1u << 7) | (1u << 10) | mn;
    else if constexpr (KIND == MOE_PEAK_F16) return (1u << 4) | mn;
    else {
        constexpr uint32_t bfmt = KIND == MOE_PEAK_E4M3_E2M1 ? 5u : 0u;
        return ((uint32_t)sf_id << 4) | (bfmt << 10) | (1u << 23) | mn | ((uint32_t)sf_id << 29);
    }
}

__device__ __forceinline__ void bs_mma(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t sfa,
                                       uint32_t sfb, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
        ::"r"(d), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
        : "memory");
}

template <int KIND>
__global__ void __launch_bounds__(kThreads, 1) tensor_peak_kernel(int64_t iters, int32_t* hdr) {
    constexpr bool kBlockScaled = KIND == MOE_PEAK_E4M3_E2M1 || KIND == MOE_PEAK_E4M3_E4M3;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint32_t* tiles = reinterpret_cast<uint32_t*>(smem);
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kABytes + kBBytes);
    uint32_t* holder = reinterpret_cast<uint32_t*>(bar + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    for (int i = threadIdx.x; i < (kABytes + kBBytes) / 4; i += kThreads)
        tiles[i] = operand_word<KIND>(mix32((uint32_t)i * 2654435761u + blockIdx.x), i >= kABytes / 4);
    fence_proxy_async_smem();  // the tiles become visible to the tensor cores' (async) reads
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(bar), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) tmem_alloc(smem_u32(holder), kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *holder;
    if constexpr (kBlockScaled) {  // every scale factor 2^0 (UE8M0 127), in all 128 lanes
        uint32_t v[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = 0x7f7f7f7fu;
        asm volatile(
            "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
            "%15, %16};" ::"r"(tmem + ((uint32_t)(32 * warp) << 16) + kSfCol),
            "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
            "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
            : "memory");
        tmem_st_wait();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    if (warp == 0 && lane == 0) {
        const uint64_t c0 = clock64(), t0 = globaltimer_ns();
        const uint32_t a = smem_u32(tiles);
        const uint64_t ad = kmajor_desc(a, 0), bd = kmajor_desc(a + kABytes, 0);
        uint32_t idesc[4];
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) idesc[kk] = probe_idesc<KIND>(kk);
        for (int64_t i = 0; i < iters; ++i) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {  // the four 32-byte K slices of the 128-byte rows
                const uint32_t acc = (i | kk) != 0;
                if constexpr (kBlockScaled)
                    bs_mma(tmem, ad + 2 * kk, bd + 2 * kk, idesc[kk], tmem + kSfCol, tmem + kSfCol + 4, acc);
                else
                    tc_mma(tmem, ad + 2 * kk, bd + 2 * kk, idesc[kk], acc);
            }
        }
        tc_commit(smem_u32(bar));
        mbar_drain(smem_u32(bar), 0, hdr);  // bounded; the MMAs in flight take microseconds
        if (blockIdx.x == 0) {  // SM clock cycles and nanoseconds of CTA 0's MMA stream
            int64_t* rec = reinterpret_cast<int64_t*>(hdr + kProbeRecordOffset / 4);
            rec[0] = (int64_t)(clock64() - c0);
            rec[1] = (int64_t)(globaltimer_ns() - t0);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

template <int KIND>
cudaError_t launch_probe(int64_t iters, int grid, int32_t* hdr, cudaStream_t s) {
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [] {
        attr = cudaFuncSetAttribute(tensor_peak_kernel<KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
    });
    if (attr != cudaSuccess) return attr;
    tensor_peak_kernel<KIND><<<grid, kThreads, kSmem, s>>>(iters, hdr);
    return cudaGetLastError();
}

}  // namespace

}  // namespace moe

using namespace moe;

extern "C" MOE_API moe_status moe_tensor_peak_probe(moe_peak_kind kind, int64_t iters_per_cta, int grid,
                                                    double* flops_out, void* workspace, size_t workspace_bytes,
                                                    moe_stream_t stream) {
    if (kind < MOE_PEAK_BF16 || kind > MOE_PEAK_E4M3_E4M3 || iters_per_cta < 1 || !flops_out)
        return MOE_ERR_INVALID_ARG;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255) || workspace_bytes < 256) return MOE_ERR_WORKSPACE;
    if (grid <= 0) grid = tc_num_sms();
    const double k = (kind == MOE_PEAK_BF16 || kind == MOE_PEAK_F16) ? 16.0 : 32.0;
    *flops_out = 2.0 * kM * kN * k * 4.0 * (double)iters_per_cta * grid;
    int32_t* hdr = static_cast<int32_t*>(workspace);
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    switch (kind) {
        case MOE_PEAK_BF16: e = launch_probe<MOE_PEAK_BF16>(iters_per_cta, grid, hdr, s); break;
        case MOE_PEAK_F16: e = launch_probe<MOE_PEAK_F16>(iters_per_cta, grid, hdr, s); break;
        case MOE_PEAK_E4M3_E2M1: e = launch_probe<MOE_PEAK_E4M3_E2M1>(iters_per_cta, grid, hdr, s); break;
        default: e = launch_probe<MOE_PEAK_E4M3_E4M3>(iters_per_cta, grid, hdr, s); break;
    }
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
