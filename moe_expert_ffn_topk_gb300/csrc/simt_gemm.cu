// CUDA-core reference kernels of the grouped GEMM stages, one template per dtype mode.
//
// They run stages S3-S5 with plain fp32 FMAs (int32 multiply-adds in the INT8 mode) on
// 64-row tiles of the per-expert pool. They are the correctness reference for the
// tensor-core kernels and the path of any mode / shape without a tensor-core kernel; they
// make no attempt at speed.
//
// L1 (Ascend mega_moe page, "Linear1 Projection" + "SwiGLU Activation"; A8W8-INT Linear1
// dequantisation H = (C * s^W1) * s^X): each CTA owns 64 pool rows and 32 output columns j of
// A, so it accumulates the gate columns j and the up columns I + j side by side and applies
// SwiGLU in its epilogue. The epilogue writes the L2 operand: bf16 A, or e4m3 + UE8M0 for a
// 1x32 block (the CTA holds the whole block), or fp32 A for the INT8 mode, whose per-row
// scale needs the whole row and runs in int8_row_quant_kernel.
//
// L2 ("Linear2 Projection" + the gate weight of "Token Combine"): 64 rows x 64 hidden
// columns per CTA; epilogue c = bf16(G[i,k] * Y) written to combine row i*K + k.
#include <cuda_runtime.h>

#include <type_traits>

#include "common.cuh"
#include "internal.h"
#include "tc_common.cuh"  // tc_num_sms

namespace moe {

namespace {

constexpr int BM = 64, BN = 64, BK = 32, NT = 256;

// Expert owning padded pool row r: the largest e with pad_off[e] <= r.
__device__ __forceinline__ int expert_of_row(const int32_t* pad_off, int E, int r) {
    int lo = 0, hi = E - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (pad_off[mid] <= r) lo = mid; else hi = mid - 1;
    }
    return lo;
}

template <int MODE>
using acc_t = typename std::conditional<int_mode(MODE), int, float>::type;

// Element k of pool row p of the L1 operand (gathered x).
template <int MODE>
__device__ __forceinline__ acc_t<MODE> load_x(const uint8_t* xp, const uint8_t* xs, int H, int64_t p, int k) {
    if constexpr (MODE == MOE_A16W16) {
        return bf16_bits_to_float(reinterpret_cast<const uint16_t*>(xp)[p * H + k]);
    } else if constexpr (MODE == MOE_A8W8_FP8 || MODE == MOE_A8W8_FP8_E5M2) {
        return fp8_to_float<MODE == MOE_A8W8_FP8_E5M2>(xp[p * H + k]) * ue8m0_to_float(xs[p * (H / 32) + k / 32]);
    } else if constexpr (int_mode(MODE)) {
        return static_cast<int>(reinterpret_cast<const int8_t*>(xp)[p * H + k]);
    } else {
        return e4m3_to_float(xp[p * H + k]) * reinterpret_cast<const float*>(xs)[p * (H / 128) + k / 128];
    }
}

// Element (k, n) of expert e's weight in the math orientation [K_in, N_out].
// A16W16 stores [E, K_in, N_out]; every other mode stores [E, N_out, K_in] (+ scales).
template <int MODE>
__device__ __forceinline__ acc_t<MODE> load_w(const uint8_t* w, const uint8_t* ws, int e, int Kin, int Nout, int k,
                                              int n) {
    const int64_t en = (int64_t)e * Nout + n;
    if constexpr (MODE == MOE_A16W16) {
        return bf16_bits_to_float(reinterpret_cast<const uint16_t*>(w)[((int64_t)e * Kin + k) * Nout + n]);
    } else if constexpr (MODE == MOE_A8W8_FP8 || MODE == MOE_A8W8_FP8_E5M2) {
        return fp8_to_float<MODE == MOE_A8W8_FP8_E5M2>(w[en * Kin + k]) * ue8m0_to_float(ws[en * (Kin / 32) + k / 32]);
    } else if constexpr (MODE == MOE_A8W8_INT8) {
        return static_cast<int>(reinterpret_cast<const int8_t*>(w)[en * Kin + k]);
    } else if constexpr (MODE == MOE_A8W4_INT) {
        const uint8_t b = w[en * (Kin / 2) + k / 2];
        const int n = (k & 1) ? (b >> 4) : (b & 0xF);
        return n >= 8 ? n - 16 : n;  // two's-complement nibble
    } else {
        const uint8_t b = w[en * (Kin / 2) + k / 2];
        return e2m1_to_float((k & 1) ? (b >> 4) : (b & 0xF)) * ue8m0_to_float(ws[en * (Kin / 32) + k / 32]);
    }
}

// Element j of pool row p of the L2 operand A.
template <int MODE>
__device__ __forceinline__ acc_t<MODE> load_a(const uint8_t* ap, const uint8_t* as, int I, int64_t p, int j) {
    if constexpr (MODE == MOE_A16W16) {
        return bf16_bits_to_float(reinterpret_cast<const uint16_t*>(ap)[p * I + j]);
    } else if constexpr (int_mode(MODE)) {
        return static_cast<int>(reinterpret_cast<const int8_t*>(ap)[p * I + j]);
    } else {
        return fp8_to_float<MODE == MOE_A8W8_FP8_E5M2>(ap[p * I + j]) * ue8m0_to_float(as[p * (I / 32) + j / 32]);
    }
}

template <int MODE>
__global__ void __launch_bounds__(NT) l1_simt_kernel(Plan p, const uint8_t* __restrict__ w1,
                                                     const uint8_t* __restrict__ w1s) {
    using T = acc_t<MODE>;
    __shared__ T As[BK][BM + 1];
    __shared__ T Bs[BK][BN + 1];
    const int r0 = blockIdx.y * BM;
    if (r0 >= p.hdr[kHdrPadRows]) return;
    const int jb = blockIdx.x;  // 32 columns of A: gate jb*32.. and up I + jb*32..
    const int H = p.H, I = p.I;
    const int e = expert_of_row(p.pad_off, p.E, r0);
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    T acc[4][4] = {};
    constexpr bool kMajorW = MODE != MOE_A16W16;
    for (int k0 = 0; k0 < H; k0 += BK) {
        for (int q = tid; q < BM * BK; q += NT) {
            const int r = q / BK, k = q % BK;
            As[k][r] = load_x<MODE>(p.x_pool, p.x_pool_scale, H, r0 + r, k0 + k);
        }
        for (int q = tid; q < BN * BK; q += NT) {
            const int c = kMajorW ? q / BK : q % BN;
            const int k = kMajorW ? q % BK : q / BN;
            const int n = c < 32 ? jb * 32 + c : I + jb * 32 + (c - 32);
            Bs[k][c] = load_w<MODE>(w1, w1s, e, H, 2 * I, k0 + k, n);
        }
        __syncthreads();
#pragma unroll 4
        for (int k = 0; k < BK; ++k) {
            T a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = As[k][ty * 4 + i];
            b[0] = Bs[k][tx * 2];
            b[1] = Bs[k][tx * 2 + 1];
            b[2] = Bs[k][32 + tx * 2];
            b[3] = Bs[k][32 + tx * 2 + 1];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[i][c] += a[i] * b[c];
        }
        __syncthreads();
    }
    // Epilogue: SwiGLU of (gate j, up j) for j = jb*32 + tx*2 + {0,1}
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t row = r0 + ty * 4 + i;
        const int j0 = jb * 32 + tx * 2;
        float g[2], u[2];
        if constexpr (int_mode(MODE)) {
            const float sx = reinterpret_cast<const float*>(p.x_pool_scale)[row];
            const float* s1 = reinterpret_cast<const float*>(w1s) + (int64_t)e * 2 * I;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                g[c] = __fmul_rn(__fmul_rn(__int2float_rn(acc[i][c]), s1[j0 + c]), sx);
                u[c] = __fmul_rn(__fmul_rn(__int2float_rn(acc[i][2 + c]), s1[I + j0 + c]), sx);
            }
        } else {
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                g[c] = acc[i][c];
                u[c] = acc[i][2 + c];
            }
        }
        float a[2];
#pragma unroll
        for (int c = 0; c < 2; ++c) a[c] = swiglu1(g[c], u[c], p.act_clamp);
        if constexpr (MODE == MOE_A16W16) {
            uint16_t* ap = reinterpret_cast<uint16_t*>(p.a_pool);
            ap[row * I + j0] = float_to_bf16_bits(a[0]);
            ap[row * I + j0 + 1] = float_to_bf16_bits(a[1]);
        } else if constexpr (int_mode(MODE)) {
            p.a_f32[row * I + j0] = a[0];
            p.a_f32[row * I + j0 + 1] = a[1];
        } else {
            // MX re-quantisation of the 1x32 block jb of this row (16 lanes hold it)
            float amax = fmaxf(fabsf(a[0]), fabsf(a[1]));
#pragma unroll
            for (int o = 8; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
            constexpr bool kE5 = MODE == MOE_A8W8_FP8_E5M2;
            const int ex = mx_exponent_fp8<kE5>(amax);
            const float inv = exp2_neg_int(ex);
            const uint8_t c0 = float_to_fp8_satfinite<kE5>(a[0] * inv), c1 = float_to_fp8_satfinite<kE5>(a[1] * inv);
            p.a_pool[row * I + j0] = c0;
            p.a_pool[row * I + j0 + 1] = c1;
            if (tx == 0) p.a_pool_scale[row * (I / 32) + jb] = static_cast<uint8_t>(ex + 127);
        }
    }
}

template <int MODE>
__global__ void __launch_bounds__(NT) l2_simt_kernel(Plan p, const uint8_t* __restrict__ w2,
                                                     const uint8_t* __restrict__ w2s,
                                                     const float* __restrict__ topk_weights) {
    using T = acc_t<MODE>;
    __shared__ T As[BK][BM + 1];
    __shared__ T Bs[BK][BN + 1];
    const int r0 = blockIdx.y * BM;
    if (r0 >= p.hdr[kHdrPadRows]) return;
    const int h0 = blockIdx.x * BN;
    const int H = p.H, I = p.I;
    const int e = expert_of_row(p.pad_off, p.E, r0);
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    T acc[4][4] = {};
    constexpr bool kMajorW = MODE != MOE_A16W16;
    for (int k0 = 0; k0 < I; k0 += BK) {
        for (int q = tid; q < BM * BK; q += NT) {
            const int r = q / BK, k = q % BK;
            As[k][r] = load_a<MODE>(p.a_pool, p.a_pool_scale, I, r0 + r, k0 + k);
        }
        for (int q = tid; q < BN * BK; q += NT) {
            const int c = kMajorW ? q / BK : q % BN;
            const int k = kMajorW ? q % BK : q / BN;
            Bs[k][c] = load_w<MODE>(w2, w2s, e, I, H, k0 + k, h0 + c);
        }
        __syncthreads();
#pragma unroll 4
        for (int k = 0; k < BK; ++k) {
            T a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = As[k][ty * 4 + i];
#pragma unroll
            for (int c = 0; c < 4; ++c) b[c] = Bs[k][tx * 4 + c];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[i][c] += a[i] * b[c];
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t row = r0 + ty * 4 + i;
        const int src = debug_row(p.hdr, p.pool_src[row], (int64_t)p.T * p.K);
        if (src < 0) continue;  // padding row
        const float g = topk_weights[src];
        uint16_t out[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            float y;
            if constexpr (int_mode(MODE)) {
                const float s2 = reinterpret_cast<const float*>(w2s)[(int64_t)e * H + h0 + tx * 4 + c];
                const float sa = reinterpret_cast<const float*>(p.a_pool_scale)[row];
                y = __fmul_rn(__fmul_rn(__int2float_rn(acc[i][c]), s2), sa);
            } else {
                y = acc[i][c];
            }
            out[c] = float_to_bf16_bits(__fmul_rn(g, y));
        }
        uint2 v = make_uint2(out[0] | ((uint32_t)out[1] << 16), out[2] | ((uint32_t)out[3] << 16));
        *reinterpret_cast<uint2*>(p.comb + (int64_t)src * H + h0 + tx * 4) = v;
    }
}

// Integer modes, Linear2 step (1) of the A8W8-INT and A8W4-INT use cases (quant_a_row): one warp
// per pool row, 64 rows in flight per SM.
constexpr int kRqWarps = 8;
__global__ void __launch_bounds__(32 * kRqWarps) int8_row_quant_kernel(Plan p) {
    const int rows = p.hdr[kHdrPadRows];
    const int lane = threadIdx.x & 31;
    for (int r = blockIdx.x * kRqWarps + (threadIdx.x >> 5); r < rows; r += gridDim.x * kRqWarps)
        quant_a_row<false, 16>(p, r, lane);
}

template <int MODE>
cudaError_t l1_launch(const Plan& p, const void* w1, const void* w1s, cudaStream_t s) {
    dim3 grid(p.I / 32, (unsigned)((p.pool_rows + BM - 1) / BM));
    l1_simt_kernel<MODE><<<grid, NT, 0, s>>>(p, static_cast<const uint8_t*>(w1), static_cast<const uint8_t*>(w1s));
    return cudaGetLastError();
}

template <int MODE>
cudaError_t l2_launch(const Plan& p, const void* w2, const void* w2s, const float* g, cudaStream_t s) {
    dim3 grid(p.H / BN, (unsigned)((p.pool_rows + BM - 1) / BM));
    l2_simt_kernel<MODE><<<grid, NT, 0, s>>>(p, static_cast<const uint8_t*>(w2), static_cast<const uint8_t*>(w2s), g);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_l1_simt(const Plan& p, const void* w1, const void* w1_scale, cudaStream_t s) {
    if (p.pool_rows == 0) return cudaSuccess;
    switch (p.mode) {
        case MOE_A16W16: return l1_launch<MOE_A16W16>(p, w1, w1_scale, s);
        case MOE_A8W8_FP8: return l1_launch<MOE_A8W8_FP8>(p, w1, w1_scale, s);
        case MOE_A8W8_FP8_E5M2: return l1_launch<MOE_A8W8_FP8_E5M2>(p, w1, w1_scale, s);
        case MOE_A8W8_INT8: return l1_launch<MOE_A8W8_INT8>(p, w1, w1_scale, s);
        case MOE_A8W4_FP8_FP4: return l1_launch<MOE_A8W4_FP8_FP4>(p, w1, w1_scale, s);
        case MOE_A8W4_INT: return l1_launch<MOE_A8W4_INT>(p, w1, w1_scale, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_l2_simt(const Plan& p, const void* w2, const void* w2_scale, const float* topk_weights,
                           cudaStream_t s) {
    if (p.pool_rows == 0) return cudaSuccess;
    switch (p.mode) {
        case MOE_A16W16: return l2_launch<MOE_A16W16>(p, w2, w2_scale, topk_weights, s);
        case MOE_A8W8_FP8: return l2_launch<MOE_A8W8_FP8>(p, w2, w2_scale, topk_weights, s);
        case MOE_A8W8_FP8_E5M2: return l2_launch<MOE_A8W8_FP8_E5M2>(p, w2, w2_scale, topk_weights, s);
        case MOE_A8W8_INT8: return l2_launch<MOE_A8W8_INT8>(p, w2, w2_scale, topk_weights, s);
        case MOE_A8W4_FP8_FP4: return l2_launch<MOE_A8W4_FP8_FP4>(p, w2, w2_scale, topk_weights, s);
        case MOE_A8W4_INT: return l2_launch<MOE_A8W4_INT>(p, w2, w2_scale, topk_weights, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_int8_row_quant(const Plan& p, cudaStream_t s) {
    if (p.pool_rows == 0) return cudaSuccess;
    // a row per warp, 64 rows in flight per SM (8 resident blocks of 8 warps)
    const int grid = (int)std::min<int64_t>((p.pool_rows + kRqWarps - 1) / kRqWarps, (int64_t)tc_num_sms() * 8);
    int8_row_quant_kernel<<<grid, 32 * kRqWarps, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace moe
