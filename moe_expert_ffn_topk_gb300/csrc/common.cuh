// Device helpers shared by the kernels of the library.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <cmath>
#include <stdint.h>

#include "internal.h"

namespace moe {

// ---------------------------------------------------------------------------------------
// Error word: the first error recorded wins.
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ void record_error(int32_t* hdr, int code) {
    atomicCAS(&hdr[kErrWord], 0, code);
}

// Index checks of the debug build (compiled with -DMOE_DEBUG): a data-dependent row index outside
// [-1, n) records MOE_ERR_BOUNDS and comes back as -1, so the caller skips the row as padding. In
// the default build both helpers return their argument and compile to nothing.
__device__ __forceinline__ int debug_row(int32_t* hdr, int idx, int64_t n) {
#ifdef MOE_DEBUG
    if (idx < -1 || idx >= n) {
        record_error(hdr, MOE_ERR_BOUNDS);
        return -1;
    }
#else
    (void)hdr;
    (void)n;
#endif
    return idx;
}

__device__ __forceinline__ bool debug_ok(int32_t* hdr, bool ok) {
#ifdef MOE_DEBUG
    if (!ok) record_error(hdr, MOE_ERR_BOUNDS);
    return ok;
#else
    (void)hdr;
    (void)ok;
    return true;
#endif
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------------------------------
// Number formats (from the bit layouts of the formats)
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__device__ __forceinline__ uint16_t float_to_bf16_bits(float v) {
    __nv_bfloat16 h = __float2bfloat16_rn(v);
    return *reinterpret_cast<uint16_t*>(&h);
}

__device__ __forceinline__ uint16_t float_to_f16_bits(float v) { return __half_as_ushort(__float2half_rn(v)); }

// e4m3fn code -> float (exact), via the fp8 conversion of cuda_fp8.h
__device__ __forceinline__ float e4m3_to_float(uint8_t c) {
    __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(c), __NV_E4M3);
    return __half2float(__half(h));
}

// float -> e4m3fn code, round to nearest even, saturating to +-448 (the PTX conversion: of the
// two converted operands the second lands in the low byte)
__device__ __forceinline__ uint8_t float_to_e4m3_satfinite(float v) {
    uint16_t pair;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(pair) : "f"(0.0f), "f"(v));
    return static_cast<uint8_t>(pair & 0xffu);
}

// e2m1 code (low 4 bits) -> float: sign | 2 exponent bits (bias 1) | 1 mantissa bit
__device__ __forceinline__ float e2m1_to_float(uint32_t c) {
    const uint32_t e = (c >> 1) & 3u, m = c & 1u;
    float mag = (e == 0) ? 0.5f * static_cast<float>(m)
                         : (1.0f + 0.5f * static_cast<float>(m)) * static_cast<float>(1u << (e - 1));
    return (c & 8u) ? -mag : mag;
}

// UE8M0 byte -> 2^(s-127) as float (s in [1, 254] is a normal float; s = 0 is 2^-127)
__device__ __forceinline__ float ue8m0_to_float(uint8_t s) {
    return s == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(static_cast<uint32_t>(s) << 23);
}

// Shared exponent of an MX block: the smallest e with amax <= emax * 2^e, clamped to
// [-127, 127]; amax = 0 gives -127. For emax = 448 = 0.875 * 2^9: with amax = m * 2^x,
// m in [0.5, 1), amax / 448 lies in (2^(x-10), 2^(x-9)] when m <= 0.875, else in
// (2^(x-9), 2^(x-8)).
// Read from the bits: a normal amax has x = (biased exponent) - 126 and m <= 0.875 exactly when
// its 23 fraction bits are <= 0.75 * 2^23; a subnormal amax gives x <= -125, so e = -127.
__device__ __forceinline__ int mx_exponent_e4m3(float amax) {
    if (!(amax > 0.0f)) return -127;
    const uint32_t bits = __float_as_uint(amax);
    const int be = (int)(bits >> 23);
    if (be == 0) return -127;
    const int e = (bits & 0x7fffffu) <= 0x600000u ? be - 126 - 9 : be - 126 - 8;
    return e > 127 ? 127 : e;
}

// e5m2 code -> float (exact), via the fp8 conversion of cuda_fp8.h
__device__ __forceinline__ float e5m2_to_float(uint8_t c) {
    __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(c), __NV_E5M2);
    return __half2float(__half(h));
}

// float -> e5m2 code, round to nearest even, saturating to +-57344 (the PTX conversion)
__device__ __forceinline__ uint8_t float_to_e5m2_satfinite(float v) {
    uint16_t pair;
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(pair) : "f"(0.0f), "f"(v));
    return static_cast<uint8_t>(pair & 0xffu);
}

// Shared exponent of an MX block for e5m2: the smallest e with amax <= 57344 * 2^e. As
// 57344 = 448 * 2^7 this is the e4m3 exponent minus 7 (clamped to [-127, 127] the same way).
__device__ __forceinline__ int mx_exponent_e5m2(float amax) {
    const int e = mx_exponent_e4m3(amax) - 7;
    return e < -127 ? -127 : e;
}

// The FP8 element type of an A8W8-FP mode: e5m2 when kE5, else e4m3.
template <bool kE5>
__device__ __forceinline__ float fp8_to_float(uint8_t c) {
    if constexpr (kE5) return e5m2_to_float(c);
    else return e4m3_to_float(c);
}
template <bool kE5>
__device__ __forceinline__ uint8_t float_to_fp8_satfinite(float v) {
    if constexpr (kE5) return float_to_e5m2_satfinite(v);
    else return float_to_e4m3_satfinite(v);
}
template <bool kE5>
__device__ __forceinline__ int mx_exponent_fp8(float amax) {
    if constexpr (kE5) return mx_exponent_e5m2(amax);
    else return mx_exponent_e4m3(amax);
}

// 2^-e as float for e in [-127, 126] (exact power of two)
__device__ __forceinline__ float exp2_neg_int(int e) {
    return __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
}

// SiLU(z) = z / (1 + e^-z) with the approximate exp and divide (a few ulp of fp32, far below
// the bf16 / e4m3 rounding that follows, and branch-free; for z < -87 the quotient is -0)
__device__ __forceinline__ float silu(float z) {
    return __fdividef(z, 1.0f + __expf(-z));
}

// SwiGLU on one (gate, up) pair with the operator's activation_clamp (Ascend page, parameter
// activation_clamp: both inputs clipped to [-c, c]; c = +inf leaves them as they are). A select,
// not a branch, so epilogue loops stay branch-free.
__device__ __forceinline__ float swiglu1(float g, float u, float c) {
    const bool on = c < INFINITY;
    g = on ? fminf(fmaxf(g, -c), c) : g;
    u = on ? fminf(fmaxf(u, -c), c) : u;
    return silu(g) * u;
}

// ---------------------------------------------------------------------------------------
// Integer modes, Linear2 step (1) of the A8W8-INT and A8W4-INT use cases (Ascend mega_moe
// page): s = max|A[row,:]| / 127 (floored at 1e-8), q = round-half-even(A / s) clamped to
// [-127, 127]; fp32 IEEE division throughout. Besides the int8 codes it writes the tensor-core
// operand planes: hi = floor(q / 16) and lo = q mod 16 as f16 for INT8; for A8W4-INT the codes
// as f16 in the order of w4_plane_pos, and the row's code sum. One warp per pool row (all 32
// lanes call it with the same r); padding rows are skipped. A row of up to 128 * kRegVec elements
// stays in registers between the amax pass and the quantisation pass (all of a lane's loads in
// flight at once); longer rows are read twice. kCoherent: A is read through L2 (ld.global.cg), for rows that
// other CTAs of the same launch wrote (the caller has ordered those writes before this call). The
// amax, the codes and the code sum do not depend on the order of the loads: the results are the
// same bits either way.
// ---------------------------------------------------------------------------------------
template <bool kCoherent>
__device__ __forceinline__ float4 load_a4(const float4* p) {
    if constexpr (kCoherent) return __ldcg(p);
    else return *p;
}

__device__ __forceinline__ float amax4(float m, float4 x) {
    return fmaxf(m, fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w))));
}

template <bool kCoherent, int kRegVec>
__device__ __forceinline__ void quant_a_row(const Plan& p, int r, int lane) {
    if (debug_row(p.hdr, __ldg(p.pool_src + r), (int64_t)p.T * p.K) < 0) return;  // padding row: never read back
    const int I = p.I, nv = p.I / 4;  // float4 vectors of a row (a multiple of 32)
    const bool split = p.mode == MOE_A8W8_INT8;  // A8W4-INT: plane 0 holds q itself
    const float4* a = reinterpret_cast<const float4*>(p.a_f32 + (int64_t)r * I);
    const bool in_regs = nv <= 32 * kRegVec;
    float4 buf[kRegVec];
    float m = 0.0f;
    if (in_regs) {
#pragma unroll
        for (int i = 0; i < kRegVec; ++i)
            if (32 * i < nv) buf[i] = load_a4<kCoherent>(a + lane + 32 * i);  // uniform: nv is a multiple of 32
#pragma unroll
        for (int i = 0; i < kRegVec; ++i)
            if (32 * i < nv) m = amax4(m, buf[i]);
    } else {
        for (int v = lane; v < nv; v += 32) m = amax4(m, load_a4<kCoherent>(a + v));
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float s = fmaxf(__fdiv_rn(m, 127.0f), 1e-8f);
    uint32_t* q = reinterpret_cast<uint32_t*>(p.a_pool + (int64_t)r * I);      // 4 codes per word
    uint2* hi = reinterpret_cast<uint2*>(p.a_planes + (int64_t)r * I);         // plane 0: floor(q/16), f16
    uint2* lo = reinterpret_cast<uint2*>(p.a_planes + (p.pool_rows + r) * I);  // plane 1: q mod 16, f16
    int code_sum = 0;
    // codes, planes and code sum of vector v of the row; lanes 2m and 2m + 1 hold the two halves of
    // a group of 8 codes together (every lane of the warp calls it with its own v)
    auto put = [&](int v, float4 x) {
        const float xv[4] = {x.x, x.y, x.z, x.w};
        uint32_t qw = 0, h[2] = {0, 0}, l[2] = {0, 0};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            float t = rintf(__fdiv_rn(xv[c], s));
            t = fminf(fmaxf(t, -127.0f), 127.0f);
            const int qi = static_cast<int>(t);
            qw |= (uint32_t)(qi & 0xff) << (8 * c);
            h[c >> 1] |= (uint32_t)float_to_f16_bits((float)(split ? qi >> 4 : qi)) << (16 * (c & 1));
            l[c >> 1] |= (uint32_t)float_to_f16_bits((float)(qi & 15)) << (16 * (c & 1));
        }
        q[v] = qw;
        if (split) {
            hi[v] = make_uint2(h[0], h[1]);
            lo[v] = make_uint2(l[0], l[1]);
        } else {
            // q0 q4 q1 q5 from the even lane of the pair, q2 q6 q3 q7 from the odd one
            const bool odd = lane & 1;
            const uint32_t got = __shfl_xor_sync(0xffffffffu, odd ? h[0] : h[1], 1);
            const uint32_t mine = odd ? h[1] : h[0];
            hi[v] = odd ? make_uint2((got & 0xffffu) | (mine << 16), (got >> 16) | (mine & 0xffff0000u))
                        : make_uint2((mine & 0xffffu) | (got << 16), (mine >> 16) | (got & 0xffff0000u));
            code_sum += (int)(int8_t)(qw & 0xff) + (int)(int8_t)((qw >> 8) & 0xff) +
                        (int)(int8_t)((qw >> 16) & 0xff) + (int)(int8_t)(qw >> 24);
        }
    };
    if (in_regs) {
#pragma unroll
        for (int i = 0; i < kRegVec; ++i)
            if (32 * i < nv) put(lane + 32 * i, buf[i]);
    } else {
        for (int v = lane; v < nv; v += 32) put(v, load_a4<kCoherent>(a + v));
    }
    if (lane == 0) reinterpret_cast<float*>(p.a_pool_scale)[r] = s;
    if (!split) {
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) code_sum += __shfl_xor_sync(0xffffffffu, code_sum, o);
        if (lane == 0) p.a_sums[r] = code_sum;
    }
}

}  // namespace moe
