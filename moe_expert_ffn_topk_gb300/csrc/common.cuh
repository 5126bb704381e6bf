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

}  // namespace moe
