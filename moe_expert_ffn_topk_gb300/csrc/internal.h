// Internal declarations shared by the translation units of the library (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_ffn.h"

namespace moe {

constexpr int kTileRows = 128;          // rows per pool tile; expert regions are padded to it
constexpr int kHeaderInts = 16;         // workspace header: [0] error word, [1] R, [2] padded rows, [3] tiles
constexpr int kErrWord = 0;
constexpr int kHdrRows = 1;
constexpr int kHdrPadRows = 2;
constexpr int kHdrTiles = 3;
constexpr int kHdrWaitFlag = 8;         // a flag that nothing sets (bounded-wait test hook)
// moe_expert_ffn of the integer modes: re-quantisation jobs per 128-row route tile, and the int32
// counters its launch uses (per route tile, then the job queue: jobs finished, head, tail, a slot
// per job); the workspace's ffn_counters region holds the largest need of any mode
constexpr int kQuantJobs = 4;
constexpr long long fused_int_counters(long long route_tiles) { return route_tiles * (1 + kQuantJobs) + 3; }
constexpr long long ffn_counter_ints(long long route_tiles, long long T) { return fused_int_counters(route_tiles) + T; }

// The integer modes (int8 activations, fp32 per-token / per-channel scales) and the number of
// f16 operand planes their tensor-core GEMMs read: the int8 codes as hi = floor(q/16) and
// lo = q mod 16 with int8 weights, the codes themselves with int4 weights.
__host__ __device__ constexpr bool int_mode(int m) { return m == MOE_A8W8_INT8 || m == MOE_A8W4_INT; }
__host__ __device__ constexpr int int_planes(int m) { return m == MOE_A8W8_INT8 ? 2 : m == MOE_A8W4_INT ? 1 : 0; }

// Device view of the workspace for one (dims, mode).
struct Plan {
    int T, H, I, E, K;     // E, K: all experts and slots, shared ones included
    int Er, Kr;            // routed experts and slots (E - Er = K - Kr = shared experts)
    int mode;
    int64_t pool_rows;
    int32_t* hdr;
    int32_t* claim;        // [E] per-expert claim counters (zeroed at the start of each plan)
    int32_t* counts;       // [E]
    int32_t* offsets;      // [E+1]
    int32_t* pad_off;      // [E+1]
    int32_t* tile_off;     // [E+1]
    int32_t* pos;          // [T*K] position of (i,k) inside its expert
    int32_t* row_src;      // [T*K]
    int32_t* pool_src;     // [pool_rows]
    int32_t* slot_row;     // [T*K]
    uint8_t* x_pool;       // [pool_rows, H * x elem bytes]
    uint8_t* x_pool_scale;
    uint8_t* a_pool;       // [pool_rows, I * a elem bytes]
    uint8_t* a_pool_scale;
    float* a_f32;          // [pool_rows, I] (integer modes)
    uint16_t* x_planes;    // integer modes: f16 [int_planes][pool_rows, H] (INT8: hi, lo of the codes)
    uint16_t* a_planes;    // integer modes: f16 [int_planes][pool_rows, I]
    int32_t* x_sums;       // A8W4-INT: sum of each x pool row's codes [pool_rows]
    int32_t* a_sums;       // A8W4-INT: sum of each A pool row's codes [pool_rows]
    uint16_t* comb;        // bf16 [T*K, H]
    int32_t* ffn_counters; // moe_expert_ffn: [pool_rows/128] route tiles, then [T] tokens
    float act_clamp;       // SwiGLU inputs clipped to [-act_clamp, act_clamp]; +inf: no clamp
    float* gates;          // shared experts: [T*K] gates, the routed ones then 1 per shared slot
};

// x / A storage properties per mode
int x_elem_bytes(int mode);            // bytes per x element (bf16 2, others 1)
int64_t x_scale_row_bytes(int mode, int H);
int a_elem_bytes(int mode);
int64_t a_scale_row_bytes(int mode, int I);

moe_status layout(const moe_dims* d, moe_dtype_mode m, moe_workspace_layout_t* out);
moe_status make_plan_view(const moe_dims* d, moe_dtype_mode m, void* ws, size_t ws_bytes, Plan* p, bool pools);

// Launchers (each returns cudaGetLastError() of its launches).
// The shape and mode checks every entry point applies to moe_dims before anything else.
bool dims_ok(const moe_dims* d, moe_dtype_mode m);

cudaError_t launch_route(const Plan& p, const int32_t* topk_ids, int32_t* counts_out, int32_t* offsets_out,
                         int32_t* row_src_out, cudaStream_t s);
cudaError_t launch_dispatch(const Plan& p, const void* x, const void* x_scale, cudaStream_t s);
cudaError_t launch_combine(const Plan& p, uint16_t* y, cudaStream_t s);
// shared experts: p.gates[t*K + k] = k < Kr ? topk_weights[t*Kr + k] : 1
cudaError_t launch_expand_gates(const Plan& p, const float* topk_weights, cudaStream_t s);
cudaError_t launch_l1_simt(const Plan& p, const void* w1, const void* w1_scale, cudaStream_t s);
cudaError_t launch_l2_simt(const Plan& p, const void* w2, const void* w2_scale, const float* topk_weights,
                           cudaStream_t s);
cudaError_t launch_int8_row_quant(const Plan& p, cudaStream_t s);
// S2 from bf16 x with the mode's activation quantisation (A16W16: the plain gather).
cudaError_t launch_dispatch_quant(const Plan& p, const void* x_bf16, cudaStream_t s);
cudaError_t launch_debug_wait(const Plan& p, uint64_t timeout_ns, cudaStream_t s);

// Tensor-core path. Returns cudaErrorNotSupported when the mode / shape has no tcgen05 kernel.
cudaError_t launch_l1_tc(const Plan& p, const void* w1, const void* w1_scale, cudaStream_t s);
cudaError_t launch_l2_tc(const Plan& p, const void* w2, const void* w2_scale, const float* topk_weights,
                         cudaStream_t s);
bool tc_supported(const Plan& p, int stage);
// bf16 L1 / L2 on CTA pairs (tcgen05.mma.cta_group::2); same outputs as launch_l1_tc / launch_l2_tc
bool pair_supported(const Plan& p, int stage);
cudaError_t launch_l1_pair(const Plan& p, const void* w1, cudaStream_t s);
cudaError_t launch_l2_pair(const Plan& p, const void* w2, const float* topk_weights, cudaStream_t s);
// S3-S5 of the bf16 mode in one cooperative launch (L1 -> L2 dependency counters)
cudaError_t launch_ffn_fused_tc(const Plan& p, const void* w1, const void* w2, const float* topk_weights,
                                uint16_t* y, cudaStream_t s);

// Tensor-core path of the integer modes (int8 or int4 weights converted to f16 in shared
// memory, the tokens' f16 planes; every partial sum an exact integer).
cudaError_t launch_l1_int8_tc(const Plan& p, const void* w1, const void* w1_scale, bool prepared, cudaStream_t s);
cudaError_t launch_l2_int8_tc(const Plan& p, const void* w2, const void* w2_scale, const float* topk_weights,
                              bool prepared, cudaStream_t s);
// int8 codes [n] -> the same values as f16 [n] (n a multiple of 16)
// S3 and S4 of the integer modes in one cooperative launch (weight-major tiles): each route tile's
// last L1 tile re-quantises its rows of A (quant_a_row) before its L2 tiles start
cudaError_t launch_ffn_fused_int8(const Plan& p, const void* w1, const void* w1_scale, const void* w2,
                                  const void* w2_scale, const float* topk_weights, bool prepared, cudaStream_t s);
cudaError_t launch_ffn_fused_w4_wm(const Plan& p, const void* w1, const void* w1_scale, const void* w2,
                                   const void* w2_scale, const float* topk_weights, cudaStream_t s);
cudaError_t launch_prepare_int8(const void* w, void* out, int64_t n, cudaStream_t s);
bool int8_tc_supported(const Plan& p, int stage);

// Token-major tensor-core path of A8W4-INT (int4 weights expanded to f16 in shared memory).
cudaError_t launch_l1_w4_tc(const Plan& p, const void* w1, const void* w1_scale, cudaStream_t s);
cudaError_t launch_l2_w4_tc(const Plan& p, const void* w2, const void* w2_scale, const float* topk_weights,
                            cudaStream_t s);
bool w4_tc_supported(const Plan& p, int stage);
// A8W4-INT weight-major (M = weight rows, N = up to 256 tokens of an expert); same results
bool w4_wm_supported(const Plan& p, int stage);
bool w4_wm_preferred(const Plan& p, int stage);
cudaError_t launch_l1_w4_wm(const Plan& p, const void* w1, const void* w1_scale, cudaStream_t s);
cudaError_t launch_l2_w4_wm(const Plan& p, const void* w2, const void* w2_scale, const float* topk_weights,
                            cudaStream_t s);

// Position of code k of a row in the A8W4-INT f16 operand planes: within each group of 8, code
// i < 4 goes to position 2i and code 4 + i to position 2i + 1.
__host__ __device__ constexpr int w4_plane_pos(int k) { return (k & ~7) | ((k & 3) << 1) | ((k >> 2) & 1); }

// Block-scaled tensor-core path of the FP8 modes (kind::mxf8f6f4.block_scale): weight-major
// tiles for decode-sized experts; for prefill-sized ones token-major tiles, or with
// MOE_FLAG_PAIR_L1 in `flags` weight-major tiles on CTA pairs, or with MOE_FLAG_WEIGHT_MAJOR one-CTA
// weight-major tiles (each where the shape has that kernel).
cudaError_t launch_l1_bs(const Plan& p, const void* w1, const void* w1_scale, uint32_t flags, cudaStream_t s);
cudaError_t launch_l2_bs(const Plan& p, const void* w2, const void* w2_scale, const float* topk_weights,
                         uint32_t flags, cudaStream_t s);
bool bs_supported(const Plan& p, int stage);
// S3 and S4 of the FP8 modes in one cooperative launch of the weight-major block-scaled kernel:
// L1 tiles first, L2 tiles after them, each L2 tile waiting (bounded) on a per-route-tile counter of
// finished L1 tiles in p.ffn_counters; L2 writes comb, which the combine stage then reduces
cudaError_t launch_ffn_fused_bs(const Plan& p, const void* w1, const void* w1_scale, const void* w2,
                                const void* w2_scale, const float* topk_weights, cudaStream_t s);
cudaError_t launch_l1_bs_tm(const Plan& p, const void* w1, const void* w1_scale, cudaStream_t s);
cudaError_t launch_l2_bs_tm(const Plan& p, const void* w2, const void* w2_scale, const float* topk_weights,
                            cudaStream_t s);
bool bs_tm_supported(const Plan& p, int stage);
cudaError_t launch_l1_bs_pair(const Plan& p, const void* w1, const void* w1_scale, cudaStream_t s);
cudaError_t launch_l2_bs_pair(const Plan& p, const void* w2, const void* w2_scale, const float* topk_weights,
                              cudaStream_t s);
bool bs_pair_supported(const Plan& p, int stage);

}  // namespace moe
