// Host side of the C ABI: argument checks, workspace layout and the stage launch sequence.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>

#include "internal.h"
#include "moe_ffn.h"

namespace moe {

int x_elem_bytes(int mode) { return mode == MOE_A16W16 ? 2 : 1; }

int64_t x_scale_row_bytes(int mode, int H) {
    switch (mode) {
        case MOE_A8W8_FP8:
        case MOE_A8W8_FP8_E5M2: return H / 32;           // UE8M0 per 1x32
        case MOE_A8W8_INT8:
        case MOE_A8W4_INT: return 4;                     // fp32 per token
        case MOE_A8W4_FP8_FP4: return (int64_t)(H / 128) * 4;  // fp32 per 1x128
        default: return 0;
    }
}

int a_elem_bytes(int mode) { return mode == MOE_A16W16 ? 2 : 1; }

int64_t a_scale_row_bytes(int mode, int I) {
    switch (mode) {
        case MOE_A8W8_FP8:
        case MOE_A8W8_FP8_E5M2:
        case MOE_A8W4_FP8_FP4: return I / 32;            // UE8M0 per 1x32
        case MOE_A8W8_INT8:
        case MOE_A8W4_INT: return 4;                     // fp32 per row
        default: return 0;
    }
}

bool dims_ok(const moe_dims* d, moe_dtype_mode m) {
    if (!d) return false;
    if (m < MOE_A16W16 || m > MOE_A8W8_FP8_E5M2) return false;
    const int S = d->num_shared_experts;
    if (d->num_tokens < 0 || d->topk < 1 || S < 0 || d->topk + S > 32) return false;
    if (d->num_experts < d->topk || d->num_experts + S > 1024) return false;
    if (d->hidden < 128 || d->hidden % 128 || d->intermediate < 128 || d->intermediate % 128) return false;
    if ((int64_t)d->num_tokens * (d->topk + S) > (int64_t(1) << 24)) return false;
    if ((int64_t)d->hidden > (1 << 16) || (int64_t)d->intermediate > (1 << 16)) return false;
    return true;
}

static size_t align_up(size_t v) { return (v + 255) & ~size_t(255); }

moe_status layout(const moe_dims* d, moe_dtype_mode m, moe_workspace_layout_t* out) {
    if (!out || !dims_ok(d, m)) return MOE_ERR_INVALID_ARG;
    // the shared experts are experts E..E+S-1 with one slot per token each
    const int64_t S = d->num_shared_experts;
    const int64_t T = d->num_tokens, H = d->hidden, I = d->intermediate, E = d->num_experts + S, K = d->topk + S;
    const int64_t R = T * K;
    const int64_t pool_rows = R + std::min<int64_t>(E, R) * (kTileRows - 1);
    moe_workspace_layout_t L;
    std::memset(&L, 0, sizeof(L));
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t at = off;
        off = align_up(off + bytes);
        return at;
    };
    L.header = take(sizeof(int32_t) * kHeaderInts);
    size_t claim = take(sizeof(int32_t) * E);
    (void)claim;  // immediately after the header; not exported
    L.counts = take(sizeof(int32_t) * E);
    L.offsets = take(sizeof(int32_t) * (E + 1));
    L.pad_offsets = take(sizeof(int32_t) * (E + 1));
    L.tile_offsets = take(sizeof(int32_t) * (E + 1));
    size_t pos = take(sizeof(int32_t) * R);
    (void)pos;
    L.row_src = take(sizeof(int32_t) * R);
    L.pool_src = take(sizeof(int32_t) * pool_rows);
    L.slot_row = take(sizeof(int32_t) * R);
    L.gates = take(S ? sizeof(float) * R : 0);
    L.comb = take((size_t)R * H * 2);
    L.ffn_counters = take(sizeof(int32_t) * (size_t)ffn_counter_ints(pool_rows / kTileRows, T));
    // everything above is the same for every mode; the pools below depend on it
    L.x_pool = take((size_t)pool_rows * H * x_elem_bytes(m));
    L.x_pool_scale = take((size_t)pool_rows * x_scale_row_bytes(m, (int)H));
    L.a_pool = take((size_t)pool_rows * I * a_elem_bytes(m));
    L.a_pool_scale = take((size_t)pool_rows * a_scale_row_bytes(m, (int)I));
    L.a_f32 = take(int_mode(m) ? (size_t)pool_rows * I * 4 : 0);
    const int planes = int_planes(m);  // the integer tensor-core path's f16 operand planes
    L.x_pool_planes = take((size_t)planes * pool_rows * H * 2);
    L.a_pool_planes = take((size_t)planes * pool_rows * I * 2);
    L.pool_sums = take(m == MOE_A8W4_INT ? (size_t)2 * pool_rows * 4 : 0);
    L.total = off;
    L.pool_rows = pool_rows;
    *out = L;
    return MOE_OK;
}

moe_status make_plan_view(const moe_dims* d, moe_dtype_mode m, void* ws, size_t ws_bytes, Plan* p, bool pools) {
    moe_workspace_layout_t L;
    moe_status st = layout(d, m, &L);
    if (st != MOE_OK) return st;
    const size_t need = pools ? L.total : L.x_pool;  // x_pool starts where the mode-free part ends
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255) || ws_bytes < need) return MOE_ERR_WORKSPACE;
    uint8_t* b = static_cast<uint8_t*>(ws);
    p->act_clamp = INFINITY;
    p->T = d->num_tokens;
    p->H = d->hidden;
    p->I = d->intermediate;
    p->E = d->num_experts + d->num_shared_experts;
    p->K = d->topk + d->num_shared_experts;
    p->Er = d->num_experts;
    p->Kr = d->topk;
    p->gates = reinterpret_cast<float*>(b + L.gates);
    p->mode = m;
    p->pool_rows = L.pool_rows;
    p->hdr = reinterpret_cast<int32_t*>(b + L.header);
    p->claim = reinterpret_cast<int32_t*>(b + align_up(L.header + sizeof(int32_t) * kHeaderInts));
    p->counts = reinterpret_cast<int32_t*>(b + L.counts);
    p->offsets = reinterpret_cast<int32_t*>(b + L.offsets);
    p->pad_off = reinterpret_cast<int32_t*>(b + L.pad_offsets);
    p->tile_off = reinterpret_cast<int32_t*>(b + L.tile_offsets);
    p->pos = reinterpret_cast<int32_t*>(b + align_up(L.tile_offsets + sizeof(int32_t) * (p->E + 1)));
    p->row_src = reinterpret_cast<int32_t*>(b + L.row_src);
    p->pool_src = reinterpret_cast<int32_t*>(b + L.pool_src);
    p->slot_row = reinterpret_cast<int32_t*>(b + L.slot_row);
    p->x_pool = b + L.x_pool;
    p->x_pool_scale = b + L.x_pool_scale;
    p->a_pool = b + L.a_pool;
    p->a_pool_scale = b + L.a_pool_scale;
    p->a_f32 = reinterpret_cast<float*>(b + L.a_f32);
    p->x_planes = reinterpret_cast<uint16_t*>(b + L.x_pool_planes);
    p->a_planes = reinterpret_cast<uint16_t*>(b + L.a_pool_planes);
    p->x_sums = reinterpret_cast<int32_t*>(b + L.pool_sums);
    p->a_sums = p->x_sums + L.pool_rows;
    p->comb = reinterpret_cast<uint16_t*>(b + L.comb);
    p->ffn_counters = reinterpret_cast<int32_t*>(b + L.ffn_counters);
    return MOE_OK;
}

static moe_status from_cuda(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

static bool operand_ok(moe_operand o, bool needs_scale) {
    if (!o.data) return false;
    if (needs_scale && !o.scale) return false;
    return true;
}

}  // namespace moe

using namespace moe;

extern "C" {

size_t moe_workspace_bytes(const moe_dims* d, moe_dtype_mode m) {
    moe_workspace_layout_t L;
    if (layout(d, m, &L) != MOE_OK) return 0;
    return L.total;
}

moe_status moe_workspace_layout(const moe_dims* d, moe_dtype_mode m, moe_workspace_layout_t* out) {
    return layout(d, m, out);
}

moe_status moe_plan(const int32_t* topk_ids, const moe_dims* d, int32_t* counts, int32_t* offsets,
                    int32_t* row_src, void* workspace, size_t workspace_bytes, moe_stream_t stream) {
    Plan p;
    moe_status st = make_plan_view(d, MOE_A16W16, workspace, workspace_bytes, &p, false);
    if (st != MOE_OK) return st;
    if (!topk_ids && d->num_tokens > 0) return MOE_ERR_INVALID_ARG;
    return from_cuda(launch_route(p, topk_ids, counts, offsets, row_src, reinterpret_cast<cudaStream_t>(stream)));
}

moe_status moe_dispatch(moe_operand x, const moe_dims* d, moe_dtype_mode m, void* workspace, size_t workspace_bytes,
                        moe_stream_t stream) {
    Plan p;
    moe_status st = make_plan_view(d, m, workspace, workspace_bytes, &p, true);
    if (st != MOE_OK) return st;
    if (d->num_tokens > 0 && !operand_ok(x, m != MOE_A16W16)) return MOE_ERR_INVALID_ARG;
    return from_cuda(launch_dispatch(p, x.data, x.scale, reinterpret_cast<cudaStream_t>(stream)));
}

moe_status moe_dispatch_quantize(const void* x_bf16, const moe_dims* d, moe_dtype_mode m, void* workspace,
                                 size_t workspace_bytes, moe_stream_t stream) {
    Plan p;
    moe_status st = make_plan_view(d, m, workspace, workspace_bytes, &p, true);
    if (st != MOE_OK) return st;
    if (d->num_tokens > 0 && !x_bf16) return MOE_ERR_INVALID_ARG;
    return from_cuda(launch_dispatch_quant(p, x_bf16, reinterpret_cast<cudaStream_t>(stream)));
}

static moe_status expert_l1(moe_operand w1, const moe_dims* d, moe_dtype_mode m, uint32_t flags, float clamp,
                            void* workspace, size_t workspace_bytes, moe_stream_t stream);

moe_status moe_expert_l1(moe_operand w1, const moe_dims* d, moe_dtype_mode m, uint32_t flags, void* workspace,
                         size_t workspace_bytes, moe_stream_t stream) {
    return expert_l1(w1, d, m, flags, INFINITY, workspace, workspace_bytes, stream);
}

// the options of the _ex entry points: flags, and the activation clamp applied through the plan
static moe_status read_options(const moe_options* opt, uint32_t* flags, float* clamp) {
    *flags = opt ? opt->flags : 0u;
    *clamp = INFINITY;
    if (opt && opt->has_activation_clamp) {
        if (!(opt->activation_clamp >= 0.0f)) return MOE_ERR_INVALID_ARG;  // also rejects NaN
        *clamp = opt->activation_clamp;
    }
    return MOE_OK;
}

static moe_status expert_l1(moe_operand w1, const moe_dims* d, moe_dtype_mode m, uint32_t flags, float clamp,
                            void* workspace, size_t workspace_bytes, moe_stream_t stream) {
    Plan p;
    moe_status st = make_plan_view(d, m, workspace, workspace_bytes, &p, true);
    if (st != MOE_OK) return st;
    p.act_clamp = clamp;
    if (!operand_ok(w1, m != MOE_A16W16)) return MOE_ERR_INVALID_ARG;
    if (d->num_tokens == 0) return MOE_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (flags & MOE_FLAG_PREPARED_WEIGHTS) {  // f16 codes from moe_prepare_weights: the INT8 tensor cores only
        if (m != MOE_A8W8_INT8 || (flags & MOE_FLAG_SIMT) || !int8_tc_supported(p, 1)) return MOE_ERR_UNSUPPORTED;
        e = launch_l1_int8_tc(p, w1.data, w1.scale, true, s);
        if (e == cudaSuccess) e = launch_int8_row_quant(p, s);
        return from_cuda(e);
    }
    if ((flags & MOE_FLAG_PAIR_L1) && !(flags & (MOE_FLAG_SIMT | MOE_FLAG_SINGLE_CTA)) && pair_supported(p, 1)) {
        e = launch_l1_pair(p, w1.data, s);
    } else if (!(flags & MOE_FLAG_SIMT) && tc_supported(p, 1)) {
        e = launch_l1_tc(p, w1.data, w1.scale, s);
    } else if (!(flags & MOE_FLAG_SIMT) && bs_supported(p, 1)) {
        e = launch_l1_bs(p, w1.data, w1.scale, flags, s);
    } else if (!(flags & MOE_FLAG_SIMT) && int8_tc_supported(p, 1)) {
        e = launch_l1_int8_tc(p, w1.data, w1.scale, false, s);
    } else if (!(flags & (MOE_FLAG_SIMT | MOE_FLAG_TOKEN_MAJOR)) && w4_wm_supported(p, 1) &&
               ((flags & MOE_FLAG_WEIGHT_MAJOR) || w4_wm_preferred(p, 1))) {
        e = launch_l1_w4_wm(p, w1.data, w1.scale, s);
    } else if (!(flags & MOE_FLAG_SIMT) && w4_tc_supported(p, 1)) {
        e = launch_l1_w4_tc(p, w1.data, w1.scale, s);
    } else {
        e = launch_l1_simt(p, w1.data, w1.scale, s);
    }
    if (e == cudaSuccess && int_mode(m)) e = launch_int8_row_quant(p, s);
    return from_cuda(e);
}

moe_status moe_expert_l1_ex(moe_operand w1, const moe_dims* d, moe_dtype_mode m, const moe_options* opt,
                            void* workspace, size_t workspace_bytes, moe_stream_t stream) {
    uint32_t flags;
    float clamp;
    const moe_status st = read_options(opt, &flags, &clamp);
    if (st != MOE_OK) return st;
    return expert_l1(w1, d, m, flags, clamp, workspace, workspace_bytes, stream);
}

moe_status moe_expert_l2(moe_operand w2, const float* topk_weights, const moe_dims* d, moe_dtype_mode m,
                         uint32_t flags, void* workspace, size_t workspace_bytes, moe_stream_t stream) {
    Plan p;
    moe_status st = make_plan_view(d, m, workspace, workspace_bytes, &p, true);
    if (st != MOE_OK) return st;
    if (!operand_ok(w2, m != MOE_A16W16)) return MOE_ERR_INVALID_ARG;
    const bool prepared = (flags & MOE_FLAG_PREPARED_WEIGHTS) != 0;
    if (prepared && (m != MOE_A8W8_INT8 || (flags & MOE_FLAG_SIMT) || !int8_tc_supported(p, 2)))
        return MOE_ERR_UNSUPPORTED;
    if (d->num_tokens == 0) return MOE_OK;
    if (!topk_weights) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (p.K != p.Kr) {  // shared experts: their slots carry weight 1
        const cudaError_t e = launch_expand_gates(p, topk_weights, s);
        if (e != cudaSuccess) return from_cuda(e);
        topk_weights = p.gates;
    }
    if (!(flags & (MOE_FLAG_SIMT | MOE_FLAG_SINGLE_CTA)) && pair_supported(p, 2))
        return from_cuda(launch_l2_pair(p, w2.data, topk_weights, s));
    if (!(flags & MOE_FLAG_SIMT) && tc_supported(p, 2))
        return from_cuda(launch_l2_tc(p, w2.data, w2.scale, topk_weights, s));
    if (!(flags & MOE_FLAG_SIMT) && bs_supported(p, 2))
        return from_cuda(launch_l2_bs(p, w2.data, w2.scale, topk_weights, flags, s));
    if (prepared || (!(flags & MOE_FLAG_SIMT) && int8_tc_supported(p, 2)))
        return from_cuda(launch_l2_int8_tc(p, w2.data, w2.scale, topk_weights, prepared, s));
    if (!(flags & (MOE_FLAG_SIMT | MOE_FLAG_TOKEN_MAJOR)) && w4_wm_supported(p, 2) &&
        ((flags & MOE_FLAG_WEIGHT_MAJOR) || w4_wm_preferred(p, 2)))
        return from_cuda(launch_l2_w4_wm(p, w2.data, w2.scale, topk_weights, s));
    if (!(flags & MOE_FLAG_SIMT) && w4_tc_supported(p, 2))
        return from_cuda(launch_l2_w4_tc(p, w2.data, w2.scale, topk_weights, s));
    return from_cuda(launch_l2_simt(p, w2.data, w2.scale, topk_weights, s));
}

moe_status moe_expert_ffn(moe_operand w1, moe_operand w2, const float* topk_weights, void* y, const moe_dims* d,
                          moe_dtype_mode m, const moe_options* opt, void* workspace, size_t workspace_bytes,
                          moe_stream_t stream) {
    Plan p;
    moe_status st = make_plan_view(d, m, workspace, workspace_bytes, &p, true);
    if (st != MOE_OK) return st;
    uint32_t flags;
    if ((st = read_options(opt, &flags, &p.act_clamp)) != MOE_OK) return st;
    if (!operand_ok(w1, m != MOE_A16W16) || !operand_ok(w2, m != MOE_A16W16)) return MOE_ERR_INVALID_ARG;
    const bool prepared = (flags & MOE_FLAG_PREPARED_WEIGHTS) != 0;
    const bool bf16 = tc_supported(p, 1) && tc_supported(p, 2);
    const bool block_scaled = bs_supported(p, 1) && bs_supported(p, 2);
    const bool int8 = int8_tc_supported(p, 1) && int8_tc_supported(p, 2);
    const bool w4 = w4_wm_supported(p, 1) && w4_wm_supported(p, 2);
    if (!(bf16 || block_scaled || int8 || w4) || (prepared && !int8)) return MOE_ERR_UNSUPPORTED;
    if (d->num_tokens == 0) return MOE_OK;
    if (!topk_weights) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (p.K != p.Kr) {  // shared experts: their slots carry weight 1
        const cudaError_t e = launch_expand_gates(p, topk_weights, s);
        if (e != cudaSuccess) return from_cuda(e);
        topk_weights = p.gates;
    }
    if (bf16) return from_cuda(launch_ffn_fused_tc(p, w1.data, w2.data, topk_weights, static_cast<uint16_t*>(y), s));
    // FP8 and integer modes: L1 and L2 in one launch (the integer modes re-quantise A inside it),
    // the combine after it
    const cudaError_t e =
        block_scaled ? launch_ffn_fused_bs(p, w1.data, w1.scale, w2.data, w2.scale, topk_weights, s)
        : int8       ? launch_ffn_fused_int8(p, w1.data, w1.scale, w2.data, w2.scale, topk_weights, prepared, s)
                     : launch_ffn_fused_w4_wm(p, w1.data, w1.scale, w2.data, w2.scale, topk_weights, s);
    if (e != cudaSuccess || !y) return from_cuda(e);
    return from_cuda(launch_combine(p, static_cast<uint16_t*>(y), s));
}

moe_status moe_combine(void* y, const moe_dims* d, void* workspace, size_t workspace_bytes, moe_stream_t stream) {
    Plan p;
    moe_status st = make_plan_view(d, MOE_A16W16, workspace, workspace_bytes, &p, false);
    if (st != MOE_OK) return st;
    if (d->num_tokens == 0) return MOE_OK;
    if (!y) return MOE_ERR_INVALID_ARG;
    return from_cuda(launch_combine(p, static_cast<uint16_t*>(y), reinterpret_cast<cudaStream_t>(stream)));
}

static moe_status forward(moe_operand x, const int32_t* topk_ids, const float* topk_weights, moe_operand w1,
                          moe_operand w2, void* y, const moe_dims* d, moe_dtype_mode m, uint32_t flags, float clamp,
                          void* workspace, size_t workspace_bytes, moe_stream_t stream) {
    Plan p;
    moe_status st = make_plan_view(d, m, workspace, workspace_bytes, &p, true);
    if (st != MOE_OK) return st;
    const bool q = m != MOE_A16W16;
    if (!operand_ok(w1, q) || !operand_ok(w2, q)) return MOE_ERR_INVALID_ARG;
    if (d->num_tokens == 0) return MOE_OK;
    const bool quantize_x = (flags & MOE_FLAG_QUANTIZE_X) != 0;
    if (!(quantize_x ? x.data != nullptr : operand_ok(x, q)) || !topk_ids || !topk_weights || !y)
        return MOE_ERR_INVALID_ARG;
    const bool fused = (flags & MOE_FLAG_FUSED) != 0;
    if (fused && (flags & MOE_FLAG_SIMT)) return MOE_ERR_INVALID_ARG;
    if (fused && !((tc_supported(p, 1) && tc_supported(p, 2)) || (bs_supported(p, 1) && bs_supported(p, 2)) ||
                   (int8_tc_supported(p, 1) && int8_tc_supported(p, 2)) ||
                   (w4_wm_supported(p, 1) && w4_wm_supported(p, 2))))
        return MOE_ERR_UNSUPPORTED;
    if ((st = moe_plan(topk_ids, d, nullptr, nullptr, nullptr, workspace, workspace_bytes, stream)) != MOE_OK) return st;
    st = quantize_x ? moe_dispatch_quantize(x.data, d, m, workspace, workspace_bytes, stream)
                    : moe_dispatch(x, d, m, workspace, workspace_bytes, stream);
    if (st != MOE_OK) return st;
    if (fused) {
        const moe_options opt{flags, 1u, clamp};
        return moe_expert_ffn(w1, w2, topk_weights, y, d, m, &opt, workspace, workspace_bytes, stream);
    }
    if ((st = expert_l1(w1, d, m, flags, clamp, workspace, workspace_bytes, stream)) != MOE_OK) return st;
    if ((st = moe_expert_l2(w2, topk_weights, d, m, flags, workspace, workspace_bytes, stream)) != MOE_OK) return st;
    return moe_combine(y, d, workspace, workspace_bytes, stream);
}

moe_status moe_forward(moe_operand x, const int32_t* topk_ids, const float* topk_weights, moe_operand w1,
                       moe_operand w2, void* y, const moe_dims* d, moe_dtype_mode m, uint32_t flags,
                       void* workspace, size_t workspace_bytes, moe_stream_t stream) {
    return forward(x, topk_ids, topk_weights, w1, w2, y, d, m, flags, INFINITY, workspace, workspace_bytes, stream);
}

moe_status moe_forward_ex(moe_operand x, const int32_t* topk_ids, const float* topk_weights, moe_operand w1,
                          moe_operand w2, void* y, const moe_dims* d, moe_dtype_mode m, const moe_options* opt,
                          void* workspace, size_t workspace_bytes, moe_stream_t stream) {
    uint32_t flags;
    float clamp;
    const moe_status st = read_options(opt, &flags, &clamp);
    if (st != MOE_OK) return st;
    return forward(x, topk_ids, topk_weights, w1, w2, y, d, m, flags, clamp, workspace, workspace_bytes, stream);
}

moe_status moe_check_device_error(void* workspace, moe_stream_t stream) {
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255)) return MOE_ERR_WORKSPACE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int32_t err = 0;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaMemcpy(&err, workspace, sizeof(err), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
    const int32_t zero = 0;
    if (cudaMemcpy(workspace, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return MOE_ERR_CUDA;
    return static_cast<moe_status>(err);
}

size_t moe_prepared_weights_bytes(const moe_dims* d, moe_dtype_mode m, int layer) {
    if (!dims_ok(d, m) || (layer != 1 && layer != 2) || m != MOE_A8W8_INT8) return 0;
    const int64_t E = d->num_experts + d->num_shared_experts;
    return sizeof(uint16_t) * (size_t)(E * (layer == 1 ? 2 * (int64_t)d->intermediate : (int64_t)d->hidden) *
                                       (layer == 1 ? (int64_t)d->hidden : (int64_t)d->intermediate));
}

moe_status moe_prepare_weights(const void* w, const moe_dims* d, moe_dtype_mode m, int layer, void* out,
                               size_t out_bytes, moe_stream_t stream) {
    if (!dims_ok(d, m) || (layer != 1 && layer != 2)) return MOE_ERR_INVALID_ARG;
    if (m != MOE_A8W8_INT8) return MOE_ERR_UNSUPPORTED;
    const size_t need = moe_prepared_weights_bytes(d, m, layer);
    if (!w || !out || out_bytes < need || (reinterpret_cast<uintptr_t>(w) & 15) || (reinterpret_cast<uintptr_t>(out) & 15))
        return MOE_ERR_INVALID_ARG;
    return from_cuda(launch_prepare_int8(w, out, (int64_t)(need / 2), reinterpret_cast<cudaStream_t>(stream)));
}

const char* moe_status_string(moe_status s) {
    switch (s) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED: return "unsupported mode or shape";
        case MOE_ERR_CUDA: return "CUDA error";
        case MOE_ERR_BAD_ROUTE: return "expert id outside [-1, num_experts)";
        case MOE_ERR_TIMEOUT: return "bounded device wait timed out";
        case MOE_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case MOE_ERR_BAD_SCALE: return "FP8 x FP4 activation scale that is not a power of two";
        case MOE_ERR_BOUNDS: return "index outside its buffer (debug build check)";
        default: return "unknown status";
    }
}

moe_status moe_debug_bounded_wait(void* workspace, size_t workspace_bytes, uint64_t timeout_ns, moe_stream_t stream) {
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255) || workspace_bytes < 256) return MOE_ERR_WORKSPACE;
    Plan p;
    std::memset(&p, 0, sizeof(p));
    p.hdr = static_cast<int32_t*>(workspace);
    return from_cuda(launch_debug_wait(p, timeout_ns, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
