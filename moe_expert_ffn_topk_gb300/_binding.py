"""ctypes binding of the C ABI in ``include/moe_ffn.h``.

Argument marshalling only: each function takes torch tensors (device memory allocated by
the caller), checks placement and contiguity, passes their addresses and the current CUDA
stream to the library function of the same name, and turns a non-OK status into
``MoeError``. Every stage of the computation runs in the library's CUDA kernels. When the
library has not been built, importing this module raises ``ImportError``.
"""
from __future__ import annotations

import ctypes
import os

import torch

# MOE_GB300_DEBUG=1 loads the bounds-checking build (compiled with -DMOE_DEBUG by build(debug=True)):
# the same kernels with every data-dependent row index checked on the device (MOE_ERR_BOUNDS)
_LIB_NAME = "libmoe_gb300_debug.so" if os.environ.get("MOE_GB300_DEBUG") == "1" else "libmoe_gb300.so"
_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", _LIB_NAME)

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA, MOE_ERR_BAD_ROUTE, MOE_ERR_TIMEOUT, \
    MOE_ERR_WORKSPACE, MOE_ERR_BAD_SCALE, MOE_ERR_BOUNDS = range(9)
MODES = {"a16w16": 0, "a8w8_fp8": 1, "a8w8_int8": 2, "a8w4_fp8_fp4": 3, "a8w4_int": 4, "a8w8_fp8_e5m2": 5}
(MOE_FLAG_NONE, MOE_FLAG_SIMT, MOE_FLAG_WEIGHT_MAJOR, MOE_FLAG_QUANTIZE_X, MOE_FLAG_FUSED, MOE_FLAG_SINGLE_CTA,
 MOE_FLAG_PAIR_L1, MOE_FLAG_TOKEN_MAJOR, MOE_FLAG_PREPARED_WEIGHTS) = 0, 1, 2, 4, 8, 16, 32, 64, 128

ABI_FUNCTIONS = ("moe_workspace_bytes", "moe_plan", "moe_dispatch", "moe_expert_l1", "moe_expert_l2",
                 "moe_combine", "moe_forward", "moe_check_device_error", "moe_status_string",
                 "moe_workspace_layout", "moe_debug_bounded_wait", "moe_plan_noalloc", "moe_dispatch_quantize",
                 "moe_expert_l1_ex", "moe_forward_ex", "moe_expert_ffn", "moe_tensor_peak_probe",
                 "moe_prepared_weights_bytes", "moe_prepare_weights")
# moe_peak_kind (include/moe_peak.h): the tcgen05 instruction kinds the probe measures
PEAK_KINDS = {"bf16": 0, "f16": 1, "e4m3_e2m1": 2, "e4m3_e4m3": 3}


class MoeDims(ctypes.Structure):
    _fields_ = [("num_tokens", ctypes.c_int32), ("hidden", ctypes.c_int32), ("intermediate", ctypes.c_int32),
                ("num_experts", ctypes.c_int32), ("topk", ctypes.c_int32), ("num_shared_experts", ctypes.c_int32)]


class MoeOptions(ctypes.Structure):
    _fields_ = [("flags", ctypes.c_uint32), ("has_activation_clamp", ctypes.c_uint32),
                ("activation_clamp", ctypes.c_float)]


class MoeOperand(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("scale", ctypes.c_void_p)]


class MoeWorkspaceLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in (
        "header", "counts", "offsets", "pad_offsets", "tile_offsets", "row_src", "pool_src", "slot_row", "gates",
        "x_pool", "x_pool_scale", "a_pool", "a_pool_scale", "a_f32", "x_pool_planes", "a_pool_planes", "pool_sums",
        "comb", "ffn_counters",
        "total")] + \
        [("pool_rows", ctypes.c_int64)]


class MoeError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {moe_status_string(status)} (status {status})")


def _load():
    if not os.path.exists(_LIB_PATH):
        raise ImportError(f"CUDA library not built ({_LIB_PATH} is missing); run __graft_entry__.build()")
    lib = ctypes.CDLL(_LIB_PATH)
    vp, sz, u32, st = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_uint32, ctypes.c_int
    dims_p = ctypes.POINTER(MoeDims)
    sig = {
        "moe_workspace_bytes": (sz, [dims_p, st]),
        "moe_plan": (st, [vp, dims_p, vp, vp, vp, vp, sz, vp]),
        "moe_dispatch": (st, [MoeOperand, dims_p, st, vp, sz, vp]),
        "moe_expert_l1": (st, [MoeOperand, dims_p, st, u32, vp, sz, vp]),
        "moe_expert_l2": (st, [MoeOperand, vp, dims_p, st, u32, vp, sz, vp]),
        "moe_combine": (st, [vp, dims_p, vp, sz, vp]),
        "moe_forward": (st, [MoeOperand, vp, vp, MoeOperand, MoeOperand, vp, dims_p, st, u32, vp, sz, vp]),
        "moe_check_device_error": (st, [vp, vp]),
        "moe_status_string": (ctypes.c_char_p, [st]),
        "moe_workspace_layout": (st, [dims_p, st, ctypes.POINTER(MoeWorkspaceLayout)]),
        "moe_debug_bounded_wait": (st, [vp, sz, ctypes.c_uint64, vp]),
        "moe_plan_noalloc": (st, [vp, dims_p, vp, vp, vp, vp]),
        "moe_dispatch_quantize": (st, [vp, dims_p, st, vp, sz, vp]),
        "moe_expert_l1_ex": (st, [MoeOperand, dims_p, st, ctypes.POINTER(MoeOptions), vp, sz, vp]),
        "moe_expert_ffn": (st, [MoeOperand, MoeOperand, vp, vp, dims_p, st, ctypes.POINTER(MoeOptions), vp, sz, vp]),
        "moe_forward_ex": (st, [MoeOperand, vp, vp, MoeOperand, MoeOperand, vp, dims_p, st, ctypes.POINTER(MoeOptions),
                                vp, sz, vp]),
        "moe_tensor_peak_probe": (st, [st, ctypes.c_int64, ctypes.c_int, ctypes.POINTER(ctypes.c_double), vp, sz, vp]),
        "moe_prepared_weights_bytes": (sz, [dims_p, st, ctypes.c_int]),
        "moe_prepare_weights": (st, [vp, dims_p, st, ctypes.c_int, vp, sz, vp]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype, f.argtypes = res, args
    return lib


LIB = _load()


# ---------------------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------------------


def dims(T: int, H: int, I: int, E: int, K: int, S: int = 0) -> MoeDims:  # noqa: E741
    """T tokens, hidden H, intermediate I, E routed experts, top-K, S shared experts."""
    return MoeDims(T, H, I, E, K, S)


def _mode(m) -> int:
    return MODES[m] if isinstance(m, str) else int(m)


def _ptr(t, what, dev=True):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{what} must be a torch.Tensor")
    if dev and not t.is_cuda:
        raise ValueError(f"{what} must be in device memory")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    return t.data_ptr() if t.numel() else None


def _operand(data, scale, what):
    return MoeOperand(_ptr(data, what), _ptr(scale, what + "_scale"))


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ws(workspace):
    return _ptr(workspace, "workspace"), workspace.numel() * workspace.element_size()


def _check(status, what):
    if status != MOE_OK:
        raise MoeError(status, what)


# ---------------------------------------------------------------------------------------
# the ABI, one function each
# ---------------------------------------------------------------------------------------


def moe_status_string(status: int) -> str:
    return LIB.moe_status_string(int(status)).decode()


def moe_workspace_bytes(d: MoeDims, mode) -> int:
    return LIB.moe_workspace_bytes(ctypes.byref(d), _mode(mode))


def moe_workspace_layout(d: MoeDims, mode) -> dict:
    out = MoeWorkspaceLayout()
    _check(LIB.moe_workspace_layout(ctypes.byref(d), _mode(mode), ctypes.byref(out)), "moe_workspace_layout")
    return {name: getattr(out, name) for name, _ in MoeWorkspaceLayout._fields_}


def moe_plan(topk_ids, d: MoeDims, workspace, counts=None, offsets=None, row_src=None, stream=None):
    ws, nb = _ws(workspace)
    _check(LIB.moe_plan(_ptr(topk_ids, "topk_ids"), ctypes.byref(d), _ptr(counts, "counts"),
                        _ptr(offsets, "offsets"), _ptr(row_src, "row_src"), ws, nb, _stream(stream)), "moe_plan")


def moe_dispatch(x, x_scale, d: MoeDims, mode, workspace, stream=None):
    ws, nb = _ws(workspace)
    _check(LIB.moe_dispatch(_operand(x, x_scale, "x"), ctypes.byref(d), _mode(mode), ws, nb, _stream(stream)),
           "moe_dispatch")


def moe_dispatch_quantize(x_bf16, d: MoeDims, mode, workspace, stream=None):
    """S2 from bf16 x with the mode's activation quantisation (x_bf16: bf16 [T, H])."""
    ws, nb = _ws(workspace)
    _check(LIB.moe_dispatch_quantize(_ptr(x_bf16, "x_bf16"), ctypes.byref(d), _mode(mode), ws, nb, _stream(stream)),
           "moe_dispatch_quantize")


def moe_expert_l1(w1, w1_scale, d: MoeDims, mode, workspace, flags=0, stream=None):
    ws, nb = _ws(workspace)
    _check(LIB.moe_expert_l1(_operand(w1, w1_scale, "w1"), ctypes.byref(d), _mode(mode), flags, ws, nb,
                             _stream(stream)), "moe_expert_l1")


def moe_expert_l2(w2, w2_scale, topk_weights, d: MoeDims, mode, workspace, flags=0, stream=None):
    ws, nb = _ws(workspace)
    _check(LIB.moe_expert_l2(_operand(w2, w2_scale, "w2"), _ptr(topk_weights, "topk_weights"), ctypes.byref(d),
                             _mode(mode), flags, ws, nb, _stream(stream)), "moe_expert_l2")


def moe_combine(y, d: MoeDims, workspace, stream=None):
    ws, nb = _ws(workspace)
    _check(LIB.moe_combine(_ptr(y, "y"), ctypes.byref(d), ws, nb, _stream(stream)), "moe_combine")


def moe_forward(x, x_scale, topk_ids, topk_weights, w1, w1_scale, w2, w2_scale, y, d: MoeDims, mode, workspace,
                flags=0, stream=None):
    ws, nb = _ws(workspace)
    _check(LIB.moe_forward(_operand(x, x_scale, "x"), _ptr(topk_ids, "topk_ids"), _ptr(topk_weights, "topk_weights"),
                           _operand(w1, w1_scale, "w1"), _operand(w2, w2_scale, "w2"), _ptr(y, "y"),
                           ctypes.byref(d), _mode(mode), flags, ws, nb, _stream(stream)), "moe_forward")


def _options(flags, activation_clamp):
    return MoeOptions(int(flags), 0 if activation_clamp is None else 1,
                      0.0 if activation_clamp is None else float(activation_clamp))


def moe_expert_l1_ex(w1, w1_scale, d: MoeDims, mode, workspace, flags=0, activation_clamp=None, stream=None):
    """moe_expert_l1 with options (activation_clamp: None or >= 0)."""
    ws, nb = _ws(workspace)
    opt = _options(flags, activation_clamp)
    _check(LIB.moe_expert_l1_ex(_operand(w1, w1_scale, "w1"), ctypes.byref(d), _mode(mode), ctypes.byref(opt), ws, nb,
                                _stream(stream)), "moe_expert_l1_ex")


def moe_expert_ffn(w1, w1_scale, w2, w2_scale, topk_weights, d: MoeDims, mode, workspace, y=None,
                   activation_clamp=None, stream=None):
    """S3-S5 (and S6 into y when given) in one launch with dependency counters; needs
    moe_dispatch first."""
    ws, nb = _ws(workspace)
    opt = _options(0, activation_clamp)
    _check(LIB.moe_expert_ffn(_operand(w1, w1_scale, "w1"), _operand(w2, w2_scale, "w2"),
                              _ptr(topk_weights, "topk_weights"), None if y is None else _ptr(y, "y"), ctypes.byref(d),
                              _mode(mode), ctypes.byref(opt), ws, nb, _stream(stream)), "moe_expert_ffn")


def moe_forward_ex(x, x_scale, topk_ids, topk_weights, w1, w1_scale, w2, w2_scale, y, d: MoeDims, mode, workspace,
                   flags=0, activation_clamp=None, stream=None):
    """moe_forward with options (activation_clamp: None or >= 0)."""
    ws, nb = _ws(workspace)
    opt = _options(flags, activation_clamp)
    _check(LIB.moe_forward_ex(_operand(x, x_scale, "x"), _ptr(topk_ids, "topk_ids"), _ptr(topk_weights, "topk_weights"),
                              _operand(w1, w1_scale, "w1"), _operand(w2, w2_scale, "w2"), _ptr(y, "y"),
                              ctypes.byref(d), _mode(mode), ctypes.byref(opt), ws, nb, _stream(stream)),
           "moe_forward_ex")


def moe_check_device_error(workspace, stream=None) -> int:
    return LIB.moe_check_device_error(_ptr(workspace, "workspace"), _stream(stream))


def moe_debug_bounded_wait(workspace, timeout_ns: int, stream=None):
    ws, nb = _ws(workspace)
    _check(LIB.moe_debug_bounded_wait(ws, nb, int(timeout_ns), _stream(stream)), "moe_debug_bounded_wait")


def moe_prepared_weights_bytes(d: MoeDims, mode, layer: int) -> int:
    return LIB.moe_prepared_weights_bytes(ctypes.byref(d), _mode(mode), int(layer))


def moe_prepare_weights(w, d: MoeDims, mode, layer: int, out=None, stream=None):
    """The layer's weights in the prepared form the GEMMs take with MOE_FLAG_PREPARED_WEIGHTS (A8W8-INT:
    every int8 code as its exact f16 value, same layout); writes `out` (allocated here when None) and
    returns it."""
    n = moe_prepared_weights_bytes(d, mode, layer)
    if out is None:
        if n == 0:
            raise MoeError(MOE_ERR_UNSUPPORTED if _mode(mode) != MODES["a8w8_int8"] else MOE_ERR_INVALID_ARG,
                           "moe_prepare_weights")
        out = torch.empty(w.shape, dtype=torch.float16, device=w.device)  # the same layout as the int8 codes
    _check(LIB.moe_prepare_weights(_ptr(w, "w"), ctypes.byref(d), _mode(mode), int(layer), _ptr(out, "out"),
                                   out.numel() * out.element_size(), _stream(stream)), "moe_prepare_weights")
    return out


def moe_tensor_peak_probe(kind, iters_per_cta: int, workspace, grid: int = 0, stream=None) -> float:
    """Launches the dense tensor-core probe of one instruction kind ("bf16", "f16", "e4m3_e2m1",
    "e4m3_e4m3"); returns the flops the launch performs (time it with events on `stream`)."""
    ws, nb = _ws(workspace)
    flops = ctypes.c_double(0.0)
    k = PEAK_KINDS[kind] if isinstance(kind, str) else int(kind)
    _check(LIB.moe_tensor_peak_probe(k, int(iters_per_cta), int(grid), ctypes.byref(flops), ws, nb, _stream(stream)),
           "moe_tensor_peak_probe")
    return flops.value


def moe_plan_noalloc(topk_ids, d: MoeDims, counts, offsets, row_src, stream=None):
    """moe_plan without a workspace (its scratch is a fixed device array inside the library)."""
    _check(LIB.moe_plan_noalloc(_ptr(topk_ids, "topk_ids"), ctypes.byref(d), _ptr(counts, "counts"),
                                _ptr(offsets, "offsets"), _ptr(row_src, "row_src"), _stream(stream)),
           "moe_plan_noalloc")
