"""The plain C statement of the method (oracle/ref.c, test infrastructure) through ctypes: the
library built by __graft_entry__.build_oracle(), and y of a whole forward pass of any mode from
numpy host inputs. Used by the oracle's own tests and as the checker of the GPU parity tests."""
import ctypes

import numpy as np

from oracle import codecs, moe

_LIB = None


def load():
    """The C oracle library (built once per process)."""
    global _LIB
    if _LIB is None:
        import __graft_entry__
        lib = ctypes.CDLL(__graft_entry__.build_oracle())
        i64p = ctypes.POINTER(ctypes.c_int64)
        vp, i64, ci = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        lib.oracle_plan.restype = ci
        lib.oracle_plan.argtypes = [vp, i64, i64, i64, i64p, i64p, i64p]
        lib.oracle_forward_a16w16.restype = ci
        lib.oracle_forward_a16w16.argtypes = [vp] * 5 + [i64] * 5 + [vp]
        lib.oracle_forward_int.restype = ci
        lib.oracle_forward_int.argtypes = [ci] + [vp] * 8 + [i64] * 5 + [vp] * 5
        lib.oracle_forward_fp8.restype = ci
        lib.oracle_forward_fp8.argtypes = [ci] + [vp] * 8 + [i64] * 5 + [vp] * 3
        lib.oracle_forward_fp8_fp4.restype = ci
        lib.oracle_forward_fp8_fp4.argtypes = [vp] * 8 + [i64] * 5 + [vp] * 3
        lib.oracle_shared_slots.restype = None
        lib.oracle_shared_slots.argtypes = [vp, vp] + [i64] * 4 + [vp, vp]
        for name in ("oracle_e4m3_encode", "oracle_e5m2_encode"):
            getattr(lib, name).restype = ctypes.c_uint8
            getattr(lib, name).argtypes = [ctypes.c_double]
        _LIB = lib
    return _LIB


def forward(lib, mode, h, ids, g, E, I):
    """y of the C statement of `mode`, and its per-pool-row records: C, q, s^A, D (integer modes) or the
    A codes and exponents (FP8 modes)."""
    c = lambda a: np.ascontiguousarray(a)
    ids, g = c(np.asarray(ids, np.int32)), c(np.asarray(g, np.float32))
    T, K = ids.shape
    H = h["x"].shape[1]
    R = int((ids >= 0).sum())
    y = np.zeros((T, H), np.float64)
    rec = {}
    if mode == "a16w16":
        args = [c(codecs.bf16_decode(h[k])) for k in ("x", "w1", "w2")]
        st = lib.oracle_forward_a16w16(args[0].ctypes.data, ids.ctypes.data, g.ctypes.data, args[1].ctypes.data,
                                       args[2].ctypes.data, T, K, E, H, I, y.ctypes.data)
        return st, y, rec
    arr = {k: c(h[k]) for k in ("x", "x_scale", "w1", "w1_scale", "w2", "w2_scale")}
    ptrs = [arr[k].ctypes.data for k in ("x", "x_scale")] + [ids.ctypes.data, g.ctypes.data] + \
           [arr[k].ctypes.data for k in ("w1", "w1_scale", "w2", "w2_scale")]
    if mode in moe.INT_MODES:
        rec = {"c": np.zeros((R, 2 * I), np.int64), "a": np.zeros((R, I), np.int32), "a_scale": np.zeros(R, np.float32),
               "d": np.zeros((R, H), np.int64)}
        st = lib.oracle_forward_int(8 if mode == "a8w8_int8" else 4, *ptrs, T, K, E, H, I, y.ctypes.data,
                                    *[rec[k].ctypes.data for k in ("c", "a", "a_scale", "d")])
    else:
        rec = {"a": np.zeros((R, I), np.uint8), "a_scale": np.zeros((R, I // 32), np.uint8)}
        if mode == "a8w4_fp8_fp4":
            st = lib.oracle_forward_fp8_fp4(*ptrs, T, K, E, H, I, y.ctypes.data, rec["a"].ctypes.data,
                                            rec["a_scale"].ctypes.data)
        else:
            st = lib.oracle_forward_fp8(0 if moe.FP8_FORMAT[mode] == "e4m3" else 1, *ptrs, T, K, E, H, I, y.ctypes.data,
                                        rec["a"].ctypes.data, rec["a_scale"].ctypes.data)
    return st, y, rec
