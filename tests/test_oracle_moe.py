"""Pins of the oracle's plan, SwiGLU and forward path against the pages' worked example,
hand-derived closed forms, invariants, brute force and library routines."""
import dataclasses
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

from oracle import codecs, moe
from workloads import Workload, make_inputs, to_numpy

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------------------------------
# plan
# ---------------------------------------------------------------------------------------


def test_plan_worked_example():
    g = _load("plan_count_prefix_scatter.json")
    counts, offsets, row_src = moe.plan(np.array(g["topk_ids"]), g["num_experts"])
    assert counts.tolist() == g["counts"]
    assert offsets.tolist() == g["offsets"]
    assert row_src.tolist() == g["row_src"]


@pytest.mark.parametrize("seed", range(6))
def test_plan_invariants(seed):
    rng = np.random.default_rng(seed)
    T, E = int(rng.integers(1, 60)), int(rng.integers(1, 20))
    K = int(rng.integers(1, min(E, 6) + 1))
    ids = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    if seed % 2:
        ids[rng.random(ids.shape) < 0.2] = -1  # masked routes
    counts, offsets, row_src = moe.plan(ids, E)
    valid = ids.reshape(-1) >= 0
    assert counts.sum() == valid.sum() == offsets[-1]
    # brute-force count and N_e = |I_e| (ids unique per token)
    for e in range(E):
        assert counts[e] == np.sum(ids == e) == len({i for i in range(T) if e in ids[i]})
    # (i,k) -> pool position is a bijection onto [0, R) and rows sit in their expert's range
    assert sorted(row_src.tolist()) == sorted(np.flatnonzero(valid).tolist())
    for e in range(E):
        for p in range(offsets[e], offsets[e + 1]):
            assert ids.reshape(-1)[row_src[p]] == e


def test_plan_rejects_bad_ids():
    with pytest.raises(ValueError):
        moe.plan(np.array([[0, 4]]), 4)
    with pytest.raises(ValueError):
        moe.plan(np.array([[-2, 1]]), 4)


# ---------------------------------------------------------------------------------------
# SiLU / SwiGLU
# ---------------------------------------------------------------------------------------


def test_silu_closed_forms():
    z = np.linspace(-30, 30, 6001)
    s = moe.silu(z)
    assert moe.silu(np.array([0.0]))[0] == 0.0
    # SiLU(z) - SiLU(-z) = z  (z*sigma(z) - (-z)*sigma(-z) = z*(sigma(z)+sigma(-z)) = z)
    assert np.allclose(s - moe.silu(-z), z, rtol=0, atol=1e-12)
    assert abs(moe.silu(np.array([1.0]))[0] - 1.0 / (1.0 + math.exp(-1.0))) < 1e-15
    assert abs(moe.silu(np.array([60.0]))[0] - 60.0) < 1e-20 * 60 + 1e-12
    assert abs(moe.silu(np.array([-60.0]))[0]) < 1e-24
    assert moe.silu(np.array([-1000.0]))[0] == 0.0
    # the global minimum is at z* = -1.2784645 with value -0.2784645 (z* = -(1 + W(1/e)))
    zs = -(1.0 + scipy.special.lambertw(1.0 / math.e).real)
    assert abs(zs + 1.2784645428) < 1e-9
    assert np.min(s) >= moe.silu(np.array([zs]))[0] - 1e-15
    assert abs(moe.silu(np.array([zs]))[0] + 0.2784645428) < 1e-9
    # sigmoid from scipy (an independent routine)
    assert np.allclose(s, z * scipy.special.expit(z), rtol=1e-14, atol=1e-300)


def test_swiglu_gate_is_first_half():
    h = np.array([[1.0, -1.0]])  # gate = 1, up = -1
    assert moe.swiglu(h, 1)[0, 0] == pytest.approx(-1.0 / (1.0 + math.exp(-1.0)), abs=1e-15)


# ---------------------------------------------------------------------------------------
# Closed-form examples
# ---------------------------------------------------------------------------------------


def test_closed_form_a16w16():
    g = _load("ffn_closed_form_a16w16.json")
    bf = lambda a: codecs.bf16_encode(np.array(a, dtype=np.float64))
    y = moe.forward("a16w16", bf(g["x"]), None, np.array(g["topk_ids"]),
                    np.array(g["topk_weights"], dtype=np.float32), bf(g["w1"]), None, bf(g["w2"]), None,
                    num_experts=2, inter=g["intermediate"])
    assert y.tolist() == g["y"]


def test_closed_form_int8():
    g = _load("ffn_closed_form_int8.json")
    q = np.array(g["q"], dtype=np.int8)
    w1 = np.array([g["w1_stored"]], dtype=np.int8)
    w2 = np.array([g["w2_stored"]], dtype=np.int8)
    y, rec = moe.expert_ffn("a8w8_int8", q.astype(np.float64), np.array(g["x_scale"], np.float32),
                            moe.decode_weight("a8w8_int8", w1, None, 0),
                            np.array(g["w1_scale"], np.float32),
                            moe.decode_weight("a8w8_int8", w2, None, 0),
                            np.array(g["w2_scale"], np.float32), inter=1)
    assert rec["c"].tolist() == g["c"] and rec["h"].tolist() == g["h"]
    assert rec["d"].tolist() == g["d"]
    a = 12.0 / (1.0 + math.exp(-3.0))
    assert rec["a"].tolist() == [[127]]
    assert y[0, 0] == pytest.approx(a, rel=2e-7) and y[0, 1] == pytest.approx(-2 * a, rel=2e-7)


# ---------------------------------------------------------------------------------------
# Whole path: brute force, reductions, linearity
# ---------------------------------------------------------------------------------------


def _np(inp):
    return to_numpy(inp)


TINY = {
    "a16w16": Workload("t", "a16w16", 12, 64, 64, 4, 2, 11, 0.1),
    "a8w8_fp8": Workload("t", "a8w8_fp8", 12, 128, 64, 4, 2, 12, 0.1),
    "a8w8_int8": Workload("t", "a8w8_int8", 12, 96, 64, 4, 3, 13, 0.1),
    "a8w4_fp8_fp4": Workload("t", "a8w4_fp8_fp4", 12, 128, 64, 4, 2, 14, 0.1),
    "a8w4_int": Workload("t", "a8w4_int", 12, 96, 64, 4, 3, 15, 0.1),
    "a8w8_fp8_e5m2": Workload("t", "a8w8_fp8_e5m2", 12, 128, 64, 4, 2, 16, 0.1),
}


def _forward(mode, d, wl, **kw):
    return moe.forward(mode, d["x"], d["x_scale"], d["topk_ids"], d["topk_weights"], d["w1"],
                       d["w1_scale"], d["w2"], d["w2_scale"], num_experts=wl.E, inter=wl.I, **kw)


@pytest.mark.parametrize("mode", list(TINY))
def test_brute_force_per_token_equals_pooled_path(mode):
    wl = TINY[mode]
    d = _np(make_inputs(wl))
    y = _forward(mode, d, wl)
    yb = moe.forward_tokens(mode, range(wl.T), d["x"], d["x_scale"], d["topk_ids"], d["topk_weights"],
                            d["w1"], d["w1_scale"], d["w2"], d["w2_scale"], inter=wl.I)
    assert np.array_equal(y, yb)
    assert np.all(np.isfinite(y)) and np.abs(y).max() > 0


def test_dense_reduction_matches_library_routines():
    """E=1, K=1, G=1: y = bf16(bf16(SwiGLU(x W1)) W2), computed with torch float64 matmul
    and torch's SiLU, an implementation independent of the oracle's."""
    wl = Workload("dense", "a16w16", 20, 64, 32, 1, 1, 21, 0.2)
    inp = make_inputs(wl)
    inp["topk_weights"] = torch.ones_like(inp["topk_weights"])
    d = _np(inp)
    y = _forward("a16w16", d, wl)
    x = inp["x"].double()
    h = x @ inp["w1"][0].double()
    a = (torch.nn.functional.silu(h[:, :32]) * h[:, 32:]).to(torch.bfloat16).double()
    ref = (a @ inp["w2"][0].double()).float().to(torch.bfloat16).double().numpy()
    assert np.array_equal(y, ref)


def test_linearity_in_gates_and_masking():
    wl = TINY["a16w16"]
    d = _np(make_inputs(wl))
    d0 = dict(d, topk_weights=np.zeros_like(d["topk_weights"]))
    assert np.all(_forward("a16w16", d0, wl) == 0.0)
    # one-hot gates select slot 0 only; masking slot 1 gives the same result
    g1 = np.zeros_like(d["topk_weights"])
    g1[:, 0] = 1.0
    y1 = _forward("a16w16", dict(d, topk_weights=g1), wl)
    ids_m = d["topk_ids"].copy()
    ids_m[:, 1] = -1
    ym = _forward("a16w16", dict(d, topk_ids=ids_m), wl)
    y1m = _forward("a16w16", dict(d, topk_ids=ids_m, topk_weights=g1), wl)
    assert np.array_equal(y1, y1m)
    _, rec = _forward("a16w16", dict(d, topk_ids=ids_m), wl, return_intermediates=True)
    assert np.all(rec["comb"].reshape(wl.T, wl.K, -1)[:, 1] == 0.0)
    assert ym.shape == y1.shape


def test_int8_path_accumulators_are_integers_in_range():
    wl = TINY["a8w8_int8"]
    d = _np(make_inputs(wl))
    _, rec = _forward("a8w8_int8", d, wl, return_intermediates=True)
    for e, r in rec["experts"].items():
        assert r["c"].dtype == np.int64 and r["d"].dtype == np.int64
        assert np.abs(r["a"].astype(np.int64)).max() <= 127


def test_fp8_mode_decoding_uses_block_scales():
    """Scaling one 32-block's UE8M0 byte by +1 doubles exactly that block's contribution."""
    wl = TINY["a8w8_fp8"]
    d = _np(make_inputs(wl))
    xd = moe.decode_x("a8w8_fp8", d["x"], d["x_scale"])
    sc = d["x_scale"].copy()
    sc[0, 1] += 1
    xd2 = moe.decode_x("a8w8_fp8", d["x"], sc)
    assert np.array_equal(xd2[0, 32:64], 2 * xd[0, 32:64])
    assert np.array_equal(xd2[0, :32], xd[0, :32]) and np.array_equal(xd2[1:], xd[1:])


# ---------------------------------------------------------------------------------------
# activation_clamp (p1 parameter: symmetric clamp of the activation function's input)
# ---------------------------------------------------------------------------------------


def _h_range(mode, d, wl):
    _, rec = _forward(mode, d, wl, return_intermediates=True)
    hs = np.concatenate([np.abs(r["h"]).ravel() for r in rec["experts"].values()])
    return hs.min(), hs.max()


@pytest.mark.parametrize("mode", list(TINY))
def test_activation_clamp_limits(mode):
    """A clamp at or above every |H| changes nothing; a clamp of 0 makes every output 0
    (SiLU(0) * 0 = 0 in every mode, so every requantised A and every Y is 0)."""
    wl = TINY[mode]
    d = _np(make_inputs(wl))
    y = _forward(mode, d, wl)
    _, hmax = _h_range(mode, d, wl)
    assert np.array_equal(_forward(mode, d, wl, clamp=float(hmax)), y)
    assert np.all(_forward(mode, d, wl, clamp=0.0) == 0.0)


@pytest.mark.parametrize("mode", ["a16w16", "a8w8_fp8"])
def test_activation_clamp_saturates(mode):
    """With the clamp at the smallest |H| every SwiGLU input sits on the clamp, so doubling W1
    (which doubles H exactly) leaves the output unchanged; without the clamp it changes."""
    wl = TINY[mode]
    d = _np(make_inputs(wl))
    hmin, _ = _h_range(mode, d, wl)
    assert hmin > 0
    d2 = dict(d)
    if mode == "a16w16":
        d2["w1"] = codecs.bf16_encode(2.0 * codecs.bf16_decode(d["w1"]))
    else:  # one more unit of the UE8M0 block exponent doubles every weight exactly
        d2["w1_scale"] = (d["w1_scale"].astype(np.int32) + 1).astype(np.uint8)
    c = float(hmin)
    assert np.array_equal(_forward(mode, d, wl, clamp=c), _forward(mode, d2, wl, clamp=c))
    assert not np.array_equal(_forward(mode, d, wl), _forward(mode, d2, wl))


@pytest.mark.parametrize("mode", list(TINY))
def test_activation_clamp_brute_force_equals_pooled_path(mode):
    wl = TINY[mode]
    d = _np(make_inputs(wl))
    hmin, hmax = _h_range(mode, d, wl)
    c = float(0.5 * (hmin + hmax) / 4)
    y = _forward(mode, d, wl, clamp=c)
    yb = moe.forward_tokens(mode, range(wl.T), d["x"], d["x_scale"], d["topk_ids"], d["topk_weights"],
                            d["w1"], d["w1_scale"], d["w2"], d["w2_scale"], inter=wl.I, clamp=c)
    assert np.array_equal(y, yb)
    assert not np.array_equal(y, _forward(mode, d, wl))


# ---------------------------------------------------------------------------------------
# Shared experts (DeepGEMM page §6): every token, weight 1, the slot after the routed ones
# ---------------------------------------------------------------------------------------


def test_shared_expert_alone_is_a_dense_ffn():
    """Routed gates all zero, one shared expert: y = bf16(bf16(SwiGLU(x W1s)) W2s) on every
    token, computed with torch float64 matmul and torch's SiLU (independent of the oracle)."""
    wl = Workload("shared_dense", "a16w16", 20, 64, 32, 3, 2, 22, 0.2)
    inp = make_inputs(wl, shared=1)
    assert inp["w1"].shape[0] == 4 and inp["w2"].shape[0] == 4
    inp["topk_weights"] = torch.zeros_like(inp["topk_weights"])
    d = _np(inp)
    y = _forward("a16w16", d, wl, num_shared=1)
    x = inp["x"].double()
    h = x @ inp["w1"][3].double()
    a = (torch.nn.functional.silu(h[:, :32]) * h[:, 32:]).to(torch.bfloat16).double()
    ref = (a @ inp["w2"][3].double()).float().to(torch.bfloat16).double().numpy()
    assert np.array_equal(y, ref)
    # masking every routed slot instead of zeroing its gate gives the same output
    ids_m = np.full_like(d["topk_ids"], -1)
    assert np.array_equal(_forward("a16w16", dict(d, topk_ids=ids_m), wl, num_shared=1), ref)


@pytest.mark.parametrize("mode", list(TINY))
def test_shared_copy_of_the_routed_expert_doubles_the_output(mode):
    """Every token routed to expert 0 with gate 1 (K = 1) and a shared expert that is a copy of
    expert 0: both slots hold the same bf16 row c, so y = bf16(c + c) = 2 y(no shared), exactly."""
    wl = dataclasses.replace(TINY[mode], K=1)
    inp = make_inputs(wl, shared=1)
    for name in ("w1", "w1_scale", "w2", "w2_scale"):
        if inp[name] is not None:
            inp[name][wl.E] = inp[name][0]
    inp["topk_ids"] = torch.zeros_like(inp["topk_ids"])
    inp["topk_weights"] = torch.ones_like(inp["topk_weights"])
    d = _np(inp)
    y0 = _forward(mode, d, wl)
    y1 = _forward(mode, d, wl, num_shared=1)
    assert np.abs(y0).max() > 0
    assert np.array_equal(y1, 2.0 * y0)


@pytest.mark.parametrize("mode", list(TINY))
def test_shared_brute_force_per_token_equals_pooled_path(mode):
    wl = TINY[mode]
    d = _np(make_inputs(wl, shared=2))
    y, rec = _forward(mode, d, wl, num_shared=2, return_intermediates=True)
    yb = moe.forward_tokens(mode, range(wl.T), d["x"], d["x_scale"], d["topk_ids"], d["topk_weights"],
                            d["w1"], d["w1_scale"], d["w2"], d["w2_scale"], inter=wl.I,
                            num_experts=wl.E, num_shared=2)
    assert np.array_equal(y, yb)
    # each shared expert sees every token; the routed experts see their routed rows only
    assert rec["counts"].tolist()[wl.E:] == [wl.T, wl.T]
    assert sum(rec["counts"].tolist()[:wl.E]) == wl.T * wl.K
    assert not np.array_equal(y, _forward(mode, d, wl))


# ---------------------------------------------------------------------------------------
# The plain C statement of the plan and of the A16W16 layer (oracle/ref.c) against this module:
# two independent implementations of the same readings
# ---------------------------------------------------------------------------------------

def _c_oracle():
    import ctypes
    import __graft_entry__
    lib = ctypes.CDLL(__graft_entry__.build_oracle())
    i64p = ctypes.POINTER(ctypes.c_int64)
    lib.oracle_plan.restype = ctypes.c_int
    lib.oracle_plan.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, i64p, i64p, i64p]
    lib.oracle_forward_a16w16.restype = ctypes.c_int
    lib.oracle_forward_a16w16.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int64] * 5 + [ctypes.c_void_p]
    lib.oracle_forward_int8.restype = ctypes.c_int
    lib.oracle_forward_int8.argtypes = [ctypes.c_void_p] * 8 + [ctypes.c_int64] * 5 + [ctypes.c_void_p]
    lib.oracle_forward_fp8_fp4.restype = ctypes.c_int
    lib.oracle_forward_fp8_fp4.argtypes = [ctypes.c_void_p] * 8 + [ctypes.c_int64] * 5 + [ctypes.c_void_p]
    return lib


def _c_plan(lib, ids, E):
    import ctypes
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    T, K = ids.shape
    counts, offsets = np.zeros(E, np.int64), np.zeros(E + 1, np.int64)
    row_src = np.zeros(max(T * K, 1), np.int64)
    p = lambda a: a.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))
    st = lib.oracle_plan(ids.ctypes.data, T, K, E, p(counts), p(offsets), p(row_src))
    return st, counts, offsets, row_src[:offsets[-1]]


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_c_plan_equals_numpy_plan(seed):
    lib = _c_oracle()
    rng = np.random.default_rng(seed)
    E = 13
    ids = rng.integers(-1, E, size=(57, 3)).astype(np.int32)  # including masked routes
    st, counts, offsets, row_src = _c_plan(lib, ids, E)
    c2, o2, r2 = moe.plan(ids, E)
    assert st == 0 and counts.tolist() == c2.tolist() and offsets.tolist() == o2.tolist()
    assert row_src.tolist() == r2.tolist()
    ids[5, 1] = E  # an id outside [-1, E)
    assert _c_plan(lib, ids, E)[0] == -1


@pytest.mark.parametrize("case", ["tiny", "ragged_masked"])
def test_c_forward_a16w16_equals_numpy_forward(case):
    wl = (Workload("tiny_c", "a16w16", 64, 256, 128, 8, 2, 50, 0.05) if case == "tiny"
          else Workload("ragged_c", "a16w16", 77, 128, 256, 5, 3, 51, 0.05))
    h = to_numpy(make_inputs(wl, device="cpu"))
    ids = np.ascontiguousarray(h["topk_ids"], dtype=np.int32)
    if case == "ragged_masked":
        ids[::4, 1] = -1
    g = np.ascontiguousarray(h["topk_weights"], dtype=np.float32)
    x = np.ascontiguousarray(codecs.bf16_decode(h["x"]))
    w1 = np.ascontiguousarray(codecs.bf16_decode(h["w1"]))
    w2 = np.ascontiguousarray(codecs.bf16_decode(h["w2"]))
    y = np.zeros((wl.T, wl.H), np.float64)
    st = _c_oracle().oracle_forward_a16w16(x.ctypes.data, ids.ctypes.data, g.ctypes.data, w1.ctypes.data,
                                           w2.ctypes.data, wl.T, wl.K, wl.E, wl.H, wl.I, y.ctypes.data)
    assert st == 0
    ref = moe.forward("a16w16", h["x"], None, ids, g, h["w1"], None, h["w2"], None, num_experts=wl.E, inter=wl.I)
    # the same rounding points in both; the float64 sums differ only in their order, which moves
    # a bf16 or fp32 rounding decision only when a value sits within ~1e-16 of a tie
    same = np.mean(y == ref)
    assert same >= 0.999, same
    assert np.abs(y - ref).max() <= 2.0 ** -7 * np.abs(ref).max()


@pytest.mark.parametrize("case", ["tiny", "ragged_masked"])
def test_c_forward_int8_equals_numpy_forward(case):
    wl = (Workload("tiny_c8", "a8w8_int8", 64, 256, 128, 8, 2, 52, 0.05) if case == "tiny"
          else Workload("ragged_c8", "a8w8_int8", 77, 128, 256, 5, 3, 53, 0.05))
    h = to_numpy(make_inputs(wl, device="cpu"))
    ids = np.ascontiguousarray(h["topk_ids"], dtype=np.int32)
    if case == "ragged_masked":
        ids[::4, 1] = -1
    g = np.ascontiguousarray(h["topk_weights"], dtype=np.float32)
    arr = {k: np.ascontiguousarray(h[k]) for k in ("x", "x_scale", "w1", "w1_scale", "w2", "w2_scale")}
    assert arr["x"].dtype == np.int8 and arr["w1"].dtype == np.int8 and arr["x_scale"].dtype == np.float32
    y = np.zeros((wl.T, wl.H), np.float64)
    st = _c_oracle().oracle_forward_int8(arr["x"].ctypes.data, arr["x_scale"].ctypes.data, ids.ctypes.data,
                                         g.ctypes.data, arr["w1"].ctypes.data, arr["w1_scale"].ctypes.data,
                                         arr["w2"].ctypes.data, arr["w2_scale"].ctypes.data, wl.T, wl.K, wl.E, wl.H,
                                         wl.I, y.ctypes.data)
    assert st == 0
    ref = moe.forward("a8w8_int8", h["x"], h["x_scale"], ids, g, h["w1"], h["w1_scale"], h["w2"], h["w2_scale"],
                      num_experts=wl.E, inter=wl.I)
    same = np.mean(y == ref)
    assert same >= 0.999, same
    assert np.abs(y - ref).max() <= 2.0 ** -7 * np.abs(ref).max()


@pytest.mark.parametrize("case", ["tiny", "ragged_masked", "skewed"])
def test_c_forward_fp8_fp4_equals_numpy_forward(case):
    wl = {"tiny": Workload("tiny_c4", "a8w4_fp8_fp4", 64, 256, 128, 8, 2, 54, 0.02),
          "ragged_masked": Workload("ragged_c4", "a8w4_fp8_fp4", 77, 256, 256, 5, 3, 55, 0.05),
          "skewed": Workload("skew_c4", "a8w4_fp8_fp4", 57, 256, 128, 16, 4, 56, 0.05, zipf_s=1.2, zipf_empty=4)}[case]
    h = to_numpy(make_inputs(wl, device="cpu"))
    ids = np.ascontiguousarray(h["topk_ids"], dtype=np.int32)
    if case == "ragged_masked":
        ids[::4, 1] = -1
    g = np.ascontiguousarray(h["topk_weights"], dtype=np.float32)
    arr = {k: np.ascontiguousarray(h[k]) for k in ("x", "x_scale", "w1", "w1_scale", "w2", "w2_scale")}
    assert arr["x"].dtype == np.uint8 and arr["x_scale"].shape == (wl.T, wl.H // 128)
    assert arr["w1"].shape == (wl.E, 2 * wl.I, wl.H // 2) and arr["w1_scale"].shape == (wl.E, 2 * wl.I, wl.H // 32)
    assert arr["w2"].shape == (wl.E, wl.H, wl.I // 2) and arr["w2_scale"].shape == (wl.E, wl.H, wl.I // 32)
    x_scale = np.ascontiguousarray(arr["x_scale"], dtype=np.float32)
    y = np.zeros((wl.T, wl.H), np.float64)
    st = _c_oracle().oracle_forward_fp8_fp4(arr["x"].ctypes.data, x_scale.ctypes.data, ids.ctypes.data,
                                            g.ctypes.data, arr["w1"].ctypes.data, arr["w1_scale"].ctypes.data,
                                            arr["w2"].ctypes.data, arr["w2_scale"].ctypes.data, wl.T, wl.K, wl.E,
                                            wl.H, wl.I, y.ctypes.data)
    assert st == 0
    ref = moe.forward("a8w4_fp8_fp4", h["x"], h["x_scale"], ids, g, h["w1"], h["w1_scale"], h["w2"],
                      h["w2_scale"], num_experts=wl.E, inter=wl.I)
    same = np.mean(y == ref)
    assert same >= 0.999, same
    assert np.abs(y - ref).max() <= 2.0 ** -7 * np.abs(ref).max()


def test_c_e4m3_codec_equals_numpy_codec():
    """The C encoder (nearest value from the format's fields) against the numpy one (table search) on
    every code's value, every midpoint between neighbours, both signs and values beyond 448."""
    import ctypes
    lib = _c_oracle()
    vals = codecs.E4M3_VALUES[:0x7F]
    mids = (vals[:-1] + vals[1:]) / 2
    probe = np.concatenate([vals, mids, mids * (1 + 1e-12), mids * (1 - 1e-12), [448.0, 460.0, 464.0, 500.0, 1e9]])
    probe = np.concatenate([probe, -probe]).astype(np.float64)
    want = codecs.e4m3_encode_rne_satfinite(probe)
    fn = lib.oracle_e4m3_encode
    fn.restype = ctypes.c_uint8
    fn.argtypes = [ctypes.c_double]
    got = np.array([fn(float(v)) for v in probe], dtype=np.uint8)
    assert np.array_equal(got, want)
