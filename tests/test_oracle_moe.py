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

import c_oracle
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


def _check_a8w4_golden():
    """Hand-derived A8W4-INT layer (tests/golden/ffn_closed_form_a8w4_int.json): the int4 packing, the
    MSD split of negative codes and codes >= 16, the compensation bias, C, H, the requantised A and D
    are exact; y equals its closed form within the fp32 rounding of s^A."""
    g = _load("ffn_closed_form_a8w4_int.json")
    w1 = np.array([[int(b, 16) for b in g["w1_packed_hex"]]], np.uint8).reshape(1, 4, 1)
    w2 = np.array([[int(b, 16) for b in g["w2_packed_hex"]]], np.uint8).reshape(1, 2, 1)
    w1m = moe.decode_weight("a8w4_int", w1, None, 0)   # math orientation [H, 2I]
    w2m = moe.decode_weight("a8w4_int", w2, None, 0)   # [I, H]
    assert w1m.T.tolist() == g["w1_int4"] and w2m.T.tolist() == g["w2_int4"]
    assert w1m.shape == (2, 4)  # a transposed decode would be (4, 2)
    q = np.array(g["q"], np.int64)
    assert np.floor_divide(q, 16).tolist() == g["q_hi"]
    assert (np.bitwise_and(q, 0x0F) - 8).tolist() == g["q_lo_offset"]
    assert (8 * w1m.astype(np.int64).sum(axis=0)).tolist() == g["bias1"]
    assert moe.msd_int_matmul(q, w1m).tolist() == g["c"]
    y, rec = moe.expert_ffn("a8w4_int", q.astype(np.float64), np.array(g["x_scale"], np.float32), w1m,
                            np.array(g["w1_scale"], np.float32), w2m, np.array(g["w2_scale"], np.float32), inter=2)
    assert rec["c"].tolist() == g["c"] and rec["h"].tolist() == g["h"]
    assert rec["a"].tolist() == g["a_codes"] and rec["d"].tolist() == g["d"]
    s_a = float(np.float32(np.float32(6122.34375) / np.float32(127.0)))
    assert y[0, 0] == pytest.approx(762 * s_a, rel=2e-7) and y[0, 1] == pytest.approx(-127 * s_a, rel=2e-7)
    assert y[0, 1] == pytest.approx(-6122.34375, rel=2.0 ** -22)


def test_a8w4_int_closed_form_golden():
    _check_a8w4_golden()


# Plausible mistakes planted in the A8W4-INT oracle: each must fail the golden.
def _msd_without_bias(q, w):
    q = q.astype(np.int64)
    wi = w.astype(np.int64)
    return 16 * (np.floor_divide(q, 16) @ wi) + ((np.bitwise_and(q, 0x0F) - 8) @ wi)


def _msd_low_nibble_not_offset(q, w):  # q_lo = q & 0x0F (the -8 dropped) while the bias stays
    q = q.astype(np.int64)
    wi = w.astype(np.int64)
    return 16 * (np.floor_divide(q, 16) @ wi) + (np.bitwise_and(q, 0x0F) @ wi) + 8 * wi.sum(axis=0)[None, :]


def _decode_int4_untransposed(mode, w, w_scale, e):
    if mode == "a8w4_int":
        return codecs.int4_unpack(w[e]).astype(np.float64)
    return ORIG_DECODE_WEIGHT(mode, w, w_scale, e)


def _decode_int4_nibbles_swapped(mode, w, w_scale, e):
    if mode == "a8w4_int":
        b = np.asarray(w[e], np.uint8)
        return codecs.int4_unpack(((b >> 4) | (b << 4)).astype(np.uint8)).astype(np.float64).T
    return ORIG_DECODE_WEIGHT(mode, w, w_scale, e)


A8W4_MUTATIONS = {"msd_bias_dropped": ("msd_int_matmul", _msd_without_bias),
                  "msd_low_nibble_not_offset": ("msd_int_matmul", _msd_low_nibble_not_offset),
                  "int4_not_transposed": ("decode_weight", _decode_int4_untransposed),
                  "int4_nibbles_swapped": ("decode_weight", _decode_int4_nibbles_swapped)}


@pytest.mark.parametrize("mutation", list(A8W4_MUTATIONS))
def test_a8w4_int_golden_catches_planted_mistakes(monkeypatch, mutation):
    attr, fn = A8W4_MUTATIONS[mutation]
    monkeypatch.setattr(moe, attr, fn)
    with pytest.raises((AssertionError, ValueError)):
        _check_a8w4_golden()


def _golden_fp8_inputs(g, mode):
    """Dense operands of a sparse FP8 golden: codes and scale bytes not listed are 0 and 127."""
    T, H, I, E = g["T"], g["H"], g["I"], g["E"]
    x = np.zeros((T, H), np.uint8)
    for t, h, c in g["x_codes"]:
        x[t, h] = int(c, 16)
    if mode == "a8w4_fp8_fp4":
        x_scale = np.array(g["x_scale"], np.float32)
        w1 = np.zeros((E, 2 * I, H // 2), np.uint8)
        w2 = np.zeros((E, H, I // 2), np.uint8)
        for arr, key in ((w1, "w1_codes"), (w2, "w2_codes")):  # two e2m1 codes per byte, element 2j low
            for e, n, k, c in g[key]:
                arr[e, n, k // 2] |= np.uint8(int(c, 16) << (4 * (k & 1)))
    else:
        x_scale = np.array(g["x_scale_bytes"], np.uint8)
        w1 = np.zeros((E, 2 * I, H), np.uint8)
        w2 = np.zeros((E, H, I), np.uint8)
        for arr, key in ((w1, "w1_codes"), (w2, "w2_codes")):
            for e, n, k, c in g[key]:
                arr[e, n, k] = int(c, 16)
    w1_scale = np.full((E, 2 * I, H // 32), 127, np.uint8)
    w2_scale = np.full((E, H, I // 32), 127, np.uint8)
    for arr, key in ((w1_scale, "w1_scale_bytes"), (w2_scale, "w2_scale_bytes")):
        for e, n, b, v in g[key]:
            arr[e, n, b] = v
    return x, x_scale, w1, w1_scale, w2, w2_scale


def _dense(pairs, n):
    v = np.zeros(n)
    for i, val in pairs:
        v[i] = float(val) if not isinstance(val, str) else int(val, 16)
    return v


FP8_GOLDENS = [("ffn_closed_form_fp8_e4m3.json", "a8w8_fp8"), ("ffn_closed_form_fp8_e5m2.json", "a8w8_fp8_e5m2"),
               ("ffn_closed_form_fp8_fp4.json", "a8w4_fp8_fp4")]


def _check_fp8_golden(name, mode):
    """The oracle on a hand-derived FP8 example: H, the re-quantised A (codes and UE8M0 exponent
    bytes), L2's rows and y, each against the derivation written in the golden file."""
    g = _load(name)
    x, xs, w1, s1, w2, s2 = _golden_fp8_inputs(g, mode)
    y, rec = moe.forward(mode, x, xs, np.array(g["topk_ids"]), np.array(g["topk_weights"], np.float32), w1, s1, w2, s2,
                         num_experts=g["E"], inter=g["I"], return_intermediates=True)
    r = rec["experts"][0]
    assert r["h"][0].tolist() == _dense(g["h_nonzero"], 2 * g["I"]).tolist(), "H"
    assert r["a"][0].tolist() == _dense(g["a_codes_nonzero"], g["I"]).astype(np.uint8).tolist(), "A codes"
    assert r["a_scale"][0].tolist() == g["a_scale_bytes"], "A exponents"
    assert r["y"][0].tolist() == _dense(g["y_row_nonzero"], g["H"]).tolist(), "L2 rows"
    assert y[0].tolist() == _dense(g["y_nonzero"], g["H"]).tolist(), "y"


@pytest.mark.parametrize("name,mode", FP8_GOLDENS, ids=[m for _, m in FP8_GOLDENS])
def test_closed_form_fp8(name, mode):
    _check_fp8_golden(name, mode)


# Plausible mistakes planted in the oracle (on the CPU): each must fail every FP8 golden, so the
# goldens are what pins decode_weight, the block scales, the nibble order and the re-quantisation.
def _decode_weight_untransposed(mode, w, w_scale, e):
    if mode in moe.FP8_FORMAT:
        return moe.fp8_decode(moe.FP8_FORMAT[mode], w[e]) * np.repeat(codecs.ue8m0_decode(w_scale[e]), 32, axis=-1)
    if mode == "a8w4_fp8_fp4":
        return codecs.e2m1_unpack_decode(w[e]) * np.repeat(codecs.ue8m0_decode(w_scale[e]), 32, axis=-1)
    raise ValueError(mode)


def _decode_weight_per_channel_scale(mode, w, w_scale, e):
    first = w_scale[e][:, :1]  # the first K block's scale for the whole row
    if mode in moe.FP8_FORMAT:
        v = moe.fp8_decode(moe.FP8_FORMAT[mode], w[e]) * codecs.ue8m0_decode(first)
    else:
        v = codecs.e2m1_unpack_decode(w[e]) * codecs.ue8m0_decode(first)
    return v.T


def _decode_weight_nibbles_swapped(mode, w, w_scale, e):
    if mode != "a8w4_fp8_fp4":
        return ORIG_DECODE_WEIGHT(mode, w, w_scale, e)
    b = np.asarray(w[e], np.uint8)
    swapped = ((b >> 4) | (b << 4)).astype(np.uint8)
    return (codecs.e2m1_unpack_decode(swapped) * np.repeat(codecs.ue8m0_decode(w_scale[e]), 32, axis=-1)).T


def _l2_operand_unrounded(mode, a):
    _, rec = ORIG_L2_OPERAND(mode, a)
    return a, rec


ORIG_DECODE_WEIGHT, ORIG_L2_OPERAND = moe.decode_weight, moe.l2_operand
MUTATIONS = {"weight_not_transposed": ("decode_weight", _decode_weight_untransposed),
             "scale_per_output_channel": ("decode_weight", _decode_weight_per_channel_scale),
             "a_not_requantised": ("l2_operand", _l2_operand_unrounded),
             "gate_up_swapped": ("swiglu", lambda h, inter, clamp=None: moe.silu(h[:, inter:]) * h[:, :inter])}


@pytest.mark.parametrize("mutation", list(MUTATIONS))
@pytest.mark.parametrize("name,mode", FP8_GOLDENS, ids=[m for _, m in FP8_GOLDENS])
def test_fp8_goldens_catch_planted_mistakes(monkeypatch, mutation, name, mode):
    attr, fn = MUTATIONS[mutation]
    monkeypatch.setattr(moe, attr, fn)
    with pytest.raises((AssertionError, ValueError)):
        _check_fp8_golden(name, mode)


def test_fp4_golden_catches_swapped_nibbles(monkeypatch):
    monkeypatch.setattr(moe, "decode_weight", _decode_weight_nibbles_swapped)
    with pytest.raises(AssertionError):
        _check_fp8_golden("ffn_closed_form_fp8_fp4.json", "a8w4_fp8_fp4")


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
# The plain C statement of the plan, the shared slots and every mode's layer (oracle/ref.c) against
# this module: two independent implementations of the same readings
# ---------------------------------------------------------------------------------------

def _c_oracle():
    return c_oracle.load()


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


def _c_forward(lib, mode, h, ids, g, E, I):
    return c_oracle.forward(lib, mode, h, ids, g, E, I)


C_CASES = {
    "a16w16": [Workload("tiny_c", "a16w16", 64, 256, 128, 8, 2, 50, 0.05),
               Workload("ragged_c", "a16w16", 77, 128, 256, 5, 3, 51, 0.05)],
    "a8w8_int8": [Workload("tiny_c8", "a8w8_int8", 64, 256, 128, 8, 2, 52, 0.05),
                  Workload("ragged_c8", "a8w8_int8", 77, 128, 256, 5, 3, 53, 0.05)],
    "a8w4_fp8_fp4": [Workload("tiny_c4", "a8w4_fp8_fp4", 64, 256, 128, 8, 2, 54, 0.02),
                     Workload("ragged_c4", "a8w4_fp8_fp4", 77, 256, 256, 5, 3, 55, 0.05),
                     Workload("skew_c4", "a8w4_fp8_fp4", 57, 256, 128, 16, 4, 56, 0.05, zipf_s=1.2, zipf_empty=4)],
    "a8w8_fp8": [Workload("tiny_cf8", "a8w8_fp8", 64, 256, 128, 8, 2, 57, 0.05),
                 Workload("ragged_cf8", "a8w8_fp8", 77, 128, 192, 5, 3, 58, 0.05)],
    "a8w8_fp8_e5m2": [Workload("tiny_ce5", "a8w8_fp8_e5m2", 64, 256, 128, 8, 2, 59, 0.05),
                      Workload("ragged_ce5", "a8w8_fp8_e5m2", 77, 128, 192, 5, 3, 60, 0.05)],
    "a8w4_int": [Workload("tiny_cw4", "a8w4_int", 64, 256, 128, 8, 2, 61, 0.05),
                 Workload("ragged_cw4", "a8w4_int", 77, 128, 256, 5, 3, 62, 0.05)],
}
C_ALL = [(m, w) for m, ws in C_CASES.items() for w in ws]


def _numpy_records(rec, keys):
    """The numpy oracle's per-expert records stacked in pool order (expert by expert, rows ascending)."""
    ex = [rec["experts"][e] for e in sorted(rec["experts"])]
    return {k: np.concatenate([r[k] for r in ex]) for k in keys}


@pytest.mark.parametrize("mode,wl", C_ALL, ids=[w.name for _, w in C_ALL])
def test_c_forward_equals_numpy_forward(mode, wl):
    h = to_numpy(make_inputs(wl, device="cpu"))
    ids = np.ascontiguousarray(h["topk_ids"], dtype=np.int32)
    if wl.name.startswith("ragged"):
        ids[::4, 1] = -1  # masked routes
    g = np.ascontiguousarray(h["topk_weights"], dtype=np.float32)
    st, y, crec = _c_forward(_c_oracle(), mode, h, ids, g, wl.E, wl.I)
    assert st == 0
    ref, rec = moe.forward(mode, h["x"], h["x_scale"], ids, g, h["w1"], h["w1_scale"], h["w2"], h["w2_scale"],
                           num_experts=wl.E, inter=wl.I, return_intermediates=True)
    if mode in moe.INT_MODES:
        # integer accumulators and the re-quantised A, decided in fp32 on both sides, are equal
        nrec = _numpy_records(rec, ("c", "a", "a_scale", "d"))
        for k in ("c", "a", "a_scale", "d"):
            assert np.array_equal(crec[k], nrec[k].astype(crec[k].dtype)), k
        assert np.array_equal(y, ref)  # every later step is the same fp32 arithmetic
        return
    if mode != "a16w16":
        nrec = _numpy_records(rec, ("a", "a_scale"))
        # the float64 L1 sums differ only in order; a code moves only for a value within ~1e-16 of a tie
        assert np.mean(crec["a"] == nrec["a"]) >= 0.999 and np.mean(crec["a_scale"] == nrec["a_scale"]) >= 0.999
    # the same rounding points in both; the float64 sums differ only in their order, which moves a
    # bf16 or fp32 rounding decision only when a value sits within ~1e-16 of a tie
    same = np.mean(y == ref)
    assert same >= 0.999, same
    assert np.abs(y - ref).max() <= 2.0 ** -7 * np.abs(ref).max()


@pytest.mark.parametrize("mode", list(C_CASES))
def test_c_shared_slots_equal_numpy_shared_slots(mode):
    """Two shared experts after the routed ones, with masked routes: the C statement of the shared slots
    and forward against the numpy oracle's."""
    import ctypes  # noqa: F401
    wl = C_CASES[mode][0]
    S = 2
    h = to_numpy(make_inputs(wl, device="cpu", shared=S))
    ids = np.ascontiguousarray(h["topk_ids"], dtype=np.int32)
    ids[::3, 0] = -1
    g = np.ascontiguousarray(h["topk_weights"], dtype=np.float32)
    lib = _c_oracle()
    ids2 = np.zeros((wl.T, wl.K + S), np.int32)
    g2 = np.zeros((wl.T, wl.K + S), np.float32)
    lib.oracle_shared_slots(ids.ctypes.data, g.ctypes.data, wl.T, wl.K, wl.E, S, ids2.ctypes.data, g2.ctypes.data)
    nid, ng = moe.with_shared_slots(ids, g, wl.E, S)
    assert np.array_equal(ids2, nid) and np.array_equal(g2, ng)
    st, y, _ = _c_forward(lib, mode, h, ids2, g2, wl.E + S, wl.I)
    assert st == 0
    ref = moe.forward(mode, h["x"], h["x_scale"], ids, g, h["w1"], h["w1_scale"], h["w2"], h["w2_scale"],
                      num_experts=wl.E, inter=wl.I, num_shared=S)
    assert np.mean(y == ref) >= 0.999
    assert np.abs(y - ref).max() <= 2.0 ** -7 * np.abs(ref).max()


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_c_fp8_codec_equals_numpy_codec(fmt):
    """The C encoders (nearest value from the format's fields) against the numpy ones on every code's value,
    every midpoint between neighbours, both signs and values beyond the largest finite one."""
    lib = _c_oracle()
    if fmt == "e4m3":
        vals, top, fn, want_fn = codecs.E4M3_VALUES[:0x7F], 448.0, lib.oracle_e4m3_encode, codecs.e4m3_encode_rne_satfinite
    else:
        vals = codecs.e5m2_decode(np.arange(0x7C, dtype=np.uint8))  # every finite non-negative code
        top, fn, want_fn = 57344.0, lib.oracle_e5m2_encode, codecs.e5m2_encode_rne_satfinite
    mids = (vals[:-1] + vals[1:]) / 2
    probe = np.concatenate([vals, mids, mids * (1 + 1e-12), mids * (1 - 1e-12), [top, top * 1.03, top * 1.2, 1e9]])
    probe = np.concatenate([probe, -probe]).astype(np.float64)
    want = want_fn(probe)
    got = np.array([fn(float(v)) for v in probe], dtype=np.uint8)
    assert np.array_equal(got, want)
