"""GPU parity of every stage of the path against the CPU oracle, through the C ABI.

Bars: counts, offsets and the per-expert multiset of row identities bit-exact; floating
point within max|y - y_ref| <= tol * max|y_ref| (2e-2 bf16 and the integer modes, 6e-2 for the
FP8/FP4 modes); integer L2 accumulators bit-exact given the kernel's own re-quantised operand.
"""
import os

import numpy as np
import pytest
import torch

import c_oracle
from gpu_util import TOL, assert_close, covering_tokens, lib, oracle_tokens, region, run_forward, slice_tokens, y_numpy
from oracle import codecs as ocodecs
from oracle import moe as omoe
from workloads import WORKLOADS, Workload, make_inputs, to_numpy

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def moe():
    return lib()


def oracle_forward(wl, inp, **kw):
    """y of the oracle for the inputs: the plain C statement (oracle/ref.c, which tests/test_oracle_moe.py
    holds equal to the numpy oracle and to the hand-derived goldens) for every case it states; the
    numpy oracle for the options only that one states (an activation clamp, shared experts, the
    intermediates) and for the full-size workloads (the C statement takes every expert's weights
    decoded to float64)."""
    h = to_numpy(inp)
    if not kw and wl.E * wl.H * wl.I <= (1 << 25):
        st, y, _ = c_oracle.forward(c_oracle.load(), wl.mode, h, h["topk_ids"], h["topk_weights"], wl.E, wl.I)
        assert st == 0, f"C oracle status {st}"
        return y
    return omoe.forward(wl.mode, h["x"], h["x_scale"], h["topk_ids"], h["topk_weights"], h["w1"], h["w1_scale"],
                        h["w2"], h["w2_scale"], num_experts=wl.E, inter=wl.I, **kw)


# Small cases that still span several 128-row tiles, several column tiles and ragged tails.
CASES = {
    "a16w16": [WORKLOADS["tiny_bf16"], Workload("ragged_bf16", "a16w16", 300, 512, 384, 6, 2, 21, 0.05)],
    "a8w8_fp8": [Workload("tiny_fp8", "a8w8_fp8", 64, 256, 128, 8, 2, 22, 0.02),
                 Workload("ragged_fp8", "a8w8_fp8", 300, 512, 384, 6, 2, 23, 0.05)],
    "a8w8_int8": [Workload("tiny_int8", "a8w8_int8", 64, 256, 128, 8, 2, 24, 0.02),
                  Workload("ragged_int8", "a8w8_int8", 300, 512, 384, 6, 3, 25, 0.05)],
    "a8w4_int": [Workload("tiny_w4", "a8w4_int", 64, 256, 128, 8, 2, 37, 0.02),
                 Workload("ragged_w4", "a8w4_int", 300, 512, 384, 6, 3, 38, 0.05)],
    "a8w4_fp8_fp4": [Workload("tiny_fp4", "a8w4_fp8_fp4", 64, 256, 128, 8, 2, 26, 0.02),
                     Workload("ragged_fp4", "a8w4_fp8_fp4", 300, 512, 384, 6, 2, 27, 0.05),
                     Workload("skew_fp4", "a8w4_fp8_fp4", 257, 256, 256, 64, 8, 28, 0.05, zipf_s=1.2, zipf_empty=8),
                     # hidden 3584 = 7 * 512 = 16 * 224: token-major L1 and the 224-column L2 tiles
                     Workload("n224_fp4", "a8w4_fp8_fp4", 260, 3584, 512, 6, 2, 29, 0.05)],
}
CASES["a8w8_fp8"].append(Workload("n224_fp8", "a8w8_fp8", 200, 3584, 512, 5, 2, 30, 0.05))
CASES["a8w8_fp8_e5m2"] = [Workload("tiny_e5m2", "a8w8_fp8_e5m2", 64, 256, 128, 8, 2, 39, 0.02),
                          Workload("ragged_e5m2", "a8w8_fp8_e5m2", 300, 512, 384, 6, 2, 40, 0.05),
                          Workload("n224_e5m2", "a8w8_fp8_e5m2", 200, 3584, 512, 5, 2, 41, 0.05)]
ALL = [(m, wl) for m, wls in CASES.items() for wl in wls]


def check_plan(out, wl, ids):
    ids_np = ids.cpu().numpy()
    counts, offsets, row_src = omoe.plan(ids_np, wl.E)
    assert out["counts"].cpu().numpy().tolist() == counts.tolist()
    assert out["offsets"].cpu().numpy().tolist() == offsets.tolist()
    got = out["row_src"].cpu().numpy()[:offsets[-1]]
    for e in range(wl.E):
        lo, hi = offsets[e], offsets[e + 1]
        assert sorted(got[lo:hi].tolist()) == sorted(row_src[lo:hi].tolist()), f"expert {e}"


@pytest.mark.parametrize("mode,wl", ALL, ids=[f"{m}-{w.name}" for m, w in ALL])
@pytest.mark.parametrize("flags", [0, 1], ids=["default", "simt"])
def test_forward_matches_oracle(moe, mode, wl, flags):
    inp = make_inputs(wl, device=DEV)
    out = run_forward(moe, wl, inp, flags=flags, stages=True)
    assert out["status"] == 0
    check_plan(out, wl, inp["topk_ids"])
    ref, rec = oracle_forward(wl, inp, return_intermediates=True)
    # weighted combine rows (stage S5) and the output (stage S6)
    L = out["layout"]
    comb = region(out["ws"], L, "comb", torch.bfloat16, wl.T * wl.K * wl.H).view(wl.T * wl.K, wl.H)
    assert_close(y_numpy(comb), rec["comb"], mode, "combine rows")
    assert_close(y_numpy(out["y"]), ref, mode)


@pytest.mark.parametrize("mode,wl", ALL[:1] + ALL[2:3], ids=["bf16", "fp8"])
def test_deterministic(moe, mode, wl):
    inp = make_inputs(wl, device=DEV)
    y1 = run_forward(moe, wl, inp)["y"]
    y2 = run_forward(moe, wl, inp)["y"]
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))


def test_dispatch_gathers_rows(moe):
    wl = CASES["a8w4_fp8_fp4"][1]
    inp = make_inputs(wl, device=DEV)
    out = run_forward(moe, wl, inp, stages=True)
    L = out["layout"]
    rows = L["pool_rows"]
    pool_src = region(out["ws"], L, "pool_src", torch.int32, rows).cpu().numpy()
    xp = region(out["ws"], L, "x_pool", torch.uint8, rows * wl.H).view(rows, wl.H).cpu().numpy()
    xs = region(out["ws"], L, "x_pool_scale", torch.float32, rows * wl.H // 128).view(rows, -1).cpu().numpy()
    x = inp["x"].cpu().numpy()
    xsc = inp["x_scale"].cpu().numpy()
    hdr = region(out["ws"], L, "header", torch.int32, 16).cpu().numpy()
    n_pad = hdr[2]
    assert n_pad % 128 == 0 and n_pad >= wl.T * wl.K
    for r in range(n_pad):
        s = pool_src[r]
        if s >= 0:
            assert np.array_equal(xp[r], x[s // wl.K]) and np.array_equal(xs[r], xsc[s // wl.K])
    # every routed (i, k) has exactly one pool row
    assert sorted(int(v) for v in pool_src[:n_pad] if v >= 0) == list(range(wl.T * wl.K))


# Per-expert row counts that put an expert's last route tile at the edges of the INT8 kernel's
# token granularity (1, 16, 17, 127 tokens; 128, 129 and 255 spill into a second tile).
TAIL_COUNTS = [1, 16, 17, 127, 128, 129, 255]


def _tail_inputs(mode, seed):
    wl = Workload(f"tail_{mode}", mode, sum(TAIL_COUNTS), 512, 256, len(TAIL_COUNTS), 1, seed, 0.05)
    inp = make_inputs(wl, device=DEV)
    inp["topk_ids"] = torch.repeat_interleave(torch.arange(wl.E, dtype=torch.int32),
                                              torch.tensor(TAIL_COUNTS))[:, None].to(DEV).contiguous()
    return wl, inp


@pytest.mark.parametrize("mode", ["a8w8_int8", "a8w4_int"])
@pytest.mark.parametrize("case", ["ragged", "tail_sizes"])
def test_int8_l2_accumulators_exact(moe, mode, case):
    """D = A^int8 . W2 must be the exact integer product: recompute the weighted rows from the
    kernel's own A^int8 and s^A with an integer GEMM and the page's fp32 dequant order, and
    require bit equality (int8 or int4 weights). The tail case gives the experts 1, 16, 17, 127,
    128, 129 and 255 rows, and also checks y against the oracle."""
    if case == "ragged":
        wl = CASES[mode][1]
        inp = make_inputs(wl, device=DEV)
    else:
        wl, inp = _tail_inputs(mode, 47)
    out = run_forward(moe, wl, inp, stages=True)
    assert out["status"] == 0
    if case == "tail_sizes":
        check_plan(out, wl, inp["topk_ids"])
        assert_close(y_numpy(out["y"]), oracle_forward(wl, inp), wl.mode)
    L = out["layout"]
    rows = L["pool_rows"]
    ws = out["ws"]
    pool_src = region(ws, L, "pool_src", torch.int32, rows).cpu().numpy()
    pad_off = region(ws, L, "pad_offsets", torch.int32, wl.E + 1).cpu().numpy()
    a_q = region(ws, L, "a_pool", torch.int8, rows * wl.I).view(rows, wl.I).cpu().numpy()
    s_a = region(ws, L, "a_pool_scale", torch.float32, rows).cpu().numpy()
    comb = region(ws, L, "comb", torch.int16, wl.T * wl.K * wl.H).view(wl.T * wl.K, wl.H).cpu().numpy()
    h = to_numpy(inp)
    g = h["topk_weights"].reshape(-1)
    n_pad = int(region(ws, L, "header", torch.int32, 16).cpu().numpy()[2])
    assert np.abs(a_q[:n_pad][pool_src[:n_pad] >= 0].astype(np.int32)).max() <= 127
    # the row quantiser, from the kernel's own fp32 A: s = max(amax / 127, 1e-8) and
    # q = clip(rint(A / s), -127, 127), every step an IEEE fp32 operation (numpy float32 divides
    # with round-to-nearest-even; rint rounds half to even)
    routed_rows = np.nonzero(pool_src[:n_pad] >= 0)[0]
    a32 = region(ws, L, "a_f32", torch.float32, rows * wl.I).view(rows, wl.I).cpu().numpy()[routed_rows]
    s_ref = np.maximum(np.abs(a32).max(axis=1) / np.float32(127.0), np.float32(1e-8)).astype(np.float32)
    q_ref = np.clip(np.rint(a32 / s_ref[:, None]), -127, 127).astype(np.int8)
    assert np.array_equal(s_a[routed_rows], s_ref)
    assert np.array_equal(a_q[routed_rows], q_ref)
    if mode == "a8w4_int":  # the row quantiser's plane and code sums of the same codes
        routed = np.nonzero(pool_src[:n_pad] >= 0)[0]
        _check_w4_operands(ws, L, "a_pool_planes", 1, rows, wl.I, routed, a_q[routed].astype(np.int64))
        x_q = region(ws, L, "x_pool", torch.int8, rows * wl.H).view(rows, wl.H).cpu().numpy()
        _check_w4_operands(ws, L, "x_pool_planes", 0, rows, wl.H, routed, x_q[routed].astype(np.int64))
    for e in range(wl.E):
        lo, hi = pad_off[e], pad_off[e + 1]
        src = pool_src[lo:hi]
        keep = src >= 0
        if not keep.any():
            continue
        w2 = (ocodecs.int4_unpack(h["w2"][e]) if mode == "a8w4_int" else h["w2"][e]).astype(np.int64).T  # [I, H]
        d = a_q[lo:hi][keep].astype(np.int64) @ w2
        y32 = (d.astype(np.float32) * h["w2_scale"][e][None, :]).astype(np.float32)
        y32 = (y32 * s_a[lo:hi][keep][:, None]).astype(np.float32)
        c = (g[src[keep]][:, None].astype(np.float32) * y32).astype(np.float32)
        ref_bits = torch.from_numpy(c).to(torch.bfloat16).view(torch.int16).numpy()
        assert np.array_equal(comb[src[keep]], ref_bits), f"expert {e}"


EDGE = [
    Workload("one_token", "a16w16", 1, 256, 128, 8, 2, 31, 0.05),
    Workload("one_expert", "a16w16", 70, 256, 128, 1, 1, 32, 0.05),
    Workload("topk1", "a8w4_fp8_fp4", 40, 256, 128, 16, 1, 33, 0.05),
    Workload("many_empty", "a8w8_fp8", 20, 256, 128, 256, 2, 34, 0.05),
    Workload("max_topk", "a16w16", 9, 128, 128, 40, 32, 35, 0.05),
]


@pytest.mark.parametrize("wl", EDGE, ids=[w.name for w in EDGE])
def test_edge_shapes(moe, wl):
    inp = make_inputs(wl, device=DEV)
    out = run_forward(moe, wl, inp, stages=True)
    assert out["status"] == 0
    check_plan(out, wl, inp["topk_ids"])
    assert_close(y_numpy(out["y"]), oracle_forward(wl, inp), wl.mode)


def test_all_rows_to_one_expert_and_masked_routes(moe):
    wl = Workload("skewed", "a16w16", 200, 256, 128, 4, 2, 36, 0.05)
    inp = make_inputs(wl, device=DEV)
    ids = inp["topk_ids"].clone()
    ids[:, 0] = 2                     # every token's first slot goes to expert 2 (N_e = 200)
    ids[:, 1] = torch.where(ids[:, 1] == 2, torch.full_like(ids[:, 1], 3), ids[:, 1])
    ids[::3, 1] = -1                  # masked routes
    inp["topk_ids"] = ids.contiguous()
    out = run_forward(moe, wl, inp, stages=True)
    assert out["status"] == 0
    check_plan(out, wl, inp["topk_ids"])
    assert_close(y_numpy(out["y"]), oracle_forward(wl, inp), wl.mode)


def test_bad_route_is_reported_and_skipped(moe):
    wl = Workload("bad", "a16w16", 16, 256, 128, 4, 2, 37, 0.05)
    inp = make_inputs(wl, device=DEV)
    ids = inp["topk_ids"].clone()
    ids[3, 1] = 99
    inp["topk_ids"] = ids
    out = run_forward(moe, wl, inp)
    assert out["status"] == 4  # MOE_ERR_BAD_ROUTE
    ids_m = ids.clone()
    ids_m[3, 1] = -1              # the bad route is skipped like a masked one
    ref = oracle_forward(wl, dict(inp, topk_ids=ids_m))
    assert_close(y_numpy(out["y"]), ref, wl.mode)


@pytest.mark.parametrize("bad", [1.5 * 2.0 ** -6, 0.0, -0.25, float("inf"), 3.0])
def test_fp8_fp4_x_scale_that_is_not_a_power_of_two_is_reported(moe, bad):
    """The FP8 x FP4 tensor cores take an x scale's exponent byte as its UE8M0 scale, so the scale must be
    2^e (-127 <= e <= 127): the dispatch stage reads every scale and reports any other value in the error
    word, with no fault; 2^-127 (a subnormal fp32) and 2^127 are accepted."""
    wl = CASES["a8w4_fp8_fp4"][0]
    inp = make_inputs(wl, device=DEV)
    inp["x_scale"] = inp["x_scale"].clone()
    inp["x_scale"][3, 1] = bad
    assert run_forward(moe, wl, inp)["status"] == moe.MOE_ERR_BAD_SCALE
    inp["x_scale"][3, 1] = 2.0 ** -127
    inp["x_scale"][5, 0] = 2.0 ** 127
    assert run_forward(moe, wl, inp)["status"] == 0


def test_zero_tokens(moe):
    wl = Workload("empty", "a16w16", 0, 256, 128, 8, 2, 38, 0.05)
    inp = make_inputs(wl, device=DEV)
    out = run_forward(moe, wl, inp, stages=True)
    assert out["status"] == 0
    assert out["counts"].cpu().numpy().tolist() == [0] * 8
    assert out["offsets"].cpu().numpy().tolist() == [0] * 9


def test_bounded_wait_times_out_and_device_stays_usable(moe):
    ws = torch.zeros(1 << 16, dtype=torch.uint8, device=DEV)
    moe.moe_debug_bounded_wait(ws, 20_000_000)  # 20 ms on a flag that nothing sets
    assert moe.moe_check_device_error(ws) == 5  # MOE_ERR_TIMEOUT
    assert moe.moe_check_device_error(ws) == 0  # cleared
    wl = WORKLOADS["tiny_bf16"]
    inp = make_inputs(wl, device=DEV)
    out = run_forward(moe, wl, inp)
    assert out["status"] == 0
    assert_close(y_numpy(out["y"]), oracle_forward(wl, inp), wl.mode)


FULL = ["mixtral_bf16_prefill", "dsv3_fp8fp4_decode", "dsv3_fp8fp4_prefill_zipf", "int8_a8w8", "int4_a8w4"]


ORACLE_WORKERS = max(1, min(12, os.cpu_count() or 1))


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled(moe, name):
    """Full-size workload in the benchmark's launch configuration; the plan is checked in full and
    y on a sample of tokens chosen so that every expert any token routes to is computed for at least
    one sampled token (every token is an independent problem): an error confined to one expert's
    tiles shows."""
    wl = WORKLOADS[name]
    inp = make_inputs(wl, device=DEV)
    out = run_forward(moe, wl, inp, stages=True)
    assert out["status"] == 0
    check_plan(out, wl, inp["topk_ids"])
    h = to_numpy(inp)
    tokens = covering_tokens(h["topk_ids"], wl.seed)
    touched = set(h["topk_ids"].ravel().tolist()) - {-1}
    assert set(h["topk_ids"][tokens].ravel().tolist()) - {-1} == touched
    ref = oracle_tokens(wl.mode, h, tokens, wl.I, ORACLE_WORKERS)
    got = y_numpy(out["y"])[tokens]
    assert_close(got, ref, wl.mode)
    # every row of the output is written and finite
    assert torch.isfinite(out["y"].float()).all()


@pytest.mark.parametrize("wl", CASES["a16w16"], ids=[w.name for w in CASES["a16w16"]])
def test_tensor_core_stages_match_reference_kernels(moe, wl):
    """The tcgen05 L1 (A pool) and L2 (combine rows) agree with the CUDA-core reference kernels
    on the same plan: equal up to one bf16 rounding step from the fp32 summation order."""
    inp = make_inputs(wl, device=DEV)
    outs = [run_forward(moe, wl, inp, flags=f, stages=True) for f in (0, 1)]
    L = outs[0]["layout"]
    rows = L["pool_rows"]
    hdr = region(outs[0]["ws"], L, "header", torch.int32, 16).cpu().numpy()
    n_pad = int(hdr[2])
    pool_src = region(outs[0]["ws"], L, "pool_src", torch.int32, rows)[:n_pad]
    valid = (pool_src >= 0).cpu().numpy()
    # both runs use the same plan only up to the order of rows inside an expert: compare the
    # A rows by their (token, slot) identity
    a = []
    for o in outs:
        ps = region(o["ws"], L, "pool_src", torch.int32, rows)[:n_pad].cpu().numpy()
        ap = region(o["ws"], L, "a_pool", torch.bfloat16, rows * wl.I).view(rows, wl.I)[:n_pad]
        order = np.argsort(np.where(ps >= 0, ps, 1 << 30), kind="stable")[:valid.sum()]
        a.append(ap.float().cpu().numpy()[order])
    diff = np.abs(a[0] - a[1])
    scale = np.abs(a[1]).max()
    assert diff.max() <= 2 ** -7 * scale, f"A pool: max diff {diff.max():.3e} vs scale {scale:.3e}"
    c = [region(o["ws"], L, "comb", torch.bfloat16, wl.T * wl.K * wl.H).float().cpu().numpy() for o in outs]
    assert np.abs(c[0] - c[1]).max() <= 2e-2 * np.abs(c[1]).max()


@pytest.mark.parametrize("prepared", [False, True], ids=["int8_weights", "prepared_weights"])
def test_int8_l1_accumulators_exact_on_adversarial_codes(moe, prepared):
    """Every x and W1 code is +-127 and K = 5120, so the int32 accumulators reach 5120*127^2
    = 82,580,480 > 2^24: a plain fp32 accumulation would round, the exact integer GEMM must
    not. With unit scales H = C exactly and SiLU(H) is H or 0, so the fp32 A of the kernel must
    equal the oracle's bit for bit (int8 weights, or the f16 codes of moe_prepare_weights)."""
    wl = Workload("adv_int8", "a8w8_int8", 96, 5120, 256, 2, 1, 51, 0.05)
    inp = make_inputs(wl, device=DEV)
    g = torch.Generator(device=DEV).manual_seed(5)
    sign = lambda shape: (torch.randint(0, 2, shape, generator=g, device=DEV) * 2 - 1).to(torch.int8) * 127
    inp["x"] = sign(inp["x"].shape)
    inp["x"][:3] = 127                  # rows whose gate and up sums are exactly +-82,580,480
    inp["x_scale"] = torch.ones_like(inp["x_scale"])
    inp["w1"] = sign(inp["w1"].shape)
    inp["w1"][0, :3] = 127
    inp["w1"][0, wl.I:wl.I + 3] = 127
    inp["w1_scale"] = torch.ones_like(inp["w1_scale"])
    inp["topk_ids"][:3] = 0
    out = (run_prepared(moe, wl, inp) if prepared else run_forward(moe, wl, inp, stages=True))
    assert out["status"] == 0
    L = out["layout"]
    rows = L["pool_rows"]
    ws = out["ws"]
    n_pad = int(region(ws, L, "header", torch.int32, 16).cpu().numpy()[2])
    pool_src = region(ws, L, "pool_src", torch.int32, rows).cpu().numpy()[:n_pad]
    a_f32 = region(ws, L, "a_f32", torch.float32, rows * wl.I).view(rows, wl.I).cpu().numpy()
    _, rec = oracle_forward(wl, inp, return_intermediates=True)
    for e, r in rec["experts"].items():
        h = r["h"]
        assert np.abs(r["c"]).max() > 2 ** 24 or e != 0
        a_ref = (omoe.swiglu(h, wl.I)).astype(np.float32)
        got_rows = {int(s): i for i, s in enumerate(pool_src) if s >= 0}
        got = np.stack([a_f32[got_rows[int(s)]] for s in r["src"]])
        # |H| >= 32258 whenever it is non-zero, so SiLU(H) = H exactly for H > 0 on both sides;
        # for H <= 0 SiLU(H) * H_up is 0 up to an fp32/float64 underflow difference
        pos = h[:, :wl.I] > 0
        assert np.array_equal(got[pos], a_ref[pos]), f"expert {e}: {np.abs(got - a_ref)[pos].max()}"
        assert np.abs(got[~pos]).max(initial=0) < 1e-20 and np.abs(a_ref[~pos]).max(initial=0) < 1e-20


def run_prepared(moe, wl, inp, **kw):
    """run_forward with the A8W8-INT weights prepared once as exact f16 codes (moe_prepare_weights)
    and MOE_FLAG_PREPARED_WEIGHTS."""
    d = moe.dims(wl.T, wl.H, wl.I, wl.E, wl.K)
    w1p = moe.moe_prepare_weights(inp["w1"], d, wl.mode, 1)
    w2p = moe.moe_prepare_weights(inp["w2"], d, wl.mode, 2)
    assert torch.equal(w1p.float(), inp["w1"].float()) and torch.equal(w2p.float(), inp["w2"].float())
    return run_forward(moe, wl, dict(inp, w1=w1p, w2=w2p), flags=moe.MOE_FLAG_PREPARED_WEIGHTS, stages=True, **kw)


@pytest.mark.parametrize("case", ["tiny", "ragged", "tail_sizes", "full_size"])
def test_int8_prepared_weights_equal_int8_weights(moe, case):
    """The INT8 GEMMs on weights prepared once as exact f16 codes give the same combine rows and y,
    bit for bit, as on the int8 weights (both accumulate the exact integer products); the tail case
    puts experts at the 16-token and 128-row edges of the tiles."""
    if case == "tail_sizes":
        wl, inp = _tail_inputs("a8w8_int8", 48)
    else:
        wl = {"tiny": CASES["a8w8_int8"][0], "ragged": CASES["a8w8_int8"][1], "full_size": WORKLOADS["int8_a8w8"]}[case]
        inp = make_inputs(wl, device=DEV)
    a = run_forward(moe, wl, inp, stages=True)
    b = run_prepared(moe, wl, inp)
    assert a["status"] == 0 and b["status"] == 0
    L = a["layout"]
    ca = region(a["ws"], L, "comb", torch.int16, wl.T * wl.K * wl.H)
    cb = region(b["ws"], L, "comb", torch.int16, wl.T * wl.K * wl.H)
    assert torch.equal(ca, cb)
    assert torch.equal(a["y"].view(torch.int16), b["y"].view(torch.int16))
    if case != "full_size":
        assert_close(y_numpy(b["y"]), oracle_forward(wl, inp), wl.mode)


def test_prepared_weights_rejections(moe):
    wl = CASES["a16w16"][0]
    inp = make_inputs(wl, device=DEV)
    d = moe.dims(wl.T, wl.H, wl.I, wl.E, wl.K)
    with pytest.raises(moe.MoeError) as err:
        moe.moe_prepare_weights(inp["w1"], d, wl.mode, 1)
    assert err.value.status == moe.MOE_ERR_UNSUPPORTED
    with pytest.raises(moe.MoeError) as err:  # the flag belongs to the A8W8-INT GEMMs only
        run_forward(moe, wl, inp, flags=moe.MOE_FLAG_PREPARED_WEIGHTS)
    assert err.value.status == moe.MOE_ERR_UNSUPPORTED
    wl8 = CASES["a8w8_int8"][0]
    inp8 = make_inputs(wl8, device=DEV)
    with pytest.raises(moe.MoeError) as err:  # no CUDA-core kernel takes prepared weights
        run_forward(moe, wl8, inp8, flags=moe.MOE_FLAG_PREPARED_WEIGHTS | moe.MOE_FLAG_SIMT)
    assert err.value.status == moe.MOE_ERR_UNSUPPORTED


def test_int4_l1_accumulators_exact_at_the_largest_k(moe):
    """A8W4-INT at K = 8704, the largest hidden size of its tensor-core path: x codes +-127,
    int4 weights +-4, and for expert 0 gate channels of all 7 and up channels of all -8 against
    rows of all 127. The kernel accumulates (w + 8) * q, which reaches 15 * 127 * 8704 =
    16,581,120 (between 2^23 and 2^24) on those gate channels. Every sum is a multiple of 1016 (an
    even count of odd multiples of 508) or of 1778, so SiLU(H) = H exactly for H > 0 and the fp32
    A must equal the oracle's bit for bit there."""
    wl = Workload("adv_w4", "a8w4_int", 96, 8704, 256, 2, 1, 52, 0.05)
    inp = make_inputs(wl, device=DEV)
    g = torch.Generator(device=DEV).manual_seed(6)
    sign = lambda shape: torch.randint(0, 2, shape, generator=g, device=DEV) * 2 - 1
    x = (sign(inp["x"].shape) * 127).to(torch.int8)
    x[:3] = 127
    w1 = sign((wl.E, 2 * wl.I, wl.H)) * 4
    w1[0, :3] = 7
    w1[0, wl.I:wl.I + 3] = -8
    nib = (w1 & 0xF).to(torch.uint8)
    inp["x"], inp["x_scale"] = x, torch.ones_like(inp["x_scale"])
    inp["w1"] = (nib[..., 0::2] | (nib[..., 1::2] << 4)).contiguous()
    inp["w1_scale"] = torch.ones_like(inp["w1_scale"])
    inp["topk_ids"][:3] = 0
    out = run_forward(moe, wl, inp, stages=True)
    assert out["status"] == 0
    L = out["layout"]
    rows = L["pool_rows"]
    ws = out["ws"]
    n_pad = int(region(ws, L, "header", torch.int32, 16).cpu().numpy()[2])
    pool_src = region(ws, L, "pool_src", torch.int32, rows).cpu().numpy()[:n_pad]
    a_f32 = region(ws, L, "a_f32", torch.float32, rows * wl.I).view(rows, wl.I).cpu().numpy()
    _, rec = oracle_forward(wl, inp, return_intermediates=True)
    got_rows = {int(s): i for i, s in enumerate(pool_src) if s >= 0}
    for e, r in rec["experts"].items():
        h = r["h"]
        if e == 0:
            assert np.abs(r["c"]).max() > 2 ** 22
        a_ref = (omoe.swiglu(h, wl.I)).astype(np.float32)
        got = np.stack([a_f32[got_rows[int(s)]] for s in r["src"]])
        pos = h[:, :wl.I] > 0
        assert np.array_equal(got[pos], a_ref[pos]), f"expert {e}: {np.abs(got - a_ref)[pos].max()}"
        assert np.abs(got[~pos]).max(initial=0) < 1e-20 and np.abs(a_ref[~pos]).max(initial=0) < 1e-20


@pytest.mark.parametrize("mode,wl", [(m, w) for m, w in ALL if m != "a16w16"],
                         ids=[f"{m}-{w.name}" for m, w in ALL if m != "a16w16"])
def test_quantised_tensor_core_path_matches_reference_kernels(moe, mode, wl):
    """The weight-major tcgen05 path and the CUDA-core reference kernels give the same weighted
    combine rows up to the fp32 summation order."""
    inp = make_inputs(wl, device=DEV)
    outs = [run_forward(moe, wl, inp, flags=f, stages=True) for f in (0, 1)]
    L = outs[0]["layout"]
    c = [region(o["ws"], L, "comb", torch.bfloat16, wl.T * wl.K * wl.H).float().cpu().numpy() for o in outs]
    assert np.abs(c[0] - c[1]).max() <= TOL[mode] * np.abs(c[1]).max()


FP8_PREFILL = [(m, w) for m, w in ALL if m in ("a8w8_fp8", "a8w4_fp8_fp4", "a8w8_fp8_e5m2") and w.T * w.K > 16 * w.E]


@pytest.mark.parametrize("mode,wl", FP8_PREFILL, ids=[f"{m}-{w.name}" for m, w in FP8_PREFILL])
def test_block_scaled_tile_choices_agree(moe, mode, wl):
    """At prefill sizes the FP8 modes run 128-token x 256-weight-row tiles; MOE_FLAG_PAIR_L1 selects
    weight-major tiles on CTA pairs (256 weight rows x up to 192 tokens) where the shape allows and
    MOE_FLAG_WEIGHT_MAJOR one-CTA 128-weight-row x 128-token tiles. All compute the same block-scaled
    products, so the combine rows and the output agree up to the fp32 summation order (within the
    mode's tolerance), and the oracle bounds each."""
    inp = make_inputs(wl, device=DEV)
    flags = (0, moe.MOE_FLAG_PAIR_L1, moe.MOE_FLAG_WEIGHT_MAJOR)
    outs = [run_forward(moe, wl, inp, flags=f, stages=True) for f in flags]
    assert all(o["status"] == 0 for o in outs)
    L = outs[0]["layout"]
    c = [region(o["ws"], L, "comb", torch.bfloat16, wl.T * wl.K * wl.H).float().cpu().numpy() for o in outs]
    for other in c[1:]:
        assert np.abs(c[0] - other).max() <= TOL[mode] * np.abs(other).max()
    ref = oracle_forward(wl, inp)
    for o in outs:
        assert_close(y_numpy(o["y"]), ref, mode)


# Per-expert token counts at the edges of the pair tiles' granularities: 16-token MMA columns, 16-row
# token boxes of a partial tile, the 96 rows a CTA stages, the 192 tokens of a full tile.
PAIR_COUNTS = [1, 15, 16, 17, 95, 96, 97, 191, 192, 193, 383, 449]


@pytest.mark.parametrize("mode", ["a8w4_fp8_fp4", "a8w8_fp8", "a8w8_fp8_e5m2"])
def test_pair_tiles_at_token_count_edges(moe, mode):
    """The CTA-pair weight-major kernel (MOE_FLAG_PAIR_L1; both GEMMs: H 512, I 512) against the oracle
    and against the token-major tiles with experts of 1 to 449 routed tokens."""
    wl = Workload(f"pair_edges_{mode}", mode, sum(PAIR_COUNTS), 512, 512, len(PAIR_COUNTS), 1, 77, 0.05)
    inp = make_inputs(wl, device=DEV)
    inp["topk_ids"] = torch.repeat_interleave(torch.arange(wl.E, dtype=torch.int32),
                                              torch.tensor(PAIR_COUNTS))[:, None].to(DEV).contiguous()
    a = run_forward(moe, wl, inp, flags=moe.MOE_FLAG_PAIR_L1, stages=True)
    b = run_forward(moe, wl, inp, stages=True)
    assert a["status"] == 0 and b["status"] == 0
    check_plan(a, wl, inp["topk_ids"])
    ref, rec = oracle_forward(wl, inp, return_intermediates=True)
    L = a["layout"]
    comb = region(a["ws"], L, "comb", torch.bfloat16, wl.T * wl.K * wl.H).view(wl.T * wl.K, wl.H)
    assert_close(y_numpy(comb), rec["comb"], mode, "combine rows")
    assert_close(y_numpy(a["y"]), ref, mode)
    assert_close(y_numpy(b["y"]), ref, mode)


W4_ORDER = np.array([0, 4, 1, 5, 2, 6, 3, 7])


def _check_w4_operands(ws, L, planes, sums_half, R, n, rows, codes):
    """A8W4-INT operand rows: plane position 8g + p holds code 8g + W4_ORDER[p] as f16, and the
    row's code sum is stored beside (x rows in the first half of the sums region, A rows in the
    second)."""
    plane = region(ws, L, planes, torch.float16, R * n).view(R, n).float().cpu().numpy()[rows]
    perm = (np.arange(n) // 8) * 8 + W4_ORDER[np.arange(n) % 8]
    assert np.array_equal(plane, codes[:, perm].astype(np.float64)), "plane"
    sums = region(ws, L, "pool_sums", torch.int32, 2 * R).view(2, R).cpu().numpy()[sums_half, rows]
    assert np.array_equal(sums, codes.sum(axis=1)), "code sums"


XQ_CASES = [(m, w) for m, w in ALL if m != "a16w16" and w.name in ("tiny_fp8", "ragged_fp8", "tiny_int8", "ragged_int8",
                                                                    "tiny_w4", "ragged_w4", "tiny_e5m2", "ragged_e5m2",
                                                                    "tiny_fp4", "skew_fp4", "n224_fp4", "n224_fp8")]


def _special_rows(x_bf16):
    """Rows that reach the corners of the quantisers: all zero, tiny, huge, one spike."""
    x = x_bf16.clone()
    x[0] = 0.0
    if x.shape[0] > 3:
        x[1] = x[1] * 1e-30
        x[2] = x[2] * 1e30
        x[3] = 0.0
        x[3, 5] = -3.0
    return x.contiguous()


@pytest.mark.parametrize("mode,wl", XQ_CASES, ids=[f"{m}-{w.name}" for m, w in XQ_CASES])
def test_dispatch_quantize_matches_oracle_bit_exactly(moe, mode, wl):
    """S2 from bf16 x: every routed pool row holds the oracle's quantisation of its token (codes
    and scales bit-exact: both sides decide in fp32), and the INT8 planes hold its hi/lo split."""
    inp = make_inputs(wl, device=DEV)
    xb = _special_rows(inp["x_bf16"])
    d = moe.dims(wl.T, wl.H, wl.I, wl.E, wl.K)
    ws = moe.alloc_workspace(d, wl.mode, DEV)
    moe.moe_plan(inp["topk_ids"], d, ws)
    moe.moe_dispatch_quantize(xb, d, wl.mode, ws)
    assert moe.moe_check_device_error(ws) == 0
    L = moe.moe_workspace_layout(d, wl.mode)
    R = L["pool_rows"]
    pool_src = region(ws, L, "pool_src", torch.int32, R).cpu().numpy()
    rows = np.nonzero(pool_src >= 0)[0]
    tok = pool_src[rows] // wl.K
    qx, sx = omoe.quantize_x(mode, to_numpy({"x": xb})["x"])
    codes = region(ws, L, "x_pool", torch.uint8, R * wl.H).view(R, wl.H).cpu().numpy()[rows]
    assert np.array_equal(codes, qx.view(np.uint8)[tok]), "codes"
    if mode in ("a8w8_fp8", "a8w8_fp8_e5m2"):
        sc = region(ws, L, "x_pool_scale", torch.uint8, R * (wl.H // 32)).view(R, -1).cpu().numpy()[rows]
        assert np.array_equal(sc, sx[tok])
    else:
        n = wl.H // 128 if mode == "a8w4_fp8_fp4" else 1
        sc = region(ws, L, "x_pool_scale", torch.float32, R * n).view(R, n).cpu().numpy()[rows]
        assert np.array_equal(sc.reshape(len(rows), -1), np.asarray(sx, np.float32)[tok].reshape(len(rows), -1))
    if mode == "a8w8_int8":
        planes = region(ws, L, "x_pool_planes", torch.float16, 2 * R * wl.H).view(2, R, wl.H).float().cpu().numpy()
        q = qx.astype(np.int64)[tok]
        assert np.array_equal(planes[0, rows], np.floor_divide(q, 16)) and np.array_equal(planes[1, rows], q % 16)
    if mode == "a8w4_int":  # one plane: the codes themselves, in the expansion's order, and their sums
        _check_w4_operands(ws, L, "x_pool_planes", 0, R, wl.H, rows, qx.astype(np.int64)[tok])


@pytest.mark.parametrize("mode,wl", XQ_CASES, ids=[f"{m}-{w.name}" for m, w in XQ_CASES])
def test_forward_quantizing_x_matches_oracle(moe, mode, wl):
    """moe_forward with MOE_FLAG_QUANTIZE_X on bf16 x equals the oracle on its own quantisation of x."""
    inp = make_inputs(wl, device=DEV)
    d = moe.dims(wl.T, wl.H, wl.I, wl.E, wl.K)
    ws = moe.alloc_workspace(d, wl.mode, DEV)
    y = torch.full((wl.T, wl.H), float("nan"), dtype=torch.bfloat16, device=DEV)
    moe.moe_forward(inp["x_bf16"], None, inp["topk_ids"], inp["topk_weights"], inp["w1"], inp["w1_scale"], inp["w2"],
                    inp["w2_scale"], y, d, wl.mode, ws, moe.MOE_FLAG_QUANTIZE_X)
    assert moe.moe_check_device_error(ws) == 0
    h = to_numpy(inp)
    qx, sx = omoe.quantize_x(mode, h["x_bf16"])
    ref = omoe.forward(mode, qx, sx, h["topk_ids"], h["topk_weights"], h["w1"], h["w1_scale"], h["w2"], h["w2_scale"],
                       num_experts=wl.E, inter=wl.I)
    assert_close(y_numpy(y), ref, mode)


@pytest.mark.parametrize("name", ["dsv3_fp8fp4_prefill_zipf", "int8_a8w8", "dsv3_fp8fp4_decode", "int4_a8w4"])
def test_full_size_quantizing_x_sampled(moe, name):
    """Full-size workload from bf16 x (the dispatch stage quantises it, as the bench's --quantize-x
    times it): on a sample of tokens that covers every routed expert, the pool codes are bit-exact
    against the oracle's quantisation and the outputs match the oracle within the mode's bound."""
    wl = WORKLOADS[name]
    inp = make_inputs(wl, device=DEV)
    d = moe.dims(wl.T, wl.H, wl.I, wl.E, wl.K)
    ws = moe.alloc_workspace(d, wl.mode, DEV)
    y = torch.full((wl.T, wl.H), float("nan"), dtype=torch.bfloat16, device=DEV)
    moe.moe_forward(inp["x_bf16"], None, inp["topk_ids"], inp["topk_weights"], inp["w1"], inp["w1_scale"], inp["w2"],
                    inp["w2_scale"], y, d, wl.mode, ws, moe.MOE_FLAG_QUANTIZE_X)
    assert moe.moe_check_device_error(ws) == 0
    h = to_numpy({k: inp[k] for k in ("x_bf16", "topk_ids", "topk_weights", "w1", "w1_scale", "w2", "w2_scale")})
    tokens = covering_tokens(h["topk_ids"], wl.seed + 100)
    qx, sx = omoe.quantize_x(wl.mode, h["x_bf16"][tokens])
    # the pool rows of the sampled tokens hold their codes
    L = moe.moe_workspace_layout(d, wl.mode)
    slot_row = region(ws, L, "slot_row", torch.int32, wl.T * wl.K).view(wl.T, wl.K)
    codes = region(ws, L, "x_pool", torch.uint8, L["pool_rows"] * wl.H).view(L["pool_rows"], wl.H)
    rows = slot_row[torch.as_tensor(tokens, device=DEV)].long()
    got_codes = codes[rows.reshape(-1)].view(len(tokens), wl.K, wl.H).cpu().numpy()
    for j, t in enumerate(tokens):
        for k in range(wl.K):
            assert np.array_equal(got_codes[j, k], qx.view(np.uint8)[j]), (t, k)
    sub = {"x": qx, "x_scale": sx, "topk_ids": h["topk_ids"][tokens], "topk_weights": h["topk_weights"][tokens],
           **{k: h[k] for k in ("w1", "w1_scale", "w2", "w2_scale")}}
    ref = oracle_tokens(wl.mode, sub, range(len(tokens)), wl.I, ORACLE_WORKERS)
    assert_close(y_numpy(y)[tokens], ref, wl.mode)
    assert torch.isfinite(y.float()).all()


CLAMP_CASES = [(m, w) for m, w in ALL if w.name in ("tiny_bf16", "ragged_bf16", "ragged_fp8", "ragged_int8", "ragged_fp4",
                                                     "skew_fp4", "n224_fp4", "ragged_w4", "ragged_e5m2")]


@pytest.mark.parametrize("mode,wl", CLAMP_CASES, ids=[f"{m}-{w.name}" for m, w in CLAMP_CASES])
@pytest.mark.parametrize("flags", [0, 1, 2], ids=["default", "simt", "weight_major"])
def test_activation_clamp_matches_oracle(moe, mode, wl, flags):
    """moe_forward_ex with activation_clamp: every L1 kernel clips both SwiGLU inputs; the clamp,
    set near the median |H| (an fp32 value), changes the output and the oracle bounds it."""
    inp = make_inputs(wl, device=DEV)
    h = to_numpy(inp)
    _, rec = omoe.forward(mode, h["x"], h["x_scale"], h["topk_ids"], h["topk_weights"], h["w1"], h["w1_scale"],
                          h["w2"], h["w2_scale"], num_experts=wl.E, inter=wl.I, return_intermediates=True)
    hs = np.concatenate([np.abs(r["h"]).ravel() for r in rec["experts"].values()])
    c = float(np.float32(np.median(hs)))
    d = moe.dims(wl.T, wl.H, wl.I, wl.E, wl.K)
    ws = moe.alloc_workspace(d, wl.mode, DEV)
    y = torch.full((wl.T, wl.H), float("nan"), dtype=torch.bfloat16, device=DEV)
    moe.moe_forward_ex(inp["x"], inp["x_scale"], inp["topk_ids"], inp["topk_weights"], inp["w1"], inp["w1_scale"],
                       inp["w2"], inp["w2_scale"], y, d, wl.mode, ws, flags=flags, activation_clamp=c)
    assert moe.moe_check_device_error(ws) == 0
    ref = omoe.forward(mode, h["x"], h["x_scale"], h["topk_ids"], h["topk_weights"], h["w1"], h["w1_scale"], h["w2"],
                       h["w2_scale"], num_experts=wl.E, inter=wl.I, clamp=c)
    assert_close(y_numpy(y), ref, mode)
    unclamped = oracle_forward(wl, inp)
    assert np.abs(ref - unclamped).max() > 10 * TOL[mode] * np.abs(unclamped).max()


def test_activation_clamp_rejects_bad_values(moe):
    wl = WORKLOADS["tiny_bf16"]
    inp = make_inputs(wl, device=DEV)
    d = moe.dims(wl.T, wl.H, wl.I, wl.E, wl.K)
    ws = moe.alloc_workspace(d, wl.mode, DEV)
    y = torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device=DEV)
    for bad in (-1.0, float("nan")):
        with pytest.raises(moe.MoeError):
            moe.moe_forward_ex(inp["x"], None, inp["topk_ids"], inp["topk_weights"], inp["w1"], None, inp["w2"], None,
                               y, d, wl.mode, ws, activation_clamp=bad)
    # no clamp through the options path is the plain forward, bit for bit
    y0 = torch.empty_like(y)
    moe.moe_forward(inp["x"], None, inp["topk_ids"], inp["topk_weights"], inp["w1"], None, inp["w2"], None, y0, d,
                    wl.mode, ws)
    moe.moe_forward_ex(inp["x"], None, inp["topk_ids"], inp["topk_weights"], inp["w1"], None, inp["w2"], None, y, d,
                       wl.mode, ws)
    assert torch.equal(y.view(torch.int16), y0.view(torch.int16))


# ---------------------------------------------------------------------------------------
# Shared experts (DeepGEMM page §6): every token, weight 1, the slot after the routed ones
# ---------------------------------------------------------------------------------------

SHARED_CASES = [(m, w) for m, w in ALL if w.name in ("tiny_bf16", "ragged_bf16", "ragged_fp8", "ragged_int8",
                                                      "ragged_w4", "ragged_fp4", "skew_fp4", "n224_fp8", "ragged_e5m2")]


@pytest.mark.parametrize("mode,wl", SHARED_CASES, ids=[f"{m}-{w.name}" for m, w in SHARED_CASES])
@pytest.mark.parametrize("shared", [1, 2])
@pytest.mark.parametrize("flags", [0, 1], ids=["default", "simt"])
def test_shared_experts_match_oracle(moe, mode, wl, shared, flags):
    inp = make_inputs(wl, device=DEV, shared=shared)
    out = run_forward(moe, wl, inp, flags=flags, stages=True, shared=shared)
    assert out["status"] == 0
    h = to_numpy(inp)
    ids_ext, _ = omoe.with_shared_slots(h["topk_ids"], h["topk_weights"], wl.E, shared)
    counts, offsets, row_src = omoe.plan(ids_ext, wl.E + shared)
    assert out["counts"].cpu().numpy().tolist() == counts.tolist()
    assert counts[wl.E:].tolist() == [wl.T] * shared
    assert out["offsets"].cpu().numpy().tolist() == offsets.tolist()
    got = out["row_src"].cpu().numpy()
    assert sorted(got.tolist()) == sorted(row_src.tolist())
    ref = omoe.forward(mode, h["x"], h["x_scale"], h["topk_ids"], h["topk_weights"], h["w1"], h["w1_scale"],
                       h["w2"], h["w2_scale"], num_experts=wl.E, inter=wl.I, num_shared=shared)
    assert_close(y_numpy(out["y"]), ref, mode)


def test_shared_experts_with_masked_routes_and_quantizing_dispatch(moe):
    """Every routed slot of half the tokens masked: those tokens get the shared experts alone;
    the quantising dispatch (row f1) feeds the shared experts' pool rows too."""
    wl = CASES["a8w8_int8"][1]
    inp = make_inputs(wl, device=DEV, shared=1)
    inp["topk_ids"][: wl.T // 2] = -1
    d = moe.dims(wl.T, wl.H, wl.I, wl.E, wl.K, 1)
    ws = moe.alloc_workspace(d, wl.mode, DEV)
    y = torch.full((wl.T, wl.H), float("nan"), dtype=torch.bfloat16, device=DEV)
    moe.moe_forward(inp["x_bf16"], None, inp["topk_ids"], inp["topk_weights"], inp["w1"], inp["w1_scale"], inp["w2"],
                    inp["w2_scale"], y, d, wl.mode, ws, moe.MOE_FLAG_QUANTIZE_X)
    assert moe.moe_check_device_error(ws) == 0
    h = to_numpy(inp)
    qx, sx = omoe.quantize_x(wl.mode, h["x_bf16"])
    ref = omoe.forward(wl.mode, qx, sx, h["topk_ids"], h["topk_weights"], h["w1"], h["w1_scale"], h["w2"],
                       h["w2_scale"], num_experts=wl.E, inter=wl.I, num_shared=1)
    assert_close(y_numpy(y), ref, wl.mode)


def test_routed_id_naming_a_shared_expert_is_a_bad_route(moe):
    wl = CASES["a16w16"][0]
    inp = make_inputs(wl, device=DEV, shared=1)
    inp["topk_ids"][0, 0] = wl.E  # the shared expert's index: not a routed expert
    out = run_forward(moe, wl, inp, shared=1)
    assert out["status"] == 4  # MOE_ERR_BAD_ROUTE
    ids = inp["topk_ids"].clone()
    ids[0, 0] = -1  # the kernel skipped the bad route: same as a masked one
    h = to_numpy(dict(inp, topk_ids=ids))
    ref = omoe.forward(wl.mode, h["x"], h["x_scale"], h["topk_ids"], h["topk_weights"], h["w1"], h["w1_scale"],
                       h["w2"], h["w2_scale"], num_experts=wl.E, inter=wl.I, num_shared=1)
    assert_close(y_numpy(out["y"]), ref, wl.mode)


# ---------------------------------------------------------------------------------------
# L1 and L2 in one launch (MOE_FLAG_FUSED, §8(f) row f3): the same tiles and arithmetic as the
# separate stages, so the output is bit-identical to them
# ---------------------------------------------------------------------------------------

# (shapes with tensor-core tiles for both stages: H a multiple of 256)
FUSED_CASES = CASES["a16w16"] + [w for w in EDGE if w.mode == "a16w16" and w.H % 256 == 0] + [
    Workload("fused_one_expert_all_rows", "a16w16", 700, 512, 384, 3, 1, 42, 0.05),
    Workload("fused_many_tiles", "a16w16", 1500, 1024, 1024, 8, 2, 43, 0.03)]


def _forward_flags(moe, wl, inp, flags, shared=0, clamp=None, x=None):
    d = moe.dims(wl.T, wl.H, wl.I, wl.E, wl.K, shared)
    ws = moe.alloc_workspace(d, wl.mode, DEV)
    y = torch.full((wl.T, wl.H), float("nan"), dtype=torch.bfloat16, device=DEV)
    moe.moe_forward_ex(inp["x"] if x is None else x, inp["x_scale"], inp["topk_ids"], inp["topk_weights"], inp["w1"],
                       inp["w1_scale"], inp["w2"], inp["w2_scale"], y, d, wl.mode, ws, flags, clamp)
    return y, moe.moe_check_device_error(ws)


@pytest.mark.parametrize("wl", FUSED_CASES, ids=[w.name for w in FUSED_CASES])
def test_fused_l1_l2_equals_the_separate_stages(moe, wl):
    inp = make_inputs(wl, device=DEV)
    if wl.name == "fused_one_expert_all_rows":
        inp["topk_ids"][:] = 1                  # 700 rows on one expert: 6 route tiles, the last ragged
        inp["topk_ids"][::7] = -1               # and some masked routes
    y0, st0 = _forward_flags(moe, wl, inp, moe.MOE_FLAG_SINGLE_CTA)
    y1, st1 = _forward_flags(moe, wl, inp, moe.MOE_FLAG_FUSED)
    assert st0 == 0 and st1 == 0
    assert torch.equal(y0.view(torch.int16), y1.view(torch.int16))
    assert_close(y_numpy(y1), oracle_forward(wl, inp), wl.mode)


def test_fused_launch_without_y_leaves_the_combine_rows(moe):
    """moe_expert_ffn without y: L1 and L2 in one launch, the combine rows left in the workspace for
    moe_combine; with y the launch also combines. Both equal the separate stages bit for bit."""
    wl = FUSED_CASES[1]
    inp = make_inputs(wl, device=DEV)
    y_ref, st = _forward_flags(moe, wl, inp, moe.MOE_FLAG_SINGLE_CTA)
    assert st == 0
    d = moe.dims(wl.T, wl.H, wl.I, wl.E, wl.K)
    for with_y in (False, True):
        ws = moe.alloc_workspace(d, wl.mode, DEV)
        y = torch.full((wl.T, wl.H), float("nan"), dtype=torch.bfloat16, device=DEV)
        moe.moe_plan(inp["topk_ids"], d, ws)
        moe.moe_dispatch(inp["x"], inp["x_scale"], d, wl.mode, ws)
        moe.moe_expert_ffn(inp["w1"], inp["w1_scale"], inp["w2"], inp["w2_scale"], inp["topk_weights"], d, wl.mode, ws,
                           y=y if with_y else None)
        if not with_y:
            moe.moe_combine(y, d, ws)
        assert moe.moe_check_device_error(ws) == 0
        assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16)), with_y


def test_fused_full_size_equals_the_separate_stages(moe):
    wl = WORKLOADS["mixtral_bf16_prefill"]
    inp = make_inputs(wl, device=DEV)
    y0, st0 = _forward_flags(moe, wl, inp, moe.MOE_FLAG_SINGLE_CTA)
    y1, st1 = _forward_flags(moe, wl, inp, moe.MOE_FLAG_FUSED)
    assert st0 == 0 and st1 == 0
    assert torch.equal(y0.view(torch.int16), y1.view(torch.int16))
    rng = np.random.default_rng(wl.seed + 7)
    tokens = sorted(rng.choice(wl.T, size=4, replace=False).tolist())
    assert_close(y_numpy(y1)[tokens], oracle_forward(wl, slice_tokens(inp, tokens)), wl.mode)


def test_fused_with_clamp_shared_experts_and_quantizing_dispatch(moe):
    wl = CASES["a16w16"][1]
    inp = make_inputs(wl, device=DEV, shared=1)
    for flags in (0, moe.MOE_FLAG_QUANTIZE_X):
        x = inp["x_bf16"] if flags else None
        y0, st0 = _forward_flags(moe, wl, inp, flags | moe.MOE_FLAG_SINGLE_CTA, shared=1, clamp=0.5, x=x)
        y1, st1 = _forward_flags(moe, wl, inp, flags | moe.MOE_FLAG_FUSED, shared=1, clamp=0.5, x=x)
        assert st0 == 0 and st1 == 0
        assert torch.equal(y0.view(torch.int16), y1.view(torch.int16))
    h = to_numpy(inp)
    ref = omoe.forward(wl.mode, h["x"], h["x_scale"], h["topk_ids"], h["topk_weights"], h["w1"], h["w1_scale"],
                       h["w2"], h["w2_scale"], num_experts=wl.E, inter=wl.I, num_shared=1, clamp=0.5)
    assert_close(y_numpy(y1), ref, wl.mode)


# FP8 modes: L1 and L2 in one cooperative launch of the weight-major block-scaled kernel (the
# combine after it), so the output equals the separate stages on weight-major tiles bit for bit.
# Decode-shaped cases (at most 16 routed rows per expert on average) run 16-token sub-tiles, the
# others 128-token ones; several route tiles per expert, ragged last sub-tiles, masked routes and
# empty experts are all exercised.
FUSED_BS_CASES = [w for m in ("a8w8_fp8", "a8w8_fp8_e5m2", "a8w4_fp8_fp4") for w in CASES[m]] + [
    w for w in EDGE if w.mode in ("a8w8_fp8", "a8w4_fp8_fp4")] + [
    Workload("fused_bs_one_expert_all_rows", "a8w4_fp8_fp4", 700, 512, 384, 3, 1, 53, 0.05),
    Workload("fused_bs_decode_deep_expert", "a8w4_fp8_fp4", 200, 512, 512, 16, 1, 54, 0.05),
    Workload("fused_bs_decode_e4m3", "a8w8_fp8", 96, 1024, 256, 64, 8, 55, 0.05)]


def _fused_bs_ids(wl, inp):
    if wl.name == "fused_bs_one_expert_all_rows":
        inp["topk_ids"][:] = 1          # 700 rows on one expert: 6 route tiles, the last ragged
        inp["topk_ids"][::7] = -1       # and some masked routes
    elif wl.name == "fused_bs_decode_deep_expert":
        inp["topk_ids"][:150] = 0       # 150 rows on expert 0: route tiles of 128 and 22 rows
        inp["topk_ids"][150:] = torch.arange(50, device=inp["topk_ids"].device).view(50, 1) % 15 + 1
    return inp


@pytest.mark.parametrize("wl", FUSED_BS_CASES, ids=[w.name for w in FUSED_BS_CASES])
def test_fused_block_scaled_equals_the_separate_stages(moe, wl):
    inp = _fused_bs_ids(wl, make_inputs(wl, device=DEV))
    assert moe.MOE_FLAG_FUSED & moe.MOE_FLAG_WEIGHT_MAJOR == 0
    y0, st0 = _forward_flags(moe, wl, inp, moe.MOE_FLAG_WEIGHT_MAJOR)
    y1, st1 = _forward_flags(moe, wl, inp, moe.MOE_FLAG_FUSED)
    assert st0 == 0 and st1 == 0
    assert torch.equal(y0.view(torch.int16), y1.view(torch.int16))
    assert_close(y_numpy(y1), oracle_forward(wl, inp), wl.mode)


def test_fused_block_scaled_shared_experts_clamp_and_quantizing_dispatch(moe):
    wl = CASES["a8w4_fp8_fp4"][1]
    inp = make_inputs(wl, device=DEV, shared=1)
    for flags in (0, moe.MOE_FLAG_QUANTIZE_X):
        x = inp["x_bf16"] if flags else None
        y0, st0 = _forward_flags(moe, wl, inp, flags | moe.MOE_FLAG_WEIGHT_MAJOR, shared=1, clamp=0.5, x=x)
        y1, st1 = _forward_flags(moe, wl, inp, flags | moe.MOE_FLAG_FUSED, shared=1, clamp=0.5, x=x)
        assert st0 == 0 and st1 == 0
        assert torch.equal(y0.view(torch.int16), y1.view(torch.int16))
    h = to_numpy(inp)
    ref = omoe.forward(wl.mode, h["x"], h["x_scale"], h["topk_ids"], h["topk_weights"], h["w1"], h["w1_scale"],
                       h["w2"], h["w2_scale"], num_experts=wl.E, inter=wl.I, num_shared=1, clamp=0.5)
    assert_close(y_numpy(y1), ref, wl.mode)


def test_fused_block_scaled_without_y_leaves_the_combine_rows(moe):
    wl = CASES["a8w8_fp8"][1]
    inp = make_inputs(wl, device=DEV)
    y_ref, st = _forward_flags(moe, wl, inp, moe.MOE_FLAG_WEIGHT_MAJOR)
    assert st == 0
    d = moe.dims(wl.T, wl.H, wl.I, wl.E, wl.K)
    for with_y in (False, True):
        ws = moe.alloc_workspace(d, wl.mode, DEV)
        y = torch.full((wl.T, wl.H), float("nan"), dtype=torch.bfloat16, device=DEV)
        moe.moe_plan(inp["topk_ids"], d, ws)
        moe.moe_dispatch(inp["x"], inp["x_scale"], d, wl.mode, ws)
        moe.moe_expert_ffn(inp["w1"], inp["w1_scale"], inp["w2"], inp["w2_scale"], inp["topk_weights"], d, wl.mode, ws,
                           y=y if with_y else None)
        if not with_y:
            moe.moe_combine(y, d, ws)
        assert moe.moe_check_device_error(ws) == 0
        assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16)), with_y


@pytest.mark.parametrize("name", ["dsv3_fp8fp4_decode", "dsv3_fp8fp4_prefill_zipf"])
def test_fused_block_scaled_full_size_equals_the_separate_stages(moe, name):
    wl = WORKLOADS[name]
    inp = make_inputs(wl, device=DEV)
    y0, st0 = _forward_flags(moe, wl, inp, moe.MOE_FLAG_WEIGHT_MAJOR)
    y1, st1 = _forward_flags(moe, wl, inp, moe.MOE_FLAG_FUSED)
    assert st0 == 0 and st1 == 0
    assert torch.equal(y0.view(torch.int16), y1.view(torch.int16))


# Integer modes: L1, the per-row re-quantisation of A (by each route tile's last L1 tile) and L2
# in one cooperative launch of the weight-major kernels, the combine after it; bit-identical to the
# separate stages on weight-major tiles (A8W4-INT: MOE_FLAG_WEIGHT_MAJOR; A8W8-INT has no other).
# A8W4-INT tiles take up to two route tiles, so an expert with more than 128 rows exercises a tile
# that publishes and waits on two route-tile counters.
FUSED_INT_CASES = CASES["a8w8_int8"] + CASES["a8w4_int"] + [
    Workload("fused_int8_one_expert_all_rows", "a8w8_int8", 700, 512, 256, 3, 1, 56, 0.05),
    Workload("fused_w4_one_expert_all_rows", "a8w4_int", 700, 512, 256, 3, 1, 57, 0.05),
    Workload("fused_w4_many_experts", "a8w4_int", 300, 768, 384, 24, 4, 58, 0.05)]


@pytest.mark.parametrize("wl", FUSED_INT_CASES, ids=[w.name for w in FUSED_INT_CASES])
def test_fused_integer_equals_the_separate_stages(moe, wl):
    inp = make_inputs(wl, device=DEV)
    if wl.name.endswith("one_expert_all_rows"):
        inp["topk_ids"][:] = 1          # 700 rows on one expert: 6 route tiles, the last ragged
        inp["topk_ids"][::7] = -1       # and some masked routes
    y0, st0 = _forward_flags(moe, wl, inp, moe.MOE_FLAG_WEIGHT_MAJOR)
    y1, st1 = _forward_flags(moe, wl, inp, moe.MOE_FLAG_FUSED)
    assert st0 == 0 and st1 == 0
    assert torch.equal(y0.view(torch.int16), y1.view(torch.int16))
    assert_close(y_numpy(y1), oracle_forward(wl, inp), wl.mode)


def test_fused_integer_pools_equal_the_separate_stages(moe):
    """The fused launch leaves the same re-quantised A (codes and row scales of every routed slot's
    pool row) and the same combine rows in the workspace as the separate stages. The plan places an
    expert's rows in the order its claims land, which may differ between runs, so the pool rows are
    compared through each slot's row (slot_row)."""
    for wl in (CASES["a8w8_int8"][1], CASES["a8w4_int"][1], FUSED_INT_CASES[-1]):
        inp = make_inputs(wl, device=DEV)
        sep = run_forward(moe, wl, inp, flags=moe.MOE_FLAG_WEIGHT_MAJOR, stages=True)
        assert sep["status"] == 0
        d, L = sep["d"], sep["layout"]
        ws = moe.alloc_workspace(d, wl.mode, DEV)
        moe.moe_plan(inp["topk_ids"], d, ws)
        moe.moe_dispatch(inp["x"], inp["x_scale"], d, wl.mode, ws)
        moe.moe_expert_ffn(inp["w1"], inp["w1_scale"], inp["w2"], inp["w2_scale"], inp["topk_weights"], d, wl.mode, ws)
        assert moe.moe_check_device_error(ws) == 0
        rows, R = L["pool_rows"], wl.T * wl.K
        slot_f = region(ws, L, "slot_row", torch.int32, R).long()
        slot_s = region(sep["ws"], L, "slot_row", torch.int32, R).long()
        assert bool((slot_f >= 0).all()) and bool((slot_s >= 0).all())  # no masked routes in these cases
        for name, dtype, n in (("x_pool", torch.int8, wl.H), ("a_pool", torch.int8, wl.I),
                               ("a_pool_scale", torch.int32, 1)):
            got = region(ws, L, name, dtype, rows * n).view(rows, n)[slot_f]
            ref = region(sep["ws"], L, name, dtype, rows * n).view(rows, n)[slot_s]
            assert torch.equal(got, ref), (wl.name, name)
        assert torch.equal(region(ws, L, "comb", torch.int16, R * wl.H),
                           region(sep["ws"], L, "comb", torch.int16, R * wl.H)), wl.name


def test_fused_integer_shared_experts_clamp_quantizing_dispatch_and_prepared_weights(moe):
    for wl in (CASES["a8w8_int8"][1], CASES["a8w4_int"][1]):
        inp = make_inputs(wl, device=DEV, shared=1)
        for flags in (0, moe.MOE_FLAG_QUANTIZE_X):
            x = inp["x_bf16"] if flags else None
            y0, st0 = _forward_flags(moe, wl, inp, flags | moe.MOE_FLAG_WEIGHT_MAJOR, shared=1, clamp=0.5, x=x)
            y1, st1 = _forward_flags(moe, wl, inp, flags | moe.MOE_FLAG_FUSED, shared=1, clamp=0.5, x=x)
            assert st0 == 0 and st1 == 0
            assert torch.equal(y0.view(torch.int16), y1.view(torch.int16)), (wl.name, flags)
        h = to_numpy(inp)
        ref = omoe.forward(wl.mode, h["x"], h["x_scale"], h["topk_ids"], h["topk_weights"], h["w1"], h["w1_scale"],
                           h["w2"], h["w2_scale"], num_experts=wl.E, inter=wl.I, num_shared=1, clamp=0.5)
        assert_close(y_numpy(y1), ref, wl.mode)
    wl = CASES["a8w8_int8"][1]
    inp = make_inputs(wl, device=DEV)
    y0, st0 = _forward_flags(moe, wl, inp, 0)
    d = moe.dims(wl.T, wl.H, wl.I, wl.E, wl.K)
    prep = dict(inp, w1=moe.moe_prepare_weights(inp["w1"], d, wl.mode, 1),
                w2=moe.moe_prepare_weights(inp["w2"], d, wl.mode, 2))
    y1, st1 = _forward_flags(moe, wl, prep, moe.MOE_FLAG_FUSED | moe.MOE_FLAG_PREPARED_WEIGHTS)
    assert st0 == 0 and st1 == 0
    assert torch.equal(y0.view(torch.int16), y1.view(torch.int16))


@pytest.mark.parametrize("name", ["int8_a8w8", "int4_a8w4"])
def test_fused_integer_full_size_equals_the_separate_stages(moe, name):
    wl = WORKLOADS[name]
    inp = make_inputs(wl, device=DEV)
    y0, st0 = _forward_flags(moe, wl, inp, moe.MOE_FLAG_WEIGHT_MAJOR)
    y1, st1 = _forward_flags(moe, wl, inp, moe.MOE_FLAG_FUSED)
    assert st0 == 0 and st1 == 0
    assert torch.equal(y0.view(torch.int16), y1.view(torch.int16))


def test_fused_flag_rejections(moe):
    wl = Workload("fused_int8_h384", "a8w8_int8", 32, 384, 128, 4, 2, 59, 0.05)
    inp = make_inputs(wl, device=DEV)
    with pytest.raises(moe.MoeError) as err:
        _forward_flags(moe, wl, inp, moe.MOE_FLAG_FUSED)
    assert err.value.status == 2  # MOE_ERR_UNSUPPORTED: H = 384 has no 256-row L2 weight tile
    wl = CASES["a8w8_fp8"][0]
    inp = make_inputs(wl, device=DEV)
    with pytest.raises(moe.MoeError) as err:  # prepared weights are the INT8 mode's only
        _forward_flags(moe, wl, inp, moe.MOE_FLAG_FUSED | moe.MOE_FLAG_PREPARED_WEIGHTS)
    assert err.value.status == 2
    wl = EDGE[-1]  # max_topk: H = 128 has no 256-column L2 tile
    assert wl.name == "max_topk"
    with pytest.raises(moe.MoeError) as err:
        _forward_flags(moe, wl, make_inputs(wl, device=DEV), moe.MOE_FLAG_FUSED)
    assert err.value.status == 2
    wl = CASES["a16w16"][0]
    inp = make_inputs(wl, device=DEV)
    with pytest.raises(moe.MoeError) as err:
        _forward_flags(moe, wl, inp, moe.MOE_FLAG_FUSED | moe.MOE_FLAG_SIMT)
    assert err.value.status == 1  # MOE_ERR_INVALID_ARG


# ---------------------------------------------------------------------------------------
# bf16 GEMMs on CTA pairs (the default) against one-CTA tiles (MOE_FLAG_SINGLE_CTA): each
# output element is the same sequence of 16-K tensor-core products in the same order, so the
# two are compared bit for bit, and both against the oracle
# ---------------------------------------------------------------------------------------

def _pair_case_ids(wl, inp):
    ids = inp["topk_ids"]
    if wl.name == "pair_odd_tile_then_expert":
        # expert 0: 300 rows (three route tiles, so its last pair's odd half lies on expert 1's
        # first tile), expert 1: 130 rows, expert 2: 130 rows
        ids[:300] = 0
        ids[300:430] = 1
        ids[430:] = 2
    elif wl.name == "pair_odd_tile_last":
        ids[:130] = 0        # two route tiles, one pair
        ids[130:] = 1        # three route tiles: the last pair's odd half is past the pool's tiles
    elif wl.name == "pair_sparse":
        ids[:, 0] = 5        # two busy experts (three route tiles each), one with a single
        ids[:, 1] = 7        # tile whose pair's odd half lies on expert 5, the others empty
        ids[::5, 0] = 1
        ids[::11, 1] = -1    # masked routes
    return inp


PAIR_CASES = FUSED_CASES + [
    Workload("pair_odd_tile_then_expert", "a16w16", 560, 512, 384, 3, 1, 44, 0.05),
    Workload("pair_odd_tile_last", "a16w16", 430, 512, 384, 4, 1, 45, 0.05),
    Workload("pair_sparse", "a16w16", 333, 768, 256, 12, 2, 46, 0.05)]


@pytest.mark.parametrize("wl", PAIR_CASES, ids=[w.name for w in PAIR_CASES])
def test_pair_tiles_equal_single_cta_tiles(moe, wl):
    """Default (L2 on pairs) and MOE_FLAG_PAIR_L1 (both stages on pairs) against one-CTA tiles."""
    inp = _pair_case_ids(wl, make_inputs(wl, device=DEV))
    y0, st0 = _forward_flags(moe, wl, inp, moe.MOE_FLAG_SINGLE_CTA)
    assert st0 == 0
    for flags in (0, moe.MOE_FLAG_PAIR_L1):
        y1, st1 = _forward_flags(moe, wl, inp, flags)
        assert st1 == 0
        assert torch.equal(y0.view(torch.int16), y1.view(torch.int16)), flags
    assert_close(y_numpy(y1), oracle_forward(wl, inp), wl.mode)


def test_pair_tiles_full_size_equal_single_cta_tiles(moe):
    wl = WORKLOADS["mixtral_bf16_prefill"]
    inp = make_inputs(wl, device=DEV)
    y0, st0 = _forward_flags(moe, wl, inp, moe.MOE_FLAG_SINGLE_CTA)
    assert st0 == 0
    for flags in (0, moe.MOE_FLAG_PAIR_L1):
        y1, st1 = _forward_flags(moe, wl, inp, flags)
        assert st1 == 0
        assert torch.equal(y0.view(torch.int16), y1.view(torch.int16)), flags


# ---------------------------------------------------------------------------------------
# A8W4-INT: weight-major tiles (MOE_FLAG_WEIGHT_MAJOR; the default when the experts' weight slabs
# fill four rounds of tiles) against token-major ones (MOE_FLAG_TOKEN_MAJOR): both compute the
# same exact integers and the same fp32 operations, so y is compared bit for bit
# ---------------------------------------------------------------------------------------

@pytest.mark.parametrize("case", ["tiny", "ragged", "tail_sizes", "full_size"])
def test_w4_weight_major_equals_token_major(moe, case):
    if case == "tail_sizes":
        wl, inp = _tail_inputs("a8w4_int", 48)
    else:
        wl = {"tiny": CASES["a8w4_int"][0], "ragged": CASES["a8w4_int"][1], "full_size": WORKLOADS["int4_a8w4"]}[case]
        inp = make_inputs(wl, device=DEV)
    y0, st0 = _forward_flags(moe, wl, inp, moe.MOE_FLAG_TOKEN_MAJOR)
    y1, st1 = _forward_flags(moe, wl, inp, moe.MOE_FLAG_WEIGHT_MAJOR)
    y2, st2 = _forward_flags(moe, wl, inp, 0)  # the tile-count rule's choice
    assert st0 == 0 and st1 == 0 and st2 == 0
    assert torch.equal(y0.view(torch.int16), y1.view(torch.int16))
    assert torch.equal(y0.view(torch.int16), y2.view(torch.int16))
    if case != "full_size":
        assert_close(y_numpy(y1), oracle_forward(wl, inp), wl.mode)


# The largest expert count the ABI takes (E = 1024) with the largest top-k (K = 32): about two rows
# per expert, so every kernel's per-expert tables, scans and tile searches run at their limits.
MAX_E = [Workload(f"max_experts_{m}", m, 64, 256, 128, 1024, 32, 49, 0.05)
         for m in ("a16w16", "a8w8_fp8", "a8w8_int8", "a8w4_int", "a8w4_fp8_fp4")]


@pytest.mark.parametrize("wl", MAX_E, ids=[w.name for w in MAX_E])
def test_max_experts_and_topk(moe, wl):
    inp = make_inputs(wl, device=DEV)
    out = run_forward(moe, wl, inp, stages=True)
    assert out["status"] == 0
    check_plan(out, wl, inp["topk_ids"])
    assert_close(y_numpy(out["y"]), oracle_forward(wl, inp), wl.mode)
