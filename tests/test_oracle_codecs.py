"""Pins of the oracle's number-format codecs and quantisers against the format definitions,
closed forms and torch's own conversions (independent library routines)."""
import math

import numpy as np
import pytest
import torch

from oracle import codecs, moe


def test_e4m3_table_matches_definition_landmarks():
    t = codecs.E4M3_VALUES
    assert t[0x00] == 0.0 and t[0x80] == 0.0
    assert t[0x01] == 2.0 ** -9          # smallest subnormal: 1/8 * 2^-6
    assert t[0x08] == 2.0 ** -6          # smallest normal
    assert t[0x38] == 1.0                # exponent field 7 = bias
    assert t[0x7E] == 448.0              # largest finite
    assert math.isnan(t[0x7F]) and math.isnan(t[0xFF])
    assert t[0xFE] == -448.0


def test_e4m3_table_matches_torch_for_every_code():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = codecs.E4M3_VALUES
    both_nan = np.isnan(ref) & np.isnan(ours)
    assert np.all(both_nan | (ref == ours))


def test_e4m3_encode_matches_torch_rne():
    rng = np.random.default_rng(7)
    v = np.concatenate([rng.standard_normal(20000) * 50, rng.standard_normal(2000) * 0.01,
                        codecs.E4M3_VALUES[:0x7F], -codecs.E4M3_VALUES[1:0x7F]])
    # midpoints between neighbouring magnitudes: ties must go to the even code
    mids = (codecs.E4M3_VALUES[1:0x7F] + codecs.E4M3_VALUES[0:0x7E]) / 2
    # values that round to +-0 (below half the smallest subnormal, and exactly half of it)
    tiny = np.array([2.0 ** -10, 2.0 ** -11, 1e-6, 0.0])
    v = np.concatenate([v, mids, -mids, tiny, -tiny])
    v = np.clip(v, -448, 448).astype(np.float32).astype(np.float64)
    ref = torch.from_numpy(v).to(torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = codecs.e4m3_encode_rne_satfinite(v)
    assert np.array_equal(ours, ref)  # including the sign of a zero result


def test_e4m3_encode_saturates():
    assert codecs.e4m3_encode_rne_satfinite(np.array([1e6]))[0] == 0x7E
    assert codecs.e4m3_encode_rne_satfinite(np.array([-500.0]))[0] == 0xFE


def test_e5m2_table_matches_definition_landmarks():
    t = codecs.E5M2_VALUES
    assert t[0x00] == 0.0 and t[0x80] == 0.0
    assert t[0x01] == 2.0 ** -16          # smallest subnormal: 1/4 * 2^-14
    assert t[0x04] == 2.0 ** -14          # smallest normal
    assert t[0x3C] == 1.0                 # exponent field 15 = bias
    assert t[0x7B] == 57344.0             # largest finite: 1.75 * 2^15
    assert t[0x7C] == math.inf and t[0xFC] == -math.inf
    assert math.isnan(t[0x7D]) and math.isnan(t[0xFF])


def test_e5m2_table_matches_torch_for_every_code():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e5m2).to(torch.float64).numpy()
    ours = codecs.E5M2_VALUES
    both_nan = np.isnan(ref) & np.isnan(ours)
    assert np.all(both_nan | (ref == ours))


def test_e5m2_encode_matches_torch_rne():
    rng = np.random.default_rng(8)
    pos = codecs.E5M2_VALUES[:0x7C]
    v = np.concatenate([rng.standard_normal(20000) * 3000, rng.standard_normal(2000) * 1e-4, pos, -pos[1:]])
    mids = (pos[1:] + pos[:-1]) / 2  # ties go to the even code
    tiny = np.array([2.0 ** -17, 2.0 ** -18, 1e-9, 0.0])
    v = np.concatenate([v, mids, -mids, tiny, -tiny])
    v = np.clip(v, -57344, 57344).astype(np.float32).astype(np.float64)
    ref = torch.from_numpy(v).to(torch.float32).to(torch.float8_e5m2).view(torch.uint8).numpy()
    assert np.array_equal(codecs.e5m2_encode_rne_satfinite(v), ref)


def test_e5m2_encode_saturates_to_the_largest_finite():
    # (torch's own conversion overflows to infinity; the satfinite rule clamps)
    assert codecs.e5m2_encode_rne_satfinite(np.array([1e9]))[0] == 0x7B
    assert codecs.e5m2_encode_rne_satfinite(np.array([-61440.0]))[0] == 0xFB


def test_mx_e5m2_quant_properties():
    rng = np.random.default_rng(9)
    a = rng.standard_normal((6, 128)) * np.exp(rng.standard_normal((6, 1)) * 4)
    a[0] = 0.0
    codes, sc = moe.quant_mx_fp8(a, 32, "e5m2")
    vals = codecs.e5m2_decode(codes) * np.repeat(codecs.ue8m0_decode(sc), 32, axis=1)
    assert np.all(vals[0] == 0.0) and np.all(sc[0] == 0)
    blocks = np.abs(a.astype(np.float32).astype(np.float64)).reshape(6, 4, 32).max(axis=2)
    e = sc.astype(np.int64) - 127
    ratio = blocks[1:] / np.ldexp(1.0, e[1:])
    # the largest element of a block lands in the top binade of e5m2: (28672, 57344]
    assert np.all(ratio > 28672) and np.all(ratio <= 57344)
    # relative rounding error of e5m2 (2 mantissa bits) is at most 2^-3 of the value's binade
    err = np.abs(vals[1:] - a[1:]) / np.maximum(np.abs(a[1:]), 2.0 ** -14 * np.ldexp(1.0, np.repeat(e[1:], 32, axis=1)))
    assert err.max() <= 2.0 ** -3 + 1e-12


def test_e2m1_table_is_the_format():
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert list(codecs.E2M1_VALUES[:8]) == mags
    assert list(codecs.E2M1_VALUES[8:]) == [-m for m in mags]


def test_e2m1_unpack_nibble_order():
    # byte 0x21: low nibble code 1 (0.5) is element 0, high nibble code 2 (1.0) is element 1
    out = codecs.e2m1_unpack_decode(np.array([[0x21, 0xF7]], dtype=np.uint8))
    assert out.tolist() == [[0.5, 1.0, 6.0, -6.0]]


def test_ue8m0():
    s = np.array([0, 1, 127, 128, 254, 255], dtype=np.uint8)
    d = codecs.ue8m0_decode(s)
    assert d[0] == 2.0 ** -127 and d[1] == 2.0 ** -126 and d[2] == 1.0 and d[3] == 2.0
    assert d[4] == 2.0 ** 127 and math.isnan(d[5])


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(3)
    v = np.concatenate([rng.standard_normal(50000), rng.standard_normal(5000) * 1e-30,
                        rng.standard_normal(5000) * 1e30])
    v32 = v.astype(np.float32)
    # exact ties: bf16 value + half a spacing (low 16 bits = 0x8000)
    ties = ((v32.view(np.uint32) & np.uint32(0xFFFF0000)) | np.uint32(0x8000)).view(np.float32)
    v32 = np.concatenate([v32, ties])
    ref = torch.from_numpy(v32).to(torch.bfloat16).to(torch.float64).numpy()
    ours = codecs.round_to_bf16(v32.astype(np.float64))
    assert np.array_equal(ref, ours)
    assert np.array_equal(codecs.bf16_decode(codecs.bf16_encode(ours)), ours)


def test_int8_row_quant_range_and_error():
    rng = np.random.default_rng(5)
    a = rng.standard_normal((64, 300)) * rng.uniform(0.01, 100, size=(64, 1))
    q, s = moe.quant_int8_rows(a)
    assert q.dtype == np.int8 and q.min() >= -127 and q.max() <= 127
    assert (q != -128).all()
    a32 = a.astype(np.float32).astype(np.float64)
    arg = np.argmax(np.abs(a32), axis=1)
    assert np.all(np.abs(q[np.arange(64), arg]) == 127)
    err = np.abs(q * s[:, None].astype(np.float64) - a32)
    assert np.all(err <= s[:, None] * 0.5 * (1 + 1e-6))


def test_int8_row_quant_zero_row():
    q, s = moe.quant_int8_rows(np.zeros((2, 8)))
    assert np.all(q == 0) and np.all(s == np.float32(1e-8))


def test_mx_exponent_rule():
    am = np.array([448.0, 449.0, 224.0, 896.0, 1.0, 0.0, 3.0e-38], dtype=np.float32)
    e = moe.mx_scale_exponent(am, 448.0)
    assert e[0] == 0 and e[1] == 1 and e[2] == -1 and e[3] == 1
    assert e[4] == math.ceil(math.log2(1.0 / 448.0)) and e[5] == -127
    assert e[6] == -127  # clamped to the smallest UE8M0 exponent


def test_mx_fp8_quant_properties():
    rng = np.random.default_rng(9)
    a = rng.standard_normal((16, 128)) * rng.uniform(1e-3, 1e3, size=(16, 1))
    a[3, 32:64] = 0.0
    codes, sc = moe.quant_mx_fp8(a)
    vals = codecs.e4m3_decode(codes)
    scale = codecs.ue8m0_decode(sc)
    assert np.all(np.abs(vals) <= 448.0)
    assert np.all(vals[3, 32:64] == 0.0)
    deq = vals * np.repeat(scale, 32, axis=1)
    a32 = a.astype(np.float32).astype(np.float64)
    # the block's largest element lands in the top binade of e4m3: |amax/2^e| > 224
    blocks = np.abs(a32).reshape(16, 4, 32).max(axis=2)
    nz = blocks > 0
    assert np.all((blocks / scale)[nz] > 224.0) and np.all((blocks / scale)[nz] <= 448.0)
    # RNE error: at most half a spacing of the element's binade (relative 2^-4)
    rel = np.abs(deq - a32) / np.maximum(np.abs(a32), 2.0 ** -6 * np.repeat(scale, 32, axis=1))
    assert np.all(rel <= 2.0 ** -4 + 1e-12)


def _bf16(v):
    return codecs.bf16_encode(codecs.round_to_bf16(np.asarray(v, dtype=np.float64)))


def test_quantize_x_int8_closed_form_and_invariants():
    # a row of small integers with max 127: s = 1 exactly and q = the row
    row = np.array([[127.0, -64.0, 1.0, 0.0, -127.0, 3.0, 100.0, -1.0]])
    q, s = moe.quantize_x("a8w8_int8", _bf16(row))
    assert s[0] == np.float32(1.0) and np.array_equal(q[0], row[0].astype(np.int8))
    rng = np.random.default_rng(11)
    x = _bf16(rng.standard_normal((32, 256)) * rng.uniform(1e-3, 1e3, size=(32, 1)))
    xv = codecs.bf16_decode(x)
    q, s = moe.quantize_x("a8w8_int8", x)
    assert q.min() >= -127 and q.max() <= 127
    arg = np.argmax(np.abs(xv), axis=1)
    assert np.all(np.abs(q[np.arange(32), arg]) == 127)
    # half a step, plus the fp32 rounding of s and of x/s (a quotient next to .5 can round to
    # the tie and then to the even integer: x = 972, max 1944 gives 63.5 -> 64)
    assert np.all(np.abs(q * s[:, None].astype(np.float64) - xv) <= s[:, None] * 0.5 * (1 + 1e-5))
    q, s = moe.quantize_x("a8w8_int8", _bf16(np.zeros((1, 16))))
    assert np.all(q == 0) and s[0] == np.float32(1e-8)


@pytest.mark.parametrize("mode,block", [("a8w8_fp8", 32), ("a8w4_fp8_fp4", 128)])
def test_quantize_x_fp8_groups(mode, block):
    rng = np.random.default_rng(12)
    x = rng.standard_normal((8, 512)) * rng.uniform(1e-2, 1e2, size=(8, 1))
    x[2, :block] = 0.0
    xb = _bf16(x)
    xv = codecs.bf16_decode(xb)
    codes, sc = moe.quantize_x(mode, xb)
    scale = codecs.ue8m0_decode(sc) if mode == "a8w8_fp8" else sc.astype(np.float64)
    assert scale.shape == (8, 512 // block)
    assert np.all(np.log2(scale[scale > 0]) == np.round(np.log2(scale[scale > 0])))  # powers of two
    vals = codecs.e4m3_decode(codes)
    full = np.repeat(scale, block, axis=1)
    amax = np.abs(xv).reshape(8, -1, block).max(axis=2)
    nz = amax > 0
    assert np.all((amax / scale)[nz] > 224.0) and np.all((amax / scale)[nz] <= 448.0)
    assert np.all(vals[2, :block] == 0.0)
    rel = np.abs(vals * full - xv) / np.maximum(np.abs(xv), 2.0 ** -6 * full)
    assert np.all(rel <= 2.0 ** -4 + 1e-12)
    # values that are e4m3 codes times the group's power of two come back exactly
    exact = np.resize(codecs.e4m3_decode(np.arange(0x30, 0x7e, dtype=np.uint8)), block) * 2.0 ** 3
    exact[0] = 448.0 * 2.0 ** 3  # the group's amax sets the exponent to 3
    c2, s2 = moe.quantize_x(mode, _bf16(np.tile(exact, (1, 512 // block))))
    s2v = codecs.ue8m0_decode(s2) if mode == "a8w8_fp8" else s2.astype(np.float64)
    assert np.all(s2v == 8.0)
    assert np.array_equal(codecs.e4m3_decode(c2) * 8.0, codecs.bf16_decode(_bf16(np.tile(exact, (1, 512 // block)))))


def test_quantize_x_a16w16_is_the_input():
    x = _bf16(np.linspace(-3, 3, 64).reshape(4, 16))
    xx, sc = moe.quantize_x("a16w16", x)
    assert sc is None and np.array_equal(xx, x)


def test_int4_pack_round_trip_exhaustive():
    v0, v1 = np.meshgrid(np.arange(-8, 8), np.arange(-8, 8), indexing="ij")
    packed = ((v0.ravel() & 0xF) | ((v1.ravel() & 0xF) << 4)).astype(np.uint8)[:, None]
    out = codecs.int4_unpack(packed)
    assert np.array_equal(out[:, 0], v0.ravel()) and np.array_equal(out[:, 1], v1.ravel())
    assert len(np.unique(packed)) == 256


def test_msd_split_equals_the_integer_product():
    """The A8W4-INT decomposition (high nibble, offset low nibble, compensation bias) gives
    q . W exactly, also at the int8 extremes."""
    rng = np.random.default_rng(21)
    q = rng.integers(-127, 128, size=(17, 96)).astype(np.int8)
    q[0] = 127
    q[1] = -127
    q[2, ::2] = -128 + 1
    w = rng.integers(-8, 8, size=(96, 40)).astype(np.int8)
    ref = q.astype(np.int64) @ w.astype(np.int64)
    assert np.array_equal(moe.msd_int_matmul(q, w), ref)


def test_int32_accumulator_guard():
    q = np.full((1, 200000), 127, dtype=np.int8)
    w = np.full((200000, 1), 127, dtype=np.int8)
    with pytest.raises(OverflowError):
        moe._int_matmul_checked(q, w)
    # the largest inner dimension of the configurations fits: 5120 * 127^2 < 2^31
    q = np.full((1, 5120), -127, dtype=np.int8)
    w = np.full((5120, 1), 127, dtype=np.int8)
    assert moe._int_matmul_checked(q, w)[0, 0] == -5120 * 127 * 127


def test_quantize_x_e5m2_round_trip_and_zero_groups():
    """A8W8-FP with the E5M2 target type (p1 Q_MX): values that are e5m2 codes times the group's
    power of two come back exactly; a group of zeros gets scale byte 0 and zero codes."""
    block = 32
    top = codecs.e5m2_decode(np.arange(0x5C, 0x7C, dtype=np.uint8))  # 32 codes up to 57344
    exact = np.tile(top, (1, 4)) * 2.0 ** -10   # fits bf16: 3 significant bits
    x = np.concatenate([exact, np.zeros((1, 128))])
    codes, sc = moe.quantize_x("a8w8_fp8_e5m2", _bf16(x))
    assert codes.dtype == np.uint8 and sc.shape == (2, 4)
    assert np.all(sc[0] == 127 - 10) and np.all(sc[1] == 0) and np.all(codes[1] == 0)
    back = codecs.e5m2_decode(codes[0]) * 2.0 ** -10
    assert np.array_equal(back, codecs.bf16_decode(_bf16(exact))[0])
