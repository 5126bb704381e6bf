"""Plain CPU definition of the fused MoE expert feed-forward with top-k combine.

TEST INFRASTRUCTURE ONLY. Nothing in the product path may import this module; only
``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` use it.
It shares no code with the CUDA path.

What it computes (Ascend ``mega_moe`` page, "Computation Process", A16W16 use case):

    y_i = sum_k G[i,k] * Y_{e_ik}[row(i,k), :],    Y_e = SwiGLU(X_e . W1[e]) . W2[e]

with the quantised use cases of the same page (A8W8-INT, A8W8-FP) and the FP8-activation x
FP4-weight recipe of the DeepGEMM MegaMoE page (§4, steps 5-7). Every floating-point step
runs in float64 except where a step's result is a quantised code or a stored rounded value:
there the rounding is written out (bf16, e4m3 + UE8M0, int8 + fp32 scale) and, where
floating point decides an integer code, the decision is taken on the fp32 value, the
precision of the kernel (the pages fix none).

Readings where the pages are silent or disagree (each listed in the design notes):
  * rows of X_e are stacked in ascending (i*K + k) order; the pages allow any fixed order;
  * the gate weight G multiplies the L2 output (p1, "Token Combine"), in fp32, and each
    weighted row is stored as bf16 before the top-k sum; the sum runs in fp32 in slot
    order k = 0..K-1 and is rounded once to bf16;
  * an expert id of -1 is a masked route: it is skipped and contributes nothing;
  * the A16W16 L2 operand A is rounded to bf16 (both GEMMs take bf16 operands);
  * the FP8 re-quantisation of A uses blocks of 32 along the intermediate dimension with a
    power-of-two scale 2^ceil(log2(amax/448)) stored as UE8M0;
  * the INT8 re-quantisation of A follows p1's per-row formula with the scale floored at
    1e-8 (the floor of p1's own weight-quantisation example);
  * a shared expert (DeepGEMM page §6) is computed like a routed one, in the same dtype mode,
    on every token, with weight 1 in the extra combine slot K + j after the routed slots.
"""
from __future__ import annotations

import numpy as np

from . import codecs

MODES = ("a16w16", "a8w8_fp8", "a8w8_int8", "a8w4_fp8_fp4", "a8w4_int", "a8w8_fp8_e5m2")
# the FP8 element format of each A8W8-FP mode (p1 A8W8-FP: FLOAT8_E4M3FN or FLOAT8_E5M2; x, both
# weights and the re-quantised A take the same type)
FP8_FORMAT = {"a8w8_fp8": "e4m3", "a8w8_fp8_e5m2": "e5m2"}
INT_MODES = ("a8w8_int8", "a8w4_int")  # integer GEMMs with per-token / per-channel fp32 scales


# ---------------------------------------------------------------------------------------
# Dispatch: I_e, N_e and row(i, k)  (p1, A16W16 "EP Dispatch"; p3 §1 count -> prefix sum
# -> scatter)
# ---------------------------------------------------------------------------------------


def plan(topk_ids: np.ndarray, num_experts: int):
    """Per-expert counts N_e, exclusive offsets and the pool order of routed rows.

    counts[e]  = #{(i,k) : E[i,k] = e}
    offsets[e] = sum_{e' < e} counts[e'], offsets[E] = number of routed rows
    row_src[p] = i*K + k of the routed row stored at pool position p; the rows of expert e
                 occupy [offsets[e], offsets[e+1]) in ascending i*K + k.
    Masked routes (id -1) are skipped. Any other id outside [0, E) raises ValueError.
    """
    ids = np.asarray(topk_ids).astype(np.int64)
    T, K = ids.shape
    flat = ids.reshape(-1)
    bad = (flat < -1) | (flat >= num_experts)
    if bad.any():
        raise ValueError("expert id outside [-1, num_experts)")
    counts = np.zeros(num_experts, dtype=np.int64)
    for e in flat:
        if e >= 0:
            counts[e] += 1
    offsets = np.zeros(num_experts + 1, dtype=np.int64)
    for e in range(num_experts):
        offsets[e + 1] = offsets[e] + counts[e]
    row_src = np.empty(offsets[-1], dtype=np.int64)
    cursor = offsets[:-1].copy()
    for r in range(T * K):  # ascending i*K + k: a stable counting sort
        e = flat[r]
        if e >= 0:
            row_src[cursor[e]] = r
            cursor[e] += 1
    return counts, offsets, row_src


# ---------------------------------------------------------------------------------------
# Operand decoding: stored codes -> exact real values
# ---------------------------------------------------------------------------------------


def fp8_decode(fmt: str, codes: np.ndarray) -> np.ndarray:
    return codecs.e4m3_decode(codes) if fmt == "e4m3" else codecs.e5m2_decode(codes)


def decode_x(mode: str, x: np.ndarray, x_scale: np.ndarray | None) -> np.ndarray:
    """Activations [T, H] as exact float64 values.

    a16w16       : x bf16 codes (uint16).
    a8w8_fp8     : x e4m3 codes, x_scale UE8M0 [T, H/32] (p1 A8W8-FP, Q_MX group 32).
    a8w8_int8    : x int8 codes q_i; x_scale fp32 [T] = s^X_i. Returns the integer codes;
                   the int8 path keeps q and s^X apart (p1 A8W8-INT).
    a8w4_fp8_fp4 : x e4m3 codes, x_scale fp32 [T, H/128] (1x128 blocks).
    a8w4_int     : as a8w8_int8 (p1 A8W4-INT: the same per-token int8 quantisation of X).
    a8w8_fp8_e5m2: as a8w8_fp8 with e5m2 codes.
    """
    if mode == "a16w16":
        return codecs.bf16_decode(x)
    if mode in FP8_FORMAT:
        v = fp8_decode(FP8_FORMAT[mode], x)
        s = np.repeat(codecs.ue8m0_decode(x_scale), 32, axis=-1)
        return v * s
    if mode in INT_MODES:
        return np.asarray(x, dtype=np.int8).astype(np.float64)
    if mode == "a8w4_fp8_fp4":
        v = codecs.e4m3_decode(x)
        s = np.repeat(np.asarray(x_scale, dtype=np.float32).astype(np.float64), 128, axis=-1)
        return v * s
    raise ValueError(mode)


def decode_weight(mode: str, w: np.ndarray, w_scale: np.ndarray | None, e: int) -> np.ndarray:
    """Weight matrix of expert e in the math orientation [K_in, N_out] as float64.

    a16w16       : w bf16 [E, K_in, N_out] (p1: W1 is hidden x 2*intermediate per expert).
    a8w8_fp8     : w e4m3 [E, N_out, K_in] (p1 950 layout, transposed) with UE8M0 scales
                   [E, N_out, K_in/32].
    a8w8_int8    : w int8 [E, N_out, K_in]; returns the integer codes (the per-output-channel
                   fp32 scale is applied after the integer GEMM).
    a8w4_fp8_fp4 : w e2m1 packed [E, N_out, K_in/2] with UE8M0 scales [E, N_out, K_in/32].
    a8w4_int     : w signed int4 packed [E, N_out, K_in/2] (element 2j in the low nibble);
                   returns the integer codes (per-output-channel fp32 scale as for a8w8_int8).
    a8w8_fp8_e5m2: as a8w8_fp8 with e5m2 codes.
    """
    if mode == "a16w16":
        return codecs.bf16_decode(w[e])
    if mode in FP8_FORMAT:
        v = fp8_decode(FP8_FORMAT[mode], w[e]) * np.repeat(codecs.ue8m0_decode(w_scale[e]), 32, axis=-1)
        return v.T
    if mode == "a8w8_int8":
        return np.asarray(w[e], dtype=np.int8).astype(np.float64).T
    if mode == "a8w4_int":
        return codecs.int4_unpack(w[e]).astype(np.float64).T
    if mode == "a8w4_fp8_fp4":
        v = codecs.e2m1_unpack_decode(w[e]) * np.repeat(codecs.ue8m0_decode(w_scale[e]), 32, axis=-1)
        return v.T
    raise ValueError(mode)


# ---------------------------------------------------------------------------------------
# SwiGLU (p1 "Conventions": SiLU(z) = z / (1 + e^-z); "SwiGLU Activation")
# ---------------------------------------------------------------------------------------


def silu(z: np.ndarray) -> np.ndarray:
    z = np.asarray(z, dtype=np.float64)
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def swiglu(h: np.ndarray, inter: int, clamp: float | None = None) -> np.ndarray:
    """A = SiLU(H[:, :I]) * H[:, I:]; gate is the first half of the columns.

    clamp (p1 parameter activation_clamp: a threshold t >= 0 that limits the input of the
    activation function to [-t, t], symmetrically): when given, both halves of H, the input of
    SwiGLU, are first clipped to [-clamp, clamp]."""
    if clamp is not None:
        h = np.clip(h, -clamp, clamp)
    return silu(h[:, :inter]) * h[:, inter:]


# ---------------------------------------------------------------------------------------
# L2-operand quantisers (the requantisation of A)
# ---------------------------------------------------------------------------------------


def quant_int8_rows(a: np.ndarray):
    """p1 A8W8-INT, Linear2 step (1): s_i = max|A[i,:]|/127, q = round(A/s) in [-127, 127].

    The decision runs in fp32 (the kernel's precision): a is first rounded to fp32, then
    s = fp32(amax / 127) floored at 1e-8, q = rint(fp32(a / s)) clamped to [-127, 127].
    Returns (q int8 [n, I], s float32 [n]).
    """
    a32 = np.asarray(a, dtype=np.float64).astype(np.float32)
    amax = np.max(np.abs(a32), axis=1)
    s = np.maximum(amax / np.float32(127.0), np.float32(1e-8)).astype(np.float32)
    q = np.rint((a32 / s[:, None]).astype(np.float32))
    q = np.clip(q, -127, 127).astype(np.int8)
    return q, s


def mx_scale_exponent(amax32: np.ndarray, elem_max: float) -> np.ndarray:
    """Smallest integer e with amax <= elem_max * 2^e, clamped to [-127, 127]; amax = 0
    gives -127. That is the shared exponent ceil(log2(amax / elem_max)) of an MX block."""
    amax = np.asarray(amax32, dtype=np.float64)
    out = np.full(amax.shape, -127, dtype=np.int64)
    nz = amax > 0
    # frexp gives amax/elem_max = m * 2^ex, 0.5 <= m < 1; ceil(log2) = ex, or ex-1 when m = 0.5
    m, ex = np.frexp(amax[nz] / elem_max)
    e = np.where(m == 0.5, ex - 1, ex)
    out[nz] = np.clip(e, -127, 127)
    return out


def quant_mx_fp8(a: np.ndarray, block: int = 32, fmt: str = "e4m3"):
    """MX quantisation with 1 x `block` groups along the last axis to an FP8 format (e4m3 or
    e5m2) + a shared power-of-two exponent (p1 A8W8-FP "Q_MX", group size 32, target type
    FLOAT8_E4M3FN or FLOAT8_E5M2; DeepGEMM §4 step 6 FP8 re-quantisation). The decision runs on
    fp32 values: a -> fp32, per-group amax, exponent e = the smallest with amax <= max * 2^e
    (max = the format's largest finite value), codes = rne_satfinite(a / 2^e).
    Returns (codes uint8 [n, m], exponents as UE8M0 bytes uint8 [n, m/block])."""
    a32 = np.asarray(a, dtype=np.float64).astype(np.float32).astype(np.float64)
    n, m = a32.shape
    blocks = a32.reshape(n, m // block, block)
    amax = np.max(np.abs(blocks), axis=2)
    elem_max = codecs.E4M3_MAX if fmt == "e4m3" else codecs.E5M2_MAX
    encode = codecs.e4m3_encode_rne_satfinite if fmt == "e4m3" else codecs.e5m2_encode_rne_satfinite
    e = mx_scale_exponent(amax, elem_max)
    scaled = blocks / np.ldexp(1.0, e.astype(np.int32))[:, :, None]
    codes = encode(scaled).reshape(n, m)
    return codes, (e + 127).astype(np.uint8)


def quantize_x(mode: str, x_bf16: np.ndarray):
    """The operator's own quantisation of the bf16 activations before dispatch, to the mode's
    x format (p1 parameter dispatch_quant_mode):
      * A8W8-INT (p1 "A8W8-INT Quantization Use Case", "EP Dispatch"): per token
        s_i = max|X[i,:]| / 127 and q_i = round(X[i,:] / s_i), as quant_int8_rows (fp32
        decision, scale floored at 1e-8);
      * A8W8-FP (p1 "A8W8-FP Quantization Use Case", first phase): Q_MX with groups of 32,
        e4m3 (or, for a8w8_fp8_e5m2, e5m2) codes and E8M0 scales;
      * FP8 activations x FP4 weights: the same shared-exponent rule on groups of 128 gives the
        mode's x format, e4m3 codes with power-of-two fp32 scales (the DeepGEMM page takes
        FP8 activations with their scales as the input of fp8_fp4_mega_moe).
    x_bf16: uint16 bf16 codes [T, H]. Returns (x, x_scale) as moe_forward's x operand takes them:
    bf16 codes and None for A16W16."""
    x = np.asarray(x_bf16, dtype=np.uint16)
    if mode == "a16w16":
        return x, None
    xv = codecs.bf16_decode(x)
    if mode in INT_MODES:
        return quant_int8_rows(xv)
    if mode in FP8_FORMAT:
        return quant_mx_fp8(xv, 32, FP8_FORMAT[mode])
    if mode == "a8w4_fp8_fp4":
        codes, sb = quant_mx_fp8(xv, 128)
        return codes, np.ldexp(np.float32(1.0), sb.astype(np.int32) - 127).astype(np.float32)
    raise ValueError(mode)


def l2_operand(mode: str, a: np.ndarray):
    """The re-quantised A of one expert as (exact float64 values, record of the codes)."""
    if mode == "a16w16":
        v = codecs.round_to_bf16(a)
        return v, {"a": codecs.bf16_encode(v)}
    if mode in ("a8w8_fp8", "a8w4_fp8_fp4", "a8w8_fp8_e5m2"):
        fmt = FP8_FORMAT.get(mode, "e4m3")  # FP8 x FP4 re-quantises A to e4m3 (DeepGEMM §4 step 6)
        codes, sc = quant_mx_fp8(a, 32, fmt)
        v = fp8_decode(fmt, codes) * np.repeat(codecs.ue8m0_decode(sc), 32, axis=1)
        return v, {"a": codes, "a_scale": sc}
    if mode in INT_MODES:
        q, s = quant_int8_rows(a)
        return q.astype(np.float64), {"a": q, "a_scale": s}
    raise ValueError(mode)


# ---------------------------------------------------------------------------------------
# One expert's FFN on the rows routed to it
# ---------------------------------------------------------------------------------------

INT32_MIN, INT32_MAX = -(2 ** 31), 2 ** 31 - 1


def _int_matmul_checked(q: np.ndarray, w: np.ndarray) -> np.ndarray:
    """Exact integer product in int64; the pages require the result to fit int32."""
    c = q.astype(np.int64) @ w.astype(np.int64)
    if c.size and (c.min() < INT32_MIN or c.max() > INT32_MAX):
        raise OverflowError("int8 GEMM accumulator outside int32")
    return c


def msd_int_matmul(q: np.ndarray, w: np.ndarray) -> np.ndarray:
    """The A8W4-INT product of p1 ("A8W4-INT Quantization Use Case", Expert Compute): the int8
    activations are split into a signed high nibble q_hi = floor(q / 16) and an offset low
    nibble q_lo = (q & 0x0F) - 8, each multiplied by the int4 weights, and recombined as
    16 * (q_hi . W) + (q_lo . W) + bias with the compensation bias = 8 * (1^T . W) that the page
    defines (computed offline there and passed to the operator). All in int64; the page applies
    the weight scale before this combination, which in exact arithmetic is the same as applying
    it to the combined integer, as done by the caller. Equals q . W exactly."""
    q = q.astype(np.int64)
    hi = np.floor_divide(q, 16)
    lo = np.bitwise_and(q, 0x0F) - 8
    wi = w.astype(np.int64)
    bias = 8 * wi.sum(axis=0)
    c = 16 * (hi @ wi) + (lo @ wi) + bias[None, :]
    if c.size and (c.min() < INT32_MIN or c.max() > INT32_MAX):
        raise OverflowError("int8 x int4 GEMM accumulator outside int32")
    return c


def expert_ffn(mode: str, xe: np.ndarray, sx: np.ndarray | None, w1e: np.ndarray,
               s_w1e: np.ndarray | None, w2e: np.ndarray, s_w2e: np.ndarray | None, inter: int,
               clamp: float | None = None):
    """Y_e for the rows X_e of one expert. Returns (Y float64 [n, H], intermediates).

    float modes : H = X_e . W1 (float64), A = SwiGLU(H), A~ = requant(A), Y = A~ . W2.
    a8w8_int8   : C = Q_e . W1 (int32), H = (C * s^W1) * s^X in fp32 (p1 Linear1),
                  A = SwiGLU(H), (A^int8, s^A) = requant(A),
                  D = A^int8 . W2 (int32), Y = (D * s^W2) * s^A in fp32 (p1 Linear2).
    a8w4_int    : the same with int4 weights, C and D by the MSD decomposition (msd_int_matmul).
    """
    if mode in INT_MODES:
        mm = _int_matmul_checked if mode == "a8w8_int8" else msd_int_matmul
        c = mm(xe, w1e)
        h32 = (c.astype(np.float32) * s_w1e[None, :].astype(np.float32)).astype(np.float32)
        h32 = (h32 * sx[:, None].astype(np.float32)).astype(np.float32)
        h = h32.astype(np.float64)
        a = swiglu(h, inter, clamp)
        q, rec = l2_operand(mode, a)
        d = mm(rec["a"], w2e)
        y32 = (d.astype(np.float32) * s_w2e[None, :].astype(np.float32)).astype(np.float32)
        y32 = (y32 * rec["a_scale"][:, None]).astype(np.float32)
        return y32.astype(np.float64), {"h": h, "c": c, "d": d, **rec}
    h = xe @ w1e
    a = swiglu(h, inter, clamp)
    a_q, rec = l2_operand(mode, a)
    y = a_q @ w2e
    return y, {"h": h, **rec}


# ---------------------------------------------------------------------------------------
# Combine (p1 "Token Combine")
# ---------------------------------------------------------------------------------------


def weighted_rows(g: np.ndarray, y_rows: np.ndarray) -> np.ndarray:
    """Combine contributions bf16( fp32( G[i,k] * Y_e[row(i,k), :] ) ) for a batch of rows:
    g [n] fp32 gate weights, y_rows [n, H]."""
    g64 = np.asarray(g, dtype=np.float32).astype(np.float64)
    prod32 = (g64[:, None] * y_rows).astype(np.float32).astype(np.float64)
    return codecs.round_to_bf16(prod32)


def combine_rows(contrib: np.ndarray) -> np.ndarray:
    """y_i = bf16( sum_{k=0..K-1} contrib[..., k, :] ), the sum taken in fp32 in slot order.
    contrib [..., K, H] -> [..., H]."""
    acc = np.zeros(contrib.shape[:-2] + contrib.shape[-1:], dtype=np.float32)
    for k in range(contrib.shape[-2]):
        acc = (acc + contrib[..., k, :].astype(np.float32)).astype(np.float32)
    return codecs.round_to_bf16(acc.astype(np.float64))


# ---------------------------------------------------------------------------------------
# The whole path
# ---------------------------------------------------------------------------------------


def with_shared_slots(topk_ids, topk_weights, num_experts: int, num_shared: int):
    """The routing with the shared experts' slots (DeepGEMM page §6, optional shared experts):
    a shared expert takes no routed id; it sees every token, and its output goes to an extra
    combine slot after the K routed ones, which the combine sums with them. Shared expert j is
    expert num_experts + j of the weight tensors; its slot K + j carries weight 1 (the page gives
    the slot no gate). Returns ids [T, K + S] and weights [T, K + S]."""
    ids = np.asarray(topk_ids)
    g = np.asarray(topk_weights, dtype=np.float32)
    T = ids.shape[0]
    shared_ids = np.tile(np.arange(num_experts, num_experts + num_shared, dtype=ids.dtype), (T, 1))
    ones = np.ones((T, num_shared), dtype=np.float32)
    return np.concatenate([ids, shared_ids], axis=1), np.concatenate([g, ones], axis=1)


def forward(mode: str, x, x_scale, topk_ids, topk_weights, w1, w1_scale, w2, w2_scale,
            num_experts: int, inter: int, return_intermediates: bool = False, clamp: float | None = None,
            num_shared: int = 0):
    """Plan -> per-expert L1 -> SwiGLU (inputs clipped to [-clamp, clamp] when clamp is given)
    -> requant -> L2 -> gate -> combine. With num_shared > 0 the weight tensors hold
    num_experts routed experts followed by the shared ones (see with_shared_slots).

    Returns y as float64 bf16 values [T, H] (and, on request, the plan and per-row
    intermediates keyed by pool position: 'comb' holds the weighted bf16 rows [T*K, H]).
    """
    if num_shared:
        topk_ids, topk_weights = with_shared_slots(topk_ids, topk_weights, num_experts, num_shared)
        num_experts += num_shared
    ids = np.asarray(topk_ids)
    T, K = ids.shape
    g = np.asarray(topk_weights, dtype=np.float32)
    counts, offsets, row_src = plan(ids, num_experts)
    xd = decode_x(mode, x, x_scale)
    hidden = xd.shape[1]
    comb = np.zeros((T * K, hidden), dtype=np.float64)
    inter_rec = {}
    for e in range(num_experts):
        lo, hi = offsets[e], offsets[e + 1]
        if hi == lo:
            continue
        src = row_src[lo:hi]
        tok = src // K
        xe = xd[tok]
        sx = None if mode not in INT_MODES else np.asarray(x_scale, dtype=np.float32)[tok]
        w1e = decode_weight(mode, w1, w1_scale, e)
        w2e = decode_weight(mode, w2, w2_scale, e)
        s1 = None if mode not in INT_MODES else np.asarray(w1_scale[e], dtype=np.float32)
        s2 = None if mode not in INT_MODES else np.asarray(w2_scale[e], dtype=np.float32)
        y_e, rec = expert_ffn(mode, xe, sx, w1e, s1, w2e, s2, inter, clamp)
        comb[src] = weighted_rows(g.reshape(-1)[src], y_e)
        if return_intermediates:
            inter_rec[e] = {"src": src, "y": y_e, **rec}
    y = combine_rows(comb.reshape(T, K, hidden))
    if return_intermediates:
        return y, {"counts": counts, "offsets": offsets, "row_src": row_src, "comb": comb,
                   "experts": inter_rec}
    return y


def forward_tokens(mode: str, tokens, x, x_scale, topk_ids, topk_weights, w1, w1_scale, w2,
                   w2_scale, inter: int, clamp: float | None = None, num_experts: int = 0, num_shared: int = 0):
    """Brute force for a subset of tokens: for each token i and each slot k, evaluate the FFN
    of expert E[i,k] on x_i alone, weight it and sum. No plan and no permutation is used, so
    this checks the pooled path (every row of an expert is computed independently). Shared
    experts (num_shared > 0, after num_experts routed ones) add their slots after the routed."""
    if num_shared:
        topk_ids, topk_weights = with_shared_slots(topk_ids, topk_weights, num_experts, num_shared)
    ids = np.asarray(topk_ids)
    T, K = ids.shape
    g = np.asarray(topk_weights, dtype=np.float32)
    out = []
    decoded = {}
    for i in tokens:
        xi = decode_x(mode, x[i:i + 1], None if x_scale is None else x_scale[i:i + 1])
        contrib = []
        for k in range(K):
            e = int(ids[i, k])
            if e < 0:
                contrib.append(np.zeros(xi.shape[1]))
                continue
            if e not in decoded:
                decoded[e] = (decode_weight(mode, w1, w1_scale, e), decode_weight(mode, w2, w2_scale, e))
            w1e, w2e = decoded[e]
            sx = None if mode not in INT_MODES else np.asarray(x_scale, dtype=np.float32)[i:i + 1]
            s1 = None if mode not in INT_MODES else np.asarray(w1_scale[e], dtype=np.float32)
            s2 = None if mode not in INT_MODES else np.asarray(w2_scale[e], dtype=np.float32)
            y_e, _ = expert_ffn(mode, xi, sx, w1e, s1, w2e, s2, inter, clamp)
            contrib.append(weighted_rows(g[i, k:k + 1], y_e)[0])
        out.append(combine_rows(np.stack(contrib)))
    return np.stack(out)
