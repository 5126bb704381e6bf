"""Seeded synthetic workloads for the fused MoE expert FFN.

This module is shared by the tests, the benchmark and the oracle-side checks as the single
source of inputs. It draws random numbers and prepares the caller-side operands the library
takes as inputs: routing (top-k ids and softmax gates) and the storage formats of x and the
expert weights. It holds none of the expert computation (no GEMM, SwiGLU, re-quantisation
or combine) and imports neither the oracle nor the CUDA package.

Distributions (the workload descriptions of the method's configurations):
  * router scores ~ N(0, 1) fp32 over the experts; ids = top-K by score, highest first;
    gates = softmax over the K chosen scores (max subtracted);
  * skewed routing: scores = log p_e + Gumbel(0, 1) with p_e proportional to rank^-s under a
    seeded permutation of the experts; a tail of experts gets p_e = 0 and is never chosen;
  * x ~ N(0, 1), weights ~ N(0, w_std).
Storage formats per mode (x, w1, w2 and their scales; row-major, contiguous):
  a16w16       : x bf16 [T,H]; w1 bf16 [E,H,2I]; w2 bf16 [E,I,H].
  a8w8_fp8     : x e4m3 [T,H] + UE8M0 [T,H/32]; w1 e4m3 [E,2I,H] + UE8M0 [E,2I,H/32];
                 w2 e4m3 [E,H,I] + UE8M0 [E,H,I/32].
  a8w8_int8    : x int8 [T,H] + fp32 [T] (per-token symmetric, [-127,127]);
                 w1 int8 [E,2I,H] + fp32 [E,2I]; w2 int8 [E,H,I] + fp32 [E,H]
                 (per-output-channel symmetric).
  a8w4_fp8_fp4 : x e4m3 [T,H] + fp32 power-of-two scales [T,H/128];
                 w1 e2m1 packed [E,2I,H/2] + UE8M0 [E,2I,H/32];
                 w2 e2m1 packed [E,H,I/2] + UE8M0 [E,H,I/32]; low nibble = even element.
  a8w4_int     : x as a8w8_int8; w1 int4 packed [E,2I,H/2] + fp32 [E,2I]; w2 int4 packed
                 [E,H,I/2] + fp32 [E,H] (per-output-channel symmetric, [-7,7]).
  a8w8_fp8_e5m2: as a8w8_fp8 with e5m2 codes.
"""
from __future__ import annotations

import dataclasses

import torch

MODES = ("a16w16", "a8w8_fp8", "a8w8_int8", "a8w4_fp8_fp4", "a8w4_int", "a8w8_fp8_e5m2")


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    mode: str
    T: int
    H: int
    I: int
    E: int
    K: int
    seed: int
    w_std: float
    zipf_s: float | None = None   # skewed routing exponent
    zipf_empty: int = 0           # experts that are never routed to in skewed routing

    @property
    def routed_rows(self) -> int:
        return self.T * self.K

    @property
    def flops(self) -> int:
        """Algorithmic work: 2*H*2I (L1) + 2*I*H (L2) per routed row."""
        return 6 * self.H * self.I * self.routed_rows


WORKLOADS = {
    "tiny_bf16": Workload("tiny_bf16", "a16w16", 64, 256, 128, 8, 2, 0, 0.02),
    "mixtral_bf16_prefill": Workload("mixtral_bf16_prefill", "a16w16", 4096, 4096, 14336, 8, 2, 1, 0.01),
    "dsv3_fp8fp4_decode": Workload("dsv3_fp8fp4_decode", "a8w4_fp8_fp4", 128, 7168, 2048, 256, 8, 2, 0.02),
    "dsv3_fp8fp4_prefill_zipf": Workload("dsv3_fp8fp4_prefill_zipf", "a8w4_fp8_fp4", 8192, 7168, 2048, 256, 8,
                                         3, 0.02, zipf_s=1.2, zipf_empty=16),
    "int8_a8w8": Workload("int8_a8w8", "a8w8_int8", 2048, 5120, 1536, 64, 6, 4, 0.02),
    # the A8W8-INT shapes with int4 weights (the A8W4-INT use case)
    "int4_a8w4": Workload("int4_a8w4", "a8w4_int", 2048, 5120, 1536, 64, 6, 5, 0.02),
}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


# ---------------------------------------------------------------------------------------
# Routing
# ---------------------------------------------------------------------------------------


def routing(T: int, E: int, K: int, g: torch.Generator, device, zipf_s=None, zipf_empty=0):
    """Top-K expert ids (int32 [T,K], highest score first) and softmax gates (fp32 [T,K])."""
    scores = torch.randn((T, E), generator=g, device=device, dtype=torch.float32)
    if zipf_s is not None:
        perm = torch.randperm(E, generator=g, device=device)
        rank = torch.empty(E, device=device, dtype=torch.float32)
        rank[perm] = torch.arange(1, E + 1, device=device, dtype=torch.float32)
        logp = -zipf_s * torch.log(rank)
        logp = torch.where(rank > E - zipf_empty, torch.full_like(logp, float("-inf")), logp)
        u = torch.rand((T, E), generator=g, device=device, dtype=torch.float32).clamp_(1e-20, 1.0)
        scores = logp[None, :] - torch.log(-torch.log(u))
    vals, ids = torch.topk(scores, K, dim=1, largest=True, sorted=True)
    gates = torch.softmax(vals - vals.max(dim=1, keepdim=True).values, dim=1)
    return ids.to(torch.int32).contiguous(), gates.to(torch.float32).contiguous()


# ---------------------------------------------------------------------------------------
# Caller-side storage formats
# ---------------------------------------------------------------------------------------


def _pow2_ceil_exponent(amax: torch.Tensor, elem_max: float) -> torch.Tensor:
    """Smallest integer e with amax <= elem_max * 2^e (amax > 0), else -127."""
    m, ex = torch.frexp(amax.double() / elem_max)
    e = torch.where(m == 0.5, ex - 1, ex)
    e = torch.where(amax > 0, e, torch.full_like(e, -127))
    return e.clamp(-127, 127).to(torch.int32)


def to_e4m3_blocks(v: torch.Tensor, block: int, fmt: str = "e4m3"):
    """Power-of-two block scales along the last axis, then e4m3 (or e5m2) codes (RNE).
    Returns (codes uint8, exponent int32 [..., n/block])."""
    shp = v.shape
    b = v.float().reshape(*shp[:-1], shp[-1] // block, block)
    top, dt = (448.0, torch.float8_e4m3fn) if fmt == "e4m3" else (57344.0, torch.float8_e5m2)
    e = _pow2_ceil_exponent(b.abs().amax(dim=-1), top)
    scaled = b / torch.ldexp(torch.ones_like(e, dtype=torch.float32), e.float())[..., None]
    codes = scaled.clamp(-top, top).to(dt).view(torch.uint8)
    return codes.reshape(shp), e


_E2M1_MIDPOINTS = (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0)


def to_e2m1_packed(v: torch.Tensor, block: int = 32):
    """UE8M0 block scales (2^ceil(log2(amax/6))) along the last axis, then e2m1 codes by
    round-to-nearest, ties to the even code, packed two per byte (low nibble = even index).
    Returns (packed uint8 [..., n/2], scale bytes uint8 [..., n/block])."""
    shp = v.shape
    b = v.float().reshape(*shp[:-1], shp[-1] // block, block)
    e = _pow2_ceil_exponent(b.abs().amax(dim=-1), 6.0)
    scaled = (b / torch.ldexp(torch.ones_like(e, dtype=torch.float32), e.float())[..., None]).reshape(shp)
    mag = scaled.abs().clamp(max=6.0)
    mids = torch.tensor(_E2M1_MIDPOINTS, device=v.device, dtype=torch.float32)
    code = torch.bucketize(mag, mids, right=False)          # ties go to the lower code
    tie = torch.isin(mag, mids) & (code % 2 == 1)
    code = code + tie.to(code.dtype)                         # ... unless it is odd
    sign = (scaled < 0) & (code != 0)
    nib = (code | (sign.to(code.dtype) << 3)).to(torch.uint8)
    packed = nib[..., 0::2] | (nib[..., 1::2] << 4)
    return packed.contiguous(), (e + 127).to(torch.uint8)


def int8_per_row(v: torch.Tensor):
    """Symmetric per-row int8: s = max|v|/127 (floored at 1e-8), q = round(v/s) in [-127,127]."""
    vf = v.float()
    s = (vf.abs().amax(dim=-1) / 127.0).clamp(min=1e-8)
    q = torch.round(vf / s[..., None]).clamp(-127, 127).to(torch.int8)
    return q.contiguous(), s.float().contiguous()


def int4_per_row_packed(v: torch.Tensor):
    """Symmetric per-row int4: s = max|v|/7 (floored at 1e-8), q = round(v/s) in [-7, 7], packed
    two per byte (element 2j in the low nibble, two's complement). Returns (packed uint8 [..., n/2],
    s float32 [...])."""
    vf = v.float()
    s = (vf.abs().amax(dim=-1) / 7.0).clamp(min=1e-8)
    q = torch.round(vf / s[..., None]).clamp(-7, 7).to(torch.int16) & 0xF
    packed = (q[..., 0::2] | (q[..., 1::2] << 4)).to(torch.uint8)
    return packed.contiguous(), s.float().contiguous()


# ---------------------------------------------------------------------------------------
# A complete set of inputs
# ---------------------------------------------------------------------------------------


def make_inputs(wl: Workload, device="cpu", mode: str | None = None, shared: int = 0):
    """Generate every input of one forward call for workload ``wl`` on ``device``.

    Returns a dict of contiguous tensors: x, x_scale, topk_ids, topk_weights, w1, w1_scale,
    w2, w2_scale (scales are None where the mode has none), and x_bf16, the bf16 activations
    (the input of the path on which the operator quantises x itself). With ``shared`` > 0 the
    weight tensors hold the wl.E routed experts (the same as without) followed by ``shared``
    shared experts drawn from a seed of their own; routing stays over the routed experts."""
    if shared:
        out = make_inputs(wl, device, mode)
        extra = make_inputs(dataclasses.replace(wl, E=shared, K=1, seed=wl.seed + 1000003, zipf_s=None), device, mode)
        for name in ("w1", "w1_scale", "w2", "w2_scale"):
            if out[name] is not None:
                out[name] = torch.cat([out[name], extra[name]]).contiguous()
        return out
    mode = mode or wl.mode
    T, H, I, E, K = wl.T, wl.H, wl.I, wl.E, wl.K
    g = _gen(wl.seed, device)
    ids, gates = routing(T, E, K, g, device, wl.zipf_s, wl.zipf_empty)
    x = torch.randn((T, H), generator=g, device=device, dtype=torch.float32)
    # the bf16 activations, for the path on which the operator quantises x itself
    out = {"topk_ids": ids, "topk_weights": gates, "x_bf16": x.to(torch.bfloat16)}

    # weights are drawn one expert at a time, which keeps the fp32 staging small at full size
    if mode == "a16w16":
        out["x"], out["x_scale"] = x.to(torch.bfloat16), None
        w1 = torch.empty((E, H, 2 * I), device=device, dtype=torch.bfloat16)
        w2 = torch.empty((E, I, H), device=device, dtype=torch.bfloat16)
        for e in range(E):
            w1[e] = (torch.randn((H, 2 * I), generator=g, device=device) * wl.w_std).to(torch.bfloat16)
        for e in range(E):
            w2[e] = (torch.randn((I, H), generator=g, device=device) * wl.w_std).to(torch.bfloat16)
        out.update(w1=w1, w1_scale=None, w2=w2, w2_scale=None)
    elif mode in ("a8w8_fp8", "a8w8_fp8_e5m2"):
        fmt = "e4m3" if mode == "a8w8_fp8" else "e5m2"
        xc, xe = to_e4m3_blocks(x, 32, fmt)
        out["x"], out["x_scale"] = xc, (xe + 127).to(torch.uint8)
        for name, (n_out, k_in) in (("w1", (2 * I, H)), ("w2", (H, I))):
            codes = torch.empty((E, n_out, k_in), device=device, dtype=torch.uint8)
            sc = torch.empty((E, n_out, k_in // 32), device=device, dtype=torch.uint8)
            for e in range(E):
                w = torch.randn((n_out, k_in), generator=g, device=device) * wl.w_std
                c, ex = to_e4m3_blocks(w, 32, fmt)
                codes[e], sc[e] = c, (ex + 127).to(torch.uint8)
            out[name], out[name + "_scale"] = codes, sc
    elif mode == "a8w8_int8":
        out["x"], out["x_scale"] = int8_per_row(x.to(torch.bfloat16))
        for name, (n_out, k_in) in (("w1", (2 * I, H)), ("w2", (H, I))):
            q = torch.empty((E, n_out, k_in), device=device, dtype=torch.int8)
            sc = torch.empty((E, n_out), device=device, dtype=torch.float32)
            for e in range(E):
                w = (torch.randn((n_out, k_in), generator=g, device=device) * wl.w_std).to(torch.bfloat16)
                q[e], sc[e] = int8_per_row(w)  # per output channel: amax over the input dim
            out[name], out[name + "_scale"] = q, sc
    elif mode == "a8w4_int":
        out["x"], out["x_scale"] = int8_per_row(x.to(torch.bfloat16))
        for name, (n_out, k_in) in (("w1", (2 * I, H)), ("w2", (H, I))):
            packed = torch.empty((E, n_out, k_in // 2), device=device, dtype=torch.uint8)
            sc = torch.empty((E, n_out), device=device, dtype=torch.float32)
            for e in range(E):
                w = (torch.randn((n_out, k_in), generator=g, device=device) * wl.w_std).to(torch.bfloat16)
                packed[e], sc[e] = int4_per_row_packed(w)  # per output channel: amax over the input dim
            out[name], out[name + "_scale"] = packed, sc
    elif mode == "a8w4_fp8_fp4":
        xc, xe = to_e4m3_blocks(x, 128)
        out["x"] = xc
        out["x_scale"] = torch.ldexp(torch.ones_like(xe, dtype=torch.float32), xe.float()).contiguous()
        for name, (n_out, k_in) in (("w1", (2 * I, H)), ("w2", (H, I))):
            packed = torch.empty((E, n_out, k_in // 2), device=device, dtype=torch.uint8)
            sc = torch.empty((E, n_out, k_in // 32), device=device, dtype=torch.uint8)
            for e in range(E):
                w = torch.randn((n_out, k_in), generator=g, device=device) * wl.w_std
                packed[e], sc[e] = to_e2m1_packed(w, 32)
            out[name], out[name + "_scale"] = packed, sc
    else:
        raise ValueError(mode)
    return out


def scaled(wl: Workload, **changes) -> Workload:
    """A copy of ``wl`` with some fields changed (smaller parity cases of the same kind)."""
    return dataclasses.replace(wl, **changes)


def to_numpy(inputs: dict) -> dict:
    """Host numpy copies of the stored codes: bf16 tensors become their uint16 bit patterns,
    every other tensor keeps its dtype."""
    out = {}
    for k, v in inputs.items():
        if v is None:
            out[k] = None
        elif v.dtype == torch.bfloat16:
            out[k] = v.detach().cpu().view(torch.int16).numpy().view("uint16")
        else:
            out[k] = v.detach().cpu().numpy()
    return out
