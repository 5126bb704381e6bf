"""Benchmark of the fused MoE expert FFN (route -> dispatch -> L1+SwiGLU -> L2+gate -> combine).

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference] [--workload NAME]

One step = one pass of the whole path (moe_plan, moe_dispatch, moe_expert_l1, moe_expert_l2,
moe_combine -- the sequence moe_forward runs) over one batch of seeded synthetic inputs
already resident in HBM. The default workload is the bf16 Mixtral-like prefill (4096 tokens,
hidden 4096, intermediate 14336, 8 experts, top-2). Its weights (2.82 GB) are larger than the
129 MB L2, so no L2 flush is needed between steps.

Prints one JSON line (rank 0). value = TFLOP/s of algorithmic work (6*H*I per routed row)
summed over ranks; under torchrun every rank runs an independent replica (weak scaling, no
collective on the data path). `--impl reference` times the CPU oracle (float64 numpy) on the
host cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused MoE FFN TFLOP/s + routed rows/s, % of tensor/HBM roofline, 1xGB300"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
DTYPE = {"a16w16": "bf16", "a8w8_fp8": "e4m3", "a8w8_int8": "int8", "a8w4_fp8_fp4": "e4m3xe2m1", "a8w4_int": "int8xint4", "a8w8_fp8_e5m2": "e5m2"}
LAUNCHES_PER_STEP = {"a16w16": 7, "a8w8_fp8": 7, "a8w8_int8": 8, "a8w4_fp8_fp4": 7, "a8w4_int": 8, "a8w8_fp8_e5m2": 7}
# launches the fused launch replaces: A16W16 runs L1, L2 and the combine in it, the FP8 modes L1 and L2,
# the integer modes L1, the re-quantisation of A and L2
FUSED_SAVES = {"a16w16": 2, "a8w8_int8": 2, "a8w4_int": 2}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="mixtral_bf16_prefill")
    ap.add_argument("--flags", type=int, default=0,
                    help="GEMM stage flags, MOE_FLAG_* of the C ABI: 1 CUDA-core reference kernels, 2 weight-major "
                         "tiles (FP8 modes at prefill sizes; A8W4-INT at any tile count), 16 one-CTA bf16 L2, "
                         "32 bf16 L1 on CTA pairs, 64 token-major A8W4-INT")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--configs", default="all", choices=["all", "none"],
                    help="all: also time the method's other configurations in the same run (each in the line's "
                         "'configs' object); none: the selected workload only")
    ap.add_argument("--no-probe", action="store_true", help="skip the tensor-core peak probe")
    ap.add_argument("--tokens", type=int, default=None, help="override the workload's token count")
    ap.add_argument("--experts", type=int, default=None, help="override the workload's expert count")
    ap.add_argument("--fused", action="store_true",
                    help="S3-S5 in one launch (moe_expert_ffn; MOE_FLAG_FUSED end to end); A16W16 and FP8 modes")
    ap.add_argument("--quantize-x", action="store_true",
                    help="bf16 x in, quantised by the dispatch stage as the mode prescribes (MOE_FLAG_QUANTIZE_X)")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return FALLBACK_PEAKS, "fallback"


L2_BYTES = 126 * 2**20  # the GPU's L2 (an input set above it leaves nothing of a step in L2 for the next)


def resident_input_bytes(wl):
    """Bytes of one step's resident inputs: W1 and W2 of every expert (with their scales) and x."""
    w = 3 * wl.E * wl.H * wl.I * WEIGHT_BYTES_PER_ELEM[wl.mode]
    return w + wl.T * wl.H * X_BYTES_PER_ELEM[wl.mode]


def workload_config(wl, quantize_x=False, fused=False, flags=0):
    big = resident_input_bytes(wl) > L2_BYTES
    cfg = {"workload": wl.name, "mode": wl.mode, "tokens": wl.T, "hidden": wl.H, "intermediate": wl.I,
           "experts": wl.E, "topk": wl.K, "routed_rows": wl.routed_rows, "seed": wl.seed,
           "l2_policy": "inputs larger than L2 (no flush)" if big else
                        "inputs fit in L2 (no flush): a warm-cache timing, not a benchmark figure"}
    if quantize_x:
        cfg["x_input"] = "bf16, quantised by the dispatch stage"
    if fused:
        cfg["gemm_launch"] = ("L1, L2 and the combine in one cooperative launch (moe_expert_ffn)" if wl.mode == "a16w16"
                              else "L1 and L2 in one cooperative launch, the combine after it (moe_expert_ffn)")
    if flags & 128:  # MOE_FLAG_PREPARED_WEIGHTS
        cfg["weights"] = ("prepared once, untimed, by moe_prepare_weights: every int8 code as its exact f16 value "
                          "(2 bytes per weight in HBM; MOE_FLAG_PREPARED_WEIGHTS)")
    elif wl.mode == "a8w8_int8":
        cfg["weights"] = "int8 in HBM, expanded to f16 in shared memory by the GEMM"
    if flags & ~128:
        cfg["flags"] = flags & ~128
    return cfg


# ---------------------------------------------------------------------------------------
# CPU oracle (the reference arm and the cpu_baseline leg)
# ---------------------------------------------------------------------------------------


def oracle_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var):
            return int(os.environ[var])
    return os.cpu_count() or 1


def oracle_sample(wl, inp_host, n_tokens, seed, quantize_x=False):
    """Run the oracle, as it stands, on a seeded sample of n_tokens tokens; returns
    (seconds, routed rows computed). With quantize_x the sampled bf16 rows are quantised by the
    oracle first (the quantisation is per token, so a sample is exact)."""
    import numpy as np
    from oracle import moe as omoe
    rng = np.random.default_rng(seed)
    tokens = np.sort(rng.choice(wl.T, size=n_tokens, replace=False))
    h = inp_host
    ids = h["topk_ids"][tokens]
    t0 = time.perf_counter()
    if quantize_x:
        x, xs = omoe.quantize_x(wl.mode, h["x_bf16"][tokens])
    else:
        x, xs = h["x"][tokens], None if h["x_scale"] is None else h["x_scale"][tokens]
    omoe.forward(wl.mode, x, xs, ids, h["topk_weights"][tokens], h["w1"], h["w1_scale"], h["w2"],
                 h["w2_scale"], num_experts=wl.E, inter=wl.I)
    dt = time.perf_counter() - t0
    return dt, int((ids >= 0).sum())


def sample_tokens_for(wl, h, seconds, quantize_x=False, seed=5):
    """Tokens per oracle sample for about `seconds` of oracle time (at least 1, at most the
    workload's tokens). The oracle's time is close to a + b*n for n tokens (a: decoding the
    touched experts' weights, b: the per-token rows), so two probes fix a and b."""
    n1, n2 = 1, min(8, wl.T)
    t1, _ = oracle_sample(wl, h, n1, seed=seed, quantize_x=quantize_x)
    t2, _ = oracle_sample(wl, h, n2, seed=seed + 1, quantize_x=quantize_x)
    b = max((t2 - t1) / max(n2 - n1, 1), 1e-4)
    a = max(t1 - b * n1, 0.0)
    return int(max(1, min(wl.T, (seconds - a) / b)))


# whole reference-arm run (warm-up + timed steps): about this many seconds of oracle time
REFERENCE_RUN_SECONDS = 150.0
# the cpu_baseline leg of the GB300 arm: one sample of about this many seconds
CPU_BASELINE_SECONDS = 12.0


def host_inputs(wl):
    from workloads import make_inputs, to_numpy
    import torch
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    return to_numpy(make_inputs(wl, device=dev))


def run_reference(args, wl, rank, world):
    if rank != 0:
        return None
    h = host_inputs(wl)
    n_tok = sample_tokens_for(wl, h, REFERENCE_RUN_SECONDS / max(args.steps + args.warmup, 1),
                              quantize_x=args.quantize_x)
    for w in range(args.warmup):
        oracle_sample(wl, h, n_tok, seed=1000 + w, quantize_x=args.quantize_x)
    total_t, total_rows = 0.0, 0
    for s in range(args.steps):
        dt, rows = oracle_sample(wl, h, n_tok, seed=2000 + s, quantize_x=args.quantize_x)
        total_t += dt
        total_rows += rows
    flops = 6.0 * wl.H * wl.I * total_rows
    value = flops / total_t / 1e12
    cores = oracle_threads()
    sample = f"{n_tok} seeded tokens per step ({total_rows / args.steps:.0f} routed rows), float64 numpy oracle"
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(wl, args.quantize_x, args.fused), "routed_rows_per_s": total_rows / total_t,
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ---------------------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------------------

CLOCK_FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    """nvidia-smi samples every 50 ms while the context is open; summary() keeps the samples
    taken between mark_start() and mark_end() (the timed region)."""

    def __init__(self, gpu_index):
        self.proc = None
        self.gpu_index = gpu_index
        self.out = os.path.join("/tmp", f"moe_clocks_{os.getpid()}.csv")
        self.t_start = self.t_end = None

    def mark_start(self):
        self.t_start = time.time()

    def mark_end(self):
        self.t_end = time.time()

    def __enter__(self):
        try:
            self.f = open(self.out, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={CLOCK_FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        import datetime
        if self.proc is None or not os.path.exists(self.out):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.out):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 10 and parts[2].replace(".", "").isdigit():
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                except ValueError:
                    ts = None
                rows.append((ts, parts[1:]))
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        inside = [r for ts, r in rows if ts is not None and self.t_start is not None and
                  self.t_start <= ts <= self.t_end]
        use = inside or [r for _, r in rows]
        sm = [float(r[1]) for r in use]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i in range(4) if r[5 + i].lower() == "active"})
        power = [float(r[3]) for r in use if r[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(use[0][2]), "reasons": reasons,
                "samples_in_timed_region": len(inside), "samples": len(use),
                "power_w_median": statistics.median(power) if power else None}


# ---------------------------------------------------------------------------------------
# the GB300 arm
# ---------------------------------------------------------------------------------------


def dominant_kernel_traffic(workload, prefix="l1_gemm"):
    """DRAM bytes per launch of the dominant kernel from the committed ncu summary of this
    workload, valid only while the kernel sources the counters were taken on are unchanged (the
    summary lists them and their sha256)."""
    path = os.path.join(ROOT, "profiles", f"{prefix}_{workload}.md")
    if not os.path.exists(path):
        return None
    txt = open(path).read()
    m = re.search(r"traffic_bytes_per_launch:\s*(\d+)", txt)
    h = re.search(r"source_sha256:\s*([0-9a-f]{64})", txt)
    f = re.search(r"source_files:\s*(.+)", txt)
    if not m or not h or not f:
        return None
    return int(m.group(1)) if h.group(1) == kernel_source_hash(f.group(1).split()) else None


def kernel_source_hash(files):
    """sha256 over the given files of the CUDA sources, in order."""
    d = os.path.join(ROOT, "moe_expert_ffn_topk_gb300", "csrc")
    sha = hashlib.sha256()
    for name in files:
        sha.update(open(os.path.join(d, name), "rb").read())
    return sha.hexdigest()


def max_over_ranks(x: float, world: int, device) -> float:
    """The largest value over all ranks (the slowest rank's time); identity on one rank."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_step: float, steps: int, elapsed_ms: float, world: int) -> float:
    """Replicas: every rank runs the full step, so the job did world * steps steps in the
    slowest rank's time."""
    return world * flops_per_step * steps / (elapsed_ms * 1e-3) / 1e12


WEIGHT_BYTES_PER_ELEM = {"a16w16": 2.0, "a8w8_fp8": 1.0 + 1 / 32, "a8w8_int8": 1.0, "a8w4_fp8_fp4": 0.5 + 1 / 32,
                         "a8w4_int": 0.5, "a8w8_fp8_e5m2": 1.0 + 1 / 32}
X_BYTES_PER_ELEM = {"a16w16": 2.0, "a8w8_fp8": 1.0 + 1 / 32, "a8w8_int8": 1.0, "a8w4_fp8_fp4": 1.0 + 4 / 128,
                    "a8w4_int": 1.0, "a8w8_fp8_e5m2": 1.0 + 1 / 32}


def is_decode(wl) -> bool:
    """Few routed rows per expert: the step streams the weights (HBM-bound)."""
    return wl.routed_rows / wl.E < 64


# The tcgen05 instruction kind each mode's GEMMs issue (include/moe_peak.h) and how many of its MACs
# one algorithmic MAC costs: the INT8 GEMM runs every int8 product as two exact f16 products (the
# hi/lo split of the tokens), A8W4-INT and the float modes one.
TENSOR_KIND = {"a16w16": ("bf16", 1), "a8w8_fp8": ("e4m3_e4m3", 1), "a8w8_fp8_e5m2": ("e4m3_e4m3", 1),
               "a8w4_fp8_fp4": ("e4m3_e2m1", 1), "a8w8_int8": ("f16", 2), "a8w4_int": ("f16", 1)}
PROBE_ITERS = 20000  # about 5 ms of MMA work per CTA at 1.9 GHz


def measure_tensor_peaks(moe, dev, kinds, sustained_s=0.0, repeats=3):
    """The dense rate of each tcgen05 kind in `kinds`, from the library's probe (one CTA per SM issuing
    back-to-back MMAs on shared-memory operands), timed with events on the launching stream. Burst: the
    best of `repeats` single launches per kind, the kinds interleaved (each after a warm-up launch), with
    the SM clock that CTA 0 measured during the launch (cycles over %globaltimer nanoseconds). With
    sustained_s > 0 also back-to-back launches for that long (under the power cap). TFLOP/s."""
    import torch
    stream = torch.cuda.current_stream()
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    out = {k: {"burst_tflops": 0.0} for k in kinds}
    with ClockSampler(dev.index or 0) as clocks:
        clocks.mark_start()
        for _ in range(repeats):
            for kind in kinds:
                moe.moe_tensor_peak_probe(kind, PROBE_ITERS // 10, ws, stream=stream)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                flops = moe.moe_tensor_peak_probe(kind, PROBE_ITERS, ws, stream=stream)
                e1.record(stream)
                torch.cuda.synchronize()
                cycles, ns = ws[128:144].view(torch.int64).tolist()  # CTA 0's SM cycles and nanoseconds
                tflops = flops / (e0.elapsed_time(e1) * 1e-3) / 1e12
                if tflops > out[kind]["burst_tflops"]:
                    out[kind] = {"burst_tflops": tflops, "sm_mhz": 1e3 * cycles / max(ns, 1),
                                 "flops_per_sm_cycle": flops / max(cycles * n_sm, 1)}
        if sustained_s > 0:
            for kind in kinds:
                total, n = 0.0, 0
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                t_end = time.time() + sustained_s
                while time.time() < t_end:
                    total += moe.moe_tensor_peak_probe(kind, PROBE_ITERS, ws, stream=stream)
                    n += 1
                    if n % 8 == 0:
                        torch.cuda.synchronize()  # keep the queue short so the loop lasts sustained_s
                e1.record(stream)
                torch.cuda.synchronize()
                out[kind]["sustained_tflops"] = total / (e0.elapsed_time(e1) * 1e-3) / 1e12
        clocks.mark_end()
    st = moe.moe_check_device_error(ws)
    if st != 0:
        raise RuntimeError(f"tensor peak probe: {moe.moe_status_string(st)}")
    out["clocks"] = clocks.summary()
    out["how"] = (f"moe_tensor_peak_probe: one CTA per SM, {PROBE_ITERS} x 4 dense MMAs (M 128, N 256) per CTA on "
                  f"shared-memory operands, CUDA events; burst = best of {repeats} launches per kind (interleaved, "
                  "each after a warm-up launch); sm_mhz = CTA 0's clock64 cycles over %globaltimer ns")
    return out


def tensor_peak(wl, pk, pk_src, probe, sustained):
    """The peak of the tensor pipe a mode's GEMMs use, in algorithmic TFLOP/s (or TOP/s): the bf16
    modes take the measured cuBLAS bf16 figure; the others the probe's measured rate of their
    own instruction kind, divided by the MACs each algorithmic MAC costs (2 for the hi/lo INT8 split)."""
    clock = "sustained" if sustained else "burst"
    kind, cost = TENSOR_KIND[wl.mode]
    if kind == "bf16":
        return float(pk["bf16_tflops_sustained" if sustained else "bf16_tflops"]), f"{pk_src} bf16 dense (cuBLAS), {clock}"
    rec = probe.get(kind, {}) if probe else {}
    key = "sustained_tflops" if sustained and "sustained_tflops" in rec else "burst_tflops"
    if key in rec:
        src = f"measured tcgen05 {kind} dense rate (moe_tensor_peak_probe, {key.split('_')[0]})"
        if cost != 1:
            src += f" / {cost} (each int8 MAC runs as {cost} exact f16 MACs)"
        return rec[key] / cost, src
    # no probe: the bf16 measurement times the nominal dense ratio of the kind
    ratio = 2.0 if kind.startswith("e4m3") else 1.0
    bf = float(pk["bf16_tflops_sustained" if sustained else "bf16_tflops"])
    return bf * ratio / cost, f"{pk_src} bf16 dense ({clock}) x nominal {kind}/bf16 ratio {ratio} / {cost}"


def touched_weight_bytes(wl, inp):
    """W1 and W2 (with their scales) of every expert with N_e > 0, and the number of such experts."""
    import numpy as np
    ids = inp["topk_ids"].cpu().numpy().reshape(-1)
    touched = len(np.unique(ids[ids >= 0]))
    return touched * 3 * wl.I * wl.H * WEIGHT_BYTES_PER_ELEM[wl.mode], touched


def l1_roofline(wl, inp, l1_ms, pk, pk_src, probe, sustained):
    """Roofline of the dominant kernel, the L1 grouped GEMM (2/3 of the flops and of the weight
    bytes). Tensor-bound workloads: algorithmic flops 4*H*I per routed row against the dense peak of
    the mode's tensor pipe (tensor_peak). Weight-streaming (decode) workloads: algorithmic bytes = W1
    (+ block scales) of every expert with N_e > 0 plus the x rows, against the measured HBM copy
    bandwidth."""
    if is_decode(wl):
        w_bytes, touched = touched_weight_bytes(wl, inp)
        nbytes = w_bytes * 2 / 3 + wl.T * wl.H * X_BYTES_PER_ELEM[wl.mode]
        achieved = nbytes / (l1_ms * 1e-3) / 1e9
        peak = float(pk["hbm_gbs"])
        return {"bound": "hbm", "kernel": "L1 grouped GEMM + SwiGLU (moe_expert_l1)", "achieved": achieved,
                "peak": peak, "unit": "GB/s", "frac": achieved / peak, "peak_source": f"{pk_src} HBM copy",
                "l1_ms": l1_ms, "algorithmic_bytes": nbytes, "experts_touched": touched,
                "traffic": dominant_kernel_traffic(wl.name)}
    l1_flops = 4.0 * wl.H * wl.I * wl.routed_rows
    achieved = l1_flops / (l1_ms * 1e-3) / 1e12
    peak, src = tensor_peak(wl, pk, pk_src, probe, sustained)
    return {"bound": "tensor", "kernel": "L1 grouped GEMM + SwiGLU (moe_expert_l1)", "achieved": achieved,
            "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak, "peak_source": src, "l1_ms": l1_ms,
            "algorithmic_flops": l1_flops, "traffic": dominant_kernel_traffic(wl.name)}


def step_roofline(wl, inp, step_ms, pk, pk_src, probe, sustained):
    """The whole step against the roofline that bounds it: for decode, every algorithmic byte (touched
    W1 + W2 with scales, x, ids, gates, y) against the HBM copy bandwidth; otherwise 6*H*I flops per
    routed row against the mode's tensor peak."""
    if is_decode(wl):
        w_bytes, touched = touched_weight_bytes(wl, inp)
        nbytes = (w_bytes + wl.T * wl.H * X_BYTES_PER_ELEM[wl.mode] + wl.T * wl.K * 8 + wl.T * wl.H * 2)
        achieved = nbytes / (step_ms * 1e-3) / 1e9
        peak = float(pk["hbm_gbs"])
        return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "peak_source": f"{pk_src} HBM copy", "algorithmic_bytes": nbytes, "experts_touched": touched,
                "step_ms": step_ms}
    achieved = wl.flops / (step_ms * 1e-3) / 1e12
    peak, src = tensor_peak(wl, pk, pk_src, probe, sustained)
    return {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
            "peak_source": src, "step_ms": step_ms}


def fused_roofline(wl, inp, ffn_ms, pk, pk_src, probe, sustained):
    """Roofline of the fused launch (moe_expert_ffn: L1 + SwiGLU + L2 + gate, and for A16W16 the combine).
    Weight-streaming (decode) workloads: algorithmic bytes = W1 + W2 (+ block scales) of every expert with
    N_e > 0, the x rows read and the bf16 combine rows written, against the measured HBM copy bandwidth.
    Otherwise algorithmic flops 6*H*I per routed row against the dense peak of the mode's tensor pipe."""
    kernel = ("L1 + SwiGLU + L2 + gate + combine in one launch (moe_expert_ffn)" if wl.mode == "a16w16"
              else "L1 + SwiGLU + L2 + gate in one launch (moe_expert_ffn; the combine is a second launch)")
    if is_decode(wl):
        w_bytes, touched = touched_weight_bytes(wl, inp)
        nbytes = w_bytes + wl.T * wl.H * X_BYTES_PER_ELEM[wl.mode] + wl.routed_rows * wl.H * 2
        achieved = nbytes / (ffn_ms * 1e-3) / 1e9
        peak = float(pk["hbm_gbs"])
        return {"bound": "hbm", "kernel": kernel, "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "peak_source": f"{pk_src} HBM copy", "ffn_ms": ffn_ms,
                "algorithmic_bytes": nbytes, "experts_touched": touched,
                "traffic": dominant_kernel_traffic(wl.name, "ffn_fused")}
    flops = 6.0 * wl.H * wl.I * wl.routed_rows
    achieved = flops / (ffn_ms * 1e-3) / 1e12
    peak, src = tensor_peak(wl, pk, pk_src, probe, sustained)
    return {"bound": "tensor", "kernel": kernel, "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
            "frac": achieved / peak, "peak_source": src, "ffn_ms": ffn_ms, "algorithmic_flops": flops,
            "traffic": dominant_kernel_traffic(wl.name, "ffn_fused")}


def measure_workload(args, wl, world, local_rank, fused=False, quantize_x=False, flags=0):
    """Times args.steps steps of one workload (after args.warmup) through the C ABI with inputs resident
    in HBM, then the same metric end to end with host buffers twice: copies overlapped with the
    neighbouring steps on two copy streams, and serial (copy in, forward, copy out on one stream).
    Returns the raw measurements of rank 0 (None on other ranks) and the inputs."""
    import torch
    import torch.distributed as dist

    import moe_expert_ffn_topk_gb300 as moe
    from workloads import make_inputs

    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.current_stream()
    inp = make_inputs(wl, device=dev)
    d = moe.dims(wl.T, wl.H, wl.I, wl.E, wl.K)
    w1, w2 = inp["w1"], inp["w2"]  # the GEMMs' weight operands (inp keeps the stored codes for the oracle)
    if flags & moe.MOE_FLAG_PREPARED_WEIGHTS:
        # one-time weight preparation (exact f16 codes of the int8 weights), before and outside every timed region
        w1 = moe.moe_prepare_weights(inp["w1"], d, wl.mode, 1)
        w2 = moe.moe_prepare_weights(inp["w2"], d, wl.mode, 2)
        torch.cuda.synchronize()
    ws = moe.alloc_workspace(d, wl.mode, dev)
    y = torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device=dev)
    fwd_flags = flags | (moe.MOE_FLAG_QUANTIZE_X if quantize_x else 0) | (moe.MOE_FLAG_FUSED if fused else 0)

    def step(ev_l1=None):
        moe.moe_plan(inp["topk_ids"], d, ws, stream=stream)
        if quantize_x:
            moe.moe_dispatch_quantize(inp["x_bf16"], d, wl.mode, ws, stream=stream)
        else:
            moe.moe_dispatch(inp["x"], inp["x_scale"], d, wl.mode, ws, stream=stream)
        if ev_l1:
            ev_l1[0].record(stream)
        if fused:  # the events bracket the one launch of S3-S6
            moe.moe_expert_ffn(w1, inp["w1_scale"], w2, inp["w2_scale"], inp["topk_weights"], d, wl.mode,
                               ws, y=y, stream=stream)
            if ev_l1:
                ev_l1[1].record(stream)
            return
        moe.moe_expert_l1(w1, inp["w1_scale"], d, wl.mode, ws, flags, stream=stream)
        if ev_l1:
            ev_l1[1].record(stream)
        moe.moe_expert_l2(w2, inp["w2_scale"], inp["topk_weights"], d, wl.mode, ws, flags, stream=stream)
        moe.moe_combine(y, d, ws, stream=stream)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        step()
    st = moe.moe_check_device_error(ws)
    if st != 0:
        raise RuntimeError(f"{wl.name}: device error during warm-up: {moe.moe_status_string(st)}")

    l1_events = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                 for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clocks:
        barrier()
        clocks.mark_start()
        t0.record(stream)
        for i in range(args.steps):
            step(l1_events[i])
        t1.record(stream)
        barrier()
        clocks.mark_end()
    elapsed_ms = t0.elapsed_time(t1)
    l1_ms = statistics.mean(a.elapsed_time(b) for a, b in l1_events)
    st = moe.moe_check_device_error(ws)
    if st != 0:
        raise RuntimeError(f"{wl.name}: device error in the timed region: {moe.moe_status_string(st)}")
    elapsed_ms = max_over_ranks(elapsed_ms, world, dev)

    # end to end through the public API with host buffers: every step copies its inputs from pinned host
    # memory, calls moe_forward and copies y back to pinned host memory
    x_keys = ("x_bf16",) if quantize_x else ("x", "x_scale")
    host_in = {k: inp[k].cpu().pin_memory() for k in x_keys + ("topk_ids", "topk_weights") if inp[k] is not None}
    dev_in = [{k: torch.empty_like(v, device=dev) for k, v in host_in.items()} for _ in range(2)]
    y_dev = [y, torch.empty_like(y)]
    y_host = [torch.empty(y.shape, dtype=y.dtype).pin_memory() for _ in range(2)]
    h2d = sum(v.numel() * v.element_size() for v in host_in.values())
    d2h = y_host[0].numel() * y_host[0].element_size()

    def forward(di, yd):
        moe.moe_forward(di["x_bf16"] if quantize_x else di["x"], di.get("x_scale"), di["topk_ids"], di["topk_weights"],
                        w1, inp["w1_scale"], w2, inp["w2_scale"], yd, d, wl.mode, ws, fwd_flags,
                        stream=stream)

    # (a) overlapped: the input and the output copies run on two more streams with double-buffered
    # device inputs and outputs, so step i+1's input copy and step i-1's y copy overlap step i's compute
    # (events order each buffer's use), as a serving loop would run
    in_stream, out_stream = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev = lambda: torch.cuda.Event()  # noqa: E731
    in_ready, fwd_done, out_read = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    state = {"i": 0}

    def e2e_step():
        b = state["i"] & 1
        state["i"] += 1
        with torch.cuda.stream(in_stream):
            in_stream.wait_event(fwd_done[b])  # the forward two steps back has read dev_in[b]
            for k, v in host_in.items():
                dev_in[b][k].copy_(v, non_blocking=True)
            in_ready[b].record(in_stream)
        stream.wait_event(in_ready[b])
        stream.wait_event(out_read[b])  # y_dev[b] of two steps back has been copied out
        forward(dev_in[b], y_dev[b])
        fwd_done[b].record(stream)
        with torch.cuda.stream(out_stream):
            out_stream.wait_event(fwd_done[b])
            y_host[b].copy_(y_dev[b], non_blocking=True)
            out_read[b].record(out_stream)

    for e in fwd_done + out_read:
        e.record(stream)
    for _ in range(max(1, args.warmup)):
        e2e_step()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    stream.wait_stream(in_stream)
    stream.wait_stream(out_stream)
    barrier()
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    stream.wait_stream(out_stream)  # the last step's y has reached the host buffer
    e1.record(stream)
    barrier()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)

    # (b) serial: copy in, forward, copy out, one after the other on one stream (a call that cannot
    # be overlapped with its neighbours)
    def serial_step():
        for k, v in host_in.items():
            dev_in[0][k].copy_(v, non_blocking=True)
        forward(dev_in[0], y_dev[0])
        y_host[0].copy_(y_dev[0], non_blocking=True)

    for _ in range(max(1, args.warmup)):
        serial_step()
    barrier()
    e0.record(stream)
    for _ in range(args.steps):
        serial_step()
    e1.record(stream)
    barrier()
    serial_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    st = moe.moe_check_device_error(ws)
    if st != 0:
        raise RuntimeError(f"{wl.name}: device error in the end-to-end runs: {moe.moe_status_string(st)}")
    res = {"elapsed_ms": elapsed_ms, "l1_ms": l1_ms, "e2e_ms": e2e_ms, "serial_ms": serial_ms, "h2d": h2d,
           "d2h": d2h, "clocks": clocks.summary()}
    del ws, y, y_dev, dev_in, w1, w2
    return res, inp


def cpu_baseline(wl, inp, seconds, quantize_x=False):
    """The oracle, as it stands, on one seeded sample of whole tokens sized to about `seconds` on the host
    cores; re-sized up to four times if it came out short (the oracle's fixed cost grows with the experts a
    sample touches, so the two-probe fit can come out short)."""
    from workloads import to_numpy
    h = to_numpy(inp)
    n_tok = sample_tokens_for(wl, h, seconds, quantize_x=quantize_x)
    for attempt in range(5):
        dt, rows = oracle_sample(wl, h, n_tok, seed=7 + attempt, quantize_x=quantize_x)
        if dt >= 0.6 * seconds or n_tok >= wl.T or attempt == 4:
            break
        n_tok = int(min(wl.T, max(n_tok + 1, n_tok * seconds / max(dt, 1e-3))))
    return {"value": 6.0 * wl.H * wl.I * rows / dt / 1e12, "unit": "TFLOP/s", "cores": oracle_threads(),
            "kind": "oracle", "sample": f"{n_tok} seeded tokens ({rows} routed rows) of {wl.name}, {dt:.1f} s, "
                                        f"float64 numpy oracle"}


def is_sustained(res):
    """The sustained (power-capped) peak when the GPU was at its power cap during the timed region, or
    the region lasted a second or more; the burst peak for a short, uncapped one."""
    return res["elapsed_ms"] >= 1000.0 or "sw_power_cap" in (res["clocks"].get("reasons") or [])


def result_fields(args, wl, res, inp, world, pk, pk_src, probe, fused, quantize_x, flags=0):
    """The per-workload measurements of the JSON line (rank 0)."""
    flops = float(wl.flops)
    ms_per_step = res["elapsed_ms"] / args.steps
    sustained = is_sustained(res)
    roof = (fused_roofline(wl, inp, res["l1_ms"], pk, pk_src, probe, sustained) if fused
            else l1_roofline(wl, inp, res["l1_ms"], pk, pk_src, probe, sustained))
    return {
        "value": whole_job_tflops(flops, args.steps, res["elapsed_ms"], world), "unit": "TFLOP/s",
        "ms_per_step": ms_per_step, "dtype": DTYPE[wl.mode], "config": workload_config(wl, quantize_x, fused, flags),
        "routed_rows_per_s": world * wl.routed_rows * args.steps / (res["elapsed_ms"] * 1e-3),
        "roofline": roof,
        "step_roofline": step_roofline(wl, inp, ms_per_step, pk, pk_src, probe, sustained),
        "e2e": {"value": whole_job_tflops(flops, args.steps, res["e2e_ms"], world), "unit": "TFLOP/s",
                "h2d_bytes_per_step": res["h2d"], "d2h_bytes_per_step": res["d2h"],
                "ms_per_step": res["e2e_ms"] / args.steps,
                "copies": "overlapped: each step's input copy and the previous step's y copy run on two more "
                          "streams beside the forward (double-buffered)",
                "serial": {"value": whole_job_tflops(flops, args.steps, res["serial_ms"], world), "unit": "TFLOP/s",
                           "ms_per_step": res["serial_ms"] / args.steps,
                           "copies": "copy in, moe_forward, copy out, one after the other on one stream"}},
        "gpu_launches": (LAUNCHES_PER_STEP[wl.mode] - (FUSED_SAVES.get(wl.mode, 1) if fused else 0)) * args.steps,
        "clocks": res["clocks"],
    }


# the other configurations of the method's benchmark, measured in the same run (each with the same steps
# and warm-up): (workload, GEMM flags, key in the line's "configs"), and the oracle's sample length for
# their cpu_baseline. A8W8-INT runs on its int8 weights and, for comparison, on weights prepared once as
# exact f16 codes (MOE_FLAG_PREPARED_WEIGHTS = 128; no cpu_baseline of its own: the same oracle sample).
# FP8 x FP4 decode and the integer modes also run L1 and L2 in one cooperative launch (MOE_FLAG_FUSED = 8,
# through moe_expert_ffn).
OTHER_CONFIGS = (("tiny_bf16", 0, "tiny_bf16"), ("dsv3_fp8fp4_decode", 0, "dsv3_fp8fp4_decode"),
                 ("dsv3_fp8fp4_decode", 8, "dsv3_fp8fp4_decode[fused L1+L2 launch]"),
                 ("dsv3_fp8fp4_prefill_zipf", 0, "dsv3_fp8fp4_prefill_zipf"), ("int8_a8w8", 0, "int8_a8w8"),
                 ("int8_a8w8", 128, "int8_a8w8[prepared f16 weights]"),
                 ("int8_a8w8", 8, "int8_a8w8[fused L1+L2 launch]"), ("int4_a8w4", 0, "int4_a8w4"),
                 ("int4_a8w4", 8, "int4_a8w4[fused L1+L2 launch]"))
FLAG_FUSED = 8
OTHER_CPU_SECONDS = 4.0


def run_gb300(args, wl, rank, world, local_rank):
    import torch

    import moe_expert_ffn_topk_gb300 as moe

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    runs = [(wl, args.fused, args.quantize_x, args.flags, wl.name, True)]
    if args.configs == "all":
        from workloads import WORKLOADS
        runs += [(WORKLOADS[n], bool(f & FLAG_FUSED), False, f & ~FLAG_FUSED, key, not key.endswith("]"))
                 for n, f, key in OTHER_CONFIGS if key != wl.name]
    measured, failed = [], {}
    for i, (w, fused, qx, flags, key, want_cpu) in enumerate(runs):
        try:
            res, inp = measure_workload(args, w, world, local_rank, fused, qx, flags)
            cpu = None
            if rank == 0 and want_cpu and not args.no_cpu_baseline:
                cpu = cpu_baseline(w, inp, CPU_BASELINE_SECONDS if w is wl else OTHER_CPU_SECONDS, qx)
        except Exception as exc:  # an extra configuration that fails is reported, not fatal
            if i == 0:
                raise
            failed[key] = {"error": f"{type(exc).__name__}: {exc}"[:500]}
            torch.cuda.synchronize()
            continue
        ids = inp["topk_ids"].cpu()
        measured.append((w, fused, qx, flags, key, res, {"topk_ids": ids}, cpu))
        del inp
        torch.cuda.empty_cache()
    # the peaks of the tensor pipes the measured modes use, after every timed region (so that the probes'
    # heat and power do not touch the measurements)
    kinds = ["bf16", "f16", "e4m3_e2m1", "e4m3_e4m3"]  # every kind the GEMM stages issue
    sustained_s = 2.0 if any(is_sustained(m[5]) for m in measured) else 0.0
    probe = measure_tensor_peaks(moe, dev, kinds, sustained_s) if not args.no_probe else None
    if rank != 0:
        return None
    pk, pk_src = peaks()
    lines = []
    for w, fused, qx, flags, key, res, inp, cpu in measured:
        f = result_fields(args, w, res, inp, world, pk, pk_src, probe, fused, qx, flags)
        if cpu is not None:
            f["cpu_baseline"] = cpu
        lines.append((key, f))
    head = lines[0][1]
    line = {"metric": METRIC, "value": head["value"], "unit": head["unit"], "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": head["dtype"], "data": "synthetic (seeded; random-init weights)"}
    line.update({k: v for k, v in head.items() if k not in line})
    # gpu_launches counts the library kernels of the headline's timed region; each entry of "configs"
    # counts those of its own timed region
    if len(lines) > 1 or failed:
        line["configs"] = {key: f for key, f in lines[1:]}
        line["configs"].update(failed)
    if probe:
        line["tensor_peaks"] = probe
    return line


def main():
    args = parse()
    from workloads import WORKLOADS, scaled
    wl = WORKLOADS[args.workload]
    if args.tokens is not None or args.experts is not None:
        wl = scaled(wl, name=f"{wl.name}[T={args.tokens or wl.T},E={args.experts or wl.E}]",
                    T=args.tokens or wl.T, E=args.experts or wl.E)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        line = run_reference(args, wl, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    line = run_gb300(args, wl, rank, world, local_rank)
    if line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
