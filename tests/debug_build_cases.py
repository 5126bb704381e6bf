"""Small parity cases run through the bounds-checking build of the library (-DMOE_DEBUG; loaded when
MOE_GB300_DEBUG=1). Run as its own process by test_debug_build.py: every case must leave the error
word clear (no index check failed) and match the oracle within the mode's bound."""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

import torch  # noqa: E402

from gpu_util import assert_close, run_forward, y_numpy  # noqa: E402
from oracle import moe as omoe  # noqa: E402
from workloads import Workload, make_inputs, to_numpy  # noqa: E402

CASES = [Workload("dbg_bf16", "a16w16", 300, 512, 384, 6, 2, 71, 0.05),
         Workload("dbg_fp8", "a8w8_fp8", 200, 512, 384, 6, 2, 72, 0.05),
         Workload("dbg_int8", "a8w8_int8", 300, 512, 384, 6, 3, 73, 0.05),
         Workload("dbg_fp4", "a8w4_fp8_fp4", 257, 256, 256, 64, 8, 74, 0.05, zipf_s=1.2, zipf_empty=8),
         Workload("dbg_w4", "a8w4_int", 300, 512, 384, 6, 3, 75, 0.05),
         Workload("dbg_e5m2", "a8w8_fp8_e5m2", 200, 512, 384, 6, 2, 76, 0.05)]


def main():
    import moe_expert_ffn_topk_gb300 as moe
    assert os.path.basename(moe._binding._LIB_PATH) == "libmoe_gb300_debug.so"
    n = 0
    for wl in CASES:
        for flags in (0, moe.MOE_FLAG_SIMT):
            inp = make_inputs(wl, device="cuda")
            inp["topk_ids"] = inp["topk_ids"].clone()
            inp["topk_ids"][::7, 0] = -1  # masked routes
            out = run_forward(moe, wl, inp, flags=flags, stages=True)
            assert out["status"] == 0, (wl.name, flags, moe.moe_status_string(out["status"]))
            h = to_numpy(inp)
            ref = omoe.forward(wl.mode, h["x"], h["x_scale"], h["topk_ids"], h["topk_weights"], h["w1"],
                               h["w1_scale"], h["w2"], h["w2_scale"], num_experts=wl.E, inter=wl.I)
            assert_close(y_numpy(out["y"]), ref, wl.mode, f"{wl.name} flags {flags}")
            n += 1
    torch.cuda.synchronize()
    print(f"debug build: {n} cases ok")


if __name__ == "__main__":
    main()
