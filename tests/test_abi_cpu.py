"""The C-ABI library loads on the CPU host, exports every symbol its header declares, and its
host-side logic (limits, workspace layout, argument checks) behaves without a GPU."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def moe():
    import __graft_entry__
    __graft_entry__.build_module().build()
    import moe_expert_ffn_topk_gb300 as m
    return m


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        names |= set(re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", src))
    return names


def test_exports_every_declared_symbol(moe):
    declared = _declared_functions()
    assert declared == set(moe.ABI_FUNCTIONS), declared ^ set(moe.ABI_FUNCTIONS)
    lib = ctypes.CDLL(moe._binding._LIB_PATH)
    for name in declared:
        assert hasattr(lib, name), name


def _header_enum(prefix):
    src = open(os.path.join(ROOT, "include", "moe_ffn.h")).read()
    return {name: int(val) for name, val in re.findall(r"\b(" + prefix + r"\w*)\s*=\s*(\d+)u?\b", src)}


def test_binding_constants_match_the_header(moe):
    """The binding's flag and mode values are the header's enum values (nothing is renumbered)."""
    flags = _header_enum("MOE_FLAG_")
    assert flags and all(getattr(moe, name) == val for name, val in flags.items()), flags
    assert len(set(flags.values())) == len(flags)
    modes = _header_enum("MOE_A")
    assert sorted(modes.values()) == sorted(moe.MODES.values()) == list(range(len(modes)))


def test_status_strings(moe):
    assert moe.moe_status_string(0) == "ok"
    assert "timed out" in moe.moe_status_string(5)
    assert moe.moe_status_string(99) == "unknown status"
    statuses = _header_enum("MOE_ERR_")
    assert statuses == {n: getattr(moe, n) for n in statuses} and len(statuses) == 8
    for v in statuses.values():  # every status has its own message
        assert moe.moe_status_string(v) != "unknown status"
    assert len({moe.moe_status_string(v) for v in statuses.values()}) == len(statuses)


CONFIGS = [(64, 256, 128, 8, 2), (4096, 4096, 14336, 8, 2), (128, 7168, 2048, 256, 8),
           (8192, 7168, 2048, 256, 8), (2048, 5120, 1536, 64, 6), (0, 256, 128, 8, 2)]


@pytest.mark.parametrize("cfg", CONFIGS)
@pytest.mark.parametrize("mode", ["a16w16", "a8w8_fp8", "a8w8_int8", "a8w4_fp8_fp4", "a8w4_int", "a8w8_fp8_e5m2"])
def test_workspace_layout(moe, cfg, mode):
    T, H, I, E, K = cfg
    d = moe.dims(*cfg)
    L = moe.moe_workspace_layout(d, mode)
    assert L["total"] == moe.moe_workspace_bytes(d, mode) > 0
    R = T * K
    assert L["pool_rows"] == R + min(E, R) * 127
    regions = {
        "header": 64, "counts": 4 * E, "offsets": 4 * (E + 1), "pad_offsets": 4 * (E + 1),
        "tile_offsets": 4 * (E + 1), "row_src": 4 * R, "pool_src": 4 * L["pool_rows"], "slot_row": 4 * R,
        "comb": 2 * R * H, "x_pool": L["pool_rows"] * H * (2 if mode == "a16w16" else 1),
        "a_pool": L["pool_rows"] * I * (2 if mode == "a16w16" else 1),
    }
    # the integer modes: fp32 A and the f16 operand planes (two for int8 weights, one for int4)
    planes = {"a8w8_int8": 2, "a8w4_int": 1}.get(mode, 0)
    if planes:
        regions.update(a_f32=4 * L["pool_rows"] * I, x_pool_planes=2 * planes * L["pool_rows"] * H,
                       a_pool_planes=2 * planes * L["pool_rows"] * I)
    if mode == "a8w4_int":
        regions["pool_sums"] = 8 * L["pool_rows"]
    spans = sorted((L[k], L[k] + n) for k, n in regions.items() if n)
    for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
        assert a1 <= b0
    assert spans[-1][1] <= L["total"]
    for k in regions:
        assert L[k] % 256 == 0


@pytest.mark.parametrize("shared", [1, 3])
def test_workspace_layout_with_shared_experts(moe, shared):
    """S shared experts: the plan regions cover E + S experts and T*(K+S) slots, and the gate
    region holds T*(K+S) fp32 values."""
    T, H, I, E, K = 64, 256, 128, 8, 2
    d = moe.dims(T, H, I, E, K, shared)
    L = moe.moe_workspace_layout(d, "a16w16")
    Et, Kt = E + shared, K + shared
    R = T * Kt
    assert L["pool_rows"] == R + min(Et, R) * 127
    regions = {"counts": 4 * Et, "offsets": 4 * (Et + 1), "row_src": 4 * R, "slot_row": 4 * R, "gates": 4 * R,
               "pool_src": 4 * L["pool_rows"], "comb": 2 * R * H, "x_pool": 2 * L["pool_rows"] * H}
    spans = sorted((L[k], L[k] + n) for k, n in regions.items())
    for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
        assert a1 <= b0
    assert L["gates"] > 0 and moe.moe_workspace_layout(moe.dims(T, H, I, E, K), "a16w16")["gates"] >= 0
    assert moe.moe_workspace_bytes(d, "a16w16") > moe.moe_workspace_bytes(moe.dims(T, H, I, E, K), "a16w16")


@pytest.mark.parametrize("bad", [(1, 256, 128, 8, 2, -1), (1, 256, 128, 8, 30, 3), (1, 256, 128, 1022, 2, 3)])
def test_shared_expert_limits(moe, bad):
    assert moe.moe_workspace_bytes(moe.dims(*bad), "a16w16") == 0


@pytest.mark.parametrize("bad", [(1, 100, 128, 8, 2), (1, 256, 96, 8, 2), (1, 256, 128, 8, 0),
                                 (1, 256, 128, 8, 33), (1, 256, 128, 2000, 2), (1, 256, 128, 2, 4),
                                 (-1, 256, 128, 8, 2)])
def test_limits(moe, bad):
    assert moe.moe_workspace_bytes(moe.dims(*bad), "a16w16") == 0


def test_host_checks_return_before_launch(moe):
    lib = moe._binding.LIB
    d = moe.dims(64, 256, 128, 8, 2)
    # no workspace
    assert lib.moe_plan(ctypes.c_void_p(16), ctypes.byref(d), None, None, None, None, 0, None) == 6
    # misaligned workspace
    assert lib.moe_plan(ctypes.c_void_p(16), ctypes.byref(d), None, None, None, ctypes.c_void_p(4096 + 8),
                        1 << 30, None) == 6
    # workspace too small
    assert lib.moe_plan(ctypes.c_void_p(16), ctypes.byref(d), None, None, None, ctypes.c_void_p(4096), 16,
                        None) == 6
    # bad dims
    bad = moe.dims(64, 100, 128, 8, 2)
    assert lib.moe_plan(ctypes.c_void_p(16), ctypes.byref(bad), None, None, None, ctypes.c_void_p(4096),
                        1 << 30, None) == 1
    # missing operands
    op = moe._binding.MoeOperand(None, None)
    assert lib.moe_expert_l1(op, ctypes.byref(d), 0, 0, ctypes.c_void_p(4096), 1 << 30, None) == 1
    w = moe._binding.MoeOperand(ctypes.c_void_p(4096), None)
    assert lib.moe_expert_l1(w, ctypes.byref(d), 3, 0, ctypes.c_void_p(4096), 1 << 30, None) == 1  # scale needed
    assert lib.moe_forward(op, None, None, w, w, None, ctypes.byref(d), 9, 0, ctypes.c_void_p(4096), 1 << 30,
                           None) == 1  # unknown mode
    # weight preparation: modes without a prepared form, bad layer, missing pointers, short output
    d8 = moe.dims(64, 256, 128, 8, 2)
    assert moe.moe_prepared_weights_bytes(d8, "a8w8_int8", 1) == 2 * 8 * 256 * 256
    assert moe.moe_prepared_weights_bytes(d8, "a8w8_int8", 2) == 2 * 8 * 256 * 128
    assert moe.moe_prepared_weights_bytes(moe.dims(64, 256, 128, 8, 2, 1), "a8w8_int8", 2) == 2 * 9 * 256 * 128
    for mode in ("a16w16", "a8w8_fp8", "a8w4_fp8_fp4", "a8w4_int", "a8w8_fp8_e5m2"):
        assert moe.moe_prepared_weights_bytes(d8, mode, 1) == 0
        assert lib.moe_prepare_weights(ctypes.c_void_p(4096), ctypes.byref(d8), moe.MODES[mode], 1,
                                       ctypes.c_void_p(8192), 1 << 30, None) == 2
    assert moe.moe_prepared_weights_bytes(d8, "a8w8_int8", 3) == 0
    assert lib.moe_prepare_weights(ctypes.c_void_p(4096), ctypes.byref(d8), 2, 3, ctypes.c_void_p(8192), 1 << 30, None) == 1
    assert lib.moe_prepare_weights(None, ctypes.byref(d8), 2, 1, ctypes.c_void_p(8192), 1 << 30, None) == 1
    assert lib.moe_prepare_weights(ctypes.c_void_p(4096), ctypes.byref(d8), 2, 1, ctypes.c_void_p(8192), 1024, None) == 1
    assert lib.moe_prepare_weights(ctypes.c_void_p(4096), ctypes.byref(d8), 2, 1, ctypes.c_void_p(8200), 1 << 30, None) == 1
    # the tensor-core peak probe: unknown kind, no iterations, no flops output, bad workspace
    flops = ctypes.c_double(0.0)
    ws = ctypes.c_void_p(4096)
    assert lib.moe_tensor_peak_probe(4, 10, 0, ctypes.byref(flops), ws, 256, None) == 1
    assert lib.moe_tensor_peak_probe(0, 0, 0, ctypes.byref(flops), ws, 256, None) == 1
    assert lib.moe_tensor_peak_probe(0, 10, 0, None, ws, 256, None) == 1
    assert lib.moe_tensor_peak_probe(0, 10, 0, ctypes.byref(flops), ctypes.c_void_p(4096 + 8), 256, None) == 6
    assert lib.moe_tensor_peak_probe(0, 10, 0, ctypes.byref(flops), ws, 128, None) == 6


def test_binding_rejects_host_tensors(moe):
    import torch
    d = moe.dims(64, 256, 128, 8, 2)
    with pytest.raises(ValueError):
        moe.moe_plan(torch.zeros((64, 2), dtype=torch.int32), d, torch.zeros(1 << 20, dtype=torch.uint8))


def test_header_is_a_c_abi(moe, tmp_path):
    """A C99 program includes include/moe_ffn.h (no CUDA or C++ headers needed), links the library and
    calls its host-only functions; the workspace size equals the binding's."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "abi.c"
    src.write_text(
        '#include "moe_ffn.h"\n#include "moe_peak.h"\n#include <stdio.h>\n'
        "int main(void) {\n"
        "    moe_dims d = {0};\n"
        "    d.num_tokens = 300; d.hidden = 512; d.intermediate = 384; d.num_experts = 6; d.topk = 2;\n"
        "    printf(\"%zu %zu %s\\n\", moe_workspace_bytes(&d, MOE_A16W16), moe_workspace_bytes(&d, MOE_A8W4_INT),\n"
        "           moe_status_string(MOE_ERR_TIMEOUT));\n"
        "    return 0;\n}\n")
    lib_dir = os.path.dirname(moe._binding._LIB_PATH)
    lib_name = os.path.basename(moe._binding._LIB_PATH)[3:-3]  # libNAME.so -> NAME
    exe = tmp_path / "abi"
    cc = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.join(ROOT, "include"),
                         str(src), "-L", lib_dir, "-l" + lib_name, "-o", str(exe)], capture_output=True, text=True)
    assert cc.returncode == 0, cc.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, env=dict(os.environ, LD_LIBRARY_PATH=lib_dir))
    assert run.returncode == 0, run.stderr
    bf16, w4, msg = run.stdout.split(maxsplit=2)
    d = moe.dims(300, 512, 384, 6, 2)
    assert int(bf16) == moe.moe_workspace_bytes(d, "a16w16")
    assert int(w4) == moe.moe_workspace_bytes(d, "a8w4_int")
    assert msg.strip() == moe.moe_status_string(5)
