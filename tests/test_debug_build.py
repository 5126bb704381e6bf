"""The bounds-checking build of the library (-DMOE_DEBUG): every data-dependent row index of the route,
dispatch and GEMM epilogue kernels checked on the device. It builds on the CPU host with every symbol the
header declares, and on a GPU it runs the small parity cases of every mode with the error word clear."""
import ctypes
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _debug_lib():
    sys.path.insert(0, ROOT)
    import __graft_entry__
    return __graft_entry__.build_module().build(debug=True)


def test_debug_build_exports_the_abi():
    path = _debug_lib()
    lib = ctypes.CDLL(path)
    from test_abi_cpu import _declared_functions
    for name in _declared_functions():
        assert hasattr(lib, name), name


@pytest.mark.gpu
def test_debug_build_passes_the_small_cases():
    _debug_lib()
    env = dict(os.environ, MOE_GB300_DEBUG="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "debug_build_cases.py")], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "cases ok" in r.stdout
