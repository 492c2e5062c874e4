"""Failure detection without a GPU fault.

* A bounded device wait that runs out: the test-only setting
  moe_debug_force_wait_timeout makes the weight-streaming kernel's down units
  wait for a count that no gate/up unit reaches, with a short poll limit.
  The kernel returns, moe_read_status reports MOE_ERR_DEVICE_TIMEOUT, and the
  next normal call is clean and correct.
* The MOE_DEBUG_BOUNDS build (index checks in the expert, gather and
  quantiser kernels) passes parity with a clean status on small cases, in a
  child process that loads that build.
"""
import os
import subprocess
import sys

import pytest
import torch

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
import gpu_helpers as gh  # noqa: E402

import expert_layer_gb300 as moe  # noqa: E402
import moe_inputs  # noqa: E402
import oracle  # noqa: E402

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
MOE_ERR_DEVICE_TIMEOUT = -6


@pytest.fixture(scope="module", autouse=True)
def _built():
    from expert_layer_gb300 import _build
    _build.build()
    moe.lib()


@pytest.mark.parametrize("fmt", ["bf16", "nvfp4_tma"])
def test_forced_wait_timeout_is_reported_and_next_call_is_clean(fmt):
    # decode-sized batch: every group on a weight-streaming kernel, whose
    # down units wait for their expert's gate/up units (bf16: the cp.async
    # kernel; NVFP4 with H, I multiples of 256: the TMA-fed kernel)
    shape = dict(T=8, H=256, E=16, top_k=4, I=128) if fmt == "bf16" else dict(T=8, H=256, E=16, top_k=4, I=256)
    inp = moe_inputs.make_inputs(dict(shape, bias=None, nvfp4=fmt != "bf16"), seed=3, device="cuda")
    lib = moe.lib()
    assert lib.moe_debug_force_wait_timeout(2000) == 0
    try:
        _, _, _, ws = gh.run_forward(inp)
        assert moe.read_status(ws) == MOE_ERR_DEVICE_TIMEOUT
    finally:
        assert lib.moe_debug_force_wait_timeout(0) == 0
    out, idx, w, ws = gh.run_forward(inp, workspace=ws)
    assert moe.read_status(ws) == 0
    orc = oracle.forward_from_inputs(inp)
    gh.check_routing(inp, idx, w, orc)
    gh.check_output(inp, out, orc)
    assert lib.moe_debug_force_wait_timeout(-1) == -1   # MOE_ERR_INVALID_ARG


def test_debug_bounds_build_passes_parity():
    from expert_layer_gb300 import _build
    lib_path = os.path.join(ROOT, "expert_layer_gb300", "libmoe_gb300_debug.so")
    _build.build(extra_flags=["-DMOE_DEBUG_BOUNDS"], build_dir=os.path.join(ROOT, "_build_debug"),
                 lib_path=lib_path)
    env = dict(os.environ, MOE_GB300_LIB=lib_path)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "debug_bounds_run.py")], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-3000:]
    assert "all cases pass" in r.stdout
