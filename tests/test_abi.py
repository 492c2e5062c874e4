"""CPU tests of the C ABI: the library builds, loads, exports every declared
symbol, sizes workspaces and rejects bad arguments on the host (no GPU call is
made on any path exercised here)."""
import ctypes
import os
import re

import pytest

import expert_layer_gb300 as moe
from expert_layer_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return moe.lib()


def declared_functions():
    with open(HEADER) as fh:
        text = fh.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_entry_points():
    names = declared_functions()
    for required in ("moe_workspace_size", "moe_route", "moe_permute", "moe_forward",
                     "moe_read_status", "moe_error_string"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_error_strings(lib):
    for code in range(0, -7, -1):
        s = lib.moe_error_string(code).decode()
        assert s.startswith("MOE_")
    assert lib.moe_version() >= 100


def test_workspace_size(lib):
    assert moe.workspace_size(8, 2048, 128, 768, 8) > 0
    assert moe.workspace_size(8192, 2048, 128, 768, 8) > moe.workspace_size(64, 2048, 128, 768, 8)
    # invalid shapes report 0
    assert moe.workspace_size(8, 2048, 128, 768, 0) == 0
    assert moe.workspace_size(8, 2048, 8, 768, 9) == 0       # top_k > E
    assert moe.workspace_size(8, 2000, 128, 768, 8) == 0     # H % 128
    assert moe.workspace_size(8, 2048, 2048, 768, 8) == 0    # E > 1024
    assert moe.workspace_size(-1, 2048, 128, 768, 8) == 0


def test_workspace_holds_the_tiled_router_pieces(lib):
    """From T = 2048 (E <= 128) the router's logits come in up to four
    stream-K pieces per token block, each with partial squares of x: the
    workspace grows by at least 4*T*E + 4*T floats at that step, beyond what
    one more token costs anywhere else."""
    for E in (32, 128):
        below = moe.workspace_size(2047, 2048, E, 768, 8)
        at = moe.workspace_size(2048, 2048, E, 768, 8)
        per_token = moe.workspace_size(2047, 2048, E, 768, 8) - moe.workspace_size(2046, 2048, E, 768, 8)
        # two 256-byte-aligned regions: up to 2 x 255 bytes of padding may be absorbed
        assert at - below - per_token >= 4 * (4 * 2048 * E + 4 * 2048) - 2 * 256
    # more than 128 experts keeps the small-batch router: no pieces
    below = moe.workspace_size(2047, 2048, 256, 768, 8)
    at = moe.workspace_size(2048, 2048, 256, 768, 8)
    per_token = below - moe.workspace_size(2046, 2048, 256, 768, 8)
    assert at - below <= per_token + 4 * 256


P = ctypes.c_void_p


def test_host_side_argument_errors(lib):
    fake = P(1 << 20)          # never dereferenced: every case fails on the host
    mis = P((1 << 20) + 4)     # not 16-byte aligned
    ws_n = moe.workspace_size(4, 256, 8, 128, 2)
    # null x
    assert lib.moe_route(None, fake, None, 4, 256, 8, 2, fake, fake, fake, ws_n, None) == -1
    # top_k > E
    assert lib.moe_route(fake, fake, None, 4, 256, 8, 9, fake, fake, fake, ws_n, None) == -1
    # misaligned gate_w
    assert lib.moe_route(fake, mis, None, 4, 256, 8, 2, fake, fake, fake, ws_n, None) == -2
    # workspace too small
    assert lib.moe_route(fake, fake, None, 4, 256, 8, 2, fake, fake, fake, ws_n - 1, None) == -3
    # T == 0 is a no-op
    assert lib.moe_route(None, None, None, 0, 256, 8, 2, None, None, None, 0, None) == 0
    assert lib.moe_permute(None, 4, 8, 2, fake, fake, fake, fake, fake, ws_n, None) == -1
    assert lib.moe_permute(fake, 4, 8, 2, fake, fake, fake, fake, fake, 16, None) == -3
    # forward: both bf16 and NVFP4 weights
    nv = moe._NVFP4(1 << 20, 1 << 20, 1 << 20, 1 << 20, 1 << 20, 1 << 20)
    ws_f = moe.workspace_size(4, 256, 8, 128, 2)
    assert lib.moe_forward(fake, fake, None, fake, fake, ctypes.byref(nv), 4, 256, 8, 128, 2, fake,
                           None, None, fake, ws_f, None) == -1
    # forward: H not a multiple of 128
    assert lib.moe_forward(fake, fake, None, fake, fake, None, 4, 200, 8, 128, 2, fake, None, None,
                           fake, ws_f, None) == -2
    # forward: missing w_down
    assert lib.moe_forward(fake, fake, None, fake, None, None, 4, 256, 8, 128, 2, fake, None, None,
                           fake, ws_f, None) == -1
    assert lib.moe_read_status(None, None) == -1


def test_python_binding_rejects_cpu_tensors(lib):
    import torch
    x = torch.zeros(4, 256, dtype=torch.bfloat16)
    with pytest.raises(moe.MoEError):
        moe.route(x, torch.zeros(8, 256, dtype=torch.bfloat16), None, 2,
                  workspace=torch.zeros(16, dtype=torch.uint8))
