"""GPU test of moe_route_noalloc, the router entry point for callers that
cannot allocate device memory (graph capture, pool-only runtimes).  It keeps
its scratch in a fixed device array inside the library instead of a
caller-provided workspace.  Two calls in a row, with different batches, must
give the same routing as moe_route on the same inputs: identical expert ids
and weights within the routing-weight bound the parity tests use.

The file name sorts last so that a run stopping at the first failure has
already run every other test."""
import ctypes
import os
import sys

import numpy as np
import pytest
import torch

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
import gpu_helpers as gh  # noqa: E402

import expert_layer_gb300 as moe  # noqa: E402
import moe_inputs  # noqa: E402
import oracle  # noqa: E402

pytestmark = pytest.mark.gpu


def _noalloc(inp):
    idx = torch.full((inp.T, inp.top_k), -1, dtype=torch.int32, device="cuda")
    w = torch.full((inp.T, inp.top_k), -1.0, dtype=torch.float32, device="cuda")
    P = ctypes.c_void_p
    rc = moe.lib().moe_route_noalloc(P(inp.x.data_ptr()), P(inp.gate_w.data_ptr()),
                                     P(inp.bias.data_ptr()) if inp.bias is not None else None,
                                     inp.T, inp.H, inp.E, inp.top_k, P(idx.data_ptr()), P(w.data_ptr()),
                                     P(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, moe.lib().moe_error_string(rc)
    return idx, w


def test_route_noalloc_matches_route_twice():
    from expert_layer_gb300 import _build
    _build.build()
    # the first two take the small-batch router, the third (T >= 2048) the
    # token-tiled router; all three share the one scratch array in turn
    batches = [moe_inputs.make_inputs(dict(T=64, H=2048, E=128, top_k=8, I=128, bias="zipf", nvfp4=False),
                                      seed=5, device="cuda"),
               moe_inputs.make_inputs(dict(T=37, H=512, E=64, top_k=6, I=128, bias=None, nvfp4=False),
                                      seed=6, device="cuda"),
               moe_inputs.make_inputs(dict(T=2048, H=256, E=32, top_k=4, I=128, bias="zipf", nvfp4=False),
                                      seed=7, device="cuda")]
    for inp in batches:                        # calls in a row on the shared scratch
        idx_n, w_n = _noalloc(inp)
        idx_r, w_r = moe.route(inp.x, inp.gate_w, inp.bias, inp.top_k)
        torch.cuda.synchronize()
        assert torch.equal(idx_n, idx_r)
        r = oracle.route_from_inputs(inp)
        gh.check_routing(inp, idx_n, w_n, r)   # ids bit-exact, weights within the bound
        bound = gh.weight_bound(inp, r["logits"])[:, None]
        wr = w_r.cpu().double().numpy()
        assert np.all(np.abs(w_n.cpu().double().numpy() - wr) <= bound * wr + 1e-12)


def test_route_noalloc_rejects_oversized_batch():
    inp = moe_inputs.make_inputs(dict(T=1024, H=256, E=128, top_k=2, I=128, bias=None, nvfp4=False),
                                 device="cuda")
    idx = torch.empty((inp.T, 2), dtype=torch.int32, device="cuda")
    w = torch.empty((inp.T, 2), dtype=torch.float32, device="cuda")
    P = ctypes.c_void_p
    rc = moe.lib().moe_route_noalloc(P(inp.x.data_ptr()), P(inp.gate_w.data_ptr()), None, inp.T, inp.H,
                                     inp.E, 2, P(idx.data_ptr()), P(w.data_ptr()), None)
    assert rc == -2   # MOE_ERR_UNSUPPORTED: T*E above the fixed scratch
