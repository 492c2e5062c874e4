"""CPU oracle package -- test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The CUDA library never calls it.
"""
from __future__ import annotations

import numpy as np

from . import moe_oracle
from .moe_oracle import (ExpertWeights, bf16_to_f64, e2m1_quantize, e2m1_to_f64, e4m3_quantize,
                         e4m3_to_f64, f16_to_f64, forward, forward_w4a4, nvfp4_dequant, nvfp4_quantize,
                         permute, q8_dequant, route, silu, softmax)


def _np(t):
    return None if t is None else t.detach().to("cpu").contiguous().numpy()


def _bits16(t):
    return t.detach().to("cpu").contiguous().view(__import__("torch").int16).numpy().view(np.uint16)


def forward_from_inputs(inp, tokens=None):
    """Run the oracle on a ``moe_inputs.MoEInputs`` bundle (torch tensors on
    any device; they are copied to the host as raw bits)."""
    if getattr(inp, "q8_gate_up", None) is not None:
        q, d = inp.q8_gate_up, inp.q8_down
        weights = ExpertWeights(q8_gate_up=(_np(q.codes), _bits16(q.scales)),
                                q8_down=(_np(d.codes), _bits16(d.scales)))
    elif inp.nvfp4_gate_up is not None:
        q = inp.nvfp4_gate_up
        d = inp.nvfp4_down
        weights = ExpertWeights(nvfp4_gate_up=(_np(q.codes), _np(q.scales), _np(q.glob)),
                                nvfp4_down=(_np(d.codes), _np(d.scales), _np(d.glob)))
    else:
        weights = ExpertWeights(_bits16(inp.w_gate_up), _bits16(inp.w_down))
    bias = _np(inp.bias)
    return forward(_bits16(inp.x), _bits16(inp.gate_w), bias, inp.top_k, weights, tokens=tokens)


def route_from_inputs(inp):
    """Oracle routing (steps 1-4) and grouping (step 5) for a whole batch."""
    x = bf16_to_f64(_bits16(inp.x))
    gw = bf16_to_f64(_bits16(inp.gate_w))
    logits, idx, w = route(x, gw, _np(inp.bias), inp.top_k)
    counts, offsets, perm, inv_perm = permute(idx, inp.E)
    return dict(logits=logits, idx=idx, w=w, counts=counts, offsets=offsets, perm=perm,
                inv_perm=inv_perm)


def forward_w4a4_from_inputs(inp, tokens=None):
    """The W4A4 oracle on a ``moe_inputs.MoEInputs`` bundle with NVFP4 weights
    and activation global scales (``inp.x_global``, ``inp.h_global``)."""
    q, d = inp.nvfp4_gate_up, inp.nvfp4_down
    weights = ExpertWeights(nvfp4_gate_up=(_np(q.codes), _np(q.scales), _np(q.glob)),
                            nvfp4_down=(_np(d.codes), _np(d.scales), _np(d.glob)))
    return forward_w4a4(_bits16(inp.x), _bits16(inp.gate_w), _np(inp.bias), inp.top_k, weights,
                        _np(inp.x_global), _np(inp.h_global), tokens=tokens)
