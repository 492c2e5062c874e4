"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
binding and compare it with the CPU oracle on the same seeded inputs."""
from __future__ import annotations

import math

import numpy as np
import torch

import expert_layer_gb300 as moe
import moe_inputs
import oracle

TOL_BF16 = 1e-2     # max|out - ref| <= TOL * max|ref|, bf16 expert weights
TOL_NVFP4 = 3e-2    # same, NVFP4 expert weights
# int8 block weights: the oracle uses the decoded weights exactly and the GPU
# path rounds only x and h to f16 (finer than the bf16 path's h), so the bf16
# tolerance applies
TOL_INT8 = TOL_BF16


def tolerance(inp) -> float:
    if inp.nvfp4_gate_up is not None:
        return TOL_NVFP4
    return TOL_INT8 if inp.q8_gate_up is not None else TOL_BF16


def run_forward(inp, workspace=None):
    T, k = inp.T, inp.top_k
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    if workspace is None:
        workspace = moe.alloc_workspace(max(T, 1), inp.H, inp.E, inp.I, k)
    if inp.q8_gate_up is not None:
        out = moe.forward_int8(inp.x, inp.gate_w, inp.bias, inp.q8_gate_up, inp.q8_down, k,
                               workspace=workspace, topk_idx=idx, topk_w=w)
    else:
        out = moe.forward(inp.x, inp.gate_w, inp.bias, inp.w_gate_up, inp.w_down, k,
                          nvfp4_gate_up=inp.nvfp4_gate_up, nvfp4_down=inp.nvfp4_down,
                          workspace=workspace, topk_idx=idx, topk_w=w)
    torch.cuda.synchronize()
    return out, idx, w, workspace


def weight_bound(inp, orc_logits) -> np.ndarray:
    """Per-token bound on |w_gpu - w_exact| / w: the fp32 logit error bound
    delta (Cauchy-Schwarz form, the larger of the two router accumulation
    schemes) enters twice through the softmax ratio, plus fp32 rounding of the
    exponentials and the normalisation."""
    H = inp.H
    n = max(H // 32 + 5, 32 + H // 32 + 1)
    u = 2.0 ** -24
    gam = n * u / (1 - n * u)
    x = oracle.bf16_to_f64(moe_inputs.bf16_bits(inp.x))
    gw = oracle.bf16_to_f64(moe_inputs.bf16_bits(inp.gate_w))
    xn = np.sqrt((x * x).sum(axis=1))
    wn = np.sqrt((gw * gw).sum(axis=1)).max()
    delta = gam * xn * wn * (1 + 2 ** -10) * 1.01 + 2 ** -22 * np.abs(orc_logits).max(axis=1) + H * 2.0 ** -149
    return 2.01 * delta + (inp.top_k + 8) * 2.0 ** -23


def check_routing(inp, idx, w, orc):
    idx_g = idx.cpu().numpy()
    w_g = w.cpu().double().numpy()
    bad = np.nonzero((idx_g != orc["idx"]).any(axis=1))[0]
    assert bad.size == 0, f"routing differs for tokens {bad[:10]}: gpu {idx_g[bad[:3]]} vs oracle {orc['idx'][bad[:3]]}"
    rel = weight_bound(inp, orc["logits"])[:, None]
    err = np.abs(w_g - orc["w"])
    assert np.all(err <= rel * orc["w"] + 1e-12), f"max weight error {err.max():.3e}"


def check_output(inp, out, orc, rows=None):
    o = out.float().cpu().double().numpy()
    if rows is not None:
        o = o[rows]
    ref = orc["out"]
    scale = np.abs(ref).max()
    err = np.abs(o - ref).max()
    tol = tolerance(inp)
    assert err <= tol * scale, f"max|out-ref| = {err:.3e} > {tol} * max|ref| = {tol * scale:.3e}"
    return err / scale


def min_topk_gap(orc_logits, k) -> float:
    s = -np.sort(-orc_logits, axis=1)
    return float(np.min(s[:, :k] - s[:, 1:k + 1])) if s.shape[1] > k else math.inf
