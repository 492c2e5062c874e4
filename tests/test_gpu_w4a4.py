"""GPU parity of the W4A4 path (NVFP4 weights and NVFP4 activations on the
block-scaled tensor cores) against the CPU oracle's W4A4 layer.

The activation quantiser must match the oracle's bit for bit (codes and
scales); routing ids bit-exact; outputs within 3e-2 * max|ref| of the W4A4
oracle (the NVFP4 tolerance: h is quantised from the GPU's own fp32 sums, so
a code of h can land one step apart where h sits on a rounding boundary).
"""
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
from oracle import moe_oracle  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from expert_layer_gb300 import _build
    _build.build()
    moe.lib()


# ------------------------------------------------------------ quantiser
def _tie_block(G):
    """A 16-element block whose quotients v / (s G) sit exactly on e2m1
    midpoints (ties) and on the grid's ends: amax = 6 G gives s = 1."""
    q = np.array([6, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5, -0.25, -0.75, -1.25, -1.75, -2.5, -3.5, -5, 0.0])
    return q * G


@pytest.mark.parametrize("K,G", [(256, 2.0 ** -7), (768, 0.0059523810), (2048, 1.0 / 3.0)])
def test_quantize_matches_oracle(K, G):
    g = torch.Generator().manual_seed(K)
    a = torch.randn(37, K, generator=g) * 1.5
    a[3, 16:32] = 0.0                                  # an all-zero block
    a[5, 40] = 4.0e4                                   # a block whose scale saturates
    if G == 2.0 ** -7:
        a[7, 0:16] = torch.from_numpy(_tie_block(G)).float()   # exact in bf16: G is a power of two
    a[9, 100] = 1e-30                                  # a tiny value (subnormal quotient)
    ab = a.to(torch.bfloat16).cuda()
    codes, scales = moe.nvfp4_quantize(ab, G)
    torch.cuda.synchronize()
    ref_c, ref_s = moe_oracle.nvfp4_quantize(moe_oracle.bf16_to_f64(moe_inputs.bf16_bits(ab)), np.float32(G))
    assert np.array_equal(scales.cpu().numpy(), ref_s), np.argwhere(scales.cpu().numpy() != ref_s)[:5]
    bad = np.argwhere(codes.cpu().numpy() != ref_c)
    assert bad.size == 0, (bad[:5], codes.cpu().numpy()[tuple(bad[0])], ref_c[tuple(bad[0])])


def test_tc_scales_layout():
    """The tensor-core scale layout against its definition (moe.h), for a
    plain tensor and for gate/up's interleaved rows."""
    g = torch.Generator().manual_seed(3)
    E, I, K = 3, 128, 512
    for rows, gate_up in ((2 * I, True), (256, False)):
        sc = torch.randint(0, 256, (E, rows, K // 16), generator=g, dtype=torch.uint8)
        out = moe.nvfp4_tc_scales(sc.cuda(), gate_up).cpu().numpy().reshape(-1)
        s = sc.numpy()
        exp = np.empty_like(out)
        nblk = rows // 128
        for e in range(E):
            for b in range(nblk):
                for ks in range(K // 64):
                    base = ((e * nblk + b) * (K // 64) + ks) * 512
                    for rho in range(128):
                        if gate_up:
                            row = (I if rho % 2 else 0) + 64 * b + rho // 2
                        else:
                            row = 128 * b + rho
                        o = base + (rho % 32) * 16 + (rho // 32) * 4
                        exp[o:o + 4] = s[e, row, 4 * ks:4 * ks + 4]
        assert np.array_equal(out, exp)


# ------------------------------------------------------------ layer parity
def _w4a4_inputs(T, H, E, k, I, bias=None, seed=0):
    rng = np.random.default_rng(seed + 100)
    xg = (rng.uniform(0.5, 2.0, E) * moe_inputs.X_BOUND / (6 * 448)).astype(np.float32)
    hg = (rng.uniform(0.5, 2.0, E) * moe_inputs.H_BOUND / (6 * 448)).astype(np.float32)
    return moe_inputs.make_inputs(dict(T=T, H=H, E=E, top_k=k, I=I, bias=bias, nvfp4=True, w4a4=True,
                                       x_global=xg, h_global=hg), seed=seed, device="cuda")


def _run(inp):
    W = moe.w4a4_weights(inp)
    idx = torch.empty((inp.T, inp.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((inp.T, inp.top_k), dtype=torch.float32, device="cuda")
    ws = moe.alloc_workspace(inp.T, inp.H, inp.E, inp.I, inp.top_k)
    out = moe.forward_w4a4(inp.x, inp.gate_w, inp.bias, W, inp.top_k, workspace=ws, topk_idx=idx, topk_w=w)
    torch.cuda.synchronize()
    return out, idx, w, ws


W4A4_CASES = {
    # groups of a few rows: one 16-column tile per expert
    "small_groups": dict(T=24, H=256, E=8, k=2, I=256),
    # groups over several 128-row token tiles with a ragged last one
    "multi_tile": dict(T=300, H=512, E=4, k=2, I=256, bias="zipf"),
    "many_experts": dict(T=200, H=256, E=64, k=8, I=256),
    "one_token": dict(T=1, H=256, E=8, k=2, I=256),
    "prefill_like": dict(T=2048, H=256, E=16, k=4, I=512, bias="zipf"),
}


@pytest.mark.parametrize("name", list(W4A4_CASES))
def test_w4a4_forward_small(name):
    c = W4A4_CASES[name]
    inp = _w4a4_inputs(c["T"], c["H"], c["E"], c["k"], c["I"], bias=c.get("bias"))
    out, idx, w, ws = _run(inp)
    assert moe.read_status(ws) == 0
    orc = oracle.forward_w4a4_from_inputs(inp)
    gh.check_routing(inp, idx, w, orc)
    rel = gh.check_output(inp, out, orc)
    # the W4A4 layer is not the W4A16 layer: the comparison is with the W4A4 oracle
    assert rel <= gh.TOL_NVFP4


def test_w4a4_deterministic():
    inp = _w4a4_inputs(300, 512, 4, 2, 256, bias="zipf")
    out1, _, _, ws = _run(inp)
    W = moe.w4a4_weights(inp)
    out2 = moe.forward_w4a4(inp.x, inp.gate_w, inp.bias, W, inp.top_k, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(out1, out2)


def test_w4a4_prefill_workload_sampled():
    inp = moe_inputs.make_inputs("prefill8192_w4a4", device="cuda")
    out, idx, w, ws = _run(inp)
    assert moe.read_status(ws) == 0
    r = oracle.route_from_inputs(inp)
    counts, offsets, perm = r["counts"], r["offsets"], r["perm"]
    hot = int(np.argmax(counts))
    rows = set(range(0, inp.T, 409)) | {inp.T - 1, int(perm[offsets[hot + 1] - 1]) // inp.top_k}
    for e in [e for e in np.argsort(counts, kind="stable") if counts[e] > 0][:3]:
        rows.add(int(perm[offsets[e]]) // inp.top_k)
    rows = sorted(rows)
    orc = oracle.forward_w4a4_from_inputs(inp, tokens=rows)
    gh.check_routing(inp, idx, w, orc)
    gh.check_output(inp, out, orc, rows=rows)
