"""CPU tests of the seeded input generator (shapes, recipe, NVFP4 encoder)."""
import math

import numpy as np
import torch

import moe_inputs
from oracle import moe_oracle


def test_shapes_and_dtypes():
    inp = moe_inputs.make_inputs("tiny")
    assert inp.x.shape == (4, 256) and inp.x.dtype == torch.bfloat16
    assert inp.gate_w.shape == (8, 256)
    assert inp.w_gate_up.shape == (8, 256, 256)
    assert inp.w_down.shape == (8, 256, 128)
    assert inp.bias is None


def test_seeded_reproducible():
    a = moe_inputs.make_inputs("tiny", seed=3)
    b = moe_inputs.make_inputs("tiny", seed=3)
    c = moe_inputs.make_inputs("tiny", seed=4)
    assert torch.equal(a.w_down, b.w_down) and not torch.equal(a.w_down, c.w_down)


def test_zipf_bias_recipe():
    b = moe_inputs.zipf_router_bias(128).double().numpy()
    z = sum(j ** -1.1 for j in range(1, 129))
    assert abs(b[0] - 0.5 * math.log(1 / z)) < 1e-6
    assert abs(b[127] - 0.5 * math.log(128 ** -1.1 / z)) < 1e-6
    assert np.all(np.diff(b) < 0)


def test_nvfp4_encode_roundtrip_error_bound():
    """Decoded NVFP4 weights (oracle decoder) lie within half an e2m1 step of
    the fp32 draws, relative to each block's scale."""
    g = torch.Generator().manual_seed(0)
    w = torch.randn(2, 8, 64, generator=g) * 0.02
    q = moe_inputs.nvfp4_encode(w)
    assert q.codes.shape == (2, 8, 32) and q.scales.shape == (2, 8, 4) and q.glob.shape == (2,)
    deq = moe_oracle.nvfp4_dequant(q.codes.numpy(), q.scales.numpy(), q.glob.numpy())
    sc = moe_oracle.e4m3_to_f64(q.scales.numpy()) * q.glob.numpy().astype(np.float64)[:, None, None]
    step = np.repeat(sc, 16, axis=2)  # largest e2m1 gap is 2 (between 4 and 6) -> half step 1
    err = np.abs(deq - w.double().numpy())
    assert np.all(err <= step * 1.0 + 1e-12)
    # the block maximum maps close to code 6
    assert np.max(np.abs(deq)) > 0.9 * float(w.abs().max())
