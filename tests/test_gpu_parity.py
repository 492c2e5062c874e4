"""GPU parity of the CUDA path (through the C ABI) against the CPU oracle.

Routing (expert ids), counts, offsets and the permutation must match bit for
bit; routing weights within the derived fp32 bound; outputs within
max|out - ref| <= 1e-2 * max|ref| (bf16 weights) or 3e-2 (NVFP4 weights).
"""
import dataclasses
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


@pytest.fixture(scope="module", autouse=True)
def _built():
    from expert_layer_gb300 import _build
    _build.build()
    moe.lib()


def _small(T, H, E, k, I, bias=None, seed=0, nvfp4=False, q8=False):
    return moe_inputs.make_inputs(dict(T=T, H=H, E=E, top_k=k, I=I, bias=bias, nvfp4=nvfp4, q8=q8), seed=seed,
                                  device="cuda")


# ------------------------------------------------------------ small, full oracle
SMALL_CASES = {
    "tiny": dict(T=4, H=256, E=8, k=2, I=128),
    "T1": dict(T=1, H=256, E=8, k=2, I=128),
    "ragged": dict(T=37, H=384, E=16, k=4, I=256),
    "k_eq_E": dict(T=6, H=256, E=8, k=8, I=128),
    "E1024_k32": dict(T=16, H=256, E=1024, k=32, I=128),
    "zipf": dict(T=50, H=512, E=32, k=4, I=256, bias="zipf"),
    "nvfp4_small": dict(T=24, H=256, E=8, k=2, I=128, nvfp4=True),
    # NVFP4 streaming with several 32-row passes per group, and with H = 1280
    # (scale rows of 80 bytes)
    "nvfp4_t96": dict(T=96, H=256, E=8, k=2, I=256, nvfp4=True),
    "nvfp4_passes": dict(T=300, H=256, E=4, k=2, I=256, nvfp4=True),
    "nvfp4_h1280": dict(T=80, H=1280, E=8, k=2, I=256, nvfp4=True),
    # more than 4096 routed slots on the weight-streaming kernel: the slot
    # permutation is read from global memory instead of shared memory (NVFP4
    # never takes the tensor-core kernels; bf16 with H % 256 != 0 neither)
    "nvfp4_global_perm": dict(T=640, H=256, E=16, k=8, I=128, nvfp4=True),
    "stream_global_perm": dict(T=600, H=384, E=16, k=8, I=128),
    # int8 block weights: one 8-row tile per pass (T <= 8), two, four (groups
    # averaging >= 24 rows) with several passes, a 1280-wide H, a batch large
    # enough for the tensor-core kernels on bf16 (int8 stays on the streaming
    # kernel) and the slot permutation in global memory
    "int8_t4": dict(T=4, H=256, E=8, k=2, I=128, q8=True),
    "int8_t24": dict(T=24, H=256, E=8, k=2, I=128, q8=True),
    "int8_passes": dict(T=300, H=256, E=4, k=2, I=256, q8=True),
    "int8_h1280": dict(T=80, H=1280, E=8, k=2, I=256, q8=True, bias="zipf"),
    "int8_global_perm": dict(T=640, H=256, E=16, k=8, I=128, q8=True),
    # H and I multiples of 256 take the TMA-fed decoded-weight kernel: one,
    # two and four token tiles per pass, and the slot permutation in global
    # memory (T*k > 4096)
    "nvfp4_tma_t4": dict(T=4, H=256, E=8, k=2, I=256, nvfp4=True),
    "nvfp4_tma_global_perm": dict(T=640, H=512, E=16, k=8, I=256, nvfp4=True, bias="zipf"),
    "int8_tma_t4": dict(T=4, H=512, E=8, k=2, I=256, q8=True),
    "int8_tma_t40": dict(T=40, H=256, E=8, k=2, I=512, q8=True),
    "int8_tma_global_perm": dict(T=640, H=256, E=16, k=8, I=256, q8=True),
    # 16 rows per expert on average: 24-row passes (three token tiles)
    "nvfp4_tma_t3": dict(T=64, H=512, E=8, k=2, I=256, nvfp4=True, bias="zipf"),
    "int8_tma_t3": dict(T=64, H=256, E=8, k=2, I=512, q8=True),
    # groups of >= 64 rows run on the tcgen05 kernels
    "tc_all": dict(T=512, H=256, E=8, k=2, I=128),
    "tc_mixed": dict(T=300, H=512, E=16, k=2, I=256, bias="zipf"),
    "tc_ragged": dict(T=200, H=256, E=2, k=1, I=384),
    # prefill-sized batch (T*k >= 8192): every group, down to a few rows, on
    # the tensor-core kernels, with the multi-block grouping
    "tc_prefill_small_groups": dict(T=1024, H=256, E=512, k=8, I=128, bias="zipf"),
    # groups of several 256-row token blocks plus a ragged last block
    "tc_multi_block": dict(T=1100, H=256, E=4, k=1, I=256, bias="zipf"),
}


@pytest.mark.parametrize("name", list(SMALL_CASES))
def test_forward_small(name):
    c = SMALL_CASES[name]
    inp = _small(c["T"], c["H"], c["E"], c["k"], c["I"], bias=c.get("bias"), nvfp4=c.get("nvfp4", False),
                 q8=c.get("q8", False))
    out, idx, w, ws = gh.run_forward(inp)
    assert moe.read_status(ws) == 0
    if name.startswith("tc_"):
        assert moe.read_diagnostics(ws)["num_large"] > 0
    orc = oracle.forward_from_inputs(inp)
    gh.check_routing(inp, idx, w, orc)
    gh.check_output(inp, out, orc)


def test_tiny_workload():
    inp = moe_inputs.make_inputs("tiny", device="cuda")
    out, idx, w, ws = gh.run_forward(inp)
    orc = oracle.forward_from_inputs(inp)
    gh.check_routing(inp, idx, w, orc)
    gh.check_output(inp, out, orc)


def test_route_and_permute_entry_points():
    inp = _small(33, 256, 16, 4, 128, bias="zipf")
    idx, w = moe.route(inp.x, inp.gate_w, inp.bias, inp.top_k)
    counts, offsets, perm, inv = moe.permute(idx, inp.E)
    torch.cuda.synchronize()
    r = oracle.route_from_inputs(inp)
    gh.check_routing(inp, idx, w, r)
    assert np.array_equal(counts.cpu().numpy(), r["counts"])
    assert np.array_equal(offsets.cpu().numpy(), r["offsets"])
    assert np.array_equal(perm.cpu().numpy(), r["perm"])
    assert np.array_equal(inv.cpu().numpy(), r["inv_perm"])


@pytest.mark.parametrize("T,E,k", [(1, 8, 1), (100, 64, 8), (512, 128, 8), (2048, 128, 8),
                                   (3000, 200, 6), (9000, 128, 8), (5000, 99, 3), (4000, 600, 4),
                                   (16384, 512, 4)])
def test_permute_matches_oracle(T, E, k):
    """Grouping alone on random expert ids, single-block and multi-block paths.

    The multi-block scan has three forms, all covered: per-block counts staged
    in shared memory with each expert's walk split over 512 // E threads (E = 128,
    200; E = 99 also takes the 4-byte staging copies), staged without the split
    (E = 600 > 512), and walked in global memory (16384 x 4 slots, E = 512: the
    counts exceed the shared-memory budget)."""
    g = torch.Generator().manual_seed(T + E)
    idx = torch.randint(0, E, (T, k), generator=g, dtype=torch.int32)
    ws = moe.alloc_workspace(T, 128, E, 128, k)
    counts, offsets, perm, inv = moe.permute(idx.cuda(), E, workspace=ws)
    assert moe.read_status(ws) == 0
    rc, ro, rp, ri = oracle.permute(idx.numpy(), E)
    assert np.array_equal(counts.cpu().numpy(), rc)
    assert np.array_equal(offsets.cpu().numpy(), ro)
    assert np.array_equal(perm.cpu().numpy(), rp)
    assert np.array_equal(inv.cpu().numpy(), ri)


def test_permute_flags_bad_expert_id():
    idx = torch.tensor([[0, 1], [5, 99]], dtype=torch.int32, device="cuda")
    ws = moe.alloc_workspace(2, 128, 8, 128, 2)
    moe.permute(idx, 8, workspace=ws)
    assert moe.read_status(ws) == -5   # MOE_ERR_DEVICE


def test_empty_batch():
    inp = _small(1, 256, 8, 2, 128)
    x0 = inp.x[:0]
    out = moe.forward(x0, inp.gate_w, None, inp.w_gate_up, inp.w_down, 2,
                      workspace=moe.alloc_workspace(1, 256, 8, 128, 2))
    assert out.shape == (0, 256)


# ------------------------------------------------------------ routing edge cases
def test_exact_ties_lower_index_wins():
    inp = _small(12, 256, 16, 4, 128)
    gw = inp.gate_w.clone()
    gw[9] = gw[2]                         # identical rows: exact logit ties
    gw[13] = gw[2]
    inp.gate_w = gw
    out, idx, w, ws = gh.run_forward(inp)
    orc = oracle.forward_from_inputs(inp)
    gh.check_routing(inp, idx, w, orc)
    gh.check_output(inp, out, orc)
    i = idx.cpu().numpy()
    for t in range(inp.T):
        row = list(i[t])
        if 2 in row and 9 in row:
            assert row.index(2) < row.index(9)


def test_zero_gate_all_tied():
    """All-zero router weights: every logit ties; experts 0..k-1, weights 1/k."""
    inp = _small(5, 256, 8, 3, 128)
    inp.gate_w = torch.zeros_like(inp.gate_w)
    out, idx, w, ws = gh.run_forward(inp)
    assert (idx.cpu().numpy() == np.arange(3)[None, :]).all()
    assert torch.allclose(w.cpu(), torch.full((5, 3), 1 / 3), atol=1e-7)
    orc = oracle.forward_from_inputs(inp)
    gh.check_output(inp, out, orc)
    d = moe.read_diagnostics(ws)
    assert d["router_fallback"] == 5 or d["router_flagged"] == 5


def test_all_tokens_one_expert():
    """A dominant bias sends every token's slot 0 to expert 3 (a group larger
    than one 32-row pass)."""
    inp = _small(100, 256, 8, 1, 128)
    b = torch.zeros(8, dtype=torch.float32, device="cuda")
    b[3] = 100.0
    inp.bias = b
    out, idx, w, ws = gh.run_forward(inp)
    assert (idx.cpu().numpy() == 3).all()
    orc = oracle.forward_from_inputs(inp)
    gh.check_output(inp, out, orc)


@pytest.mark.parametrize("T,H,E", [(2304, 256, 64), (5000, 256, 64), (2085, 1280, 100), (4100, 2048, 128)])
def test_large_router_path(T, H, E):
    """T >= 2048 uses the token-tiled router (stream-K over (32-token block,
    K chunk) items: a block's logits arrive in up to four pieces that the
    select kernel adds) and the multi-block grouping.  The cases cover ragged
    last token blocks (5000, 2085, 4100), blocks of two, three and four
    pieces on a 152-SM device (H = 1280 and 2048 reach four), pieces that
    split a block mid-way at the layer's own H, and an expert count that ends
    inside a lane's group of four (E = 100)."""
    inp = _small(T, H, E, 4, 128, bias="zipf")
    idx, w = moe.route(inp.x, inp.gate_w, inp.bias, inp.top_k)
    counts, offsets, perm, inv = moe.permute(idx, inp.E)
    torch.cuda.synchronize()
    r = oracle.route_from_inputs(inp)
    gh.check_routing(inp, idx, w, r)
    assert np.array_equal(perm.cpu().numpy(), r["perm"])


# ------------------------------------------------------------ determinism / invariance
def test_deterministic_and_token_order_invariant():
    inp = moe_inputs.make_inputs("decode64", device="cuda")
    out1, _, _, ws = gh.run_forward(inp)
    out2, _, _, _ = gh.run_forward(inp, workspace=ws)
    assert torch.equal(out1, out2)
    p = torch.randperm(inp.T, generator=torch.Generator().manual_seed(1)).cuda()
    inp2 = moe_inputs.MoEInputs(inp.T, inp.H, inp.E, inp.top_k, inp.I, inp.x[p].contiguous(), inp.gate_w,
                                inp.bias, inp.w_gate_up, inp.w_down)
    out3, _, _, _ = gh.run_forward(inp2)
    assert torch.equal(out1[p], out3)


# ------------------------------------------------------------ full-size workloads
@pytest.mark.parametrize("name", ["decode8", "decode64"])
def test_decode_workloads_full(name):
    inp = moe_inputs.make_inputs(name, device="cuda")
    out, idx, w, ws = gh.run_forward(inp)
    assert moe.read_status(ws) == 0
    orc = oracle.forward_from_inputs(inp)
    gh.check_routing(inp, idx, w, orc)
    gh.check_output(inp, out, orc)
    r = oracle.route_from_inputs(inp)
    assert moe.read_diagnostics(ws)["num_active"] == int((r["counts"] > 0).sum())


def test_nvfp4_workload_sampled():
    inp = moe_inputs.make_inputs("nvfp4_256", device="cuda")
    out, idx, w, ws = gh.run_forward(inp)
    assert moe.read_status(ws) == 0
    r = oracle.route_from_inputs(inp)
    rows = sorted(set(range(0, inp.T, 8)) | {inp.T - 1} | set(_edge_rows(r, inp.top_k)))
    orc = oracle.forward_from_inputs(inp, tokens=rows)
    gh.check_routing(inp, idx, w, orc)
    gh.check_output(inp, out, orc, rows=rows)


def test_int8_workload_sampled():
    inp = moe_inputs.make_inputs("int8_256", device="cuda")
    out, idx, w, ws = gh.run_forward(inp)
    assert moe.read_status(ws) == 0
    r = oracle.route_from_inputs(inp)
    rows = sorted(set(range(0, inp.T, 8)) | {inp.T - 1} | set(_edge_rows(r, inp.top_k)))
    orc = oracle.forward_from_inputs(inp, tokens=rows)
    gh.check_routing(inp, idx, w, orc)
    gh.check_output(inp, out, orc, rows=rows)


def test_int8_activation_beyond_f16_is_flagged():
    """The int8 expert path multiplies in f16 too: an activation beyond the
    f16 range is reported as MOE_ERR_DEVICE."""
    inp = _small(24, 256, 8, 2, 128, q8=True)
    x = inp.x.clone()
    x[3, 5] = 1.0e5
    inp.x = x
    _, _, _, ws = gh.run_forward(inp)
    assert moe.read_status(ws) == -5   # MOE_ERR_DEVICE


def _edge_rows(r, k, n_small=4):
    """Tokens whose slots sit in the last (ragged) token block of the most
    loaded expert, at the first row of that expert's group, and in the
    n_small least loaded active experts."""
    counts, offsets, perm = r["counts"], r["offsets"], r["perm"]
    hot = int(np.argmax(counts))
    picks = {int(perm[offsets[hot + 1] - 1]) // k, int(perm[offsets[hot]]) // k,
             int(perm[offsets[hot] + (counts[hot] // 256) * 256]) // k}
    active = [e for e in np.argsort(counts, kind="stable") if counts[e] > 0][:n_small]
    for e in active:
        picks.add(int(perm[offsets[e]]) // k)
        picks.add(int(perm[offsets[e + 1] - 1]) // k)
    return sorted(picks)


def test_prefill_workload_sampled():
    inp = moe_inputs.make_inputs("prefill8192", device="cuda")
    out, idx, w, ws = gh.run_forward(inp)
    assert moe.read_status(ws) == 0
    r = oracle.route_from_inputs(inp)
    rows = sorted(set(range(0, inp.T, 331)) | {inp.T - 1} | set(_edge_rows(r, inp.top_k)))
    orc = oracle.forward_from_inputs(inp, tokens=rows)
    gh.check_routing(inp, idx, w, orc)
    gh.check_output(inp, out, orc, rows=rows)


# ------------------------------------------------------------ verify sweep T = 1..16
@pytest.fixture(scope="module")
def verify_batch():
    """Decode-shaped layer (H=2048, E=128, top_k=8, I=768) with 16 token rows;
    each sweep case takes the first T rows (a token's routing and output do
    not depend on the other tokens of the batch)."""
    inp = moe_inputs.make_inputs("decode8", T=16, device="cuda")
    W = oracle.ExpertWeights(moe_inputs.bf16_bits(inp.w_gate_up), moe_inputs.bf16_bits(inp.w_down))
    return inp, W, moe_inputs.bf16_bits(inp.x), moe_inputs.bf16_bits(inp.gate_w)


@pytest.mark.parametrize("T", list(range(1, 17)))
def test_verify_sweep(verify_batch, T):
    """Speculative-verify batch sizes T = 1..16 at decode shapes, no per-group
    row ceiling: routing bit-exact and output within tolerance for every T."""
    full, W, xb, gb = verify_batch
    inp = dataclasses.replace(full, T=T, x=full.x[:T].contiguous())
    out, idx, w, ws = gh.run_forward(inp)
    assert moe.read_status(ws) == 0
    orc = oracle.forward(xb[:T], gb, None, inp.top_k, W)
    gh.check_routing(inp, idx, w, orc)
    gh.check_output(inp, out, orc)


def test_nvfp4_activation_beyond_f16_is_flagged():
    """The NVFP4 expert path multiplies in f16: an activation beyond the f16
    range is reported as MOE_ERR_DEVICE instead of silently overflowing."""
    inp = _small(24, 256, 8, 2, 128, nvfp4=True)
    x = inp.x.clone()
    x[3, 5] = 1.0e5
    inp.x = x
    _, _, _, ws = gh.run_forward(inp)
    assert moe.read_status(ws) == -5   # MOE_ERR_DEVICE
    # in range: clean status
    _, _, _, ws2 = gh.run_forward(_small(24, 256, 8, 2, 128, nvfp4=True))
    assert moe.read_status(ws2) == 0
