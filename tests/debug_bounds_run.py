"""Parity of the MOE_DEBUG_BOUNDS build of the library on small cases (run in
a child process by test_gpu_failure.py with MOE_GB300_LIB pointing at that
build).  Every case must pass its parity check with a clean device status:
the index checks find nothing out of range on valid inputs."""
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import gpu_helpers as gh  # noqa: E402

import expert_layer_gb300 as moe  # noqa: E402
import moe_inputs  # noqa: E402
import oracle  # noqa: E402

CASES = [
    dict(T=4, H=256, E=8, top_k=2, I=128, bias=None, nvfp4=False),              # streaming, fused grouping
    dict(T=37, H=384, E=16, top_k=4, I=256, bias=None, nvfp4=False),            # ragged
    dict(T=600, H=384, E=16, top_k=8, I=128, bias=None, nvfp4=False),           # permutation in global memory
    dict(T=300, H=512, E=16, top_k=2, I=256, bias="zipf", nvfp4=False),         # streaming + tensor cores
    dict(T=1024, H=256, E=512, top_k=8, I=128, bias="zipf", nvfp4=False),       # prefill-sized grouping
    dict(T=24, H=256, E=8, top_k=2, I=128, bias=None, nvfp4=True),              # NVFP4 weights
    dict(T=640, H=256, E=16, top_k=8, I=256, bias=None, nvfp4=True),            # NVFP4, TMA-fed kernel
    dict(T=40, H=256, E=8, top_k=2, I=256, bias=None, q8=True),                 # int8, TMA-fed kernel
    dict(T=24, H=256, E=8, top_k=2, I=128, bias=None, q8=True),                 # int8, cp.async kernel
    dict(T=300, H=512, E=4, top_k=2, I=256, bias="zipf", nvfp4=True, w4a4=True),  # W4A4
]


def main():
    assert os.path.abspath(moe.LIB_PATH) == os.path.abspath(os.environ["MOE_GB300_LIB"]), moe.LIB_PATH
    for c in CASES:
        inp = moe_inputs.make_inputs(c, seed=1, device="cuda")
        if c.get("w4a4"):
            import torch
            W = moe.w4a4_weights(inp)
            idx = torch.empty((inp.T, inp.top_k), dtype=torch.int32, device="cuda")
            w = torch.empty((inp.T, inp.top_k), dtype=torch.float32, device="cuda")
            ws = moe.alloc_workspace(inp.T, inp.H, inp.E, inp.I, inp.top_k)
            out = moe.forward_w4a4(inp.x, inp.gate_w, inp.bias, W, inp.top_k, workspace=ws, topk_idx=idx,
                                   topk_w=w)
            orc = oracle.forward_w4a4_from_inputs(inp)
        else:
            out, idx, w, ws = gh.run_forward(inp)
            orc = oracle.forward_from_inputs(inp)
        st = moe.read_status(ws)
        assert st == 0, (c, st)
        gh.check_routing(inp, idx, w, orc)
        gh.check_output(inp, out, orc)
    print("debug-bounds build: all cases pass")


if __name__ == "__main__":
    main()
