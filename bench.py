#!/usr/bin/env python
"""MoE FFN layer forward benchmark on GB300 -- prints one JSON line (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one moe_forward (router, grouping, gate/up + SwiGLU, down, combine)
over one batch of the workload.  Inputs are seeded synthetic tensors with the
workload's shapes; they stay resident in HBM during the device-timed region.
Consecutive steps cycle through several copies of the expert weights (more
bytes than L2 between two uses of a copy), so no step reads another step's
weights from L2.  The e2e figure repeats the steps with each step's input
copied in from pinned host memory and its result copied back, the copies of
neighbouring steps overlapping the current step's kernels as in a serving
loop.  Under torchrun each rank runs an independent replica
(weak scaling, no collective on the data path); the reported time is the max
over ranks.

--impl reference times the CPU oracle (the plain fp64 definition of the
layer) on this host's cores instead; rank 0 only.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

if "reference" in sys.argv:
    # the oracle's BLAS runs single-threaded so that the core count is exact
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[v] = "1"

DEFAULT_WORKLOAD = "decode8"
WEIGHT_SETS = 4
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
STAGES = ["route", "permute", "stream", "tc", "combine"]


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=None)
    p.add_argument("--warmup", type=int, default=None)
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--weight-sets", type=int, default=WEIGHT_SETS,
                   help="copies of the expert weights cycled across steps")
    p.add_argument("--tokens", type=int, default=None,
                   help="batch size T in place of the workload's own (e.g. a T = 1..16 verify sweep "
                        "at decode shapes); the workload is then named <workload>_T<T>")
    p.add_argument("--target-seconds", type=float, default=2.0,
                   help="timed-region length used to pick K when --steps is not given")
    return p.parse_args()


def max_over_ranks(x: float, device) -> float:
    """The largest of every rank's x (the slowest rank's time); x itself with
    one process or no process group."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world: int, steps: int, tokens: int, max_ms: float) -> float:
    """Whole-job throughput of `world` independent replicas, each running
    `steps` steps of `tokens` tokens, timed by the slowest rank."""
    return world * steps * tokens / (max_ms / 1e3)


def workload_name(args) -> str:
    return args.workload if args.tokens is None else f"{args.workload}_T{args.tokens}"


STAGE_SOURCES = {
    "stream": ["expert_layer_gb300/csrc/stream_gemm.cu", "expert_layer_gb300/csrc/common.cuh",
               "expert_layer_gb300/csrc/kernels.h"],
    # the tensor-core stage: token-row gather + gate/up + down kernels
    "tc": ["expert_layer_gb300/csrc/tc_gemm.cu", "expert_layer_gb300/csrc/tc_ptx.cuh",
           "expert_layer_gb300/csrc/common.cuh", "expert_layer_gb300/csrc/kernels.h"],
}


def measured_traffic(workload: str, stage: str):
    """DRAM bytes per launch recorded from an ncu capture (profiles/traffic.txt),
    or None when none was taken or the kernel sources changed since."""
    import hashlib
    srcs = STAGE_SOURCES.get(stage)
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not srcs or not os.path.exists(path):
        return None
    h = hashlib.sha256()
    for f in srcs:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    digest = h.hexdigest()[:16]
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 4 and not line.startswith("#") and parts[0] == workload and parts[1] == stage:
                return int(parts[3]) if parts[2] == digest else None
    return None


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    FIELDS = ("pci.bus_id,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id: str | None):
        self.bus_id = bus_id
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                if self.bus_id and self.bus_id.lower() not in parts[0].lower():
                    continue
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


def pci_bus_id(dev_index: int):
    import torch
    try:
        p = torch.cuda.get_device_properties(dev_index)
        return f"{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0"
    except Exception:
        return None


# ------------------------------------------------------------------ work model
def group_split(inp, counts):
    """Experts and routed rows served by the weight-streaming kernel (small
    groups) and by the tensor-core kernels (large groups), with the same
    threshold rule as the library."""
    T, H, k = inp.T, inp.H, inp.top_k
    thr = 32 if T * k >= 8192 else 65
    use_tc = inp.nvfp4_gate_up is None and T >= thr and H % 256 == 0
    act = [int(c) for c in counts if c > 0]
    large = [c for c in act if use_tc and c >= thr]
    small = [c for c in act if not (use_tc and c >= thr)]
    return {"A_s": len(small), "S_s": sum(small), "A_l": len(large), "S_l": sum(large)}


def algorithmic_bytes(inp, split):
    """Compulsory HBM bytes per stage for one forward."""
    T, H, E, k, I = inp.T, inp.H, inp.E, inp.top_k, inp.I
    S = T * k
    wb = 0.5 + 1.0 / 16 if inp.nvfp4_gate_up is not None else 2.0   # bytes per weight
    pb = 4 if S * H * 4 <= (32 << 20) else 2                        # bytes per partial
    per_row = H * 2 + 2 * I * 2 + H * pb   # token row in, h out and back in, partial out
    A = split["A_s"] + split["A_l"]
    return {
        "route": E * H * 2 + T * H * 2 + S * 8,
        "permute": S * 4 * 4 + E * 12,
        "stream": split["A_s"] * 3 * I * H * wb + split["S_s"] * per_row,
        "tc": split["A_l"] * 3 * I * H * 2 + split["S_l"] * per_row,
        "combine": S * H * pb + T * H * 2,
        "weights": A * 3 * I * H * wb,
    }


def algorithmic_flops(inp, split):
    return {"route": 2 * inp.T * inp.E * inp.H, "stream": 2 * split["S_s"] * 3 * inp.I * inp.H,
            "tc": 2 * split["S_l"] * 3 * inp.I * inp.H}


# ------------------------------------------------------------------ CPU baseline (oracle)
ORACLE_SNIPPET = r"""
import json, os, sys, time
import numpy as np
sys.path.insert(0, sys.argv[1])
import oracle
d = sys.argv[2]
ld = lambda n: np.load(os.path.join(d, n + ".npy"), mmap_mode="r")
meta = json.load(open(os.path.join(d, "meta.json")))
bias = ld("bias") if meta["bias"] else None
if meta["nvfp4"]:
    W = oracle.ExpertWeights(nvfp4_gate_up=(ld("gu_codes"), ld("gu_scales"), ld("gu_glob")),
                             nvfp4_down=(ld("dn_codes"), ld("dn_scales"), ld("dn_glob")))
else:
    W = oracle.ExpertWeights(ld("w_gate_up"), ld("w_down"))
x, gw = np.array(ld("x")), np.array(ld("gate_w"))
budget, max_reps = float(sys.argv[3]), int(sys.argv[4])
tokens = meta["tokens"]
t0 = time.perf_counter(); reps = 0; done = 0
while True:
    oracle.forward(x, gw, bias, meta["top_k"], W, tokens=tokens)
    reps += 1; done += len(tokens)
    if time.perf_counter() - t0 >= budget or reps >= max_reps:
        break
el = time.perf_counter() - t0
print(json.dumps({"tokens": done, "seconds": el, "reps": reps}))
"""


def dump_inputs(inp, d, tokens):
    import numpy as np
    import moe_inputs as mi

    def save(name, arr):
        np.save(os.path.join(d, name + ".npy"), arr)

    save("x", mi.bf16_bits(inp.x))
    save("gate_w", mi.bf16_bits(inp.gate_w))
    if inp.bias is not None:
        save("bias", inp.bias.cpu().numpy())
    if inp.nvfp4_gate_up is not None:
        for pre, q in (("gu", inp.nvfp4_gate_up), ("dn", inp.nvfp4_down)):
            save(pre + "_codes", q.codes.cpu().numpy())
            save(pre + "_scales", q.scales.cpu().numpy())
            save(pre + "_glob", q.glob.cpu().numpy())
    else:
        save("w_gate_up", mi.bf16_bits(inp.w_gate_up))
        save("w_down", mi.bf16_bits(inp.w_down))
    with open(os.path.join(d, "meta.json"), "w") as f:
        json.dump({"bias": inp.bias is not None, "nvfp4": inp.nvfp4_gate_up is not None,
                   "top_k": inp.top_k, "tokens": list(tokens)}, f)


def cpu_baseline(inp, workload, budget_s=12.0, max_reps=1000):
    """Time the oracle, as it stands, single-threaded in a child process."""
    T = inp.T
    tokens = list(range(T)) if T <= 64 else list(range(0, T, max(1, T // 16)))[:16]
    with tempfile.TemporaryDirectory() as d:
        dump_inputs(inp, d, tokens)
        env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
        r = subprocess.run([sys.executable, "-c", ORACLE_SNIPPET, ROOT, d, str(budget_s), str(max_reps)],
                           capture_output=True, text=True, env=env, timeout=600)
    if r.returncode != 0:
        return {"value": None, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                "error": r.stderr.strip().splitlines()[-1:]}
    res = json.loads(r.stdout.strip().splitlines()[-1])
    sample = (f"{workload}: oracle forward of {len(tokens)} of the batch's {T} tokens "
              f"(routing and grouping of the whole batch each time), {res['reps']} repetitions, "
              f"{res['seconds']:.1f} s, fp64 numpy, 1 thread")
    return {"value": res["tokens"] / res["seconds"], "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": sample}


# ------------------------------------------------------------------ our arm
def run_ours(args):
    import ctypes

    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import expert_layer_gb300 as moe
    from expert_layer_gb300 import _build
    import moe_inputs

    if not os.path.exists(moe.LIB_PATH):
        _build.build()
    lib = moe.lib()
    over = {} if args.tokens is None else {"T": args.tokens}
    inp = moe_inputs.make_inputs(args.workload, seed=args.seed + rank, device=dev, **over)
    T, H, E, k, I = inp.T, inp.H, inp.E, inp.top_k, inp.I
    nv = inp.nvfp4_gate_up is not None

    # weight sets cycled across steps
    sets = []
    nsets = max(1, args.weight_sets)
    for r in range(nsets):
        if nv:
            q = inp.nvfp4_gate_up if r == 0 else moe_inputs.NVFP4Tensor(
                inp.nvfp4_gate_up.codes.clone(), inp.nvfp4_gate_up.scales.clone(), inp.nvfp4_gate_up.glob.clone())
            d = inp.nvfp4_down if r == 0 else moe_inputs.NVFP4Tensor(
                inp.nvfp4_down.codes.clone(), inp.nvfp4_down.scales.clone(), inp.nvfp4_down.glob.clone())
            st = moe._NVFP4(q.codes.data_ptr(), q.scales.data_ptr(), q.glob.data_ptr(),
                            d.codes.data_ptr(), d.scales.data_ptr(), d.glob.data_ptr())
            sets.append((None, None, ctypes.byref(st), (q, d, st)))
        else:
            gu = inp.w_gate_up if r == 0 else inp.w_gate_up.clone()
            dn = inp.w_down if r == 0 else inp.w_down.clone()
            sets.append((ctypes.c_void_p(gu.data_ptr()), ctypes.c_void_p(dn.data_ptr()), None, (gu, dn)))
    weight_bytes_per_set = (sum(t.numel() * t.element_size() for t in (
        [inp.nvfp4_gate_up.codes, inp.nvfp4_gate_up.scales, inp.nvfp4_down.codes, inp.nvfp4_down.scales]
        if nv else [inp.w_gate_up, inp.w_down])))

    ws = moe.alloc_workspace(T, H, E, I, k, dev)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)
    sptr = ctypes.c_void_p(stream.cuda_stream)
    P = ctypes.c_void_p
    x_p, g_p, o_p, ws_p = P(inp.x.data_ptr()), P(inp.gate_w.data_ptr()), P(out.data_ptr()), P(ws.data_ptr())
    b_p = P(inp.bias.data_ptr()) if inp.bias is not None else None
    wsn = ws.numel()

    def step(i, xp=x_p, op=o_p):
        gu, dn, nvp, _ = sets[i % nsets]
        rc = lib.moe_forward(xp, g_p, b_p, gu, dn, nvp, T, H, E, I, k, op, None, None, ws_p, wsn, sptr)
        if rc != 0:
            raise moe.MoEError(lib.moe_error_string(rc).decode())

    # warm-up (also sizes K when not given)
    W = args.warmup if args.warmup is not None else 20
    W = max(W, 3)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(W):
        step(i)
    torch.cuda.synchronize()
    per_step = (time.perf_counter() - t0) / W
    K = args.steps if args.steps is not None else int(min(200000, max(20, args.target_seconds / per_step)))

    diag = moe.read_diagnostics(ws)
    A = diag["num_active"]
    idx_probe = torch.empty((T, k), dtype=torch.int32, device=dev)
    moe.forward(inp.x, inp.gate_w, inp.bias, inp.w_gate_up, inp.w_down, k, nvfp4_gate_up=inp.nvfp4_gate_up,
                nvfp4_down=inp.nvfp4_down, workspace=ws, topk_idx=idx_probe)
    split = group_split(inp, torch.bincount(idx_probe.flatten().long(), minlength=E).cpu().tolist())
    router_diag = {"tokens_fp64_checked": diag["router_flagged"], "tokens_fp64_all": diag["router_fallback"],
                   "experts_on_tensor_cores": diag["num_large"]}
    assert moe.read_status(ws) == 0

    # ---- device-timed region
    sampler = ClockSampler(pci_bus_id(local))
    sampler.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(K):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    ms = max_over_ranks(e0.elapsed_time(e1), dev)
    value = job_tokens_per_s(world, K, T, ms)

    # ---- per-stage times (same steps, events at stage boundaries)
    K2 = min(K, 2000)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(K2)]
    for row in evs:          # torch creates the CUDA event on first record
        for e in row:
            e.record(stream)
    torch.cuda.synchronize()
    ev_ptrs = [(P * 6)(*[P(e.cuda_event) for e in row]) for row in evs]
    nk = ctypes.c_int32(0)
    for i in range(K2):
        gu, dn, nvp, _ = sets[i % nsets]
        rc = lib.moe_forward_profiled(x_p, g_p, b_p, gu, dn, nvp, T, H, E, I, k, o_p, None, None, ws_p,
                                      wsn, sptr, ev_ptrs[i], ctypes.byref(nk))
        assert rc == 0
    torch.cuda.synchronize()
    stage_ms = {s: statistics.fmean(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(K2))
                for j, s in enumerate(STAGES)}
    kernels_per_step = nk.value

    # ---- end to end through the C ABI with host buffers: every step copies its
    # input from pinned host memory and reads its result back, all inside the
    # timed region.  As a serving loop would, the copies of neighbouring steps
    # overlap the current step's kernels: two device input and output buffers,
    # one copy stream per direction, events ordering each buffer's reuse.
    x_h = inp.x.cpu().pin_memory()
    out_h = [torch.empty((T, H), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    x_d = [torch.empty_like(inp.x) for _ in range(2)]
    o_d = [torch.empty_like(out) for _ in range(2)]
    xd_p = [P(t.data_ptr()) for t in x_d]
    od_p = [P(t.data_ptr()) for t in o_d]
    h2d_s, d2h_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ready = [torch.cuda.Event() for _ in range(2)]   # input b copied in
    used = [torch.cuda.Event() for _ in range(2)]    # the step's kernels are done with buffers b
    read = [torch.cuda.Event() for _ in range(2)]    # result b copied out
    K3 = K
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    t0 = time.perf_counter()
    f0 = torch.cuda.Event(enable_timing=True)
    f1 = torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    h2d_s.wait_stream(stream)
    d2h_s.wait_stream(stream)
    for i in range(K3):
        b = i % 2
        with torch.cuda.stream(h2d_s):
            if i >= 2:
                h2d_s.wait_event(used[b])   # step i-2 has read x_d[b]
            x_d[b].copy_(x_h, non_blocking=True)
            ready[b].record(h2d_s)
        stream.wait_event(ready[b])
        if i >= 2:
            stream.wait_event(read[b])      # step i-2's result has left o_d[b]
        step(i, xp=xd_p[b], op=od_p[b])
        used[b].record(stream)
        with torch.cuda.stream(d2h_s):
            d2h_s.wait_event(used[b])
            out_h[b].copy_(o_d[b], non_blocking=True)
            read[b].record(d2h_s)
    stream.wait_stream(h2d_s)
    stream.wait_stream(d2h_s)
    f1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(f0.elapsed_time(f1), dev)
    e2e_value = job_tokens_per_s(world, K3, T, e2e_ms)

    if rank != 0:
        dist.destroy_process_group()
        return

    # ---- roofline of the dominant kernel
    peaks, peak_src = load_peaks()
    byt = algorithmic_bytes(inp, split)
    flops = algorithmic_flops(inp, split)
    dom = max(("stream", "tc", "route", "combine", "permute"), key=lambda s: stage_ms[s])
    dom_s = stage_ms[dom] / 1e3
    if dom == "tc":
        peak = peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
        achieved = flops[dom] / dom_s / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": measured_traffic(workload_name(args), dom)}
    else:
        peak = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
        achieved = byt[dom] / dom_s / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": measured_traffic(workload_name(args), dom)}
    roof.update({"kernel": dom, "peak_source": f"{peak_src} MEASURED_PEAKS.json" if peak_src == "measured"
                 else "fallback", "algorithmic_bytes": byt[dom],
                 "algorithmic_flops": flops.get(dom), "launch_us": stage_ms[dom] * 1e3})
    step_ms = ms / K
    layer = {"weights_bytes": byt["weights"], "weights_gbs": byt["weights"] / (step_ms / 1e3) / 1e9,
             "weights_frac_of_hbm": byt["weights"] / (step_ms / 1e3) / 1e9 / peaks.get("hbm_gbs", 6800.0),
             "active_experts": A, "groups": split, "stage_us": {s: round(stage_ms[s] * 1e3, 2) for s in STAGES},
             "router": router_diag}

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(inp, workload_name(args))

    h2d = T * H * 2
    d2h = T * H * 2
    line = {
        "metric": "MoE-layer tokens/s",
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": step_ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "nvfp4-w4a16/bf16/f32acc" if nv else "bf16/f32acc",
        "data": "synthetic",
        "config": {"workload": workload_name(args), "T": T, "H": H, "E": E, "top_k": k, "I": I,
                   "weights": "nvfp4" if nv else "bf16",
                   "router_bias": "0.5*log-Zipf(1.1)" if inp.bias is not None else None,
                   "seed": args.seed, "parallelism": f"replicas x{world}",
                   "l2": f"{nsets} rotating expert-weight sets of {weight_bytes_per_set / 1e9:.2f} GB "
                         f"(> 129 MB L2) cycled across steps"},
        "roofline": roof,
        "layer": layer,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": kernels_per_step * K,
        "kernels_per_step": kernels_per_step,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


# ------------------------------------------------------------------ reference arm (oracle)
def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import numpy as np
    import torch

    import moe_inputs
    import oracle

    dev = "cuda" if torch.cuda.is_available() else "cpu"
    over = {} if args.tokens is None else {"T": args.tokens}
    inp = moe_inputs.make_inputs(args.workload, seed=args.seed, device=dev, **over)
    x = moe_inputs.bf16_bits(inp.x)
    gw = moe_inputs.bf16_bits(inp.gate_w)
    bias = inp.bias.cpu().numpy() if inp.bias is not None else None
    if inp.nvfp4_gate_up is not None:
        q, d = inp.nvfp4_gate_up, inp.nvfp4_down
        W = oracle.ExpertWeights(nvfp4_gate_up=(q.codes.cpu().numpy(), q.scales.cpu().numpy(), q.glob.cpu().numpy()),
                                 nvfp4_down=(d.codes.cpu().numpy(), d.scales.cpu().numpy(), d.glob.cpu().numpy()))
    else:
        W = oracle.ExpertWeights(moe_inputs.bf16_bits(inp.w_gate_up), moe_inputs.bf16_bits(inp.w_down))
    del inp
    T = x.shape[0]
    K = args.steps if args.steps is not None else 5
    Wm = args.warmup if args.warmup is not None else 1
    # size each step's token sample so that the whole run stays within ~2 minutes
    t0 = time.perf_counter()
    oracle.forward(x, gw, bias, int(moe_inputs.WORKLOADS[args.workload]["top_k"]), W, tokens=[0])
    t_one = time.perf_counter() - t0
    budget = 120.0 / max(1, K + Wm)
    n_tok = int(max(1, min(T, budget / max(t_one, 1e-3))))
    tokens = list(range(0, T, max(1, T // n_tok)))[:n_tok]
    top_k = int(moe_inputs.WORKLOADS[args.workload]["top_k"])
    for _ in range(Wm):
        oracle.forward(x, gw, bias, top_k, W, tokens=tokens)
    t0 = time.perf_counter()
    for _ in range(K):
        oracle.forward(x, gw, bias, top_k, W, tokens=tokens)
    el = time.perf_counter() - t0
    value = K * len(tokens) / el
    sample = (f"{workload_name(args)}: oracle forward of {len(tokens)} of the batch's {T} tokens per step "
              f"(routing and grouping of the whole batch each step), fp64 numpy, 1 thread")
    line = {"impl": "reference", "metric": "MoE-layer tokens/s", "value": value, "unit": "tokens/s",
            "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": K, "warmup": Wm,
            "ms_per_step": el / K * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic", "config": {"workload": workload_name(args)},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
