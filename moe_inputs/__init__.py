"""Seeded synthetic inputs for the MoE FFN layer forward.

This module is shared by the CUDA path's tests/bench and by the CPU oracle's
tests.  It holds only input generation: random draws, the router-bias recipe
and the NVFP4 *encoder* that turns fp32 draws into e2m1 codes plus e4m3 block
scales.  It holds none of the layer's arithmetic (no routing, no expert MLP,
no decoding of the NVFP4 format); each side implements that on its own.

Workloads (Qwen3-style A3B MoE layer shapes):

=============  =====  =====  ===  =====  ====  =========================
name             T      H     E   top_k    I   structure
=============  =====  =====  ===  =====  ====  =========================
tiny             4     256    8     2     128  uniform router
decode8          8    2048  128     8     768  uniform router
decode64        64    2048  128     8     768  0.5*log-Zipf(1.1) bias
prefill8192   8192    2048  128     8     768  0.5*log-Zipf(1.1) bias
nvfp4_256      256    2048  128     8     768  NVFP4 expert weights
prefill8192_w4a4 8192 2048  128     8     768  NVFP4 weights and activations,
                                               0.5*log-Zipf(1.1) bias
int8_256       256    2048  128     8     768  int8 block expert weights
=============  =====  =====  ===  =====  ====  =========================

Recipe: one ``torch.Generator`` on the requested device seeded with ``seed``;
draw order x, gate_w, w_gate_up, w_down, each an fp32 ``randn`` (weights times
0.02) rounded to bf16 (round-to-nearest-even).  For the NVFP4 workload the
expert weights are drawn the same way in fp32 and encoded to NVFP4 instead of
bf16.  The values depend on the generator's device (CPU and CUDA generators
produce different streams for the same seed); every consumer of one call sees
the same bytes.

W4A4 workloads also carry the activations' NVFP4 global scales, one fp32 per
expert for the token rows (x_global) and for the SwiGLU output (h_global),
as an NVFP4 checkpoint stores calibrated input scales.  The recipe sets them
from a bound on the activations' magnitude, G = bound / (6 * 448) (6 is the
largest e2m1 value, 448 the largest e4m3 value): bound 8 for x ~ N(0,1) and
bound 32 for the SwiGLU output, the same for every expert.  Tests pass other
values (different per expert) through ``make_inputs(..., x_global=...,
h_global=...)``.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

WORKLOADS = {
    "tiny": dict(T=4, H=256, E=8, top_k=2, I=128, bias=None, nvfp4=False),
    "decode8": dict(T=8, H=2048, E=128, top_k=8, I=768, bias=None, nvfp4=False),
    "decode64": dict(T=64, H=2048, E=128, top_k=8, I=768, bias="zipf", nvfp4=False),
    "prefill8192": dict(T=8192, H=2048, E=128, top_k=8, I=768, bias="zipf", nvfp4=False),
    "nvfp4_256": dict(T=256, H=2048, E=128, top_k=8, I=768, bias=None, nvfp4=True),
    "prefill8192_w4a4": dict(T=8192, H=2048, E=128, top_k=8, I=768, bias="zipf", nvfp4=True, w4a4=True),
    "int8_256": dict(T=256, H=2048, E=128, top_k=8, I=768, bias=None, nvfp4=False, q8=True),
}

X_BOUND, H_BOUND = 8.0, 32.0


@dataclass
class NVFP4Tensor:
    """One NVFP4-encoded weight tensor of logical shape [E, R, K].

    codes  uint8 [E, R, K/2]  two e2m1 codes per byte, the even K index in the
                              low nibble
    scales uint8 [E, R, K/16] e4m3 bit patterns, one per 16 consecutive K
    glob   fp32  [E]          one global scale per expert
    """
    codes: torch.Tensor
    scales: torch.Tensor
    glob: torch.Tensor


@dataclass
class Q8Tensor:
    """One int8 block-quantised weight tensor of logical shape [E, R, K]:
    codes int8 [E, R, K], scales fp16 [E, R, K/32] (one per 32 consecutive K);
    W = code * scale."""
    codes: torch.Tensor
    scales: torch.Tensor


@dataclass
class MoEInputs:
    T: int
    H: int
    E: int
    top_k: int
    I: int
    x: torch.Tensor                 # bf16 [T, H]
    gate_w: torch.Tensor            # bf16 [E, H]
    bias: torch.Tensor | None       # fp32 [E] or None
    w_gate_up: torch.Tensor | None  # bf16 [E, 2I, H]  (None for NVFP4)
    w_down: torch.Tensor | None     # bf16 [E, H, I]   (None for NVFP4)
    nvfp4_gate_up: NVFP4Tensor | None = None
    nvfp4_down: NVFP4Tensor | None = None
    meta: dict = field(default_factory=dict)
    x_global: torch.Tensor | None = None  # fp32 [E], W4A4 only
    h_global: torch.Tensor | None = None  # fp32 [E], W4A4 only
    q8_gate_up: Q8Tensor | None = None    # int8 block weights
    q8_down: Q8Tensor | None = None

    def to(self, device) -> "MoEInputs":
        def mv(t):
            return None if t is None else t.to(device)

        def mvq(q):
            return None if q is None else NVFP4Tensor(mv(q.codes), mv(q.scales), mv(q.glob))

        def mv8(q):
            return None if q is None else Q8Tensor(mv(q.codes), mv(q.scales))

        return MoEInputs(self.T, self.H, self.E, self.top_k, self.I, mv(self.x), mv(self.gate_w),
                         mv(self.bias), mv(self.w_gate_up), mv(self.w_down),
                         mvq(self.nvfp4_gate_up), mvq(self.nvfp4_down), dict(self.meta),
                         mv(self.x_global), mv(self.h_global), mv8(self.q8_gate_up), mv8(self.q8_down))


def zipf_router_bias(E: int, s: float = 1.1, scale: float = 0.5) -> torch.Tensor:
    """Per-expert router bias 0.5*log-Zipf(s): b[e] = scale*ln(p_e), with
    p_e = (e+1)^-s / sum_j j^-s, so expert 0 is the most popular.  Returned in
    fp32 (the rounding from the fp64 formula happens once, here)."""
    z = sum((j + 1) ** -s for j in range(E))
    return torch.tensor([scale * math.log(((e + 1) ** -s) / z) for e in range(E)], dtype=torch.float32)


# ---------------------------------------------------------------- NVFP4 encode
_E2M1_GRID = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)


def _e2m1_encode_magnitude(a: torch.Tensor) -> torch.Tensor:
    """Round |v| (fp32) to the nearest e2m1 magnitude code 0..7, ties to the
    code with an even mantissa bit; values above 6 saturate to 6."""
    # midpoints between neighbouring grid values; a tie goes to the neighbour
    # whose mantissa bit is 0 (codes 0, 2, 4, 6 are the even ones)
    code = torch.zeros_like(a, dtype=torch.uint8)
    # (threshold, code assigned above it, tie goes up?)
    steps = ((0.25, 1, False), (0.75, 2, True), (1.25, 3, False), (1.75, 4, True),
             (2.5, 5, False), (3.5, 6, True), (5.0, 7, False))
    for thr, c, tie_up in steps:
        above = (a >= thr) if tie_up else (a > thr)
        code = torch.where(above, torch.full_like(code, c), code)
    return code


def nvfp4_encode(w: torch.Tensor) -> NVFP4Tensor:
    """Encode fp32 weights [E, R, K] (K % 16 == 0) to NVFP4.

    global_e = amax(|w_e|) / (6*448); block scale = e4m3(amax_block / (6*global))
    rounded to nearest even by torch's float8_e4m3fn cast; element code =
    e2m1 nearest-even of w / (scale*global).  Works on whatever device w is on.
    """
    E, R, K = w.shape
    assert K % 16 == 0
    w = w.float()
    amax_e = w.abs().amax(dim=(1, 2))
    glob = amax_e / (6.0 * 448.0)
    glob = torch.where(glob > 0, glob, torch.ones_like(glob))
    blocks = w.view(E, R, K // 16, 16)
    amax_b = blocks.abs().amax(dim=-1)
    scale_f = (amax_b / (6.0 * glob.view(E, 1, 1))).to(torch.float8_e4m3fn)
    scales = scale_f.view(torch.uint8)
    denom = scale_f.float() * glob.view(E, 1, 1)
    q = torch.where(denom.unsqueeze(-1) > 0, blocks / denom.unsqueeze(-1), torch.zeros_like(blocks))
    mag = _e2m1_encode_magnitude(q.abs())
    sign = ((q < 0) & (mag > 0)).to(torch.uint8) << 3
    nib = (mag | sign).view(E, R, K)
    codes = (nib[..., 0::2] | (nib[..., 1::2] << 4)).contiguous()
    return NVFP4Tensor(codes, scales.contiguous(), glob.float().contiguous())


# ---------------------------------------------------------------- int8 encode
def q8_encode(w: torch.Tensor) -> Q8Tensor:
    """Encode fp32 weights [E, R, K] (K % 32 == 0) to int8 blocks: per 32
    consecutive K the scale d = fp16(amax / 127) (torch's round to nearest
    even) and the codes round(w / d) (half to even) clamped to [-127, 127]."""
    E, R, K = w.shape
    assert K % 32 == 0
    blocks = w.float().view(E, R, K // 32, 32)
    d = (blocks.abs().amax(dim=-1) / 127.0).to(torch.float16)
    d32 = d.float().unsqueeze(-1)
    q = torch.where(d32 > 0, blocks / d32, torch.zeros_like(blocks))
    codes = torch.round(q).clamp(-127, 127).to(torch.int8).view(E, R, K)
    return Q8Tensor(codes.contiguous(), d.contiguous())


# ---------------------------------------------------------------- generator
def make_inputs(workload: str | dict, seed: int = 0, device: str | torch.device = "cpu",
                **overrides) -> MoEInputs:
    """Draw one workload's inputs.  ``workload`` is a key of WORKLOADS or a
    dict with the same fields; ``overrides`` replace single fields (e.g. T)."""
    cfg = dict(WORKLOADS[workload]) if isinstance(workload, str) else dict(workload)
    cfg.update(overrides)
    T, H, E, k, I = cfg["T"], cfg["H"], cfg["E"], cfg["top_k"], cfg["I"]
    dev = torch.device(device)
    g = torch.Generator(device=dev).manual_seed(seed)

    def draw(shape, std):
        t = torch.randn(*shape, generator=g, device=dev, dtype=torch.float32)
        return t * std if std != 1.0 else t

    x = draw((T, H), 1.0).to(torch.bfloat16)
    gate_w = draw((E, H), 0.02).to(torch.bfloat16)
    bias = zipf_router_bias(E).to(dev) if cfg.get("bias") == "zipf" else None
    if cfg.get("nvfp4"):
        gu = nvfp4_encode(draw((E, 2 * I, H), 0.02))
        dn = nvfp4_encode(draw((E, H, I), 0.02))
        xg = hg = None
        if cfg.get("w4a4"):
            xg = cfg.get("x_global")
            hg = cfg.get("h_global")
            xg = (torch.full((E,), X_BOUND / (6.0 * 448.0), dtype=torch.float32) if xg is None
                  else torch.as_tensor(xg, dtype=torch.float32)).to(dev)
            hg = (torch.full((E,), H_BOUND / (6.0 * 448.0), dtype=torch.float32) if hg is None
                  else torch.as_tensor(hg, dtype=torch.float32)).to(dev)
        return MoEInputs(T, H, E, k, I, x, gate_w, bias, None, None, gu, dn, meta=cfg, x_global=xg,
                         h_global=hg)
    if cfg.get("q8"):
        gu = q8_encode(draw((E, 2 * I, H), 0.02))
        dn = q8_encode(draw((E, H, I), 0.02))
        return MoEInputs(T, H, E, k, I, x, gate_w, bias, None, None, meta=cfg, q8_gate_up=gu, q8_down=dn)
    w_gate_up = draw((E, 2 * I, H), 0.02).to(torch.bfloat16)
    w_down = draw((E, H, I), 0.02).to(torch.bfloat16)
    return MoEInputs(T, H, E, k, I, x, gate_w, bias, w_gate_up, w_down, meta=cfg)


def bf16_bits(t: torch.Tensor):
    """Raw bf16 bit patterns of a tensor as a numpy uint16 array (host copy)."""
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view("uint16")
