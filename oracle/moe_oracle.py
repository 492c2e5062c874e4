"""CPU oracle for the MoE FFN layer forward -- TEST INFRASTRUCTURE ONLY.

Only the test-suite, the smoke check and the benchmark's CPU-baseline leg may
import this module.  The product path (the CUDA library and its Python
binding) never calls it; the two share no code, tables or helpers.

What it computes (plain definition, fp64 throughout):

The pages name the layer's phases -- the router ("MoE gate"), then "topk,
expert kernel, activation, sum" inside the fused-MoE path (page "Decode 吞吐专项
实验分析报告", section "下一步 profiling 方向", items 2-3) -- and the Strata
chapter ("第 9 章 prefill：最大的瓶颈", sec. 9.5 and 9.9) groups routed rows by
expert on the GPU before the expert GEMMs.  The pages never write the layer
out as formulas, so the steps below take the plainest reading of those phases
for a Qwen3-style SwiGLU MoE layer:

  1. router logits   l[t,e] = sum_h x[t,h]*gate_w[e,h] (+ bias[e])
  2. softmax         p[t,:] = softmax(l[t,:]) over all E experts
  3. top-k           experts ranked by logit, larger first, lower index first
                     on equal logits; the first k are slots s = 0..k-1
  4. renormalise     w[t,s] = p[t,e_s] / sum_{s'} p[t,e_s']
  5. grouping        counts[e], exclusive offsets, stable permutation of the
                     flat slot index f = t*k+s (by expert, then ascending f)
  6. expert SwiGLU   g = W_gate[e] x_t, u = W_up[e] x_t (rows [0,I) and [I,2I)
                     of w_gate_up[e]), h = silu(g)*u, y = W_down[e] h
  7. combine         out[t] = sum_{s=0..k-1} w[t,s]*y[t,s], summed in s order

NVFP4 weights are decoded exactly to fp64 (e2m1 code x e4m3 block scale x fp32
global) and then used as in step 6.  Int8 block weights (``q8_dequant``:
int8 code x fp16 scale per 32 consecutive elements along K) likewise.

W4A4 (``forward_w4a4``): NVFP4 weights and NVFP4 activations.  The pages
name the NVFP4 deployment (page "vLLM 0.32 升级试验：TEP2 prefill 诅咒解除 +
decode 本机纪录", header and "背景与动机": the 176B NVFP4 MoE served through
the "nvfp4-sm80" graft) but not its activation numerics; the reading taken
here is the format's own recipe applied to each routed row: for expert e the
token row x_t (step 6's input) and the SwiGLU output h (rounded to bf16, as
on the bf16-weight path) are each cut into 16-element blocks along the
contraction axis; a block with largest magnitude a gets the e4m3 scale
s = RNE_e4m3(a / (6*G)) and its elements the e2m1 codes RNE_e2m1(v * r) with
r = 1 / (s*G) (one reciprocal per block, as the format's deployed
quantisers compute it),
G = x_global[e] or h_global[e] (fp32 constants given with the weights, like
the calibrated input scales of NVFP4 checkpoints).  Each quotient and product
in these decisions is taken in fp32 (the precision a kernel takes them in);
both roundings are to nearest, ties to the even code, and saturate at the
format's largest finite value (448 and 6).  The GEMMs then use the decoded
values exactly in fp64.

Inputs are the raw bit patterns (uint16 bf16, uint8 e2m1/e4m3) or fp32 arrays
produced by the seeded input module; the oracle decodes them itself.
"""
from __future__ import annotations

import numpy as np

# ----------------------------------------------------------------- formats


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Decode bf16 bit patterns: a bf16 value is the fp32 value whose upper 16
    bits are the pattern and whose lower 16 bits are zero (exact in fp64)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def e2m1_to_f64(code: np.ndarray) -> np.ndarray:
    """Decode 4-bit e2m1 codes (OCP Microscaling Formats v1.0, FP4 E2M1):
    1 sign bit, 2 exponent bits with bias 1, 1 mantissa bit; exponent field 0
    is subnormal (0.m x 2^0); no infinities or NaN."""
    c = np.asarray(code, dtype=np.int64) & 0xF
    sign = np.where(c >> 3, -1.0, 1.0)
    e = (c >> 1) & 3
    m = c & 1
    mag = np.where(e == 0, 0.5 * m, np.ldexp(1.0 + 0.5 * m, e - 1))
    return sign * mag


def e4m3_to_f64(byte: np.ndarray) -> np.ndarray:
    """Decode e4m3 bytes (OCP 8-bit Floating Point Specification, E4M3):
    1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits; exponent field 0
    is subnormal (0.mmm x 2^-6); S.1111.111 is NaN; there are no infinities."""
    b = np.asarray(byte, dtype=np.int64) & 0xFF
    sign = np.where(b >> 7, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = b & 7
    mag = np.where(e == 0, np.ldexp(m / 8.0, -6), np.ldexp(1.0 + m / 8.0, e - 7))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


def nvfp4_dequant(codes: np.ndarray, scales: np.ndarray, glob: np.ndarray) -> np.ndarray:
    """Decode NVFP4 weights [E, R, K] to fp64.

    codes  uint8 [E, R, K/2]: element k is in byte k//2, low nibble for even k
    scales uint8 [E, R, K/16]: e4m3 scale of the 16-element block k//16
    glob   fp32  [E]: one global scale per expert tensor
    W[e,r,k] = e2m1(code) * e4m3(scale[e,r,k//16]) * glob[e]; each product is
    exact in fp64 (a 2-bit, a 4-bit and a 24-bit significand)."""
    codes = np.asarray(codes, dtype=np.uint8)
    E, R, K2 = codes.shape
    K = 2 * K2
    elem = np.empty((E, R, K), dtype=np.float64)
    elem[:, :, 0::2] = e2m1_to_f64(codes & 0xF)
    elem[:, :, 1::2] = e2m1_to_f64(codes >> 4)
    sc = e4m3_to_f64(np.asarray(scales, dtype=np.uint8))
    elem *= np.repeat(sc, 16, axis=2)
    elem *= np.asarray(glob, dtype=np.float32).astype(np.float64).reshape(E, 1, 1)
    return elem


def f16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Decode IEEE binary16 bit patterns: 1 sign bit, 5 exponent bits (bias
    15), 10 fraction bits; exponent field 0 is subnormal (0.f x 2^-14),
    field 31 is infinity / NaN."""
    b = np.asarray(bits, dtype=np.int64) & 0xFFFF
    sign = np.where(b >> 15, -1.0, 1.0)
    e = (b >> 10) & 0x1F
    f = b & 0x3FF
    mag = np.where(e == 0, np.ldexp(f / 1024.0, -14), np.ldexp(1.0 + f / 1024.0, e - 15))
    mag = np.where(e == 31, np.where(f == 0, np.inf, np.nan), mag)
    return sign * mag


def q8_dequant(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Decode int8 block weights [E, R, K] to fp64.

    codes  int8 [E, R, K]: one signed byte per element
    scales fp16 bits (uint16) [E, R, K/32]: the scale of the 32-element block k//32
    W[e,r,k] = code * scale[e,r,k//32]; each product is exact in fp64 (an
    8-bit and an 11-bit significand)."""
    c = np.asarray(codes, dtype=np.int8).astype(np.float64)
    sc = f16_to_f64(np.asarray(scales, dtype=np.uint16))
    return c * np.repeat(sc, 32, axis=2)


# ----------------------------------------------------------------- router


def router_logits(x: np.ndarray, gate_w: np.ndarray, bias: np.ndarray | None) -> np.ndarray:
    """Step 1: l[t,e] = sum_h x[t,h]*gate_w[e,h] + bias[e], in fp64.

    x and gate_w are fp64 arrays holding bf16 values, so every product is exact;
    each (t,e) sum runs through the same numpy reduction, so experts with equal
    gate rows get bitwise-equal logits."""
    T = x.shape[0]
    E = gate_w.shape[0]
    out = np.empty((T, E), dtype=np.float64)
    for t in range(T):
        out[t] = (gate_w * x[t]).sum(axis=1)
    if bias is not None:
        out += np.asarray(bias, dtype=np.float32).astype(np.float64)[None, :]
    return out


def softmax(l: np.ndarray) -> np.ndarray:
    """Step 2: softmax over the last axis, max subtracted, fp64."""
    z = np.exp(l - l.max(axis=-1, keepdims=True))
    return z / z.sum(axis=-1, keepdims=True)


def topk_order(l_row: np.ndarray, k: int) -> np.ndarray:
    """Step 3: the k experts with the largest logits, larger first, ties by
    lower expert index (lexsort: last key is primary)."""
    E = l_row.shape[0]
    order = np.lexsort((np.arange(E), -l_row))
    return order[:k]


def route(x: np.ndarray, gate_w: np.ndarray, bias: np.ndarray | None, top_k: int):
    """Steps 1-4.  Returns (logits fp64 [T,E], idx int32 [T,k], w fp64 [T,k])."""
    l = router_logits(x, gate_w, bias)
    p = softmax(l)
    T = l.shape[0]
    idx = np.empty((T, top_k), dtype=np.int32)
    w = np.empty((T, top_k), dtype=np.float64)
    for t in range(T):
        sel = topk_order(l[t], top_k)
        idx[t] = sel
        w[t] = p[t, sel] / p[t, sel].sum()
    return l, idx, w


# ----------------------------------------------------------------- grouping


def permute(idx: np.ndarray, E: int):
    """Step 5: counts, exclusive offsets (E+1), stable permutation and inverse.

    perm[r] is the flat slot f = t*k+s at sorted position r (sorted by expert,
    then ascending f); inv_perm[f] is the position of f."""
    flat = np.asarray(idx, dtype=np.int64).reshape(-1)
    S = flat.shape[0]
    counts = np.zeros(E, dtype=np.int32)
    for f in range(S):
        counts[flat[f]] += 1
    offsets = np.zeros(E + 1, dtype=np.int32)
    for e in range(E):
        offsets[e + 1] = offsets[e] + counts[e]
    fill = offsets[:E].copy()
    perm = np.empty(S, dtype=np.int32)
    inv_perm = np.empty(S, dtype=np.int32)
    for f in range(S):
        e = flat[f]
        perm[fill[e]] = f
        inv_perm[f] = fill[e]
        fill[e] += 1
    return counts, offsets, perm, inv_perm


# ----------------------------------------------------------------- experts


def silu(z: np.ndarray) -> np.ndarray:
    """silu(z) = z * sigmoid(z) = z / (1 + exp(-z))."""
    return z / (1.0 + np.exp(-z))


def expert_swiglu(X: np.ndarray, w_gu: np.ndarray, w_dn: np.ndarray) -> np.ndarray:
    """Step 6 for the token rows X [m, H] routed to one expert.

    w_gu [2I, H]: rows [0, I) are the gate projection, rows [I, 2I) the up
    projection; w_dn [H, I].  Each output row depends only on its own input
    row: y_r = W_down (silu(W_gate x_r) * (W_up x_r)), evaluated one row at a
    time (matrix-vector products), so a row's value never depends on which
    other rows share the expert."""
    I = w_gu.shape[0] // 2
    w_gate, w_up = w_gu[:I], w_gu[I:]
    Y = np.empty((X.shape[0], w_dn.shape[0]), dtype=np.float64)
    for r in range(X.shape[0]):
        g = w_gate @ X[r]
        u = w_up @ X[r]
        h = silu(g) * u
        Y[r] = w_dn @ h
    return Y


class ExpertWeights:
    """Expert weights decoded to fp64 on demand, one expert at a time."""

    def __init__(self, w_gate_up_bits=None, w_down_bits=None, nvfp4_gate_up=None, nvfp4_down=None,
                 q8_gate_up=None, q8_down=None):
        self.gu_bits, self.dn_bits = w_gate_up_bits, w_down_bits
        self.q_gu, self.q_dn = nvfp4_gate_up, nvfp4_down
        self.q8_gu, self.q8_dn = q8_gate_up, q8_down

    def get(self, e: int):
        if self.q8_gu is not None:
            c, s = self.q8_gu
            gu = q8_dequant(c[e:e + 1], s[e:e + 1])[0]
            c, s = self.q8_dn
            dn = q8_dequant(c[e:e + 1], s[e:e + 1])[0]
            return gu, dn
        if self.q_gu is not None:
            c, s, g = self.q_gu
            gu = nvfp4_dequant(c[e:e + 1], s[e:e + 1], g[e:e + 1])[0]
            c, s, g = self.q_dn
            dn = nvfp4_dequant(c[e:e + 1], s[e:e + 1], g[e:e + 1])[0]
            return gu, dn
        return bf16_to_f64(self.gu_bits[e]), bf16_to_f64(self.dn_bits[e])


# ----------------------------------------------------------------- forward


def forward(x_bits, gate_w_bits, bias, top_k, weights: ExpertWeights, tokens=None):
    """Steps 1-7.  Returns a dict with fp64 ``out`` for the requested tokens
    (all tokens when ``tokens`` is None) and the full-batch routing: logits,
    idx, w, counts, offsets, perm, inv_perm.

    Routing and grouping always cover the whole batch; the expert MLP runs only
    for the slots of the requested tokens.  The y rows of one expert are
    computed together (each row on its own, step 6); the per-token sum then
    runs over s = 0..k-1 in order."""
    x = bf16_to_f64(x_bits)
    gw = bf16_to_f64(gate_w_bits)
    T = x.shape[0]
    E = gw.shape[0]
    logits, idx, w = route(x, gw, bias, top_k)
    counts, offsets, perm, inv_perm = permute(idx, E)
    toks = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    y = {}
    for e in np.unique(idx[toks].reshape(-1)):
        slots = [(int(t), s) for t in toks for s in range(top_k) if idx[t, s] == e]
        gu, dn = weights.get(int(e))
        Y = expert_swiglu(x[[t for t, _ in slots]], gu, dn)
        for (t, s), row in zip(slots, Y):
            y[(t, s)] = row
    out = np.zeros((len(toks), x.shape[1]), dtype=np.float64)
    for i, t in enumerate(toks):
        acc = np.zeros(x.shape[1], dtype=np.float64)
        for s in range(top_k):
            acc = acc + w[t, s] * y[(int(t), s)]
        out[i] = acc
    return dict(out=out, tokens=toks, logits=logits, idx=idx, w=w, counts=counts,
                offsets=offsets, perm=perm, inv_perm=inv_perm)


# ----------------------------------------------------------------- W4A4


def e4m3_quantize(v: np.ndarray) -> np.ndarray:
    """fp32 values -> e4m3 bytes (OCP FP8 E4M3): round to nearest, ties to the
    even mantissa, magnitudes beyond 448 saturate to 448.

    Normal numbers are (1 + m/8) * 2^(e-7), e = 1..15; exponent field 0 is
    subnormal m/8 * 2^-6.  A magnitude v >= 2^-6 is rounded on the grid of
    its binade, 2^(floor(log2 v) - 3); below 2^-6 on the subnormal grid
    2^-9.  Rounding up into the next binade carries into the exponent field
    (mantissa 8 becomes exponent + 1, mantissa 0)."""
    a = np.abs(np.asarray(v, dtype=np.float32).astype(np.float64))
    sign = np.signbit(np.asarray(v, dtype=np.float32)).astype(np.int64)
    code = np.zeros(a.shape, dtype=np.int64)
    sub = a < 2.0 ** -6
    code[sub] = np.rint(a[sub] / 2.0 ** -9).astype(np.int64)          # 0..8 (8 = 2^-6)
    nrm = ~sub
    e = np.floor(np.log2(np.where(nrm, a, 1.0))).astype(np.int64)
    # log2 of an exact power of two is exact; guard the binade anyway
    e = np.where(np.ldexp(1.0, e) > a, e - 1, e)
    e = np.where(np.ldexp(1.0, e + 1) <= a, e + 1, e)
    m = np.rint(a / np.ldexp(1.0, e - 3)).astype(np.int64)             # 8..16
    code[nrm] = ((e[nrm] + 7) << 3) + (m[nrm] - 8)
    code = np.minimum(code, 0x7E)                                       # 448
    return ((sign << 7) | code).astype(np.uint8)


def e2m1_quantize(v: np.ndarray) -> np.ndarray:
    """fp32 values -> 4-bit e2m1 codes (OCP MX FP4 E2M1): nearest of
    0, 0.5, 1, 1.5, 2, 3, 4, 6 in magnitude, ties to the even code (mantissa
    bit 0), saturating at 6.  The grid is 0.5-spaced below 2, 1-spaced on
    [2, 4), 2-spaced from 4."""
    f = np.asarray(v, dtype=np.float32)
    a = np.abs(f.astype(np.float64))
    sign = np.signbit(f).astype(np.int64)
    code = np.where(a < 2.0, np.rint(a / 0.5),                          # codes 0..4
                    np.where(a < 4.0, np.rint(a) + 2.0,                 # 2,3,4 -> 4,5,6
                             np.minimum(np.rint(a / 2.0), 3.0) + 4.0))  # 4,6 -> 6,7
    return ((sign << 3) | code.astype(np.int64)).astype(np.uint8)


def nvfp4_quantize(a: np.ndarray, glob: float):
    """NVFP4-encode rows a [R, K] (values exact in fp32) with global scale
    glob: per 16-element block the e4m3 scale of fp32(amax / fp32(6*glob)),
    the block's reciprocal r = fp32(1 / fp32(scale*glob)), then the e2m1 code
    of fp32(v * r) per element (code 0 when scale*glob is 0).  Returns codes
    uint8 [R, K/2] (even k in the low nibble) and scales uint8 [R, K/16]."""
    a32 = np.asarray(a, dtype=np.float32)
    R, K = a32.shape
    g = np.float32(glob)
    blocks = a32.reshape(R, K // 16, 16)
    amax = np.abs(blocks).max(axis=2)
    scales = e4m3_quantize(amax / (np.float32(6.0) * g))
    denom = (e4m3_to_f64(scales).astype(np.float32) * g).astype(np.float32)
    recip = (np.float32(1.0) / np.where(denom > 0, denom, np.float32(1.0))).astype(np.float32)
    q = (blocks * recip[:, :, None]).astype(np.float32)
    nib = np.where(denom[:, :, None] > 0, e2m1_quantize(q), 0).astype(np.uint8).reshape(R, K)
    codes = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
    return codes, scales


def nvfp4_fake_quant(a: np.ndarray, glob: float) -> np.ndarray:
    """Rows a [R, K] quantised to NVFP4 and decoded back to fp64."""
    codes, scales = nvfp4_quantize(a, glob)
    return nvfp4_dequant(codes[None], scales[None], np.array([glob], dtype=np.float32))[0]


def bf16_round(a: np.ndarray) -> np.ndarray:
    """Round fp64 values to the nearest bf16 value (ties to even), via fp32
    (an fp64 -> fp32 -> bf16 double rounding can only differ from a direct
    rounding on values within 2^-24 relative of a bf16 midpoint)."""
    b = np.asarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint32) << np.uint32(16)
    return r.view(np.float32).astype(np.float64)


def forward_w4a4(x_bits, gate_w_bits, bias, top_k, weights: ExpertWeights, x_global, h_global,
                 tokens=None):
    """The layer with NVFP4 weights and NVFP4 activations (the W4A4 reading in
    the module docstring): routing and grouping as in ``forward``; for each
    routed slot (t, s) of expert e the token row is quantised with
    x_global[e], g and u are exact fp64 products of the decoded values,
    h = bf16(silu(g) * u) is quantised with h_global[e], and y = W_down h.
    The combine is step 7.  Returns the same dict as ``forward``."""
    x = bf16_to_f64(x_bits)
    gw = bf16_to_f64(gate_w_bits)
    T, H = x.shape
    E = gw.shape[0]
    xg = np.asarray(x_global, dtype=np.float32)
    hg = np.asarray(h_global, dtype=np.float32)
    logits, idx, w = route(x, gw, bias, top_k)
    counts, offsets, perm, inv_perm = permute(idx, E)
    toks = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    y = {}
    for e in np.unique(idx[toks].reshape(-1)):
        slots = [(int(t), s) for t in toks for s in range(top_k) if idx[t, s] == e]
        gu, dn = weights.get(int(e))
        I = gu.shape[0] // 2
        Xq = nvfp4_fake_quant(x[[t for t, _ in slots]], xg[e])
        for (t, s), xr in zip(slots, Xq):
            g = gu[:I] @ xr
            u = gu[I:] @ xr
            h = bf16_round(silu(g) * u)
            hq = nvfp4_fake_quant(h[None, :], hg[e])[0]
            y[(t, s)] = dn @ hq
    out = np.zeros((len(toks), H), dtype=np.float64)
    for i, t in enumerate(toks):
        acc = np.zeros(H, dtype=np.float64)
        for s in range(top_k):
            acc = acc + w[t, s] * y[(int(t), s)]
        out[i] = acc
    return dict(out=out, tokens=toks, logits=logits, idx=idx, w=w, counts=counts,
                offsets=offsets, perm=perm, inv_perm=inv_perm)
