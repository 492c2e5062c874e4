"""Pins that tie the CPU oracle to facts outside itself.

Each pin takes the oracle module as an argument so that the mutation test can
run the same pins against copies of the oracle with a planted mistake.  A pin
raises AssertionError when the oracle disagrees with:

* the published format tables (bf16, OCP FP4 E2M1, OCP FP8 E4M3) kept as text
  fixtures under tests/golden/,
* closed forms (zero router weights, silu at ln 3, saturated silu),
* library routines for special cases (torch fp64 matmul / silu for a dense
  SwiGLU MLP, scipy softmax for top_k = E, numpy's stable argsort for the
  grouping),
* brute force over all k-subsets on tiny routers,
* exact invariants (token-order equivariance, exact scaling by 2).
"""
from __future__ import annotations

import itertools
import math
import os
from fractions import Fraction

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _read_table(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            code, val = line.split()
            rows.append((int(code, 16), val))
    return rows


def _val(s):
    if s == "nan":
        return float("nan")
    if s == "-0":
        return -0.0
    return float(Fraction(s))


def _rng(seed):
    return np.random.default_rng(seed)


def _bf16_round(a):
    """Round fp32 values to bf16 bit patterns (nearest even) -- builds inputs."""
    b = np.asarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def _rand_bf16(rng, shape, std):
    return _bf16_round(rng.standard_normal(shape).astype(np.float32) * np.float32(std))


# ------------------------------------------------------------------ formats

def pin_bf16_table(o):
    for code, val in _read_table("bf16_bits.txt"):
        got = o.bf16_to_f64(np.array([code], dtype=np.uint16))[0]
        assert got == _val(val), (hex(code), got, val)


def pin_e2m1_table(o):
    for code, val in _read_table("e2m1_codes.txt"):
        got = o.e2m1_to_f64(np.array([code]))[0]
        exp = _val(val)
        assert got == exp and math.copysign(1, got) == math.copysign(1, exp), (hex(code), got, val)


def pin_e4m3_table(o):
    for code, val in _read_table("e4m3_codes.txt"):
        got = o.e4m3_to_f64(np.array([code]))[0]
        exp = _val(val)
        if math.isnan(exp):
            assert math.isnan(got), hex(code)
        else:
            assert got == exp and math.copysign(1, got) == math.copysign(1, exp), (hex(code), got, val)


def pin_nvfp4_layout(o):
    """Element k of a row sits in byte k//2 (low nibble for even k) and uses
    scale k//16; values from the two format tables times the global scale."""
    e2m1 = {c: _val(v) for c, v in _read_table("e2m1_codes.txt")}
    e4m3 = {c: _val(v) for c, v in _read_table("e4m3_codes.txt")}
    rng = _rng(7)
    E, R, K = 2, 3, 64
    codes = rng.integers(0, 256, size=(E, R, K // 2), dtype=np.uint8)
    scale_codes = np.array([c for c in e4m3 if not math.isnan(e4m3[c])], dtype=np.uint8)
    scales = rng.choice(scale_codes, size=(E, R, K // 16)).astype(np.uint8)
    glob = np.array([0.75, 1.0 / 3.0], dtype=np.float32)
    W = o.nvfp4_dequant(codes, scales, glob)
    assert W.shape == (E, R, K)
    for e in range(E):
        for r in range(R):
            for k in range(K):
                byte = int(codes[e, r, k // 2])
                nib = (byte & 0xF) if k % 2 == 0 else (byte >> 4)
                exp = e2m1[nib] * e4m3[int(scales[e, r, k // 16])] * float(glob[e])
                assert W[e, r, k] == exp, (e, r, k, W[e, r, k], exp)


def pin_nvfp4_forward_matches_bf16(o):
    """The layer with NVFP4 expert weights equals the layer with the same
    weights given as bf16 bits.  Every decoded weight (an e2m1 value times an
    e4m3 value times a global with two significant bits) has at most 8
    significant bits, so it is exact in bf16; the bf16 copies are built from
    the two format tables, not from the oracle's decoder.  The globals differ
    per expert and per projection, so taking one projection's global for the
    other, or one expert's slice for another, changes the output."""
    e2m1 = {c: _val(v) for c, v in _read_table("e2m1_codes.txt")}
    e4m3 = {c: _val(v) for c, v in _read_table("e4m3_codes.txt")}
    rng = _rng(13)
    T, H, E, k, I = 7, 32, 3, 2, 16
    scale_codes = np.array([c for c, v in e4m3.items() if not math.isnan(v) and 2.0 ** -9 <= abs(v) <= 8],
                           dtype=np.uint8)
    glob_gu = np.array([0.75, 0.375, 1.5], dtype=np.float32)
    glob_dn = np.array([0.5, 3.0, 0.1875], dtype=np.float32)

    def quantised(R, K, glob):
        codes = rng.integers(0, 256, size=(E, R, K // 2), dtype=np.uint8)
        scales = rng.choice(scale_codes, size=(E, R, K // 16)).astype(np.uint8)
        vals = np.empty((E, R, K), dtype=np.float64)
        for e in range(E):
            for r in range(R):
                for kk in range(K):
                    byte = int(codes[e, r, kk // 2])
                    nib = (byte & 0xF) if kk % 2 == 0 else (byte >> 4)
                    vals[e, r, kk] = e2m1[nib] * e4m3[int(scales[e, r, kk // 16])] * float(glob[e])
        bits = _bf16_round(vals.astype(np.float32))
        back = (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
        assert np.array_equal(back, vals)   # the construction is bf16-exact
        return (codes, scales, glob), bits

    q_gu, b_gu = quantised(2 * I, H, glob_gu)
    q_dn, b_dn = quantised(H, I, glob_dn)
    xb = _rand_bf16(rng, (T, H), 1.0)
    gb = _rand_bf16(rng, (E, H), 0.5)
    a = o.forward(xb, gb, None, k, o.ExpertWeights(nvfp4_gate_up=q_gu, nvfp4_down=q_dn))
    b = o.forward(xb, gb, None, k, o.ExpertWeights(b_gu, b_dn))
    assert set(np.unique(a["idx"])) == set(range(E)), a["idx"]   # every expert's slice is used
    assert np.array_equal(a["out"], b["out"]), np.abs(a["out"] - b["out"]).max()


# ------------------------------------------------------------------ int8 block weights

def pin_f16_table(o):
    """fp16 decoding against the binary16 table (exact fractions) and numpy's
    float16 (a library routine) on every pattern."""
    for code, val in _read_table("f16_bits.txt"):
        got = o.f16_to_f64(np.array([code], dtype=np.uint16))[0]
        if val == "nan":
            assert math.isnan(got), hex(code)
        elif val in ("inf", "-inf"):
            assert got == float(val), hex(code)
        else:
            exp = _val(val)
            assert got == exp and math.copysign(1, got) == math.copysign(1, exp), (hex(code), got, val)
    allb = np.arange(65536, dtype=np.uint16)
    lib = allb.view(np.float16).astype(np.float64)
    got = o.f16_to_f64(allb)
    fin = np.isfinite(lib)
    assert np.array_equal(got[fin], lib[fin]) and np.array_equal(np.isnan(got), np.isnan(lib))


def pin_q8_layout(o):
    """Element k of an int8 block row is its signed code times the fp16 scale
    of block k//32 (numpy's float16 decoding, exact products)."""
    rng = _rng(17)
    E, R, K = 2, 3, 96
    codes = rng.integers(-128, 128, size=(E, R, K)).astype(np.int8)
    scales = rng.integers(0, 0x7C00, size=(E, R, K // 32)).astype(np.uint16)
    W = o.q8_dequant(codes, scales)
    sc = scales.view(np.float16).astype(np.float64)
    for e in range(E):
        for r in range(R):
            for k in range(K):
                assert W[e, r, k] == float(codes[e, r, k]) * sc[e, r, k // 32], (e, r, k)


def pin_q8_forward_matches_bf16(o):
    """The layer with int8 block weights equals the layer with the same
    weights as bf16 bits: scales that are powers of two (different per
    expert, projection and block) times 8-bit codes are exact in bf16."""
    rng = _rng(18)
    T, H, E, k, I = 7, 64, 3, 2, 32

    def q8(R, K, lo, hi):
        codes = rng.integers(-127, 128, size=(E, R, K)).astype(np.int8)
        exps = rng.integers(lo, hi, size=(E, R, K // 32))
        scales = np.ldexp(1.0, exps).astype(np.float16).view(np.uint16)
        vals = codes.astype(np.float64) * np.repeat(np.ldexp(1.0, exps), 32, axis=2)
        bits = _bf16_round(vals.astype(np.float32))
        back = (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
        assert np.array_equal(back, vals)   # the construction is bf16-exact
        return (codes, scales), bits

    q_gu, b_gu = q8(2 * I, H, -9, -5)
    q_dn, b_dn = q8(H, I, -8, -4)
    xb = _rand_bf16(rng, (T, H), 1.0)
    gb = _rand_bf16(rng, (E, H), 0.5)
    a = o.forward(xb, gb, None, k, o.ExpertWeights(q8_gate_up=q_gu, q8_down=q_dn))
    b = o.forward(xb, gb, None, k, o.ExpertWeights(b_gu, b_dn))
    assert set(np.unique(a["idx"])) == set(range(E)), a["idx"]
    assert np.array_equal(a["out"], b["out"]), np.abs(a["out"] - b["out"]).max()


# ------------------------------------------------------------------ W4A4 quantiser

def _torch_e4m3_bytes(v32):
    import torch
    return torch.from_numpy(np.asarray(v32, dtype=np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def pin_e4m3_quantize_library(o):
    """fp32 -> e4m3 rounding equals torch's float8_e4m3fn cast (round to
    nearest even) on every e4m3 value, every midpoint between neighbours, the
    subnormal range and random values below 464; above that the quantiser
    saturates to 448 (0x7E) where the cast gives NaN."""
    import torch
    allv = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    pos = np.unique(allv[np.isfinite(allv) & (allv >= 0)]).astype(np.float64)
    mids = (pos[:-1] + pos[1:]) / 2
    rng = _rng(14)
    vals = np.concatenate([pos, mids, np.nextafter(mids.astype(np.float32), np.float32(0)),
                           np.nextafter(mids.astype(np.float32), np.float32(1e9)),
                           rng.uniform(0, 2.0 ** -6, 500), rng.uniform(0, 463.9, 2000)]).astype(np.float32)
    vals = np.concatenate([vals, -vals])
    got = o.e4m3_quantize(vals)
    exp = _torch_e4m3_bytes(vals)
    bad = np.nonzero(got != exp)[0]
    assert bad.size == 0, (vals[bad[:5]], got[bad[:5]], exp[bad[:5]])
    sat = np.array([464.5, 500.0, 1e6, 3e38], dtype=np.float32)
    assert (o.e4m3_quantize(sat) == 0x7E).all() and (o.e4m3_quantize(-sat) == 0xFE).all()


def pin_e2m1_quantize_table(o):
    """fp32 -> e2m1 rounding against the OCP FP4 E2M1 table: every table value
    maps to its code, a midpoint between neighbours to the neighbour with the
    even code, a value just past a midpoint to the upper neighbour, anything
    at or above 6 to 6; negative values mirror positive ones."""
    e2m1 = {c: _val(v) for c, v in _read_table("e2m1_codes.txt")}
    mags = sorted((v, c) for c, v in e2m1.items() if c < 8)
    for v, c in mags:
        assert o.e2m1_quantize(np.array([v], dtype=np.float32))[0] == c, (v, c)
        if v > 0:
            assert o.e2m1_quantize(np.array([-v], dtype=np.float32))[0] == c | 8, (v, c)
    for (v0, c0), (v1, c1) in zip(mags[:-1], mags[1:]):
        mid = np.float32((v0 + v1) / 2)
        even = c0 if c0 % 2 == 0 else c1
        assert o.e2m1_quantize(np.array([mid], dtype=np.float32))[0] == even, (mid, even)
        assert o.e2m1_quantize(np.array([-mid], dtype=np.float32))[0] == even | 8, (mid, even)
        above = np.nextafter(mid, np.float32(10))
        assert o.e2m1_quantize(np.array([above], dtype=np.float32))[0] == c1, (above, c1)
        below = np.nextafter(mid, np.float32(-10))
        assert o.e2m1_quantize(np.array([below], dtype=np.float32))[0] == c0, (below, c0)
    big = np.array([6.0, 6.5, 7.0, 100.0, 3e38], dtype=np.float32)
    assert (o.e2m1_quantize(big) == 7).all() and (o.e2m1_quantize(-big) == 15).all()


def pin_nvfp4_quantize_blocks(o):
    """NVFP4 encoding of activation rows, by brute force: per 16-element block
    the scale byte is torch's e4m3 cast of fp32(amax / fp32(6*G)) (448 when
    that quotient is beyond the format's range: one block here is); each
    element's code (decoded with the format tables, even k in the low nibble)
    is a nearest e2m1 value to fp32(v * fp32(1 / fp32(scale*G))), ties to the
    even code, saturating at 6; an all-zero block gets scale 0 and codes 0."""
    e2m1 = {c: _val(v) for c, v in _read_table("e2m1_codes.txt")}
    rng = _rng(15)
    R, K = 5, 96
    for G in (np.float32(0.0030517578), np.float32(1.0 / 3.0), np.float32(2.0 ** -7)):
        a = o.bf16_to_f64(_rand_bf16(rng, (R, K), 1.0))
        a[2, 16:32] = 0.0
        a[3, 40] = 300.0          # a block whose scale is far above the others
        codes, scales = o.nvfp4_quantize(a, G)
        assert codes.shape == (R, K // 2) and scales.shape == (R, K // 16)
        a32 = a.astype(np.float32)
        for r in range(R):
            for b in range(K // 16):
                blk = a32[r, 16 * b:16 * b + 16]
                amax = np.float32(np.abs(blk).max())
                sv = np.float32(amax / np.float32(np.float32(6.0) * G))
                # beyond 464 the cast gives NaN; the quantiser saturates to 448
                exp_s = _torch_e4m3_bytes(np.array([sv]))[0] if sv < 464 else np.uint8(0x7E)
                assert scales[r, b] == exp_s, (G, r, b, scales[r, b], exp_s)
                sdec = np.float32(o.e4m3_to_f64(np.array([exp_s]))[0])
                den = np.float32(sdec * G)
                for i in range(16):
                    kk = 16 * b + i
                    byte = int(codes[r, kk // 2])
                    nib = (byte & 0xF) if kk % 2 == 0 else (byte >> 4)
                    if den == 0:
                        assert nib == 0
                        continue
                    q = float(np.float32(blk[i] * np.float32(np.float32(1.0) / den)))
                    got = e2m1[nib]
                    best = min(abs(v - q) for v in e2m1.values())
                    assert abs(got - q) == best, (G, r, kk, q, got)
                    if abs(q) < 6 and sum(1 for c, v in e2m1.items() if abs(v - q) == best and
                                          (v != 0 or c == (nib & 8))) > 1:
                        assert nib % 2 == 0, (q, nib)        # a tie went to the even code
                    if q != 0 and got != 0:
                        assert (got < 0) == (q < 0)


def pin_w4a4_forward_composition(o):
    """The W4A4 layer on a tiny case equals its definition composed by hand:
    routing as in the bf16 layer; per slot of expert e the token row
    quantised with x_global[e] and decoded with the e2m1 table and torch's
    e4m3 decoding; g and u
    as exactly rounded sums (math.fsum) of the decoded products; h rounded to
    bf16 by torch; h quantised with h_global[e]; y = W_down h in torch fp64;
    the weighted sum over slots.  Globals differ per expert and between x and
    h, so mixing them up changes the output."""
    import torch
    e2m1 = {c: _val(v) for c, v in _read_table("e2m1_codes.txt")}
    e4m3 = {c: _val(v) for c, v in _read_table("e4m3_codes.txt")}
    # every e4m3 byte decoded by torch's float8_e4m3fn (activation scales take
    # any code, the table holds a sweep)
    e4m3_all = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    rng = _rng(16)
    T, H, E, k, I = 6, 32, 3, 2, 16
    scale_codes = np.array([c for c, v in e4m3.items() if not math.isnan(v) and 2.0 ** -9 <= abs(v) <= 8],
                           dtype=np.uint8)

    def weights(R, K, glob):
        codes = rng.integers(0, 256, size=(E, R, K // 2), dtype=np.uint8)
        scales = rng.choice(scale_codes, size=(E, R, K // 16)).astype(np.uint8)
        return codes, scales, glob

    def decode(codes, scales, glob):   # [R, K/2], [R, K/16], float -> fp64 [R, K] via the tables
        R, K2 = codes.shape
        out = np.empty((R, 2 * K2))
        for r in range(R):
            for kk in range(2 * K2):
                byte = int(codes[r, kk // 2])
                nib = (byte & 0xF) if kk % 2 == 0 else (byte >> 4)
                out[r, kk] = e2m1[nib] * e4m3_all[int(scales[r, kk // 16])] * float(glob)
        return out

    q_gu = weights(2 * I, H, np.array([0.75, 0.375, 1.5], dtype=np.float32))
    q_dn = weights(H, I, np.array([0.5, 3.0, 0.1875], dtype=np.float32))
    xg = np.array([0.0078125, 0.0055, 0.0021], dtype=np.float32)
    hg = np.array([0.9, 0.41, 0.23], dtype=np.float32)
    xb = _rand_bf16(rng, (T, H), 1.0)
    gb = _rand_bf16(rng, (E, H), 0.5)
    res = o.forward_w4a4(xb, gb, None, k, o.ExpertWeights(nvfp4_gate_up=q_gu, nvfp4_down=q_dn), xg, hg)
    assert set(np.unique(res["idx"])) == set(range(E)), res["idx"]
    x = o.bf16_to_f64(xb)
    ref = np.zeros((T, H))
    for t in range(T):
        for s in range(k):
            e = int(res["idx"][t, s])
            gu = decode(q_gu[0][e], q_gu[1][e], q_gu[2][e])
            dn = decode(q_dn[0][e], q_dn[1][e], q_dn[2][e])
            xc, xs = o.nvfp4_quantize(x[t:t + 1], xg[e])
            xq = decode(xc, xs, xg[e])[0]
            g = np.array([math.fsum(gu[j] * xq) for j in range(I)])
            u = np.array([math.fsum(gu[I + j] * xq) for j in range(I)])
            h = torch.from_numpy(g / (1.0 + np.exp(-g)) * u).float().bfloat16().double().numpy()
            hc, hs = o.nvfp4_quantize(h[None, :], hg[e])
            hq = decode(hc, hs, hg[e])[0]
            y = (torch.from_numpy(dn) @ torch.from_numpy(hq)).numpy()
            ref[t] += res["w"][t, s] * y
    assert np.allclose(res["out"], ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max()), \
        np.abs(res["out"] - ref).max()


# ------------------------------------------------------------------ router

def pin_router_zero_gate(o):
    """All-zero gate weights give equal logits: experts 0..k-1 in index order,
    each with weight exactly 1/k (closed form)."""
    T, H, E, k = 3, 16, 6, 4
    x = o.bf16_to_f64(_rand_bf16(_rng(1), (T, H), 1.0))
    gw = np.zeros((E, H))
    _, idx, w = o.route(x, gw, None, k)
    assert (idx == np.arange(k)[None, :]).all(), idx
    assert np.all(w == 1.0 / k), w


def pin_router_bias_only(o):
    """Zero gate weights plus a bias: the logits are the bias, so the ranking is
    numpy's stable argsort of -bias and the weights are scipy's softmax of the
    selected biases."""
    from scipy.special import softmax as sp_softmax
    T, H, E, k = 2, 8, 7, 3
    bias = np.array([0.3, -1.0, 2.5, 0.3, 1.25, -0.5, 2.0], dtype=np.float32)
    x = o.bf16_to_f64(_rand_bf16(_rng(2), (T, H), 1.0))
    _, idx, w = o.route(x, np.zeros((E, H)), bias, k)
    exp_idx = np.argsort(-bias.astype(np.float64), kind="stable")[:k]
    for t in range(T):
        assert (idx[t] == exp_idx).all(), (idx[t], exp_idx)
        assert np.allclose(w[t], sp_softmax(bias[exp_idx].astype(np.float64)), rtol=0, atol=1e-15)


def pin_router_brute_force(o):
    """Tiny routers: the selected set is the k-subset with the largest logit
    sum (checked over all subsets), slots are ordered by descending logit, the
    weights equal exp(l_s)/sum exp(l_sel) evaluated without max subtraction,
    and the logits equal torch's fp64 matmul."""
    import torch
    rng = _rng(3)
    for trial in range(12):
        T = int(rng.integers(1, 5))
        H = int(rng.integers(2, 24))
        E = int(rng.integers(2, 9))
        k = int(rng.integers(1, E + 1))
        x = o.bf16_to_f64(_rand_bf16(rng, (T, H), 1.0))
        gw = o.bf16_to_f64(_rand_bf16(rng, (E, H), 0.5))
        bias = (rng.standard_normal(E).astype(np.float32) * 0.1) if trial % 2 else None
        l, idx, w = o.route(x, gw, bias, k)
        ref_l = (torch.from_numpy(x) @ torch.from_numpy(gw).T).numpy()
        if bias is not None:
            ref_l = ref_l + bias.astype(np.float64)[None, :]
        assert np.allclose(l, ref_l, rtol=1e-12, atol=1e-12)
        for t in range(T):
            best = max(itertools.combinations(range(E), k), key=lambda c: sum(ref_l[t, e] for e in c))
            exp_order = sorted(best, key=lambda e: -ref_l[t, e])
            assert list(idx[t]) == exp_order, (trial, t, idx[t], exp_order)
            den = sum(math.exp(ref_l[t, e]) for e in exp_order)
            for s, e in enumerate(exp_order):
                assert abs(w[t, s] - math.exp(ref_l[t, e]) / den) <= 1e-14, (trial, t, s)


def pin_router_exact_ties(o):
    """Two identical gate rows tie exactly; the lower expert index wins."""
    rng = _rng(4)
    T, H, E, k = 4, 32, 8, 3
    x = o.bf16_to_f64(_rand_bf16(rng, (T, H), 1.0))
    gw = o.bf16_to_f64(_rand_bf16(rng, (E, H), 0.05))
    gw[6] = gw[2]
    # make experts 2 and 6 the two largest logits for every token
    gw[2] = gw[6] = np.sign(x[0]) * 0.5
    x[:] = np.abs(x) * np.sign(x[0])[None, :]
    _, idx, w = o.route(x, gw, None, k)
    for t in range(T):
        assert idx[t, 0] == 2 and idx[t, 1] == 6, idx[t]
        assert w[t, 0] == w[t, 1]


def pin_topk_all_is_softmax(o):
    """With top_k = E the weights are the full softmax (scipy) in rank order."""
    from scipy.special import softmax as sp_softmax
    rng = _rng(5)
    T, H, E = 5, 40, 6
    x = o.bf16_to_f64(_rand_bf16(rng, (T, H), 1.0))
    gw = o.bf16_to_f64(_rand_bf16(rng, (E, H), 0.1))
    l, idx, w = o.route(x, gw, None, E)
    p = sp_softmax(l, axis=1)
    for t in range(T):
        assert np.allclose(w[t], p[t, idx[t]], rtol=0, atol=1e-15)
        assert abs(w[t].sum() - 1.0) <= 1e-15


# ------------------------------------------------------------------ grouping

def pin_permute_stable_argsort(o):
    """Counts = bincount, offsets = exclusive cumsum, perm = numpy's stable
    argsort of the flat expert ids, inv_perm its inverse."""
    rng = _rng(6)
    for T, k, E in ((1, 1, 1), (7, 2, 5), (33, 4, 16), (64, 8, 128)):
        idx = rng.integers(0, E, size=(T, k)).astype(np.int32)
        counts, offsets, perm, inv_perm = o.permute(idx, E)
        flat = idx.reshape(-1)
        assert (counts == np.bincount(flat, minlength=E)).all()
        assert (offsets == np.concatenate([[0], np.cumsum(np.bincount(flat, minlength=E))])).all()
        assert (perm == np.argsort(flat, kind="stable")).all()
        assert (inv_perm[perm] == np.arange(T * k)).all()


# ------------------------------------------------------------------ experts

def pin_silu_closed_forms(o):
    """sigmoid(ln 3) = 3/4, sigmoid(-ln 3) = 1/4, silu(0) = 0, and silu(z)
    equals z to within z*e^-z for large z and vanishes for large -z."""
    ln3 = math.log(3.0)
    z = np.array([0.0, ln3, -ln3, 40.0, -40.0])
    s = o.silu(z)
    assert s[0] == 0.0
    assert abs(s[1] - 0.75 * ln3) <= 1e-15
    assert abs(s[2] + 0.25 * ln3) <= 1e-15
    assert abs(s[3] - 40.0) <= 40.0 * math.exp(-40.0) * 2
    assert abs(s[4]) <= 40.0 * math.exp(-40.0) * 2


def _dense_swiglu_torch(x, gu, dn):
    import torch
    X = torch.from_numpy(x)
    I = gu.shape[0] // 2
    g = X @ torch.from_numpy(gu[:I]).T
    u = X @ torch.from_numpy(gu[I:]).T
    return (torch.nn.functional.silu(g) * u @ torch.from_numpy(dn).T).numpy()


def pin_single_expert_dense(o):
    """E = 1, top_k = 1: the layer is a dense SwiGLU MLP (torch fp64)."""
    rng = _rng(8)
    T, H, I = 6, 48, 20
    xb = _rand_bf16(rng, (T, H), 1.0)
    gb = _rand_bf16(rng, (1, H), 0.1)
    gub = _rand_bf16(rng, (1, 2 * I, H), 0.2)
    dnb = _rand_bf16(rng, (1, H, I), 0.2)
    res = o.forward(xb, gb, None, 1, o.ExpertWeights(gub, dnb))
    ref = _dense_swiglu_torch(o.bf16_to_f64(xb), o.bf16_to_f64(gub[0]), o.bf16_to_f64(dnb[0]))
    assert np.allclose(res["out"], ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    assert (res["w"] == 1.0).all()


def pin_topk_all_mixture(o):
    """top_k = E: the output is the softmax-weighted sum of every expert's MLP
    (torch fp64 softmax and einsum)."""
    import torch
    rng = _rng(9)
    T, H, I, E = 5, 32, 12, 4
    xb = _rand_bf16(rng, (T, H), 1.0)
    gb = _rand_bf16(rng, (E, H), 0.2)
    gub = _rand_bf16(rng, (E, 2 * I, H), 0.2)
    dnb = _rand_bf16(rng, (E, H, I), 0.2)
    res = o.forward(xb, gb, None, E, o.ExpertWeights(gub, dnb))
    x = o.bf16_to_f64(xb)
    p = torch.softmax(torch.from_numpy(x) @ torch.from_numpy(o.bf16_to_f64(gb)).T, dim=1)
    ys = torch.stack([torch.from_numpy(_dense_swiglu_torch(x, o.bf16_to_f64(gub[e]), o.bf16_to_f64(dnb[e])))
                      for e in range(E)], dim=1)  # [T, E, H]
    ref = torch.einsum("te,teh->th", p, ys).numpy()
    assert np.allclose(res["out"], ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def pin_hand_case(o):
    """H = 2, I = 1, E = 2, top_k = 2, worked by hand.

    x = (1, 0); gate rows (1, 0) and (2, 0) give logits 1 and 2, so expert 1 is
    slot 0 with weight e^2/(e+e^2) = e/(1+e) and expert 0 is slot 1.
    Expert 1: gate row (40, 0), up row (3, 0), down column (2, -1):
      g = 40, u = 3, silu(40) = 40 to within 40e^-40, so y = (240, -120).
    Expert 0: gate row (0, 0) makes silu(g) = 0, so y = 0.
    out = e/(1+e) * (240, -120)."""
    f = o.bf16_to_f64  # noqa: F841  (inputs below are bf16-exact integers)
    xb = _bf16_round(np.array([[1.0, 0.0]], dtype=np.float32))
    gb = _bf16_round(np.array([[1.0, 0.0], [2.0, 0.0]], dtype=np.float32))
    gu = np.array([[[0.0, 0.0], [5.0, 0.0]], [[40.0, 0.0], [3.0, 0.0]]], dtype=np.float32)
    dn = np.array([[[7.0], [7.0]], [[2.0], [-1.0]]], dtype=np.float32)
    res = o.forward(xb, gb, None, 2, o.ExpertWeights(_bf16_round(gu), _bf16_round(dn)))
    assert list(res["idx"][0]) == [1, 0]
    c = math.e / (1.0 + math.e)
    exp = np.array([240.0 * c, -120.0 * c])
    assert np.allclose(res["out"][0], exp, rtol=1e-14, atol=0), (res["out"], exp)
    assert abs(res["w"][0, 0] - c) <= 1e-15 and abs(res["w"][0, 1] - (1 - c)) <= 1e-15


def _small_layer(rng, T=9, H=24, I=8, E=6, k=3):
    return dict(xb=_rand_bf16(rng, (T, H), 1.0), gb=_rand_bf16(rng, (E, H), 0.3),
                gub=_rand_bf16(rng, (E, 2 * I, H), 0.2), dnb=_rand_bf16(rng, (E, H, I), 0.2), k=k)


def pin_token_order_equivariance(o):
    """Permuting the tokens permutes the output rows exactly."""
    rng = _rng(10)
    L = _small_layer(rng)
    a = o.forward(L["xb"], L["gb"], None, L["k"], o.ExpertWeights(L["gub"], L["dnb"]))["out"]
    p = rng.permutation(L["xb"].shape[0])
    b = o.forward(L["xb"][p], L["gb"], None, L["k"], o.ExpertWeights(L["gub"], L["dnb"]))["out"]
    assert np.array_equal(a[p], b)


def pin_down_scaling(o):
    """Doubling w_down (exact in bf16) doubles the output exactly; the routing
    does not depend on the expert weights."""
    rng = _rng(11)
    L = _small_layer(rng)
    a = o.forward(L["xb"], L["gb"], None, L["k"], o.ExpertWeights(L["gub"], L["dnb"]))
    dn2 = _bf16_round(o.bf16_to_f64(L["dnb"]).astype(np.float32) * 2)
    b = o.forward(L["xb"], L["gb"], None, L["k"], o.ExpertWeights(L["gub"], dn2))
    assert np.array_equal(2 * a["out"], b["out"])
    assert np.array_equal(a["idx"], b["idx"])


def pin_sampled_tokens(o):
    """Asking for a subset of tokens returns exactly those rows of the full
    output, and the routing of the whole batch is unchanged."""
    rng = _rng(12)
    L = _small_layer(rng)
    W = o.ExpertWeights(L["gub"], L["dnb"])
    full = o.forward(L["xb"], L["gb"], None, L["k"], W)
    sub = o.forward(L["xb"], L["gb"], None, L["k"], W, tokens=[7, 2])
    assert np.array_equal(sub["out"], full["out"][[7, 2]])
    assert np.array_equal(sub["perm"], full["perm"])


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
