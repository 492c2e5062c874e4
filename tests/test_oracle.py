"""CPU tests of the oracle against its pins, plus planted-mistake checks.

The second half loads fresh copies of the oracle module, plants one plausible
mistake in each (a wrong sign, a dropped term, a swapped operand, a wrong
index or layout) and checks that at least one pin catches it, so that the
pins are known to constrain every step of the oracle.
"""
import importlib.util
import os
import sys

import numpy as np
import pytest

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
import oracle_pins  # noqa: E402

from oracle import moe_oracle  # noqa: E402

ORACLE_FILE = moe_oracle.__file__


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin(moe_oracle)


def _fresh_copy(tag):
    spec = importlib.util.spec_from_file_location(f"oracle_mutant_{tag}", ORACLE_FILE)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _mut_silu_sign(m):
    m.silu = lambda z: z / (1.0 + np.exp(z))


def _mut_no_renorm(m):
    orig_softmax = m.softmax

    def route(x, gate_w, bias, top_k):
        l = m.router_logits(x, gate_w, bias)
        p = orig_softmax(l)
        idx = np.stack([m.topk_order(l[t], top_k) for t in range(l.shape[0])]).astype(np.int32)
        w = np.take_along_axis(p, idx.astype(np.int64), axis=1)
        return l, idx, w
    m.route = route


def _mut_tie_high_index(m):
    m.topk_order = lambda l_row, k: np.lexsort((-np.arange(l_row.shape[0]), -l_row))[:k]


def _mut_topk_smallest(m):
    m.topk_order = lambda l_row, k: np.lexsort((np.arange(l_row.shape[0]), l_row))[:k]


def _mut_gate_up_swapped(m):
    def expert_swiglu(X, w_gu, w_dn):
        I = w_gu.shape[0] // 2
        return np.stack([w_dn @ (m.silu(w_gu[I:] @ x) * (w_gu[:I] @ x)) for x in X])
    m.expert_swiglu = expert_swiglu


def _mut_down_layout(m):
    def expert_swiglu(X, w_gu, w_dn):
        I = w_gu.shape[0] // 2
        return np.stack([(m.silu(w_gu[:I] @ x) * (w_gu[I:] @ x)) @ w_dn.reshape(I, -1) for x in X])
    m.expert_swiglu = expert_swiglu


def _mut_bias_sign(m):
    orig = m.router_logits

    def router_logits(x, gate_w, bias):
        return orig(x, gate_w, None if bias is None else -np.asarray(bias))
    m.router_logits = router_logits


def _mut_logit_drop_last_h(m):
    orig = m.router_logits

    def router_logits(x, gate_w, bias):
        return orig(x[:, :-1], gate_w[:, :-1], bias)
    m.router_logits = router_logits


def _mut_perm_unstable(m):
    orig = m.permute

    def permute(idx, E):
        counts, offsets, perm, inv = orig(idx, E)
        perm = perm.copy()
        for e in range(E):
            perm[offsets[e]:offsets[e + 1]] = perm[offsets[e]:offsets[e + 1]][::-1]
        inv = np.empty_like(perm)
        inv[perm] = np.arange(perm.shape[0])
        return counts, offsets, perm, inv
    m.permute = permute


def _mut_combine_drops_slot(m):
    # the combine loses the last slot's contribution
    orig_route = m.route

    def route(x, gate_w, bias, top_k):
        l, idx, w = orig_route(x, gate_w, bias, top_k)
        if top_k > 1:
            w = w.copy()
            w[:, -1] = 0.0
        return l, idx, w
    m.route = route


def _mut_bf16_shift(m):
    m.bf16_to_f64 = lambda bits: (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32)
                                  << np.uint32(15)).view(np.float32).astype(np.float64)


def _mut_e2m1_mantissa(m):
    def e2m1_to_f64(code):
        c = np.asarray(code, dtype=np.int64) & 0xF
        sign = np.where(c >> 3, -1.0, 1.0)
        e = (c >> 1) & 3
        mm = c & 1
        mag = np.where(e == 0, 0.5 * mm, np.ldexp(1.0 + mm, e - 1))
        return sign * mag
    m.e2m1_to_f64 = e2m1_to_f64


def _mut_e4m3_bias(m):
    orig = m.e4m3_to_f64
    m.e4m3_to_f64 = lambda b: orig(b) * 0.5


def _mut_nibble_order(m):
    orig = m.nvfp4_dequant

    def nvfp4_dequant(codes, scales, glob):
        c = np.asarray(codes, dtype=np.uint8)
        swapped = ((c & 0xF) << 4) | (c >> 4)
        return orig(swapped.astype(np.uint8), scales, glob)
    m.nvfp4_dequant = nvfp4_dequant


def _mut_scale_block(m):
    orig = m.nvfp4_dequant

    def nvfp4_dequant(codes, scales, glob):
        s = np.asarray(scales)
        return orig(codes, s[:, :, ::-1].copy(), glob)
    m.nvfp4_dequant = nvfp4_dequant


def _mut_softmax_no_exp(m):
    m.softmax = lambda l: (l - l.min(axis=-1, keepdims=True)) / (l - l.min(axis=-1, keepdims=True)).sum(
        axis=-1, keepdims=True)


def _mut_nvfp4_globals_swapped(m):
    # the gate/up tensor decoded with the down tensor's global and vice versa
    def get(self, e):
        if self.q_gu is not None:
            (cg, sg, gg), (cd, sd, gd) = self.q_gu, self.q_dn
            gu = m.nvfp4_dequant(cg[e:e + 1], sg[e:e + 1], gd[e:e + 1])[0]
            dn = m.nvfp4_dequant(cd[e:e + 1], sd[e:e + 1], gg[e:e + 1])[0]
            return gu, dn
        return m.bf16_to_f64(self.gu_bits[e]), m.bf16_to_f64(self.dn_bits[e])
    m.ExpertWeights.get = get


def _mut_nvfp4_expert0_global(m):
    # every expert decoded with expert 0's global scale
    def get(self, e):
        if self.q_gu is not None:
            (cg, sg, gg), (cd, sd, gd) = self.q_gu, self.q_dn
            gu = m.nvfp4_dequant(cg[e:e + 1], sg[e:e + 1], gg[0:1])[0]
            dn = m.nvfp4_dequant(cd[e:e + 1], sd[e:e + 1], gd[0:1])[0]
            return gu, dn
        return m.bf16_to_f64(self.gu_bits[e]), m.bf16_to_f64(self.dn_bits[e])
    m.ExpertWeights.get = get


def _mut_nvfp4_expert0_codes(m):
    # every expert decoded from expert 0's codes
    def get(self, e):
        if self.q_gu is not None:
            (cg, sg, gg), (cd, sd, gd) = self.q_gu, self.q_dn
            gu = m.nvfp4_dequant(cg[0:1], sg[e:e + 1], gg[e:e + 1])[0]
            dn = m.nvfp4_dequant(cd[0:1], sd[e:e + 1], gd[e:e + 1])[0]
            return gu, dn
        return m.bf16_to_f64(self.gu_bits[e]), m.bf16_to_f64(self.dn_bits[e])
    m.ExpertWeights.get = get


def _mut_w4a4_globals_swapped(m):
    # the token rows quantised with h's global and h with x's
    orig = m.forward_w4a4

    def forward_w4a4(x_bits, gate_w_bits, bias, top_k, weights, x_global, h_global, tokens=None):
        return orig(x_bits, gate_w_bits, bias, top_k, weights, h_global, x_global, tokens=tokens)
    m.forward_w4a4 = forward_w4a4


def _mut_w4a4_expert0_global(m):
    # every expert quantises with expert 0's activation globals
    orig = m.forward_w4a4

    def forward_w4a4(x_bits, gate_w_bits, bias, top_k, weights, x_global, h_global, tokens=None):
        xg = np.full_like(np.asarray(x_global), np.asarray(x_global)[0])
        hg = np.full_like(np.asarray(h_global), np.asarray(h_global)[0])
        return orig(x_bits, gate_w_bits, bias, top_k, weights, xg, hg, tokens=tokens)
    m.forward_w4a4 = forward_w4a4


def _mut_w4a4_h_unquantised(m):
    # h goes to the down projection in bf16, without the NVFP4 step
    def forward_w4a4(x_bits, gate_w_bits, bias, top_k, weights, x_global, h_global, tokens=None):
        x = m.bf16_to_f64(x_bits)
        logits, idx, w = m.route(x, m.bf16_to_f64(gate_w_bits), bias, top_k)
        out = np.zeros_like(x)
        for t in range(x.shape[0]):
            for s in range(top_k):
                e = int(idx[t, s])
                gu, dn = weights.get(e)
                I = gu.shape[0] // 2
                xq = m.nvfp4_fake_quant(x[t:t + 1], np.asarray(x_global)[e])[0]
                out[t] += w[t, s] * (dn @ m.bf16_round(m.silu(gu[:I] @ xq) * (gu[I:] @ xq)))
        return dict(out=out, idx=idx, w=w, logits=logits)
    m.forward_w4a4 = forward_w4a4


def _mut_nvfp4_quant_block32(m):
    # one scale per 32 elements: each pair of 16-element blocks shares the
    # scale of the pair's larger magnitude
    def nvfp4_quantize(a, glob):
        a32 = np.asarray(a, dtype=np.float32)
        R, K = a32.shape
        g = np.float32(glob)
        amax = np.repeat(np.abs(a32.reshape(R, K // 32, 32)).max(axis=2), 2, axis=1)
        scales = m.e4m3_quantize(amax / (np.float32(6.0) * g))
        denom = (m.e4m3_to_f64(scales).astype(np.float32) * g).astype(np.float32)
        recip = (np.float32(1.0) / np.where(denom > 0, denom, np.float32(1.0))).astype(np.float32)
        q = (a32.reshape(R, K // 16, 16) * recip[:, :, None]).astype(np.float32)
        nib = np.where(denom[:, :, None] > 0, m.e2m1_quantize(q), 0).astype(np.uint8).reshape(R, K)
        return (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8), scales
    m.nvfp4_quantize = nvfp4_quantize


def _mut_e2m1_ties_away(m):
    # ties rounded away from zero instead of to the even code
    def e2m1_quantize(v):
        f = np.asarray(v, dtype=np.float32)
        a = np.abs(f.astype(np.float64))
        grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
        d = np.abs(a[..., None] - grid)
        best = d.min(axis=-1, keepdims=True)
        code = (d == best)[..., ::-1].argmax(axis=-1)
        code = 7 - code
        return ((np.signbit(f).astype(np.int64) << 3) | code).astype(np.uint8)
    m.e2m1_quantize = e2m1_quantize


def _mut_e4m3_truncate(m):
    # scales truncated toward zero instead of rounded to nearest
    def e4m3_quantize(v):
        a = np.abs(np.asarray(v, dtype=np.float32).astype(np.float64))
        out = np.zeros(a.shape, dtype=np.uint8)
        import torch
        vals = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).float().numpy()
        pos = [(float(vals[c]), c) for c in range(0x7F) if np.isfinite(vals[c])]
        for i, x in np.ndenumerate(a):
            out[i] = max(c for val, c in pos if val <= max(x, 0.0))
        return out
    m.e4m3_quantize = e4m3_quantize


def _mut_nvfp4_scale_without_global(m):
    # the block scale ignores the global: e4m3(amax / 6)
    orig = m.nvfp4_quantize

    def nvfp4_quantize(a, glob):
        codes, _ = orig(a, glob)
        a32 = np.asarray(a, dtype=np.float32)
        R, K = a32.shape
        amax = np.abs(a32.reshape(R, K // 16, 16)).max(axis=2)
        return codes, m.e4m3_quantize(amax / np.float32(6.0))
    m.nvfp4_quantize = nvfp4_quantize


def _mut_q8_block16(m):
    # one scale per 16 elements instead of 32
    def q8_dequant(codes, scales):
        c = np.asarray(codes, dtype=np.int8).astype(np.float64)
        sc = m.f16_to_f64(np.asarray(scales, dtype=np.uint16))
        rep = np.repeat(sc, 16, axis=2)
        rep = np.concatenate([rep, rep], axis=2)[:, :, :c.shape[2]]
        return c * rep
    m.q8_dequant = q8_dequant


def _mut_q8_unsigned(m):
    # codes read as unsigned bytes
    def q8_dequant(codes, scales):
        c = np.asarray(codes, dtype=np.int8).view(np.uint8).astype(np.float64)
        return c * np.repeat(m.f16_to_f64(np.asarray(scales, dtype=np.uint16)), 32, axis=2)
    m.q8_dequant = q8_dequant


def _mut_f16_bias(m):
    # fp16 exponent bias taken as 16
    orig = m.f16_to_f64
    m.f16_to_f64 = lambda bits: orig(bits) * 0.5


def _mut_q8_expert0_scales(m):
    # every expert decoded with expert 0's scales
    def get(self, e):
        if self.q8_gu is not None:
            (cg, sg), (cd, sd) = self.q8_gu, self.q8_dn
            return m.q8_dequant(cg[e:e + 1], sg[0:1])[0], m.q8_dequant(cd[e:e + 1], sd[0:1])[0]
        if self.q_gu is not None:
            c, s, g = self.q_gu
            gu = m.nvfp4_dequant(c[e:e + 1], s[e:e + 1], g[e:e + 1])[0]
            c, s, g = self.q_dn
            dn = m.nvfp4_dequant(c[e:e + 1], s[e:e + 1], g[e:e + 1])[0]
            return gu, dn
        return m.bf16_to_f64(self.gu_bits[e]), m.bf16_to_f64(self.dn_bits[e])
    m.ExpertWeights.get = get


MUTANTS = [v for k, v in sorted(globals().items()) if k.startswith("_mut_")]


@pytest.mark.parametrize("mutant", MUTANTS, ids=lambda f: f.__name__[5:])
def test_pins_catch_planted_mistake(mutant):
    m = _fresh_copy(mutant.__name__)
    mutant(m)
    failures = 0
    for pin in oracle_pins.ALL_PINS:
        try:
            with np.errstate(all="ignore"):   # a planted mistake may divide by zero
                pin(m)
        except Exception:
            failures += 1
    assert failures > 0, f"no pin caught mutant {mutant.__name__}"
