"""Pins for the oracle's FP8 input path (oracle.dequant_e4m3, oracle.case_inputs_f64).

The FP8 inputs of the "FlashAttention-3 (BN)" page, section "Low precision (FP8)
and reducing quantisation error", are e4m3 codes with one fp32 dequantisation
scale per (batch, head).  The oracle turns them into float64 values before the
exact attention; these tests pin that step to hand-derived products
(tests/golden/e4m3_dequant_cases.json), not to a second copy of the formula:
B = N differs from H, so a scale broadcast over the wrong axis still runs but
gives other numbers, and q, k, v carry different scales, so a tensor
dequantised with another tensor's scale fails too.  The single-key case pins
the whole FP8 oracle path end to end (N_k = 1: the softmax weight is 1).
Planted mistakes (wrong broadcast axis, scale ignored, v dequantised with k's
scale) are shown to fail the pins.
"""

import json
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3_dequant_cases.json")


def _load():
    with open(GOLDEN) as f:
        g = json.load(f)
    B, N, H, d = g["shape"]
    inputs = {}
    for col, name in ((5, "q"), (6, "k"), (7, "v")):
        codes = torch.zeros((B, N, H, d), dtype=torch.float32)
        for e in g["entries"]:
            codes[e[0], e[1], e[2], e[3]] = e[4]
        c8 = codes.to(torch.float8_e4m3fn)
        # every listed code must be exactly representable
        assert torch.equal(c8.to(torch.float32), codes)
        inputs[name] = c8
        inputs[name + "_descale"] = torch.tensor(g["descale"][name], dtype=torch.float32)
    return g, inputs


def _expected(g, col):
    B, N, H, d = g["shape"]
    x = np.zeros((B, N, H, d))
    for e in g["entries"]:
        x[e[0], e[1], e[2], e[3]] = e[col]
    return x


def _check_dequant(fn_inputs):
    g, inputs = _load()
    q, k, v = fn_inputs(inputs)
    for got, col in ((q, 5), (k, 6), (v, 7)):
        exp = _expected(g, col)
        if got.shape != exp.shape or not np.array_equal(got, exp):
            return False
    return True


def test_dequant_matches_hand_products():
    assert _check_dequant(oracle.case_inputs_f64)
    g, inputs = _load()
    for col, name in ((5, "q"), (6, "k"), (7, "v")):
        x = oracle.dequant_e4m3(inputs[name], inputs[name + "_descale"])
        assert x.dtype == np.float64
        assert np.array_equal(x, _expected(g, col))


def test_single_key_attention_through_fp8_inputs():
    g, inputs = _load()
    q, k, v = oracle.case_inputs_f64(inputs)
    sk = g["single_key"]
    O, lse = oracle.attention(q, k[:, :1], v[:, :1], sk["scale"], False)
    B, N, H, d = g["shape"]
    O_exp = np.zeros((B, N, H, d))
    for b, h, t, val in sk["O_nonzero"]:
        O_exp[b, :, h, t] = val
    lse_exp = np.zeros((B, H, N))
    for b, h, i, val in sk["lse_nonzero"]:
        lse_exp[b, h, i] = val
    assert np.array_equal(O, O_exp)
    assert np.allclose(lse, lse_exp, rtol=1e-15, atol=0.0)


def _wrong_axis(inputs):
    out = []
    for n in ("q", "k", "v"):
        x = oracle.to_f64(inputs[n])
        s = oracle.to_f64(inputs[n + "_descale"])
        out.append(x * s[None, :, :, None])          # scale indexed by (n, h)
    return tuple(out)


def _scale_ignored(inputs):
    return tuple(oracle.to_f64(inputs[n]) for n in ("q", "k", "v"))


def _v_with_k_scale(inputs):
    return (oracle.dequant_e4m3(inputs["q"], inputs["q_descale"]),
            oracle.dequant_e4m3(inputs["k"], inputs["k_descale"]),
            oracle.dequant_e4m3(inputs["v"], inputs["k_descale"]))


@pytest.mark.parametrize("mutant", [_wrong_axis, _scale_ignored, _v_with_k_scale],
                         ids=lambda f: f.__name__.strip("_"))
def test_planted_mistakes_fail_the_pin(mutant):
    assert not _check_dequant(mutant)
