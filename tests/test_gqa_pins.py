"""Pins of the grouped-query references the GPU parity tests use, on the CPU.

Grouped-query / multi-query attention (the Multi-Query Attention support that
the "FlashAttention (HI)" page lists under "Development and further research",
FlashAttention-2) shares each K/V head among H / H_kv query heads.  The parity
references expand K and V so that query head h reads K/V head h // (H / H_kv),
run the fp64 oracle (forward) or the fp64 gradient oracle (backward) on the
expanded problem, and sum dk, dv over each K/V head's copies.  Here both are checked against torch's own grouped-query attention
(`scaled_dot_product_attention(..., enable_gqa=True)`, fp64 math on the CPU,
gradients by autograd), which groups consecutive query heads the same way.
A planted mistake, the other grouping (query head h with K/V head h % H_kv),
fails the pin.
"""

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import parity
import synthetic


def _bhnd(a):
    return torch.from_numpy(np.ascontiguousarray(a)).permute(0, 2, 1, 3)   # [B, H, N, d]


def _library(q, k, v, scale, causal):
    return F.scaled_dot_product_attention(_bhnd(q), _bhnd(k), _bhnd(v), is_causal=causal,
                                          scale=scale, enable_gqa=True)


# B, H, H_kv, N_q, N_k, d, causal (causal cases square: the library's top-left
# causal mask equals the bottom-right one there)
SHAPES = [(2, 6, 2, 33, 33, 16, True), (1, 4, 1, 20, 45, 8, False), (2, 8, 4, 17, 17, 8, False)]


def _inputs(shape, seed):
    B, H, H_kv, N_q, N_k, d, causal = shape
    case = synthetic.custom_case(B, H, N_q, N_k, d, causal, "bf16", outliers=False, H_kv=H_kv,
                                 seed=seed)
    return case, synthetic.make_inputs(case)


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_forward_reference_matches_the_library_grouping(oracle_lib, shape):
    case, inputs = _inputs(shape, 300 + SHAPES.index(shape))
    O, lse = parity.oracle_full(case, inputs)
    q, k, v = oracle.case_inputs_f64(inputs)
    ref = _library(q, k, v, case.scale, case.causal).permute(0, 2, 1, 3).numpy()
    assert np.abs(O - ref).max() < 1e-12


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_backward_reference_matches_library_autograd(shape):
    case, inputs = _inputs(shape, 400 + SHAPES.index(shape))
    q, k, v = oracle.case_inputs_f64(inputs)
    dO = oracle.to_f64(synthetic.make_grad(case))
    rq, rk, rv = parity.backward_gqa_reference(q, k, v, dO, case.scale, case.causal)
    tq, tk, tv = (_bhnd(a).clone().requires_grad_(True) for a in (q, k, v))
    out = F.scaled_dot_product_attention(tq, tk, tv, is_causal=case.causal, scale=case.scale,
                                         enable_gqa=True)
    out.backward(_bhnd(dO))
    for name, mine, lib in (("dq", rq, tq.grad), ("dk", rk, tk.grad), ("dv", rv, tv.grad)):
        lib = lib.permute(0, 2, 1, 3).numpy()
        assert mine.shape == lib.shape, name
        assert np.abs(mine - lib).max() < 1e-10, name


def test_the_other_grouping_fails_the_pin(oracle_lib):
    # planted mistake: query head h with K/V head h % H_kv (np.tile instead of np.repeat)
    case, inputs = _inputs(SHAPES[0], 300)
    q, k, v = oracle.case_inputs_f64(inputs)
    g = q.shape[2] // k.shape[2]
    O_wrong, _ = oracle.attention(q, np.tile(k, (1, 1, g, 1)), np.tile(v, (1, 1, g, 1)),
                                  case.scale, case.causal)
    ref = _library(q, k, v, case.scale, case.causal).permute(0, 2, 1, 3).numpy()
    assert np.abs(O_wrong - ref).max() > 1e-3
