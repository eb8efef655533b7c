"""Pins for the backward-pass oracle (oracle/backward.py), on the CPU.

The gradients are checked against facts other than the oracle's own formulas:
  * brute force: central finite differences of L = <dO, O(q, k, v)> through the
    already pinned forward oracle (oracle.attention), element by element, on
    tiny inputs (causal and not, N_q != N_k, rows with no allowed key);
  * invariants of the softmax: every row of dS sums to zero, so the key
    gradients sum to zero over keys; the rows of P sum to one, so the value
    gradients sum to the sum of dO over rows that see a key;
  * a special case: with one key, O does not depend on q or k (dq = dk = 0)
    and dv is the sum of dO.
Each planted mistake (a dropped scale, a missing subtraction of D, a
transposed dS, a top-left causal mask) must fail at least one pin.
"""

import numpy as np
import pytest

import oracle
from oracle import backward

FD_EPS = 1e-6
FD_TOL = 1e-6   # central differences of smooth fp64 functions: O(eps^2) + rounding / eps

SHAPES = [
    # B, H, N_q, N_k, d, causal
    (1, 1, 4, 4, 3, False),
    (1, 2, 5, 3, 4, True),      # N_q > N_k: rows 0 and 1 see no key
    (2, 1, 3, 6, 2, True),      # N_q < N_k: bottom-right alignment
    (1, 1, 6, 6, 3, True),
]


def _inputs(shape, seed):
    B, H, N_q, N_k, d, causal = shape
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, N_q, H, d))
    k = rng.standard_normal((B, N_k, H, d))
    v = rng.standard_normal((B, N_k, H, d))
    dO = rng.standard_normal((B, N_q, H, d))
    return q, k, v, dO, 0.7, causal


def _loss(q, k, v, dO, scale, causal):
    o, _ = oracle.attention(q, k, v, scale, causal, n_threads=1)
    return float((o * dO).sum())


def _finite_diff(q, k, v, dO, scale, causal):
    """Central differences of <dO, O> w.r.t. every element of q, k, v."""
    grads = []
    for which in range(3):
        base = [q.copy(), k.copy(), v.copy()]
        g = np.zeros_like(base[which])
        for idx in np.ndindex(*g.shape):
            plus = [x.copy() for x in base]
            minus = [x.copy() for x in base]
            plus[which][idx] += FD_EPS
            minus[which][idx] -= FD_EPS
            g[idx] = (_loss(*plus, dO, scale, causal) - _loss(*minus, dO, scale, causal)) / (2 * FD_EPS)
        grads.append(g)
    return grads


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_gradients_match_finite_differences(shape):
    q, k, v, dO, scale, causal = _inputs(shape, 7)
    fd = _finite_diff(q, k, v, dO, scale, causal)
    got = backward.attention_backward(q, k, v, dO, scale, causal)
    for name, a, b in zip(("dq", "dk", "dv"), got, fd):
        assert np.abs(a - b).max() < FD_TOL, name


@pytest.mark.parametrize("causal", [False, True])
def test_key_gradients_sum_to_zero_and_value_gradients_to_dO(causal):
    B, H, N_q, N_k, d = 2, 3, 40, 33, 8
    q, k, v, dO, scale, _ = _inputs((B, H, N_q, N_k, d, causal), 11)
    dq, dk, dv = backward.attention_backward(q, k, v, dO, scale, causal)
    assert np.abs(dk.sum(axis=1)).max() < 1e-12
    sees = np.array([min(N_k, max(0, i + N_k - N_q + 1)) if causal else N_k for i in range(N_q)]) > 0
    want = dO[:, sees].sum(axis=1)
    assert np.abs(dv.sum(axis=1) - want).max() < 1e-12


def test_one_key_gives_zero_q_k_gradients():
    q, k, v, dO, scale, _ = _inputs((2, 2, 7, 1, 5, False), 3)
    dq, dk, dv = backward.attention_backward(q, k, v, dO, scale, False)
    assert np.abs(dq).max() == 0.0 and np.abs(dk).max() == 0.0
    assert np.abs(dv[:, 0] - dO.sum(axis=1)).max() < 1e-12


def test_rows_without_keys_contribute_nothing():
    # N_q > N_k, causal: rows 0 .. N_q - N_k - 1 see no key; their dO must not matter
    q, k, v, dO, scale, _ = _inputs((1, 2, 9, 4, 3, True), 5)
    base = backward.attention_backward(q, k, v, dO, scale, True)
    dO2 = dO.copy()
    dO2[:, :5] = 123.0
    other = backward.attention_backward(q, k, v, dO2, scale, True)
    for a, b in zip(base, other):
        assert np.array_equal(a[:, 5:] if a.shape[1] == 9 else a, b[:, 5:] if b.shape[1] == 9 else b)
    assert np.abs(base[0][:, :5]).max() == 0.0


@pytest.mark.parametrize("mutant", [1, 2, 3, 4])
def test_planted_mistakes_are_caught(mutant):
    caught = False
    for shape in SHAPES:
        q, k, v, dO, scale, causal = _inputs(shape, 7)
        if mutant == 3 and shape[2] != shape[3]:
            continue  # dS^T @ K needs a square score matrix
        fd = _finite_diff(q, k, v, dO, scale, causal)
        got = backward.attention_backward(q, k, v, dO, scale, causal, mutant=mutant)
        if any(np.abs(a - b).max() > FD_TOL for a, b in zip(got, fd)):
            caught = True
            break
    assert caught
