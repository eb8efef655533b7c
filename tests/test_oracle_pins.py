"""Pins for the CPU oracle, checked against things other than itself.

Each pin is a fact fixed by the pages or by mathematics:
  * hand-derived closed forms (tests/golden/closed_form_cases.json);
  * brute force: a pure-Python triple loop over the definition on tiny inputs;
  * special cases with closed forms: N_k = 1, identical key rows, Q = 0 causal;
  * invariances: shifting every key by one vector, permuting keys with values;
  * the online (one-pass) result equals the two-pass softmax (the online-softmax
    claim of the "FlashAttention (HI)" page, section "Online softmax computation");
  * a library special case: torch's fp64 math attention on the CPU.
The mutant tests rebuild the oracle with one planted mistake each (a dropped
scale, a wrong sign, a wrong index, an off-by-one mask, a missing rescale, a
wrong lse) and require at least one pin to fail.
"""

import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import two_pass
import synthetic

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_form_cases.json")
TOL = 1e-12


def _num(x):
    return -math.inf if x == "-Infinity" else float(x)


def _as4(rows):
    """[N][d] nested list -> array [1, N, 1, d]."""
    a = np.asarray(rows, dtype=np.float64)
    return a[None, :, None, :]


def brute_force(q, k, v, scale, causal):
    """Pure-Python loops over the definition softmax(scale * q K^T) V."""
    B, N_q, H, d = q.shape
    N_k = k.shape[1]
    O = np.zeros((B, N_q, H, d))
    lse = np.zeros((B, H, N_q))
    for b in range(B):
        for h in range(H):
            for i in range(N_q):
                keys = [j for j in range(N_k) if (not causal) or j <= i + N_k - N_q]
                if not keys:
                    lse[b, h, i] = -math.inf
                    continue
                s = {}
                for j in keys:
                    acc = 0.0
                    for t in range(d):
                        acc += float(q[b, i, h, t]) * float(k[b, j, h, t])
                    s[j] = scale * acc
                mx = max(s.values())
                w = {j: math.exp(s[j] - mx) for j in keys}
                tot = sum(w.values())
                for t in range(d):
                    O[b, i, h, t] = sum(w[j] * float(v[b, j, h, t]) for j in keys) / tot
                lse[b, h, i] = mx + math.log(tot)
    return O, lse


def _close(a, b, tol=TOL):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    if a.shape != b.shape:
        return False
    both_inf = np.isinf(a) & np.isinf(b) & (np.sign(a) == np.sign(b))
    with np.errstate(invalid="ignore"):
        diff = np.where(both_inf, 0.0, np.abs(a - b))
    return bool(np.all(np.isfinite(diff)) and diff.max(initial=0.0) <= tol * max(1.0, np.abs(np.where(both_inf, 0, b)).max(initial=0.0)))


def _rng_case(seed, B, H, N_q, N_k, d):
    r = np.random.default_rng(seed)
    return r.standard_normal((B, N_q, H, d)), r.standard_normal((B, N_k, H, d)), r.standard_normal((B, N_k, H, d))


# ---------------------------------------------------------------- the pins
def pin_golden(mutant):
    fails = []
    for c in json.load(open(GOLDEN))["cases"]:
        q, k, v = _as4(c["q"]), _as4(c["k"]), _as4(c["v"])
        O, lse = oracle.attention(q, k, v, c["scale"], c["causal"], n_threads=1, mutant=mutant)
        exp_O = _as4(c["O"])
        exp_lse = np.asarray([_num(x) for x in c["lse"]])[None, None, :]
        if not (_close(O, exp_O) and _close(lse, exp_lse)):
            fails.append(c["name"])
    return fails


def pin_brute_force(mutant):
    fails = []
    for (B, H, N_q, N_k, d, causal, seed) in [(2, 3, 5, 7, 4, False, 1), (2, 3, 5, 7, 4, True, 2),
                                               (1, 2, 7, 5, 3, True, 3), (1, 2, 6, 6, 8, True, 4),
                                               (2, 1, 1, 9, 5, False, 5)]:
        q, k, v = _rng_case(seed, B, H, N_q, N_k, d)
        k = k * 2.0   # spread the scores so rescaling happens often
        scale = 1.0 / math.sqrt(d)
        O_bf, lse_bf = brute_force(q, k, v, scale, causal)
        O, lse = oracle.attention(q, k, v, scale, causal, n_threads=2, mutant=mutant)
        if not (_close(O, O_bf, 1e-12) and _close(lse, lse_bf, 1e-12)):
            fails.append((B, H, N_q, N_k, d, causal))
    return fails


def pin_nk_one(mutant):
    q, k, v = _rng_case(11, 2, 3, 6, 1, 16)
    scale = 0.25
    O, lse = oracle.attention(q, k, v, scale, False, mutant=mutant)
    exp_O = np.broadcast_to(v[:, 0:1, :, :], O.shape)
    exp_lse = scale * np.einsum("bihd,bhd->bhi", q, k[:, 0, :, :])
    return [] if (_close(O, exp_O) and _close(lse, exp_lse)) else ["N_k=1"]


def pin_identical_keys(mutant):
    fails = []
    for causal in (False, True):
        B, H, N, d = 2, 2, 9, 8
        q, _, v = _rng_case(12, B, H, N, N, d)
        kv = np.random.default_rng(13).standard_normal((B, 1, H, d))
        k = np.broadcast_to(kv, (B, N, H, d)).copy()
        scale = 1.0 / math.sqrt(d)
        O, lse = oracle.attention(q, k, v, scale, causal, mutant=mutant)
        cnt = np.array([two_pass.allowed_keys(i, N, N, causal) for i in range(N)])
        exp_O = np.zeros_like(O)
        for i in range(N):
            exp_O[:, i] = v[:, :cnt[i]].mean(axis=1)
        exp_lse = scale * np.einsum("bihd,bhd->bhi", q, kv[:, 0]) + np.log(cnt)[None, None, :]
        if not (_close(O, exp_O) and _close(lse, exp_lse)):
            fails.append(causal)
    return fails


def pin_zero_q_causal(mutant):
    B, H, N, d = 1, 3, 12, 4
    _, k, v = _rng_case(14, B, H, N, N, d)
    q = np.zeros((B, N, H, d))
    O, lse = oracle.attention(q, k, v, 0.5, True, mutant=mutant)
    exp_O = np.cumsum(v, axis=1) / np.arange(1, N + 1)[None, :, None, None]
    exp_lse = np.broadcast_to(np.log(np.arange(1, N + 1))[None, None, :], lse.shape)
    return [] if (_close(O, exp_O) and _close(lse, exp_lse)) else ["Q=0 causal"]


def pin_shift(mutant):
    q, k, v = _rng_case(15, 2, 2, 7, 10, 6)
    u = np.random.default_rng(16).standard_normal((1, 1, 2, 6))
    scale = 0.4
    O1, l1 = oracle.attention(q, k, v, scale, False, mutant=mutant)
    O2, l2 = oracle.attention(q, k + u, v, scale, False, mutant=mutant)
    shift = scale * np.einsum("bihd,hd->bhi", q, u[0, 0])
    return [] if (_close(O1, O2, 1e-11) and _close(l2, l1 + shift, 1e-11)) else ["shift"]


def pin_permutation(mutant):
    q, k, v = _rng_case(17, 1, 2, 5, 11, 4)
    perm = np.random.default_rng(18).permutation(11)
    O1, l1 = oracle.attention(q, k, v, 0.5, False, mutant=mutant)
    O2, l2 = oracle.attention(q, k[:, perm], v[:, perm], 0.5, False, mutant=mutant)
    return [] if (_close(O1, O2, 1e-11) and _close(l1, l2, 1e-11)) else ["permutation"]


PINS = [pin_golden, pin_brute_force, pin_nk_one, pin_identical_keys, pin_zero_q_causal,
        pin_shift, pin_permutation]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin_holds(oracle_lib, pin):
    assert pin(0) == []


@pytest.mark.parametrize("mutant", [1, 2, 3, 4, 5, 6])
def test_planted_mistake_is_caught(oracle_lib, mutant):
    failed = [p.__name__ for p in PINS if p(mutant)]
    assert failed, f"mutant {mutant} passed every pin"


def test_two_pass_matches_brute_force():
    q, k, v = _rng_case(19, 2, 2, 6, 8, 5)
    for causal in (False, True):
        O_bf, lse_bf = brute_force(q, k, v, 0.3, causal)
        O, lse = two_pass.attention_full(q, k, v, 0.3, causal)
        assert _close(O, O_bf) and _close(lse, lse_bf)


# --------------------------------------------- one-pass == two-pass on the cases
def test_one_pass_equals_two_pass_full_C1_C2(oracle_lib):
    for name in ("C1", "C2"):
        case = synthetic.CASES[name]
        q, k, v = oracle.case_inputs_f64(synthetic.make_inputs(case))
        O1, l1 = oracle.attention(q, k, v, case.scale, case.causal)
        O2, l2 = two_pass.attention_full(q, k, v, case.scale, case.causal)
        assert np.abs(O1 - O2).max() < 1e-12
        assert np.abs(l1 - l2).max() < 1e-12


@pytest.mark.parametrize("name", ["C3", "C4", "C5", "LKV", "D256", "D256F"])
def test_one_pass_equals_two_pass_sampled(oracle_lib, name):
    case = synthetic.CASES.get(name) or synthetic.EXTRA_CASES[name]
    q, k, v = oracle.case_inputs_f64(synthetic.make_inputs(case))
    rows = synthetic.sample_rows(case, 64)
    O1, l1 = oracle.attention_rows(q, k, v, case.scale, case.causal, rows)
    O2, l2 = two_pass.attention_rows(q, k, v, case.scale, case.causal, rows)
    assert np.abs(O1 - O2).max() < 1e-12
    assert np.abs(l1 - l2).max() < 1e-12


def test_library_special_case_sdpa(oracle_lib):
    """torch's fp64 math attention on the CPU (top-left causal == bottom-right when square)."""
    import torch
    import torch.nn.functional as F
    for causal, seed in ((False, 21), (True, 22)):
        q, k, v = _rng_case(seed, 2, 3, 33, 33, 16)
        O, lse = oracle.attention(q, k, v, 0.25, causal)
        t = lambda a: torch.from_numpy(a).permute(0, 2, 1, 3)   # [B,H,N,d]
        ref = F.scaled_dot_product_attention(t(q), t(k), t(v), is_causal=causal, scale=0.25)
        ref = ref.permute(0, 2, 1, 3).numpy()
        assert np.abs(O - ref).max() < 1e-12


def test_rows_call_matches_full_call(oracle_lib):
    q, k, v = _rng_case(23, 2, 3, 20, 20, 8)
    case = synthetic.custom_case(2, 3, 20, 20, 8, True)
    rows = synthetic.sample_rows(case, 40)
    O, lse = oracle.attention(q, k, v, 0.35, True)
    Or, lr = oracle.attention_rows(q, k, v, 0.35, True, rows)
    assert np.array_equal(Or, O[rows[:, 0], rows[:, 2], rows[:, 1]])
    assert np.array_equal(lr, lse[rows[:, 0], rows[:, 1], rows[:, 2]])
