"""Shared helpers for the GPU parity tests: run a case through the C ABI and
compare element by element with the fp64 CPU oracle."""

from __future__ import annotations

import numpy as np
import torch

import io_aware_exact_03_gb300 as attn
import oracle
import synthetic

# Tolerances stated for this path (O max / mean absolute error, lse absolute error).
# e4m3: O is written as bf16, whose spacing is 0.125 for |O| in [16, 32) and
# 0.25 in [32, 64) (C5's x10 outliers put |O| near 40 on some rows), so the
# 6e-2 bound is read as a bound on the computation: each element may also be
# off by half a bf16 ulp of the exact value, its own output rounding.
TOL = {
    "bf16": dict(o_max=1e-2, o_mean=1e-3, lse=1e-3),
    "fp16": dict(o_max=1e-2, o_mean=1e-3, lse=1e-3),
    "e4m3": dict(o_max=6e-2, o_mean=None, lse=1e-3, out_half_ulp=True),
}


def bf16_half_ulp(x):
    """Half the spacing of bf16 values (8 significant bits) at |x|."""
    ax = np.maximum(np.abs(np.asarray(x, dtype=np.float64)), 2.0 ** -126)
    return np.exp2(np.floor(np.log2(ax)) - 8.0)


def to_device(inputs: dict) -> dict:
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inputs.items()}


def run_gpu(case: synthetic.Case, dev: dict, impl: str = "tc"):
    """O [B,N_q,H,d] and lse [B,H,N_q] from the GPU, as float64 numpy arrays."""
    q, k, v = dev["q"], dev["k"], dev["v"]
    kw = dict(scale=case.scale, causal=case.causal)
    if impl == "tc":
        if case.dtype == "e4m3":
            o, lse = attn.attn_fwd_fp8(q, k, v, dev["q_descale"], dev["k_descale"],
                                       dev["v_descale"], **kw)
        else:
            o, lse = attn.attn_fwd(q, k, v, **kw)
    elif impl == "fp8ws":
        o, lse = attn.attn_fwd_fp8_ws(q, k, v, dev["q_descale"], dev["k_descale"],
                                      dev["v_descale"], **kw)
    elif impl == "gqa":
        o, lse = attn.attn_fwd_gqa(q, k, v, q_descale=dev.get("q_descale"),
                                   k_descale=dev.get("k_descale"),
                                   v_descale=dev.get("v_descale"), **kw)
    elif impl.startswith("split"):
        n = int(impl[len("split"):])
        o, lse = attn.attn_fwd_splitkv(q, k, v, n, q_descale=dev.get("q_descale"),
                                       k_descale=dev.get("k_descale"),
                                       v_descale=dev.get("v_descale"), **kw)
    elif impl == "simt":
        o, lse = attn.attn_fwd_simt(q, k, v, q_descale=dev.get("q_descale"),
                                    k_descale=dev.get("k_descale"),
                                    v_descale=dev.get("v_descale"), **kw)
    else:
        raise ValueError(impl)
    attn.attn_check_status()
    return o.double().cpu().numpy(), lse.double().cpu().numpy()


def oracle_full(case, inputs):
    q, k, v = oracle.case_inputs_f64(inputs)
    if k.shape[2] != q.shape[2]:
        # grouped-query attention: query head h attends with K/V head h // group
        g = q.shape[2] // k.shape[2]
        k, v = np.repeat(k, g, axis=2), np.repeat(v, g, axis=2)
    return oracle.attention(q, k, v, case.scale, case.causal)


def backward_gqa_reference(q, k, v, dO, scale, causal):
    """fp64 gradients with K/V shared by H / H_kv query heads: the oracle
    differentiates the expanded problem (query head h with its own copy of K/V
    head h // group) and dk, dv are summed over each head's copies, which is
    the gradient of the shared tensors.  Arrays [B, N, heads, d]."""
    from oracle import backward
    B, N_k, H_kv, d = k.shape
    g = q.shape[2] // H_kv
    rq, rk, rv = backward.attention_backward(q, np.repeat(k, g, axis=2), np.repeat(v, g, axis=2),
                                             dO, scale, causal)
    return rq, rk.reshape(B, N_k, H_kv, g, d).sum(axis=3), rv.reshape(B, N_k, H_kv, g, d).sum(axis=3)


def compare(case, O_gpu, lse_gpu, O_ref, lse_ref, tol=None):
    """Element-wise check; rows with lse = -inf must have O == 0 exactly."""
    tol = tol or TOL[case.dtype]
    O_gpu = np.asarray(O_gpu)
    O_ref = np.asarray(O_ref)
    assert O_gpu.shape == O_ref.shape
    assert np.all(np.isfinite(O_gpu)), "non-finite output"
    err = np.abs(O_gpu - O_ref)
    bound = tol["o_max"] + (bf16_half_ulp(O_ref) if tol.get("out_half_ulp") else 0.0)
    msg = (f"{case.name}: O max err {err.max():.3e} mean {err.mean():.3e}, "
           f"worst excess over the bound {(err - bound).max():.3e}")
    assert np.all(err <= bound), msg
    if tol["o_mean"] is not None:
        assert err.mean() <= tol["o_mean"], msg
    lse_gpu = np.asarray(lse_gpu)
    lse_ref = np.asarray(lse_ref)
    inf_ref = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse_gpu), inf_ref), f"{case.name}: -inf rows differ"
    if (~inf_ref).any():
        le = np.abs(lse_gpu[~inf_ref] - lse_ref[~inf_ref])
        assert le.max() <= tol["lse"], f"{case.name}: lse max err {le.max():.3e}"
    return dict(o_max=float(err.max()), o_mean=float(err.mean()))


def check_full(case, impl="tc"):
    inputs = synthetic.make_inputs(case)
    O, lse = run_gpu(case, to_device(inputs), impl)
    O_ref, lse_ref = oracle_full(case, inputs)
    return compare(case, O, lse, O_ref, lse_ref)


def check_sampled(case, impl="tc", n=256, inputs=None, dev=None):
    inputs = inputs if inputs is not None else synthetic.make_inputs(case)
    dev = dev if dev is not None else to_device(inputs)
    O, lse = run_gpu(case, dev, impl)
    rows = synthetic.sample_rows(case, n)
    q, k, v = oracle.case_inputs_f64(inputs)
    O_ref, lse_ref = oracle.attention_rows(q, k, v, case.scale, case.causal, rows)
    O_s = O[rows[:, 0], rows[:, 2], rows[:, 1]]
    lse_s = lse[rows[:, 0], rows[:, 1], rows[:, 2]]
    return compare(case, O_s, lse_s, O_ref, lse_ref)
