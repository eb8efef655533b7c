"""GPU parity of the backward pass (attn_bwd) against the fp64 gradient oracle.

The GPU path runs the tensor-core forward for o and lse, then attn_bwd; the
oracle (oracle/backward.py) differentiates the exact definition on the same
rounded q, k, v and dO.  Cases cover ragged tiles, N_q != N_k under the causal
mask (keys no row attends, rows with no key), N_k = 1, both head dimensions and
both 16-bit types; the BWD workload (C3's shape) is checked on sampled key and
query rows.

Tolerance (no figure on the pages or in the workloads for gradients), from the
arithmetic: each gradient is rounded once to bf16 on output (relative 2^-9),
and its terms use P and dS rounded to bf16 (relative 2^-9 each) and the
forward's bf16 o (in D), accumulated in fp32.  The rounding errors of a sum of
n terms grow like sqrt(n) times one term's, while the sum itself is bounded by
the largest gradient, so the bound is stated against max |reference| of each
tensor: max |err| <= 2e-2 * max|ref| + 1e-4 and mean |err| <= 2e-3 * max|ref|.
"""

import zlib

import numpy as np
import pytest
import torch

import io_aware_exact_03_gb300 as attn
import oracle
from oracle import backward
import parity
import synthetic

pytestmark = pytest.mark.gpu

MAX_REL, MEAN_REL, ABS = 2e-2, 2e-3, 1e-4

CASES = [
    # B, H, N_q, N_k, d, causal, dtype
    (1, 1, 1, 1, 64, False, "bf16"),
    (1, 1, 128, 128, 64, False, "bf16"),
    (2, 3, 200, 200, 64, True, "bf16"),
    (1, 2, 300, 300, 128, True, "bf16"),
    (2, 2, 129, 383, 128, False, "fp16"),
    (1, 2, 100, 300, 128, True, "bf16"),     # N_q < N_k: bottom-right alignment
    (1, 2, 300, 100, 64, True, "bf16"),      # rows 0..199 see no key
    (1, 1, 256, 1, 128, False, "bf16"),      # N_k = 1: dq = dk = 0
    (1, 1, 384, 384, 128, True, "fp16"),
]


@pytest.fixture(scope="module", autouse=True)
def _built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    attn.build()
    attn.lib()


def _run(case, inputs, dO):
    dev = {k: v.cuda() for k, v in inputs.items() if isinstance(v, torch.Tensor)}
    g = dO.cuda()
    o, lse = attn.attn_fwd(dev["q"], dev["k"], dev["v"], scale=case.scale, causal=case.causal)
    dq, dk, dv = attn.attn_bwd(dev["q"], dev["k"], dev["v"], o, lse, g, scale=case.scale,
                               causal=case.causal)
    attn.attn_check_status()
    return [t.double().cpu().numpy() for t in (dq, dk, dv)]


def _compare(got, ref, where=""):
    for name, a, b in zip(("dq", "dk", "dv"), got, ref):
        assert np.all(np.isfinite(a)), f"{where} {name}: non-finite"
        scale = float(np.abs(b).max()) if b.size else 0.0
        err = np.abs(a - b)
        msg = f"{where} {name}: max err {err.max():.3e} mean {err.mean():.3e} (max |ref| {scale:.3e})"
        print(msg)
        assert err.max() <= MAX_REL * scale + ABS, msg
        assert err.mean() <= MEAN_REL * scale + ABS, msg


@pytest.mark.parametrize("shape", CASES, ids=lambda s: "x".join(map(str, s)))
def test_backward_matches_oracle(shape):
    B, H, N_q, N_k, d, causal, dtype = shape
    case = synthetic.custom_case(B, H, N_q, N_k, d, causal, dtype,
                                 seed=zlib.crc32(repr(shape).encode()) % 10000, outliers=False)
    inputs = synthetic.make_inputs(case)
    dO = synthetic.make_grad(case)
    got = _run(case, inputs, dO)
    q, k, v = oracle.case_inputs_f64(inputs)
    ref = backward.attention_backward(q, k, v, oracle.to_f64(dO), case.scale, case.causal)
    _compare(got, ref, repr(shape))


def test_backward_is_deterministic():
    case = synthetic.custom_case(1, 4, 700, 700, 128, True, "bf16", seed=9, outliers=False)
    inputs = synthetic.make_inputs(case)
    dO = synthetic.make_grad(case)
    a = _run(case, inputs, dO)
    b = _run(case, inputs, dO)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_backward_workload_sampled():
    """BWD (B2 H16 N4096 d128, causal bf16) at full size: oracle gradients of
    one (b, h) slice restricted to sampled query rows (dq) and sampled keys (dk, dv)."""
    case = synthetic.EXTRA_CASES["BWD"]
    inputs = synthetic.make_inputs(case)
    dO = synthetic.make_grad(case)
    dq, dk, dv = _run(case, inputs, dO)
    q, k, v = oracle.case_inputs_f64(inputs)
    g = oracle.to_f64(dO)
    rng = np.random.default_rng(case.seed)
    for b, h in ((0, 0), (1, case.H - 1)):
        sl = lambda x: x[b:b + 1, :, h:h + 1, :]
        rq, rk, rv = backward.attention_backward(sl(q), sl(k), sl(v), sl(g), case.scale, case.causal)
        rows = np.unique(np.concatenate([[0, 1, 127, 128, case.N_q - 1], rng.integers(0, case.N_q, 60)]))
        keys = np.unique(np.concatenate([[0, 127, 128, case.N_k - 1], rng.integers(0, case.N_k, 60)]))
        got = [dq[b:b + 1, rows, h:h + 1], dk[b:b + 1, keys, h:h + 1], dv[b:b + 1, keys, h:h + 1]]
        ref = [rq[:, rows], rk[:, keys], rv[:, keys]]
        _compare(got, ref, f"BWD b{b} h{h}")


def test_fp8_backward_is_refused():
    q = torch.zeros(1, 128, 1, 64, device="cuda").to(torch.float8_e4m3fn)
    o = torch.zeros(1, 128, 1, 64, device="cuda", dtype=torch.bfloat16)
    lse = torch.zeros(1, 1, 128, device="cuda")
    ws = torch.empty(attn.attn_bwd_workspace_bytes(1, 1, 128), dtype=torch.uint8, device="cuda")
    P = lambda t: __import__("ctypes").c_void_p(t.data_ptr())
    st = attn.lib().attn_bwd(P(q), P(q), P(q), P(o), P(lse), P(o), P(o), P(o), P(o), 1, 1, 128, 128,
                             64, 0.125, 0, attn.ATTN_FP8_E4M3, P(ws), ws.numel(), None)
    assert st == attn.ATTN_ERR_UNSUPPORTED


GQA = [
    # B, H, H_kv, N_q, N_k, d, causal, dtype
    (2, 8, 2, 300, 300, 128, True, "bf16"),
    (1, 6, 1, 257, 500, 64, False, "fp16"),     # multi-query
    (1, 4, 2, 200, 130, 64, True, "bf16"),      # rows with no key
]


@pytest.mark.parametrize("shape", GQA, ids=lambda s: "x".join(map(str, s)))
def test_backward_gqa_matches_oracle(shape):
    """K/V shared by H / H_kv query heads: the oracle differentiates the
    expanded problem (each query head with its own copy of its K/V head) and
    sums dk, dv over the copies, which is the gradient of the shared tensors."""
    B, H, H_kv, N_q, N_k, d, causal, dtype = shape
    case = synthetic.custom_case(B, H, N_q, N_k, d, causal, dtype, outliers=False, H_kv=H_kv,
                                 seed=zlib.crc32(repr(shape).encode()) % 10000)
    inputs = synthetic.make_inputs(case)
    dO = synthetic.make_grad(case)
    dev = {k: v.cuda() for k, v in inputs.items() if isinstance(v, torch.Tensor)}
    o, lse = attn.attn_fwd_gqa(dev["q"], dev["k"], dev["v"], scale=case.scale, causal=causal)
    dq, dk, dv = attn.attn_bwd(dev["q"], dev["k"], dev["v"], o, lse, dO.cuda(), scale=case.scale,
                               causal=causal)
    attn.attn_check_status()
    got = [t.double().cpu().numpy() for t in (dq, dk, dv)]
    q, k, v = oracle.case_inputs_f64(inputs)
    ref = parity.backward_gqa_reference(q, k, v, oracle.to_f64(dO), case.scale, causal)
    _compare(got, list(ref), repr(shape))
