"""attn_fwd_fp8_ws: e4m3 attention whose V is widened to fp16 once, into a
caller workspace, by an elementwise kernel; the attention kernel then loads
fp16 V tiles by TMA instead of widening every V tile in every CTA that reads
it.  The fp16 V values and the MMAs (their order included) are those of
attn_fwd_fp8, so the two results must agree bit for bit; against the fp64
oracle the FP8 bound applies as for attn_fwd_fp8 ("FlashAttention-3 (BN)",
section "Low precision (FP8) and reducing quantisation error")."""

import zlib

import pytest
import torch

import io_aware_exact_03_gb300 as attn
import synthetic
from parity import check_sampled, compare, oracle_full, run_gpu, to_device

pytestmark = pytest.mark.gpu

SHAPES = [
    # B, H, N_q, N_k, d, causal
    (2, 2, 129, 383, 128, True),
    (1, 3, 256, 256, 64, False),
    (1, 2, 640, 640, 128, True),
    (3, 2, 100, 300, 64, True),
    (1, 1, 1, 1, 128, False),
    (2, 3, 300, 100, 128, True),    # the first 200 rows see no key
    (1, 2, 130, 1, 64, False),      # N_k = 1: O = v row 0 (times its descale)
    (1, 2, 384, 1000, 128, False),  # ragged last key tile
]


@pytest.fixture(scope="module", autouse=True)
def _built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    attn.build()
    attn.lib()


def _both(case, dev, workspace=None):
    kw = dict(scale=case.scale, causal=case.causal)
    args = (dev["q"], dev["k"], dev["v"], dev["q_descale"], dev["k_descale"], dev["v_descale"])
    o1, l1 = attn.attn_fwd_fp8(*args, **kw)
    o2, l2 = attn.attn_fwd_fp8_ws(*args, workspace=workspace, **kw)
    attn.attn_check_status()
    return (o1, l1), (o2, l2)


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_bitwise_equal_to_fp8_and_within_the_fp8_bound(shape):
    B, H, N_q, N_k, d, causal = shape
    case = synthetic.custom_case(B, H, N_q, N_k, d, causal, "e4m3",
                                 seed=zlib.crc32(repr(shape).encode()) % 10000, outliers=True)
    inputs = synthetic.make_inputs(case)
    (o1, l1), (o2, l2) = _both(case, to_device(inputs))
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    O_ref, lse_ref = oracle_full(case, inputs)
    compare(case, o2.double().cpu().numpy(), l2.double().cpu().numpy(), O_ref, lse_ref)


def test_c5_full_size():
    """C5 (B2 H16 N8192 d128, 0.1 % x10 outliers) as the benchmark runs it: the
    whole output bit for bit equal to attn_fwd_fp8's, and 256 seeded rows
    against the oracle."""
    case = synthetic.CASES["C5"]
    inputs = synthetic.make_inputs(case)
    dev = to_device(inputs)
    (o1, l1), (o2, l2) = _both(case, dev)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    check_sampled(case, "fp8ws", inputs=inputs, dev=dev)


def test_workspace_contents_do_not_matter():
    """The workspace is overwritten before it is read: a workspace full of fp16
    NaN patterns gives the same result as a fresh one."""
    case = synthetic.custom_case(1, 2, 300, 500, 128, False, "e4m3", seed=41, outliers=True)
    dev = to_device(synthetic.make_inputs(case))
    need = attn.attn_fwd_fp8_workspace_bytes(case.B, case.H, case.N_k, case.d)
    assert need == 2 * case.B * case.N_k * case.H * case.d
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device="cuda")
    (o1, l1), (o2, l2) = _both(case, dev, workspace=ws)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_too_small_workspace_is_rejected():
    case = synthetic.custom_case(1, 1, 128, 128, 64, False, "e4m3", seed=3, outliers=False)
    dev = to_device(synthetic.make_inputs(case))
    need = attn.attn_fwd_fp8_workspace_bytes(1, 1, 128, 64)
    ws = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(attn.AttnError) as err:
        attn.attn_fwd_fp8_ws(dev["q"], dev["k"], dev["v"], dev["q_descale"], dev["k_descale"],
                             dev["v_descale"], scale=case.scale, workspace=ws)
    assert err.value.status == attn.ATTN_ERR_INVALID_ARG


@pytest.mark.parametrize("shape", [(1, 2, 300, 300, 128, False), (1, 2, 300, 300, 64, True)],
                         ids=lambda s: "x".join(map(str, s)))
def test_abort_path(shape):
    """The fp16-V kernel's own abort path: the V widening runs in full, then the
    attention kernel's K/V loader stops after the first tile and every wait is
    limited to 500 us; the waits for the missing tiles run out, every role
    drains what it issued and TMEM is freed.  The timeout is reported and
    cleared, and the next call is correct."""
    B, H, N_q, N_k, d, causal = shape
    case = synthetic.custom_case(B, H, N_q, N_k, d, causal, "e4m3", outliers=False,
                                 seed=zlib.crc32(repr(shape).encode()) % 10000)
    inputs = synthetic.make_inputs(case)
    dev = to_device(inputs)
    ws = torch.empty(attn.attn_fwd_fp8_workspace_bytes(B, H, N_k, d), dtype=torch.uint8,
                     device="cuda")
    attn.attn_selftest_abort(dev["q"], dev["k"], dev["v"], dev["q_descale"], dev["k_descale"],
                             dev["v_descale"], scale=case.scale, causal=causal, timeout_us=500,
                             workspace=ws)
    with pytest.raises(attn.AttnError) as err:
        attn.attn_check_status()
    assert err.value.status == attn.ATTN_ERR_TIMEOUT
    assert attn.attn_check_status() == attn.ATTN_OK
    O, lse = run_gpu(case, dev, "fp8ws")
    O_ref, lse_ref = oracle_full(case, inputs)
    compare(case, O, lse, O_ref, lse_ref)


def test_no_keys_needs_no_workspace():
    """N_k = 0: nothing to widen (the workspace size is 0 and none is needed);
    every row gets O = 0 and lse = -inf, as from attn_fwd_fp8."""
    f8 = torch.float8_e4m3fn
    q = (torch.randn(2, 70, 2, 128, device="cuda") * 4).to(f8)
    kv = torch.empty(2, 0, 2, 128, device="cuda", dtype=f8)
    ones = torch.ones(2, 2, device="cuda")
    assert attn.attn_fwd_fp8_workspace_bytes(2, 2, 0, 128) == 0
    o = torch.full((2, 70, 2, 128), 7.0, device="cuda", dtype=torch.bfloat16)
    lse = torch.zeros(2, 2, 70, device="cuda")
    attn.attn_fwd_fp8_ws(q, kv, kv, ones, ones, ones, o=o, lse=lse, scale=0.1)
    attn.attn_check_status()
    assert torch.all(o == 0)
    assert torch.all(torch.isneginf(lse))
