"""The allocation-free split-KV entry point against the one that takes a workspace.

attn_fwd_splitkv_static is for callers that cannot allocate device memory (a
plugin inside a host program that owns all device memory through its own pool,
or a latency-critical loop that cannot afford an allocation's synchronisation).
Its scratch is a fixed array inside the library that every call reuses, so the
test runs it twice in a row on different problems (the second call finds the
first call's data in the array) and checks each result against
attn_fwd_splitkv with a caller-allocated workspace, within the tolerances of
the parity tests (bf16 / fp16, then e4m3 with descales and head dimension
256, whose partials come from a kernel of their own).  It also checks that a
warm call leaves the device's free memory unchanged, that a misaligned descale
pointer and a problem too large for the array are refused before anything
runs.

The file name makes pytest collect it last, so a run that stops at the first
failure has already run every other test.
"""

import ctypes

import pytest
import torch

import io_aware_exact_03_gb300 as attn
import synthetic
from parity import TOL, to_device

pytestmark = pytest.mark.gpu

CODES = {"bf16": attn.ATTN_BF16, "fp16": attn.ATTN_FP16, "e4m3": attn.ATTN_FP8_E4M3}


@pytest.fixture(scope="module")
def L():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    attn.build()
    return attn.lib()


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _run_static(L, case, dev, n_splits):
    o = torch.full((case.B, case.N_q, case.H, case.d), 3.0, device="cuda",
                   dtype=torch.float16 if case.dtype == "fp16" else torch.bfloat16)
    lse = torch.full((case.B, case.H, case.N_q), 3.0, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = L.attn_fwd_splitkv_static(_p(dev["q"]), _p(dev["k"]), _p(dev["v"]), _p(o), _p(lse),
                                   _p(dev.get("q_descale")), _p(dev.get("k_descale")),
                                   _p(dev.get("v_descale")), case.B, case.H, case.N_q, case.N_k,
                                   case.d, case.scale, int(case.causal), CODES[case.dtype],
                                   n_splits, stream)
    assert st == attn.ATTN_OK, attn.attn_status_string(st)
    attn.attn_check_status()
    return o, lse


def _run_workspace(case, dev, n_splits):
    o, lse = attn.attn_fwd_splitkv(dev["q"], dev["k"], dev["v"], n_splits, scale=case.scale,
                                   causal=case.causal, q_descale=dev.get("q_descale"),
                                   k_descale=dev.get("k_descale"),
                                   v_descale=dev.get("v_descale"))
    attn.attn_check_status()
    return o, lse


def _check(case, got, ref):
    tol = TOL[case.dtype]
    o_err = (got[0].double() - ref[0].double()).abs().max().item()
    assert o_err <= tol["o_max"], f"O differs by {o_err}"
    l_got, l_ref = got[1].double(), ref[1].double()
    inf = torch.isneginf(l_ref)
    assert torch.equal(torch.isneginf(l_got), inf)
    if (~inf).any():
        assert (l_got[~inf] - l_ref[~inf]).abs().max().item() <= tol["lse"]


def test_two_calls_in_a_row_match_the_workspace_entry_point(L):
    first = (synthetic.custom_case(1, 4, 300, 3000, 128, True, "bf16", seed=71, outliers=False), 4)
    second = (synthetic.custom_case(2, 2, 129, 2000, 64, False, "fp16", seed=72, outliers=False), 3)
    devs = [to_device(synthetic.make_inputs(c)) for c, _ in (first, second)]
    got = [_run_static(L, c, d, n) for (c, n), d in zip((first, second), devs)]
    for ((c, n), d), g in zip(zip((first, second), devs), got):
        _check(c, g, _run_workspace(c, d, n))


def test_e4m3_and_d256_calls_in_a_row(L):
    # e4m3 with per-head descales, then head dimension 256 (its own kernel
    # and partial indexing), back to back on the shared array
    first = (synthetic.custom_case(1, 3, 256, 2500, 128, False, "e4m3", seed=73, outliers=True), 5)
    second = (synthetic.custom_case(1, 2, 200, 1500, 256, True, "bf16", seed=74, outliers=False), 4)
    devs = [to_device(synthetic.make_inputs(c)) for c, _ in (first, second)]
    got = [_run_static(L, c, d, n) for (c, n), d in zip((first, second), devs)]
    for ((c, n), d), g in zip(zip((first, second), devs), got):
        _check(c, g, _run_workspace(c, d, n))


def test_a_warm_call_takes_no_device_memory(L):
    # once the library is loaded and the array's address looked up on this
    # device, a call must leave the free device memory unchanged
    case = synthetic.custom_case(1, 4, 300, 3000, 128, True, "bf16", seed=75, outliers=False)
    dev = to_device(synthetic.make_inputs(case))
    o = torch.empty((case.B, case.N_q, case.H, case.d), device="cuda", dtype=torch.bfloat16)
    lse = torch.empty((case.B, case.H, case.N_q), device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    def call():
        st = L.attn_fwd_splitkv_static(_p(dev["q"]), _p(dev["k"]), _p(dev["v"]), _p(o), _p(lse),
                                       None, None, None, case.B, case.H, case.N_q, case.N_k,
                                       case.d, case.scale, 1, attn.ATTN_BF16, 4, stream)
        assert st == attn.ATTN_OK
        torch.cuda.synchronize()

    call()  # warm: module loaded, address looked up
    free_before, _ = torch.cuda.mem_get_info()
    call()
    free_after, _ = torch.cuda.mem_get_info()
    attn.attn_check_status()
    assert free_after == free_before


def test_misaligned_descale_is_refused(L):
    case = synthetic.custom_case(1, 2, 128, 256, 64, False, "e4m3", seed=76, outliers=False)
    dev = to_device(synthetic.make_inputs(case))
    o = torch.empty((case.B, case.N_q, case.H, case.d), device="cuda", dtype=torch.bfloat16)
    bad = ctypes.c_void_p(dev["q_descale"].data_ptr() + 2)
    st = L.attn_fwd_splitkv_static(_p(dev["q"]), _p(dev["k"]), _p(dev["v"]), _p(o), None, bad,
                                   _p(dev["k_descale"]), _p(dev["v_descale"]), case.B, case.H,
                                   case.N_q, case.N_k, case.d, case.scale, 0,
                                   attn.ATTN_FP8_E4M3, 2, None)
    assert st == attn.ATTN_ERR_INVALID_ARG


def test_problem_beyond_the_scratch_is_refused(L):
    # 4 splits of B1 H16 N_q 4096 d128 need 4*16*4096*129*4 bytes > 32 MiB
    need = L.attn_splitkv_workspace_bytes(1, 16, 4096, 128, 4)
    assert need > attn.ATTN_STATIC_SCRATCH_BYTES
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: refused before any CUDA call
    st = L.attn_fwd_splitkv_static(fake, fake, fake, fake, fake, None, None, None, 1, 16, 4096,
                                   4096, 128, 0.088, 1, attn.ATTN_BF16, 4, None)
    assert st == attn.ATTN_ERR_SCRATCH_LIMIT
    assert "scratch" in attn.attn_status_string(st)
