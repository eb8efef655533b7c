"""GPU tests of attn_fwd_host: the forward pass on host-resident tensors, with
the copies to and from the device pipelined against the kernel over chunks of
heads.

Every (batch, head) is computed exactly as a single attn_fwd / attn_fwd_fp8
call computes it, so the host path must equal the device path bit for bit on
the same inputs, whatever the chunking (heads not dividing evenly, several
batch rows, one head per chunk); one case is also compared with the fp64
oracle directly.
"""

import zlib

import numpy as np
import pytest
import torch

import io_aware_exact_03_gb300 as attn
import synthetic
from parity import compare, oracle_full, run_gpu, to_device

pytestmark = pytest.mark.gpu

CASES = [
    # B, H, N_q, N_k, d, causal, dtype
    (1, 16, 1024, 1024, 128, True, "bf16"),   # four chunks of four heads
    (2, 5, 300, 300, 64, False, "fp16"),      # uneven head chunks, ragged tiles
    (2, 16, 640, 640, 128, False, "e4m3"),    # descales travel with their heads
    (1, 3, 200, 777, 128, True, "bf16"),      # N_q != N_k under the causal mask
    (3, 1, 129, 129, 256, True, "bf16"),      # d = 256, one chunk per batch row
    (1, 2, 64, 0, 128, False, "bf16"),        # no keys: o = 0, lse = -inf
]


@pytest.fixture(scope="module", autouse=True)
def _built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    attn.build()
    attn.lib()


def _host_call(case, inputs, pinned=True):
    def h(t):
        t = t.contiguous()
        return t.pin_memory() if pinned else t.clone()
    kw = dict(scale=case.scale, causal=case.causal)
    if case.dtype == "e4m3":
        kw.update(q_descale=h(inputs["q_descale"]), k_descale=h(inputs["k_descale"]),
                  v_descale=h(inputs["v_descale"]))
    o, lse = attn.attn_fwd_host(h(inputs["q"]), h(inputs["k"]), h(inputs["v"]), **kw)
    torch.cuda.synchronize()
    attn.attn_check_status()
    return o.double().numpy(), lse.double().numpy()


@pytest.mark.parametrize("shape", CASES, ids=lambda s: "x".join(map(str, s)))
def test_host_path_equals_device_path_bitwise(shape):
    B, H, N_q, N_k, d, causal, dtype = shape
    case = synthetic.custom_case(B, H, N_q, N_k, d, causal, dtype,
                                 seed=zlib.crc32(repr(shape).encode()) % 10000)
    inputs = synthetic.make_inputs(case)
    O_h, lse_h = _host_call(case, inputs)
    O_d, lse_d = run_gpu(case, to_device(inputs))
    assert np.array_equal(O_h, O_d)
    assert np.array_equal(lse_h, lse_d)


def test_host_path_matches_oracle():
    case = synthetic.custom_case(2, 6, 257, 257, 128, True, "bf16", seed=4242)
    inputs = synthetic.make_inputs(case)
    O_h, lse_h = _host_call(case, inputs)
    O_ref, lse_ref = oracle_full(case, inputs)
    compare(case, O_h, lse_h, O_ref, lse_ref)


def test_pageable_host_memory_gives_the_same_result():
    case = synthetic.custom_case(1, 8, 384, 384, 128, False, "bf16", seed=99)
    inputs = synthetic.make_inputs(case)
    a = _host_call(case, inputs, pinned=True)
    b = _host_call(case, inputs, pinned=False)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_ordered_on_the_callers_stream():
    # two calls back to back on a side stream into the same outputs and
    # workspace: the second must see the first one's copies finished
    case = synthetic.custom_case(1, 8, 512, 512, 128, True, "bf16", seed=5)
    inputs = synthetic.make_inputs(case)
    q, k, v = (inputs[n].pin_memory() for n in ("q", "k", "v"))
    s = torch.cuda.Stream()
    ws = torch.empty(attn.attn_fwd_host_workspace_bytes(1, 8, 512, 512, 128, attn.ATTN_BF16),
                     dtype=torch.uint8, device="cuda")
    o, lse = attn.attn_fwd_host(q, k, v, scale=case.scale, causal=True, workspace=ws, stream=s)
    q2 = (q.float() * 0.5).to(q.dtype).pin_memory()
    o2, lse2 = attn.attn_fwd_host(q2, k, v, scale=case.scale, causal=True, workspace=ws, stream=s)
    s.synchronize()
    ref1 = run_gpu(case, to_device(inputs))
    inputs2 = dict(inputs, q=q2)
    ref2 = run_gpu(case, to_device(inputs2))
    assert np.array_equal(o.double().numpy(), ref1[0])
    assert np.array_equal(o2.double().numpy(), ref2[0])
