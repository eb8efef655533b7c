"""Host-side checks of the C ABI: the library loads, exports every function the
header declares, and rejects bad arguments before touching the GPU (no call
here reaches a kernel launch, so these run without a GPU)."""

import ctypes
import glob
import os
import re

import pytest

import io_aware_exact_03_gb300 as attn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    attn.build()
    return attn.lib()


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"\b(attn_\w+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("attn_fwd", "attn_fwd_fp8", "attn_fwd_simt", "attn_fwd_splitkv", "attn_fwd_gqa",
              "attn_quantize_e4m3",
              "attn_splitkv_workspace_bytes", "attn_selftest_wait", "attn_check_status",
              "attn_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for n in declared_functions():
        assert hasattr(L, n), f"{n} declared in include/ but not exported"


def test_only_the_c_abi_is_exported():
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", attn.ext_build.LIB_PATH],
                         capture_output=True, text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    assert exported == set(declared_functions())


def test_status_strings(L):
    for s, txt in [(0, b"ok"), (1, b"invalid argument"), (4, b"bounded wait timed out inside a kernel")]:
        assert L.attn_status_string(s) == txt
    assert L.attn_status_string(99) == b"unknown status"


def test_last_cuda_error_names_a_cuda_error(L):
    # "none" until a call returns ATTN_ERR_CUDA on this thread, then the
    # cudaGetErrorName of its cause (calls made without a GPU can set it)
    L.attn_last_cuda_error.restype = ctypes.c_char_p
    name = L.attn_last_cuda_error()
    assert name == b"none" or name.startswith(b"cuda"), name


P = 0x10000  # a 16-byte aligned fake address; never dereferenced by these calls


def call_fwd(L, q=P, k=P, v=P, o=P, lse=P, B=1, H=1, N_q=16, N_k=16, d=64, scale=0.125,
             causal=0, dtype=0):
    return L.attn_fwd(q, k, v, o, lse, B, H, N_q, N_k, d, scale, causal, dtype, None)


def test_rejects_bad_arguments(L):
    assert call_fwd(L, q=None) == attn.ATTN_ERR_INVALID_ARG
    assert call_fwd(L, o=None) == attn.ATTN_ERR_INVALID_ARG
    assert call_fwd(L, k=None) == attn.ATTN_ERR_INVALID_ARG
    assert call_fwd(L, B=-1) == attn.ATTN_ERR_INVALID_ARG
    assert call_fwd(L, N_k=-5) == attn.ATTN_ERR_INVALID_ARG
    assert call_fwd(L, scale=0.0) == attn.ATTN_ERR_INVALID_ARG
    assert call_fwd(L, scale=float("nan")) == attn.ATTN_ERR_INVALID_ARG
    assert call_fwd(L, scale=float("inf")) == attn.ATTN_ERR_INVALID_ARG
    assert call_fwd(L, scale=-1.0) == attn.ATTN_ERR_INVALID_ARG
    assert call_fwd(L, q=P + 8) == attn.ATTN_ERR_INVALID_ARG      # misaligned
    assert call_fwd(L, lse=P + 2) == attn.ATTN_ERR_INVALID_ARG
    assert call_fwd(L, dtype=7) == attn.ATTN_ERR_INVALID_ARG
    assert call_fwd(L, d=96) == attn.ATTN_ERR_UNSUPPORTED
    assert call_fwd(L, d=32) == attn.ATTN_ERR_UNSUPPORTED
    assert call_fwd(L, d=512) == attn.ATTN_ERR_UNSUPPORTED


def test_sequence_length_limit(L):
    # N_q or N_k above ATTN_MAX_SEQ_LEN is refused by every entry point before
    # any CUDA call (even for an otherwise empty problem); the limit itself is
    # accepted (B = 0 keeps these calls from launching)
    over, top = attn.ATTN_MAX_SEQ_LEN + 1, attn.ATTN_MAX_SEQ_LEN
    U, OK = attn.ATTN_ERR_UNSUPPORTED, attn.ATTN_OK
    for B, N_q, N_k, want in ((1, over, 16, U), (1, 16, over, U), (0, top, top, OK)):
        assert call_fwd(L, B=B, N_q=N_q, N_k=N_k) == want
        fp8 = (P, P, P, P, P, P, P, P, B, 1, N_q, N_k, 128, 0.1, 0)
        assert L.attn_fwd_fp8(*fp8, None) == want
        assert L.attn_fwd_fp8_ws(*fp8, P, 1 << 40, None) == want
        assert L.attn_fwd_simt(*fp8, attn.ATTN_BF16, None) == want
        assert L.attn_fwd_gqa(P, P, P, P, P, None, None, None, B, 2, 1, N_q, N_k, 64, 0.1, 0,
                              attn.ATTN_BF16, None) == want
        assert L.attn_fwd_splitkv(P, P, P, P, P, None, None, None, B, 1, N_q, N_k, 64, 0.1, 0,
                                  attn.ATTN_BF16, 2, P, 1 << 40, None) == want
        assert L.attn_fwd_splitkv_static(P, P, P, P, P, None, None, None, B, 1, N_q, N_k, 64,
                                         0.1, 0, attn.ATTN_BF16, 2, None) == want
        assert L.attn_bwd(P, P, P, P, P, P, P, P, P, B, 1, N_q, N_k, 64, 0.1, 0, attn.ATTN_BF16,
                          P, 1 << 40, None) == want
        assert L.attn_fwd_host(P, P, P, P, P, None, None, None, B, 1, N_q, N_k, 64, 0.1, 0,
                               attn.ATTN_BF16, 0x100000, 1 << 40, None) == want
    assert L.attn_quantize_e4m3(P, attn.ATTN_FP32, P, P, 1, over, 1, 64, None, None) == U
    assert L.attn_quantize_e4m3(P, attn.ATTN_FP32, P, P, 0, top, 1, 64, None, None) == OK


def test_empty_problems_launch_nothing(L):
    # B, H or N_q == 0: nothing to compute; returns before any CUDA call
    assert call_fwd(L, B=0, q=None, k=None, v=None, o=None, lse=None) == attn.ATTN_OK
    assert call_fwd(L, H=0) == attn.ATTN_OK
    assert call_fwd(L, N_q=0) == attn.ATTN_OK


def test_fp8_requires_descales(L):
    st = L.attn_fwd_fp8(P, P, P, P, P, None, P, P, 1, 1, 16, 16, 128, 0.1, 0, None)
    assert st == attn.ATTN_ERR_INVALID_ARG
    st = L.attn_fwd_simt(None, P, P, P, P, None, None, None, 1, 1, 16, 16, 128, 0.1, 0, 2, None)
    assert st == attn.ATTN_ERR_INVALID_ARG


def test_python_binding_refuses_cpu_tensors():
    import torch
    q = torch.zeros(1, 8, 1, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        attn.attn_fwd(q, q, q)
    with pytest.raises(ValueError):
        attn.attn_fwd_splitkv_static(q, q, q, 2)


def test_binding_has_every_declared_entry_point():
    # the Python binding carries the C ABI's names, one function per entry point
    declared = set(declared_functions())
    assert len(declared) >= 20
    missing = sorted(n for n in declared if not callable(getattr(attn, n, None)))
    assert not missing, missing
    assert declared <= set(attn.__all__)


def test_last_cuda_error_through_the_binding(L):
    assert isinstance(attn.attn_last_cuda_error(), str)


def test_splitkv_workspace_size(L):
    # fp32 partial outputs [splits][B*H][N_q][d] plus fp32 partial lse [splits][B*H][N_q]
    assert L.attn_splitkv_workspace_bytes(2, 3, 100, 128, 4) == 4 * 2 * 3 * 100 * (128 + 1) * 4
    assert L.attn_splitkv_workspace_bytes(2, 3, 100, 64, 1) == 0
    assert L.attn_splitkv_workspace_bytes(2, 3, 100, 96, 4) == 0
    assert L.attn_splitkv_workspace_bytes(2, 3, 100, 64, 33) == 0


def test_fp8_ws_workspace_size(L):
    # the fp16 copy of v: 2 * B * N_k * H * d bytes for d = 64 / 128, else 0
    assert L.attn_fwd_fp8_workspace_bytes(2, 16, 8192, 128) == 2 * 2 * 8192 * 16 * 128
    assert L.attn_fwd_fp8_workspace_bytes(3, 5, 129, 64) == 2 * 3 * 129 * 5 * 64
    assert L.attn_fwd_fp8_workspace_bytes(2, 8, 8192, 256) == 0
    assert L.attn_fwd_fp8_workspace_bytes(1, 1, 16, 96) == 0
    assert L.attn_fwd_fp8_workspace_bytes(-1, 1, 16, 64) == 0
    assert L.attn_fwd_fp8_workspace_bytes(1, 1, 0, 64) == 0


def test_fp8_ws_rejects_bad_arguments(L):
    # every check below returns before anything is launched
    need = L.attn_fwd_fp8_workspace_bytes(1, 1, 16, 64)
    base = (P, P, P, P, P)
    args = (1, 1, 16, 16, 64, 0.125, 0)
    ok_ds = (P, P, P)
    assert L.attn_fwd_fp8_ws(*base, *ok_ds, *args, None, need, None) == attn.ATTN_ERR_INVALID_ARG
    assert L.attn_fwd_fp8_ws(*base, *ok_ds, *args, P, need - 1, None) == attn.ATTN_ERR_INVALID_ARG
    assert L.attn_fwd_fp8_ws(*base, *ok_ds, *args, P + 8, need, None) == attn.ATTN_ERR_INVALID_ARG
    assert L.attn_fwd_fp8_ws(*base, None, P, P, *args, P, need, None) == attn.ATTN_ERR_INVALID_ARG
    assert L.attn_fwd_fp8_ws(*base, *ok_ds, 1, 1, 16, 16, 96, 0.125, 0, P, need,
                             None) == attn.ATTN_ERR_UNSUPPORTED
    # nothing to compute: returns at once, workspace or not
    assert L.attn_fwd_fp8_ws(*base, *ok_ds, 0, 1, 16, 16, 64, 0.125, 0, None, 0,
                             None) == attn.ATTN_OK


def test_splitkv_num_splits(L):
    # long K/V, few query tiles: B1 H8 N_q 512 N_k 65536 has 16 CTAs unsplit; 9 splits fill
    # 144 of 152 SMs in one wave (8 would leave 24 idle, 10 would need a second wave)
    assert L.attn_splitkv_num_splits(1, 8, 512, 65536, 128, 152) == 9
    # a single query row against 65536 keys, 8 heads: 19 splits = 152 CTAs, one wave
    assert L.attn_splitkv_num_splits(1, 8, 1, 65536, 128, 152) == 19
    # enough query tiles to fill the GPU: no split
    assert L.attn_splitkv_num_splits(1, 16, 16384, 16384, 128, 152) == 1
    assert L.attn_splitkv_num_splits(2, 16, 8192, 8192, 128, 152) == 1
    # never more splits than key tiles, never more than 32
    assert L.attn_splitkv_num_splits(1, 1, 128, 300, 64, 152) <= 3
    assert 1 <= L.attn_splitkv_num_splits(1, 1, 1, 1 << 24, 256, 1024) <= 32
    # degenerate or invalid arguments: 1
    for args in [(0, 8, 512, 65536, 128, 152), (1, 8, 512, 0, 128, 152),
                 (1, 8, 512, 65536, 96, 152), (1, 8, 512, 65536, 128, 0)]:
        assert L.attn_splitkv_num_splits(*args) == 1


def test_splitkv_rejects_bad_workspace(L):
    need = L.attn_splitkv_workspace_bytes(1, 1, 16, 64, 4)
    args = (P, P, P, P, P, None, None, None, 1, 1, 16, 16, 64, 0.125, 0, 0)
    assert L.attn_fwd_splitkv(*args, 4, None, need, None) == attn.ATTN_ERR_INVALID_ARG
    assert L.attn_fwd_splitkv(*args, 4, P, need - 1, None) == attn.ATTN_ERR_INVALID_ARG
    assert L.attn_fwd_splitkv(*args, 4, P + 4, need, None) == attn.ATTN_ERR_INVALID_ARG
    assert L.attn_fwd_splitkv(*args, 0, P, need, None) == attn.ATTN_ERR_INVALID_ARG
    assert L.attn_fwd_splitkv(*args, 33, P, need, None) == attn.ATTN_ERR_INVALID_ARG


def test_selftest_wait_rejects_bad_limits(L):
    # the abort-path check: limit out of range, or nothing to cut short
    fp = ctypes.c_void_p(P)
    assert L.attn_selftest_abort(fp, fp, fp, fp, None, None, None, None, 1, 1, 128, 128, 64,
                                 0.125, 0, attn.ATTN_BF16, None, 0, 0, None) == attn.ATTN_ERR_INVALID_ARG
    assert L.attn_selftest_abort(fp, fp, fp, fp, None, None, None, None, 1, 1, 128, 0, 64,
                                 0.125, 0, attn.ATTN_BF16, None, 0, 500, None) == attn.ATTN_ERR_INVALID_ARG
    assert L.attn_selftest_abort(fp, fp, fp, fp, None, None, None, None, 1, 1, 128, 128, 96,
                                 0.125, 0, attn.ATTN_BF16, None, 0, 500, None) == attn.ATTN_ERR_UNSUPPORTED
    # a workspace only for e4m3 at d = 64 / 128, aligned and large enough
    need = L.attn_fwd_fp8_workspace_bytes(1, 1, 128, 64)
    assert L.attn_selftest_abort(fp, fp, fp, fp, None, None, None, None, 1, 1, 128, 128, 64,
                                 0.125, 0, attn.ATTN_BF16, fp, need, 500, None) == attn.ATTN_ERR_INVALID_ARG
    assert L.attn_selftest_abort(fp, fp, fp, fp, None, fp, fp, fp, 1, 1, 128, 128, 64, 0.125, 0,
                                 attn.ATTN_FP8_E4M3, fp, need - 1, 500, None) == attn.ATTN_ERR_INVALID_ARG
    assert L.attn_selftest_abort(fp, fp, fp, fp, None, fp, fp, fp, 1, 1, 128, 128, 64, 0.125, 0,
                                 attn.ATTN_FP8_E4M3, ctypes.c_void_p(P + 4), need, 500,
                                 None) == attn.ATTN_ERR_INVALID_ARG
    assert L.attn_selftest_wait(0, None) == attn.ATTN_ERR_INVALID_ARG
    assert L.attn_selftest_wait(20 * 1000 * 1000, None) == attn.ATTN_ERR_INVALID_ARG


def test_gqa_rejects_bad_head_counts(L):
    args = (P, P, P, P, P, None, None, None, 1)
    assert L.attn_fwd_gqa(*args, 8, 3, 16, 16, 64, 0.125, 0, 0, None) == attn.ATTN_ERR_INVALID_ARG
    assert L.attn_fwd_gqa(*args, 8, 0, 16, 16, 64, 0.125, 0, 0, None) == attn.ATTN_ERR_INVALID_ARG


def test_attention_rejects_the_quantiser_only_input_type(L):
    assert call_fwd(L, dtype=attn.ATTN_FP32) == attn.ATTN_ERR_INVALID_ARG


def test_quantiser_rejects_bad_arguments(L):
    assert L.attn_quantize_e4m3(P, attn.ATTN_FP8_E4M3, P, P, 1, 4, 1, 64, None, None) == attn.ATTN_ERR_INVALID_ARG
    assert L.attn_quantize_e4m3(P, attn.ATTN_FP32, P, P, 1, 4, 1, 96, None, None) == attn.ATTN_ERR_UNSUPPORTED
    assert L.attn_quantize_e4m3(P, attn.ATTN_FP32, P + 4, P, 1, 4, 1, 64, None, None) == attn.ATTN_ERR_INVALID_ARG
    assert L.attn_quantize_e4m3(P, attn.ATTN_FP32, P, None, 1, 4, 1, 64, None, None) == attn.ATTN_ERR_INVALID_ARG
    assert L.attn_quantize_e4m3(None, attn.ATTN_FP32, None, None, 0, 4, 1, 64, None, None) == attn.ATTN_OK


def test_host_forward_rejects_bad_arguments(L):
    # every check below returns before any CUDA call (no GPU needed)
    ws = 0x100000  # 256-byte aligned fake device address
    big = 1 << 40

    def call(q=P, k=P, v=P, o=P, lse=P, qd=None, kd=None, vd=None, B=1, H=4, N_q=64, N_k=64,
             d=128, scale=0.125, dtype=0, w=ws, wb=big):
        return L.attn_fwd_host(q, k, v, o, lse, qd, kd, vd, B, H, N_q, N_k, d, scale, 0, dtype, w,
                               wb, None)

    assert call(scale=0.0) == attn.ATTN_ERR_INVALID_ARG
    assert call(scale=float("inf")) == attn.ATTN_ERR_INVALID_ARG
    assert call(d=32) == attn.ATTN_ERR_UNSUPPORTED
    assert call(dtype=3) == attn.ATTN_ERR_INVALID_ARG
    assert call(q=None) == attn.ATTN_ERR_INVALID_ARG
    assert call(dtype=2) == attn.ATTN_ERR_INVALID_ARG          # e4m3 without descales
    assert call(w=None) == attn.ATTN_ERR_INVALID_ARG
    assert call(w=ws + 16) == attn.ATTN_ERR_INVALID_ARG        # workspace not 256-byte aligned
    need = L.attn_fwd_host_workspace_bytes(1, 4, 64, 64, 128, 0)
    assert call(wb=need - 1) == attn.ATTN_ERR_INVALID_ARG
    assert call(B=0) == attn.ATTN_OK and call(N_q=0) == attn.ATTN_OK


def test_host_forward_workspace_bytes(L):
    f = L.attn_fwd_host_workspace_bytes
    assert f(0, 4, 64, 64, 128, 0) == 0 and f(1, 4, 64, 64, 32, 0) == 0 and f(1, 4, 64, 64, 128, 3) == 0
    # bf16, B1 H16 N16384 d128: four chunks of four heads, three slots of
    # q, k, v, o (16 MiB each) + lse (256 KiB)
    assert f(1, 16, 16384, 16384, 128, 0) == 3 * (4 * (16 << 20) + (256 << 10))
    # one head, one chunk: a single slot
    assert f(1, 1, 100, 100, 64, 0) == 12800 + 2 * 12800 + 12800 + 512


def test_host_forward_binding_checks_arguments(L):
    import torch
    q = torch.zeros(1, 8, 2, 64, dtype=torch.bfloat16)
    k = torch.zeros(1, 8, 2, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        attn.attn_fwd_host(q, k, torch.zeros(1, 9, 2, 64, dtype=torch.bfloat16))   # v shape
    with pytest.raises(TypeError):
        attn.attn_fwd_host(q, k, k.to(torch.float16))                              # mixed dtypes
    with pytest.raises(ValueError):
        attn.attn_fwd_host(q[:, :, :1], k, k)                                       # q not contiguous
    f8 = torch.zeros(1, 8, 2, 64).to(torch.float8_e4m3fn)
    with pytest.raises(ValueError):
        attn.attn_fwd_host(f8, f8, f8)                                              # e4m3 without descales
