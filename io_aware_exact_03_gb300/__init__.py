"""GB300-native fused exact-attention forward pass (sm_103a).

A thin Python binding over the C ABI of libattn_gb300.so (include/attn_gb300.h):
it only marshals arguments (torch tensors -> device pointers, sizes, the
current CUDA stream).  Every step of the computation runs in the library's
CUDA kernels.  There is no CPU path: if the extension is not built, or no GPU
is present, the calls raise.

Operation: O = softmax(Q K^T * scale [+ causal mask]) V and the per-row
logsumexp ("FlashAttention (HI)" page, section "Problems of standard attention",
computed as in its sections "Tiling and block processing", "Online softmax
computation" and "Combining operations in one CUDA kernel").  Layout
[B, N, H, d], lse [B, H, N_q].
"""

from __future__ import annotations

import ctypes
import math
import os

from . import ext_build as _build

__all__ = ["attn_fwd", "attn_fwd_fp8", "attn_fwd_fp8_ws", "attn_fwd_fp8_workspace_bytes",
           "attn_fwd_simt", "attn_fwd_splitkv", "attn_fwd_splitkv_static", "attn_fwd_gqa",
           "attn_quantize_e4m3",
           "attn_splitkv_workspace_bytes", "attn_splitkv_num_splits", "attn_check_status",
           "attn_status_string",
           "attn_bwd", "attn_bwd_gqa", "attn_bwd_workspace_bytes", "attn_fwd_host",
           "attn_fwd_host_workspace_bytes", "attn_selftest_wait", "attn_selftest_abort",
           "attn_last_cuda_error",
           "AttnError", "lib", "build"]

(ATTN_OK, ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED, ATTN_ERR_CUDA, ATTN_ERR_TIMEOUT,
 ATTN_ERR_SCRATCH_LIMIT) = range(6)
ATTN_STATIC_SCRATCH_BYTES = 32 * 1024 * 1024
ATTN_MAX_SEQ_LEN = 2147483647 - 256
ATTN_BF16, ATTN_FP16, ATTN_FP8_E4M3, ATTN_FP32 = range(4)

_LIB = None


class AttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = f"{where}: {attn_status_string(status)} (status {status})"
        if status == ATTN_ERR_CUDA and _LIB is not None:
            msg += f" [{_LIB.attn_last_cuda_error().decode()}]"
        super().__init__(msg)


def build(force: bool = False) -> str:
    """Compile the CUDA extension in-tree (nvcc, sm_103a)."""
    return _build.build(force=force)


def lib() -> ctypes.CDLL:
    """The loaded C library (raises if it was never built)."""
    global _LIB
    if _LIB is None:
        path = _build.LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError(
                f"CUDA extension {os.path.basename(path)} is not built; run "
                "io_aware_exact_03_gb300.build() (nvcc, sm_103a) first")
        L = ctypes.CDLL(path)
        vp, fp, i, f = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        L.attn_fwd.argtypes = [vp, vp, vp, vp, fp, i, i, i, i, i, f, i, i, vp]
        L.attn_fwd.restype = i
        L.attn_fwd_fp8.argtypes = [vp, vp, vp, vp, fp, fp, fp, fp, i, i, i, i, i, f, i, vp]
        L.attn_fwd_fp8.restype = i
        L.attn_fwd_fp8_ws.argtypes = [vp, vp, vp, vp, fp, fp, fp, fp, i, i, i, i, i, f, i, vp,
                                      ctypes.c_size_t, vp]
        L.attn_fwd_fp8_ws.restype = i
        L.attn_fwd_fp8_workspace_bytes.argtypes = [i, i, i, i]
        L.attn_fwd_fp8_workspace_bytes.restype = ctypes.c_size_t
        L.attn_fwd_simt.argtypes = [vp, vp, vp, vp, fp, fp, fp, fp, i, i, i, i, i, f, i, i, vp]
        L.attn_fwd_simt.restype = i
        sz = ctypes.c_size_t
        L.attn_fwd_splitkv.argtypes = [vp, vp, vp, vp, fp, fp, fp, fp, i, i, i, i, i, f, i, i, i,
                                       vp, sz, vp]
        L.attn_fwd_splitkv.restype = i
        L.attn_splitkv_workspace_bytes.argtypes = [i, i, i, i, i]
        L.attn_splitkv_workspace_bytes.restype = sz
        L.attn_splitkv_num_splits.argtypes = [i, i, i, i, i, i]
        L.attn_splitkv_num_splits.restype = i
        L.attn_fwd_splitkv_static.argtypes = [vp, vp, vp, vp, fp, fp, fp, fp, i, i, i, i, i, f,
                                              i, i, i, vp]
        L.attn_fwd_splitkv_static.restype = i
        L.attn_fwd_gqa.argtypes = [vp, vp, vp, vp, fp, fp, fp, fp, i, i, i, i, i, i, f, i, i, vp]
        L.attn_fwd_gqa.restype = i
        L.attn_quantize_e4m3.argtypes = [vp, i, vp, fp, i, i, i, i, fp, vp]
        L.attn_quantize_e4m3.restype = i
        L.attn_bwd.argtypes = [vp, vp, vp, vp, fp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp, sz,
                               vp]
        L.attn_bwd.restype = i
        L.attn_bwd_gqa.argtypes = [vp, vp, vp, vp, fp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, i,
                                   vp, sz, vp]
        L.attn_bwd_gqa.restype = i
        L.attn_bwd_workspace_bytes.argtypes = [i, i, i]
        L.attn_bwd_workspace_bytes.restype = sz
        L.attn_fwd_host.argtypes = [vp, vp, vp, vp, fp, fp, fp, fp, i, i, i, i, i, f, i, i, vp, sz, vp]
        L.attn_fwd_host.restype = i
        L.attn_fwd_host_workspace_bytes.argtypes = [i, i, i, i, i, i]
        L.attn_fwd_host_workspace_bytes.restype = sz
        L.attn_selftest_wait.argtypes = [ctypes.c_uint, vp]
        L.attn_selftest_wait.restype = i
        L.attn_selftest_abort.argtypes = [vp, vp, vp, vp, fp, fp, fp, fp, i, i, i, i, i, f, i, i,
                                          vp, ctypes.c_size_t, ctypes.c_uint, vp]
        L.attn_selftest_abort.restype = i
        L.attn_check_status.argtypes = [vp]
        L.attn_check_status.restype = i
        L.attn_status_string.argtypes = [i]
        L.attn_status_string.restype = ctypes.c_char_p
        L.attn_last_cuda_error.argtypes = []
        L.attn_last_cuda_error.restype = ctypes.c_char_p
        _LIB = L
    return _LIB


def attn_status_string(status: int) -> str:
    names = {0: "ok", 1: "invalid argument", 2: "unsupported shape or dtype",
             3: "CUDA error", 4: "bounded wait timed out inside a kernel",
             5: "problem needs more scratch than the library's fixed scratch array holds"}
    if _LIB is not None:
        return _LIB.attn_status_string(int(status)).decode()
    return names.get(int(status), "unknown status")


def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return ATTN_BF16
    if t.dtype == torch.float16:
        return ATTN_FP16
    if t.dtype == torch.float8_e4m3fn:
        return ATTN_FP8_E4M3
    raise TypeError(f"unsupported input dtype {t.dtype}")


def _check_inputs(q, k, v, gqa=False):
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous [B, N, H, d]")
        if t.dim() != 4:
            raise ValueError(f"{name} must be 4-D [B, N, H, d]")
    if q.dtype != k.dtype or q.dtype != v.dtype:
        raise TypeError("q, k, v must share one dtype")
    B, N_q, H, d = q.shape
    if k.shape != v.shape or k.shape[0] != B or k.shape[3] != d or (
            k.shape[2] != H if not gqa else (k.shape[2] < 1 or H % k.shape[2] != 0)):
        raise ValueError("k and v must be [B, N_k, H, d] matching q "
                         "([B, N_k, H_kv, d] with H % H_kv == 0 for grouped-query attention)")
    return B, N_q, H, d, k.shape[1]


def _outputs(q, o, lse, B, N_q, H, d):
    torch = _torch()
    out_dtype = torch.float16 if q.dtype == torch.float16 else torch.bfloat16
    if o is None:
        o = torch.empty((B, N_q, H, d), dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, N_q), dtype=torch.float32, device=q.device)
    if o.dtype != out_dtype or tuple(o.shape) != (B, N_q, H, d) or not o.is_contiguous():
        raise ValueError("o must be a contiguous [B, N_q, H, d] tensor of the output dtype")
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, N_q) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 [B, H, N_q] tensor")
    return o, lse


def _stream(stream, device):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _raise(st, where):
    if st != ATTN_OK:
        raise AttnError(st, where)


def attn_fwd(q, k, v, o=None, lse=None, scale=None, causal=False, stream=None):
    """Tensor-core forward pass. bf16 / fp16 / e4m3 (unit descales) inputs.

    Returns (o, lse); outputs are allocated when not given.
    """
    B, N_q, H, d, N_k = _check_inputs(q, k, v)
    o, lse = _outputs(q, o, lse, B, N_q, H, d)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    st = lib().attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N_q, N_k, d,
                        scale, int(bool(causal)), _dtype_code(q), _stream(stream, q.device))
    _raise(st, "attn_fwd")
    return o, lse


def _check_fp8(q, q_descale, k_descale, v_descale, B, H, where):
    torch = _torch()
    if q.dtype != torch.float8_e4m3fn:
        raise TypeError(f"{where} takes float8_e4m3fn inputs")
    for name, t in (("q_descale", q_descale), ("k_descale", k_descale), ("v_descale", v_descale)):
        if not (t.is_cuda and t.dtype == torch.float32 and t.numel() == B * H and t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous CUDA float32 tensor of B*H values")


def attn_fwd_fp8(q, k, v, q_descale, k_descale, v_descale, o=None, lse=None, scale=None,
                 causal=False, stream=None):
    """Tensor-core forward pass on e4m3 codes with per-(batch, head) fp32 descales [B, H]."""
    B, N_q, H, d, N_k = _check_inputs(q, k, v)
    _check_fp8(q, q_descale, k_descale, v_descale, B, H, "attn_fwd_fp8")
    o, lse = _outputs(q, o, lse, B, N_q, H, d)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    st = lib().attn_fwd_fp8(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(q_descale),
                            _ptr(k_descale), _ptr(v_descale), B, H, N_q, N_k, d, scale,
                            int(bool(causal)), _stream(stream, q.device))
    _raise(st, "attn_fwd_fp8")
    return o, lse


def attn_fwd_fp8_workspace_bytes(B, H, N_k, d) -> int:
    return int(lib().attn_fwd_fp8_workspace_bytes(B, H, N_k, d))


def attn_fwd_fp8_ws(q, k, v, q_descale, k_descale, v_descale, o=None, lse=None, scale=None,
                    causal=False, workspace=None, stream=None):
    """attn_fwd_fp8 with V widened to fp16 once into a workspace (allocated when not
    given) before the attention kernel; the same result bit for bit."""
    B, N_q, H, d, N_k = _check_inputs(q, k, v)
    _check_fp8(q, q_descale, k_descale, v_descale, B, H, "attn_fwd_fp8_ws")
    o, lse = _outputs(q, o, lse, B, N_q, H, d)
    need = attn_fwd_fp8_workspace_bytes(B, H, N_k, d)
    if workspace is None and need > 0:
        workspace = _torch().empty(need, dtype=_torch().uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    st = lib().attn_fwd_fp8_ws(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(q_descale),
                               _ptr(k_descale), _ptr(v_descale), B, H, N_q, N_k, d, scale,
                               int(bool(causal)), _ptr(workspace), ws_bytes,
                               _stream(stream, q.device))
    _raise(st, "attn_fwd_fp8_ws")
    return o, lse


def attn_fwd_simt(q, k, v, o=None, lse=None, scale=None, causal=False, q_descale=None,
                  k_descale=None, v_descale=None, stream=None):
    """CUDA-core (no tensor core) forward pass: the independent GPU cross-check."""
    B, N_q, H, d, N_k = _check_inputs(q, k, v)
    o, lse = _outputs(q, o, lse, B, N_q, H, d)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    st = lib().attn_fwd_simt(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(q_descale),
                             _ptr(k_descale), _ptr(v_descale), B, H, N_q, N_k, d, scale,
                             int(bool(causal)), _dtype_code(q), _stream(stream, q.device))
    _raise(st, "attn_fwd_simt")
    return o, lse


def attn_fwd_gqa(q, k, v, o=None, lse=None, scale=None, causal=False, q_descale=None,
                 k_descale=None, v_descale=None, stream=None):
    """Grouped-query / multi-query attention: k, v are [B, N_k, H_kv, d]."""
    B, N_q, H, d, N_k = _check_inputs(q, k, v, gqa=True)
    H_kv = k.shape[2]
    o, lse = _outputs(q, o, lse, B, N_q, H, d)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    st = lib().attn_fwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(q_descale),
                            _ptr(k_descale), _ptr(v_descale), B, H, H_kv, N_q, N_k, d, scale,
                            int(bool(causal)), _dtype_code(q), _stream(stream, q.device))
    _raise(st, "attn_fwd_gqa")
    return o, lse


def attn_quantize_e4m3(x, signs=None, codes=None, descale=None, stream=None):
    """Rotate rows of x [B, N, H, d] by diag(signs) H_d / sqrt(d) (skipped when signs is
    None) and quantise to e4m3 with one fp32 descale per (batch, head)."""
    torch = _torch()
    if not (x.is_cuda and x.is_contiguous() and x.dim() == 4):
        raise ValueError("x must be a contiguous CUDA tensor [B, N, H, d]")
    codes_t = {torch.bfloat16: ATTN_BF16, torch.float16: ATTN_FP16, torch.float32: ATTN_FP32}
    if x.dtype not in codes_t:
        raise TypeError(f"unsupported input dtype {x.dtype}")
    B, N, H, d = x.shape
    if codes is None:
        codes = torch.empty(x.shape, dtype=torch.float8_e4m3fn, device=x.device)
    if descale is None:
        descale = torch.empty((B, H), dtype=torch.float32, device=x.device)
    if signs is not None and not (signs.is_cuda and signs.dtype == torch.float32
                                  and signs.numel() == d):
        raise ValueError("signs must be a CUDA float32 tensor of d values")
    st = lib().attn_quantize_e4m3(_ptr(x), codes_t[x.dtype], _ptr(codes), _ptr(descale), B, N,
                                  H, d, _ptr(signs), _stream(stream, x.device))
    _raise(st, "attn_quantize_e4m3")
    return codes, descale


def attn_splitkv_num_splits(B, H, N_q, N_k, d, num_sms=None) -> int:
    """Suggested num_splits for attn_fwd_splitkv (num_sms: of the current CUDA
    device when not given)."""
    if num_sms is None:
        torch = _torch()
        num_sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    return int(lib().attn_splitkv_num_splits(int(B), int(H), int(N_q), int(N_k), int(d), int(num_sms)))


def attn_splitkv_workspace_bytes(B, H, N_q, d, num_splits) -> int:
    return int(lib().attn_splitkv_workspace_bytes(B, H, N_q, d, num_splits))


def attn_fwd_splitkv(q, k, v, num_splits, o=None, lse=None, scale=None, causal=False,
                     q_descale=None, k_descale=None, v_descale=None, workspace=None,
                     stream=None):
    """Split-KV tensor-core forward pass; the workspace is allocated when not given."""
    B, N_q, H, d, N_k = _check_inputs(q, k, v)
    o, lse = _outputs(q, o, lse, B, N_q, H, d)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    need = attn_splitkv_workspace_bytes(B, H, N_q, d, num_splits)
    if workspace is None and need > 0:
        workspace = _torch().empty(need, dtype=_torch().uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().attn_fwd_splitkv(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(q_descale),
                                _ptr(k_descale), _ptr(v_descale), B, H, N_q, N_k, d, scale,
                                int(bool(causal)), _dtype_code(q), int(num_splits),
                                _ptr(workspace), ws_bytes, _stream(stream, q.device))
    _raise(st, "attn_fwd_splitkv")
    return o, lse


def attn_fwd_splitkv_static(q, k, v, num_splits, o=None, lse=None, scale=None, causal=False,
                            q_descale=None, k_descale=None, v_descale=None, stream=None):
    """attn_fwd_splitkv with no caller workspace: the partials go to the
    library's fixed ATTN_STATIC_SCRATCH_BYTES device array (calls whose work
    overlaps on the GPU share it).  Pass o and lse to allocate nothing here."""
    B, N_q, H, d, N_k = _check_inputs(q, k, v)
    o, lse = _outputs(q, o, lse, B, N_q, H, d)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    st = lib().attn_fwd_splitkv_static(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                       _ptr(q_descale), _ptr(k_descale), _ptr(v_descale), B, H,
                                       N_q, N_k, d, scale, int(bool(causal)), _dtype_code(q),
                                       int(num_splits), _stream(stream, q.device))
    _raise(st, "attn_fwd_splitkv_static")
    return o, lse


def attn_bwd_workspace_bytes(B, H, N_q):
    return int(lib().attn_bwd_workspace_bytes(int(B), int(H), int(N_q)))


def attn_fwd_host_workspace_bytes(B, H, N_q, N_k, d, dtype_code) -> int:
    return int(lib().attn_fwd_host_workspace_bytes(int(B), int(H), int(N_q), int(N_k), int(d),
                                                   int(dtype_code)))


def attn_fwd_host(q, k, v, o=None, lse=None, scale=None, causal=False, q_descale=None,
                  k_descale=None, v_descale=None, workspace=None, stream=None, device=None):
    """Forward pass on host (CPU) tensors, copies pipelined with the kernel.

    q, k, v: contiguous CPU tensors [B, N, H, d] (pinned for overlap); for
    float8_e4m3fn inputs the descales are CPU float32 tensors of B*H values.
    o, lse: CPU outputs (allocated pinned when not given).  workspace: a CUDA
    tensor of at least attn_fwd_host_workspace_bytes(...) bytes (allocated
    when not given).  The call returns once the work is queued on `stream`;
    synchronise that stream before reading o and lse.
    """
    torch = _torch()
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.is_cuda or not t.is_contiguous() or t.dim() != 4:
            raise ValueError(f"{name} must be a contiguous 4-D CPU tensor [B, N, H, d]")
    if q.dtype != k.dtype or q.dtype != v.dtype:
        raise TypeError("q, k, v must share one dtype")
    B, N_q, H, d = q.shape
    N_k = k.shape[1]
    if k.shape != v.shape or tuple(k.shape) != (B, N_k, H, d):
        raise ValueError("k and v must be [B, N_k, H, d] matching q")
    code = _dtype_code(q)
    fp8 = code == ATTN_FP8_E4M3
    if fp8:
        for name, t in (("q_descale", q_descale), ("k_descale", k_descale), ("v_descale", v_descale)):
            if t is None or t.is_cuda or t.dtype != torch.float32 or t.numel() != B * H or not t.is_contiguous():
                raise ValueError(f"{name} must be a contiguous CPU float32 tensor of B*H values")
    out_dtype = torch.float16 if q.dtype == torch.float16 else torch.bfloat16
    if o is None:
        o = torch.empty((B, N_q, H, d), dtype=out_dtype).pin_memory()
    if lse is None:
        lse = torch.empty((B, H, N_q), dtype=torch.float32).pin_memory()
    if o.is_cuda or o.dtype != out_dtype or tuple(o.shape) != (B, N_q, H, d) or not o.is_contiguous():
        raise ValueError("o must be a contiguous CPU [B, N_q, H, d] tensor of the output dtype")
    if lse.is_cuda or lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, N_q) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous CPU float32 [B, H, N_q] tensor")
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    ws_bytes = attn_fwd_host_workspace_bytes(B, H, N_q, N_k, d, code)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=device)
    elif workspace.numel() * workspace.element_size() < ws_bytes:
        raise ValueError(f"workspace needs {ws_bytes} bytes")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    with torch.cuda.device(device):
        st = lib().attn_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                 _ptr(q_descale if fp8 else None), _ptr(k_descale if fp8 else None),
                                 _ptr(v_descale if fp8 else None), B, H, N_q, N_k, d, scale,
                                 int(bool(causal)), code, _ptr(workspace),
                                 workspace.numel() * workspace.element_size(), _stream(stream, device))
    _raise(st, "attn_fwd_host")
    return o, lse


def attn_bwd(q, k, v, o, lse, dO, scale=None, causal=False, dq=None, dk=None, dv=None,
             workspace=None, stream=None):
    """Backward pass: (dq, dk, dv) for upstream gradient dO; o and lse from attn_fwd
    (or attn_fwd_gqa: k, v may have H_kv heads dividing H)."""
    torch = _torch()
    B, N_q, H, d, N_k = _check_inputs(q, k, v, gqa=True)
    H_kv = k.shape[2]
    for name, t, shape in (("o", o, q.shape), ("dO", dO, q.shape)):
        if tuple(t.shape) != tuple(shape) or t.dtype != q.dtype or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous {q.dtype} tensor of shape {tuple(shape)}")
    if tuple(lse.shape) != (B, H, N_q) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 tensor [B, H, N_q]")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    need = attn_bwd_workspace_bytes(B, H, N_q)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    st = lib().attn_bwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq),
                            _ptr(dk), _ptr(dv), B, H, H_kv, N_q, N_k, d, scale, int(bool(causal)),
                            _dtype_code(q), _ptr(workspace), ws_bytes, _stream(stream, q.device))
    _raise(st, "attn_bwd")
    return dq, dk, dv


# attn_bwd already takes k, v with H_kv heads dividing H (it calls the C
# attn_bwd_gqa); the same-name entry point of the C ABI.
attn_bwd_gqa = attn_bwd


def attn_last_cuda_error() -> str:
    """Name of the CUDA error behind the calling thread's last ATTN_ERR_CUDA."""
    return lib().attn_last_cuda_error().decode()


def attn_selftest_wait(timeout_us=1000, stream=None, device=None):
    """Launch the bounded-wait health check (its wait runs out after timeout_us)."""
    torch = _torch()
    dev = device if device is not None else torch.device("cuda", torch.cuda.current_device())
    st = lib().attn_selftest_wait(int(timeout_us), _stream(stream, dev))
    _raise(st, "attn_selftest_wait")


def attn_selftest_abort(q, k, v, q_descale=None, k_descale=None, v_descale=None, scale=None,
                        causal=False, timeout_us=500, workspace=None, stream=None):
    """Run the attention kernel with its K/V loader stopped after the first
    tile and every wait limited to timeout_us: the abort path's health check.
    With a workspace (e4m3, d = 64 / 128) attn_fwd_fp8_ws's kernels run.
    The next attn_check_status raises AttnError(ATTN_ERR_TIMEOUT)."""
    B, N_q, H, d, N_k = _check_inputs(q, k, v)
    o, lse = _outputs(q, None, None, B, N_q, H, d)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().attn_selftest_abort(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(q_descale),
                                   _ptr(k_descale), _ptr(v_descale), B, H, N_q, N_k, d, scale,
                                   int(bool(causal)), _dtype_code(q), _ptr(workspace), ws_bytes,
                                   int(timeout_us), _stream(stream, q.device))
    _raise(st, "attn_selftest_abort")


def attn_check_status(stream=None, device=None):
    """Synchronise the stream and raise AttnError if a kernel's bounded wait ran out."""
    torch = _torch()
    dev = device if device is not None else torch.device("cuda", torch.cuda.current_device())
    st = lib().attn_check_status(_stream(stream, dev))
    _raise(st, "attn_check_status")
    return st
