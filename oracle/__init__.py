"""CPU fp64 oracle for the exact-attention forward pass.

TEST INFRASTRUCTURE ONLY.  Only the tests, the package smoke check and the
benchmark's CPU-baseline / reference legs may import this package.  The GPU
product path never calls it and shares no code with it: the one-pass recurrence
lives in attn_oracle.c (built here with gcc, no CUDA), the two-pass cross-check
in two_pass.py (numpy), the gradients of the backward pass in backward.py
(numpy), incoherent processing in incoherent.py (numpy).

Definition followed: Attention(Q,K,V) = softmax(Q K^T / sqrt(d_k)) V from the
"FlashAttention (HI)" page, section "Problems of standard attention"; the one-pass
form follows the same page, section "Online softmax computation".  Inputs are the rounded
values the GPU sees: bf16 / fp16 are converted to float64 exactly; e4m3 codes
are converted exactly and multiplied by their fp32 per-(batch, head) descale in
float64 (the FP8 inputs of the "FlashAttention-3 (BN)" page, section "Low precision
(FP8) and reducing quantisation error").  The oracle does not imitate any rounding the GPU applies inside the
computation; the tolerances cover that.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from . import two_pass  # noqa: F401  (re-exported)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB = None
_LOCK = threading.Lock()


def lib_path(mutant: int = 0) -> str:
    name = "liboracle.so" if mutant == 0 else f"liboracle_mut{mutant}.so"
    return os.path.join(_HERE, name)


def build(mutant: int = 0, force: bool = False) -> str:
    """Compile attn_oracle.c with gcc (OpenMP, strict IEEE, no fast-math)."""
    out = lib_path(mutant)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
           f"-DORACLE_MUTANT={mutant}", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _bind(path: str):
    lib = ctypes.CDLL(path)
    dp = ctypes.POINTER(ctypes.c_double)
    ip = ctypes.POINTER(ctypes.c_int64)
    i64 = ctypes.c_int64
    lib.oracle_attn_rows.argtypes = [dp, dp, dp, i64, i64, i64, i64, i64, ctypes.c_double,
                                     ctypes.c_int, ip, i64, dp, dp, ctypes.c_int]
    lib.oracle_attn_rows.restype = ctypes.c_int
    lib.oracle_attn_full.argtypes = [dp, dp, dp, i64, i64, i64, i64, i64, ctypes.c_double,
                                     ctypes.c_int, dp, dp, ctypes.c_int]
    lib.oracle_attn_full.restype = ctypes.c_int
    return lib


def load(mutant: int = 0):
    global _LIB
    if mutant != 0:
        return _bind(build(mutant))
    with _LOCK:
        if _LIB is None:
            _LIB = _bind(build(0))
    return _LIB


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _prep(q, k, v):
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    if q.ndim != 4 or k.shape != v.shape or q.shape[0] != k.shape[0] \
            or q.shape[2] != k.shape[2] or q.shape[3] != k.shape[3]:
        raise ValueError("expected q [B,N_q,H,d], k/v [B,N_k,H,d]")
    return q, k, v


def attention(q, k, v, scale, causal, n_threads=None, mutant=0):
    """One-pass fp64 oracle over every row: (O [B,N_q,H,d], lse [B,H,N_q])."""
    q, k, v = _prep(q, k, v)
    B, N_q, H, d = q.shape
    N_k = k.shape[1]
    o = np.empty_like(q)
    lse = np.empty((B, H, N_q))
    rc = load(mutant).oracle_attn_full(
        _ptr(q, ctypes.c_double), _ptr(k, ctypes.c_double), _ptr(v, ctypes.c_double),
        B, H, N_q, N_k, d, float(scale), int(bool(causal)),
        _ptr(o, ctypes.c_double), _ptr(lse, ctypes.c_double),
        int(n_threads or default_threads()))
    if rc != 0:
        raise RuntimeError(f"oracle_attn_full failed ({rc})")
    return o, lse


def attention_rows(q, k, v, scale, causal, rows, n_threads=None, mutant=0):
    """One-pass fp64 oracle on sampled (b, h, i) rows: (O [n,d], lse [n])."""
    q, k, v = _prep(q, k, v)
    B, N_q, H, d = q.shape
    N_k = k.shape[1]
    rows = np.ascontiguousarray(rows, dtype=np.int64).reshape(-1, 3)
    o = np.empty((len(rows), d))
    lse = np.empty(len(rows))
    rc = load(mutant).oracle_attn_rows(
        _ptr(q, ctypes.c_double), _ptr(k, ctypes.c_double), _ptr(v, ctypes.c_double),
        B, H, N_q, N_k, d, float(scale), int(bool(causal)),
        _ptr(rows, ctypes.c_int64), len(rows),
        _ptr(o, ctypes.c_double), _ptr(lse, ctypes.c_double),
        int(n_threads or default_threads()))
    if rc != 0:
        raise RuntimeError(f"oracle_attn_rows failed ({rc})")
    return o, lse


def to_f64(t) -> np.ndarray:
    """Exact float64 copy of a CPU tensor stored as bf16, fp16, fp32 or e4m3."""
    import torch
    return t.detach().to("cpu").to(torch.float64).numpy()


def dequant_e4m3(codes, descale) -> np.ndarray:
    """codes [B,N,H,d] (e4m3) times descale [B,H] (fp32), in float64."""
    x = to_f64(codes)
    s = to_f64(descale)
    return x * s[:, None, :, None]


def case_inputs_f64(inputs: dict):
    """float64 (q, k, v) of an input dict made by the synthetic generator."""
    if "q_descale" in inputs:
        return tuple(dequant_e4m3(inputs[n], inputs[n + "_descale"]) for n in ("q", "k", "v"))
    return tuple(to_f64(inputs[n]) for n in ("q", "k", "v"))
