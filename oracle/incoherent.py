"""Incoherent processing before FP8 quantisation, in float64 (oracle side).

TEST INFRASTRUCTURE ONLY.  "FlashAttention-3 (BN)" page, section "Low
precision (FP8) and reducing quantisation error": before attention, the query
and key vectors are multiplied by a random orthogonal matrix (a Hadamard matrix
is the example given), which spreads outlier values over all coordinates; the
result is then quantised to FP8; since the matrix is orthogonal, Q K^T is
unchanged.  Reading taken (the page fixes neither the randomisation nor the
quantisation granularity): M = diag(signs) H_d / sqrt(d) with H_d the
Sylvester Hadamard matrix and signs a seeded +-1 vector (an input), and one
fp32 scale per (batch, head) = amax / 448 with round-to-nearest-even codes
saturated to +-448.  V is quantised without rotation.
"""

from __future__ import annotations

import numpy as np
import torch

E4M3_MAX = 448.0


def hadamard(d: int) -> np.ndarray:
    """Sylvester Hadamard matrix H_d (d a power of two): H_1 = [1], H_2n = [[H, H], [H, -H]]."""
    if d < 1 or d & (d - 1):
        raise ValueError("d must be a power of two")
    h = np.ones((1, 1))
    while h.shape[0] < d:
        h = np.block([[h, h], [h, -h]])
    return h


def rotation(signs) -> np.ndarray:
    """The orthogonal matrix M = diag(signs) H_d / sqrt(d)."""
    s = np.asarray(signs, dtype=np.float64)
    d = s.shape[0]
    return (s[:, None] * hadamard(d)) / np.sqrt(d)


def rotate(x, signs) -> np.ndarray:
    """x [.., d] times M, in float64."""
    return np.asarray(x, dtype=np.float64) @ rotation(signs)


def quantize_e4m3_per_head(y: np.ndarray):
    """Per-(batch, head) e4m3 quantisation of y [B, N, H, d] (float64 in).

    Returns (codes as float64 values of the e4m3 codes, descale [B, H] fp32).
    The scale is computed in fp32 as amax / 448, the code as
    clamp(y / s, -448, 448) rounded to nearest even on the e4m3 grid.
    """
    yt = torch.from_numpy(np.asarray(y, dtype=np.float64))
    amax = yt.abs().amax(dim=(1, 3)).to(torch.float32)
    amax = torch.where(amax > 0, amax, torch.ones_like(amax))
    s = (amax / E4M3_MAX).to(torch.float32)
    z = (yt.to(torch.float32) / s[:, None, :, None]).clamp(-E4M3_MAX, E4M3_MAX)
    codes = z.to(torch.float8_e4m3fn).to(torch.float64).numpy()
    return codes, s.numpy()


def dequantize(codes, descale) -> np.ndarray:
    return np.asarray(codes, dtype=np.float64) * np.asarray(descale, dtype=np.float64)[:, None, :, None]


def incoherent_inputs(q, k, v, signs):
    """fp64 (q, k, v) that the FP8 attention sees after incoherent processing:
    q and k rotated then quantised, v quantised as is."""
    qc, qs = quantize_e4m3_per_head(rotate(q, signs))
    kc, ks = quantize_e4m3_per_head(rotate(k, signs))
    vc, vs = quantize_e4m3_per_head(np.asarray(v, dtype=np.float64))
    return dequantize(qc, qs), dequantize(kc, ks), dequantize(vc, vs)


def plain_fp8_inputs(q, k, v):
    """fp64 (q, k, v) after per-head e4m3 quantisation without rotation."""
    out = []
    for x in (q, k, v):
        c, s = quantize_e4m3_per_head(np.asarray(x, dtype=np.float64))
        out.append(dequantize(c, s))
    return tuple(out)
