"""Seeded synthetic inputs for the exact-attention forward pass.

This module is shared by the CPU oracle, the GPU parity tests and the benchmark.
It draws and rounds inputs only; it holds none of the attention arithmetic.

Workloads (shapes, dtypes, distributions) are the five attention-forward cases
the FlashAttention pages motivate: a tiny exact check, a short-sequence batch,
two causal long-context cases and an FP8 case with outliers ("FlashAttention-3 (BN)"
page, section "Low precision (FP8) and reducing quantisation error").

Recipe (all on the CPU, one ``torch.Generator`` per case):
  * seed = 1000 + case number (C1 -> 1001 ... C5 -> 1005);
  * q, k, v drawn in that order as float32 ``randn`` of shape [B, N, H, d];
  * bf16 / fp16 cases: each tensor rounded to the storage type (round to
    nearest even, torch's cast);
  * e4m3 case: after each ``randn`` draw, a ``rand`` draw of the same shape
    marks outliers (u < 0.001) whose value is multiplied by 10; then one fp32
    scale per (batch, head) s = amax|x[b, :, h, :]| / 448 and the stored code is
    clamp(x / s, -448, 448) cast to float8_e4m3fn (round to nearest even).
    The kernel receives the codes and the dequantisation scales ("descales").
"""

from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

E4M3_MAX = 448.0
OUTLIER_RATE = 1e-3
OUTLIER_GAIN = 10.0


@dataclasses.dataclass(frozen=True)
class Case:
    name: str
    B: int
    H: int
    N_q: int
    N_k: int
    d: int
    causal: bool
    dtype: str  # "bf16" | "fp16" | "e4m3"
    seed: int
    outliers: bool = False
    H_kv: int | None = None   # K/V heads (grouped-query attention); None = H

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def flops(self) -> float:
        """Counted FLOPs: 4*B*H*N_q*N_k*d, halved for causal."""
        f = 4.0 * self.B * self.H * self.N_q * self.N_k * self.d
        return f / 2.0 if self.causal else f


CASES = {
    "C1": Case("C1", 1, 1, 128, 128, 64, False, "bf16", 1001),
    "C2": Case("C2", 4, 16, 1024, 1024, 64, False, "bf16", 1002),
    "C3": Case("C3", 2, 16, 4096, 4096, 128, True, "bf16", 1003),
    "C4": Case("C4", 1, 16, 16384, 16384, 128, True, "bf16", 1004),
    "C5": Case("C5", 2, 16, 8192, 8192, 128, False, "e4m3", 1005, outliers=True),
}

# Extra workloads for the rows beyond the five cases (not benchmark headlines):
# a long K/V range with few query rows, where one CTA per query-tile pair leaves
# most SMs idle and the K/V range is split across CTAs.
EXTRA_CASES = {
    "LKV": Case("LKV", 1, 8, 512, 65536, 128, False, "bf16", 1101),
    # head dimension 256 (the largest head size the pages name), causal bf16
    "D256": Case("D256", 2, 8, 8192, 8192, 256, True, "bf16", 1102),
    # head dimension 256 in e4m3 (non-causal, 0.1 % x10 outliers like C5)
    "D256F": Case("D256F", 2, 8, 8192, 8192, 256, False, "e4m3", 1104, outliers=True),
    # backward pass: C3's shape (B2 H16 N4096 d128, causal bf16)
    "BWD": Case("BWD", 2, 16, 4096, 4096, 128, True, "bf16", 1103),
}


def custom_case(B, H, N_q, N_k, d, causal, dtype="bf16", seed=7, outliers=None, name="custom",
                H_kv=None):
    if outliers is None:
        outliers = dtype == "e4m3"
    return Case(name, B, H, N_q, N_k, d, bool(causal), dtype, seed, outliers, H_kv)


def _draw(g: torch.Generator, shape, outliers: bool) -> torch.Tensor:
    x = torch.randn(shape, generator=g, dtype=torch.float32)
    if outliers:
        u = torch.rand(shape, generator=g, dtype=torch.float32)
        x = torch.where(u < OUTLIER_RATE, x * OUTLIER_GAIN, x)
    return x


def quantize_e4m3_per_head(x: torch.Tensor):
    """Per-(batch, head) e4m3 codes of x [B, N, H, d] and their fp32 descales [B, H]."""
    amax = x.abs().amax(dim=(1, 3)).to(torch.float32)            # [B, H]
    amax = torch.where(amax > 0, amax, torch.ones_like(amax))
    descale = (amax / E4M3_MAX).to(torch.float32)
    y = x / descale[:, None, :, None]
    codes = y.clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn)
    return codes, descale.contiguous()


def make_inputs(case: Case) -> dict:
    """Inputs of one case as CPU tensors in [B, N, H, d] layout.

    Returns a dict with q, k, v (bf16 / fp16 / float8_e4m3fn) and, for e4m3,
    q_descale, k_descale, v_descale (float32 [B, H]); plus ``scale``.
    """
    g = torch.Generator().manual_seed(case.seed)
    out = {"scale": case.scale}
    h_kv = case.H if case.H_kv is None else case.H_kv
    shapes = {"q": (case.B, case.N_q, case.H, case.d),
              "k": (case.B, case.N_k, h_kv, case.d),
              "v": (case.B, case.N_k, h_kv, case.d)}
    for name in ("q", "k", "v"):
        x = _draw(g, shapes[name], case.outliers)
        if case.dtype == "bf16":
            out[name] = x.to(torch.bfloat16)
        elif case.dtype == "fp16":
            out[name] = x.to(torch.float16)
        elif case.dtype == "e4m3":
            codes, ds = quantize_e4m3_per_head(x)
            out[name] = codes
            out[name + "_descale"] = ds
        else:
            raise ValueError(f"unknown dtype {case.dtype}")
    return out


def make_raw_inputs(case: Case) -> dict:
    """The fp32 q, k, v of a case before any rounding (same draws as make_inputs)."""
    g = torch.Generator().manual_seed(case.seed)
    h_kv = case.H if case.H_kv is None else case.H_kv
    shapes = {"q": (case.B, case.N_q, case.H, case.d),
              "k": (case.B, case.N_k, h_kv, case.d),
              "v": (case.B, case.N_k, h_kv, case.d)}
    return {n: _draw(g, shapes[n], case.outliers) for n in ("q", "k", "v")}


def make_grad(case: Case) -> torch.Tensor:
    """Seeded upstream gradient dO [B, N_q, H, d] for the backward pass: fp32
    randn from its own generator (seed + 500 000, so the forward's q, k, v
    draws are unchanged), rounded to the case's dtype."""
    if case.dtype not in ("bf16", "fp16"):
        raise ValueError("the backward pass takes bf16 or fp16")
    g = torch.Generator().manual_seed(case.seed + 500_000)
    x = torch.randn((case.B, case.N_q, case.H, case.d), generator=g, dtype=torch.float32)
    return x.to(torch.bfloat16 if case.dtype == "bf16" else torch.float16)


def random_signs(d: int, seed: int) -> torch.Tensor:
    """A seeded vector of d random signs (+1 / -1), float32."""
    g = torch.Generator().manual_seed(seed)
    return (torch.randint(0, 2, (d,), generator=g) * 2 - 1).to(torch.float32)


def sample_rows(case: Case, n: int = 256, seed: int | None = None) -> np.ndarray:
    """Seeded (b, h, i) query-row triples, int64 [n, 3].

    Always contains rows 0, 1, 127, 128, 129 and N_q-1 (tile edges and the
    causal start) when they exist; the rest are uniform draws.
    """
    rng = np.random.default_rng(case.seed + 77 if seed is None else seed)
    edges = [i for i in (0, 1, 127, 128, 129, case.N_q - 1) if 0 <= i < case.N_q]
    rows = []
    for j, i in enumerate(edges):
        rows.append((j % case.B, (j * 7) % case.H, i))
    while len(rows) < n:
        rows.append((int(rng.integers(case.B)), int(rng.integers(case.H)), int(rng.integers(case.N_q))))
    return np.asarray(rows[:n], dtype=np.int64)
