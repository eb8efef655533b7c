"""Gradients of exact attention in numpy float64 (the backward pass).

TEST INFRASTRUCTURE ONLY.  Only the tests and the benchmark's CPU legs may
import this module; the GPU product path never calls it and shares no code
with it.

The pages name training speedups ("FlashAttention (HI)" page, section
"Empirical results") but never write the backward pass out, so this is the plain
derivative of the forward definition ("FlashAttention (HI)" page, section
"Problems of standard attention"), O = softmax(scale Q K^T [mask]) V, for an
upstream gradient dO of the same shape as O.  Per (batch, head), with the
row softmax P (masked entries 0; a row with no allowed key has P = 0, O = 0):

    dV = P^T dO
    dP = dO V^T
    D_i = sum_j P_ij dP_ij  (= sum_t dO_it O_it)
    dS = P * (dP - D)        (the softmax Jacobian applied row by row)
    dQ = scale dS K
    dK = scale dS^T Q

The causal mask is the forward's: key j is allowed for query i iff
j <= i + N_k - N_q.  Every matrix is materialised (O(N^2) memory); the
sizes used are small.

`mutant` plants one plausible mistake so the tests can show their pins catch
it: 1 drops the scale from dK, 2 skips the subtraction of D, 3 uses dS^T in
place of dS for dQ (square cases), 4 aligns the causal mask top-left.
"""

from __future__ import annotations

import numpy as np


def _allowed(N_q: int, N_k: int, causal: bool, top_left: bool = False) -> np.ndarray:
    """[N_q, N_k] boolean mask of allowed (query, key) pairs."""
    i = np.arange(N_q)[:, None]
    j = np.arange(N_k)[None, :]
    if not causal:
        return np.ones((N_q, N_k), dtype=bool)
    shift = 0 if top_left else N_k - N_q
    return j <= i + shift


def softmax_rows(S: np.ndarray, mask: np.ndarray) -> np.ndarray:
    """Row softmax of S over the allowed entries; rows with none are all zero."""
    S = np.where(mask, S, -np.inf)
    M = S.max(axis=1, initial=-np.inf)
    Msafe = np.where(np.isfinite(M), M, 0.0)
    W = np.where(mask, np.exp(S - Msafe[:, None]), 0.0)
    L = W.sum(axis=1)
    return W / np.where(L > 0, L, 1.0)[:, None]


def attention_backward(q, k, v, dO, scale, causal, mutant: int = 0):
    """(dq, dk, dv), float64, for q, dO [B, N_q, H, d] and k, v [B, N_k, H, d]."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    dO = np.asarray(dO, dtype=np.float64)
    B, N_q, H, d = q.shape
    N_k = k.shape[1]
    if k.shape != (B, N_k, H, d) or v.shape != k.shape or dO.shape != q.shape:
        raise ValueError("expected q, dO [B,N_q,H,d] and k, v [B,N_k,H,d]")
    mask = _allowed(N_q, N_k, causal, top_left=(mutant == 4))
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        for h in range(H):
            Q, K, V, G = q[b, :, h, :], k[b, :, h, :], v[b, :, h, :], dO[b, :, h, :]
            P = softmax_rows(scale * (Q @ K.T), mask)          # [N_q, N_k]
            dv[b, :, h, :] = P.T @ G
            dP = G @ V.T
            Drow = (P * dP).sum(axis=1)                        # [N_q]
            dS = P * (dP - (0.0 if mutant == 2 else Drow[:, None]))
            dq[b, :, h, :] = scale * ((dS.T if mutant == 3 else dS) @ K)
            dk[b, :, h, :] = (1.0 if mutant == 1 else scale) * (dS.T @ Q)
    return dq, dk, dv

