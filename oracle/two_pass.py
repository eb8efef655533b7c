"""Two-pass (materialised) softmax attention in numpy float64.

TEST INFRASTRUCTURE ONLY: the oracle's own cross-check.  It follows the
standard-attention definition on the "FlashAttention (HI)" page, section "Problems
of standard attention": build the whole score row S = scale * q K^T, apply the
mask, take the softmax with the row maximum subtracted, multiply by V.  It is
the "naive" O(N^2)-memory method the pages contrast with the fused kernel, so
it shares nothing with the one-pass recurrence in attn_oracle.c.
"""

from __future__ import annotations

import numpy as np


def allowed_keys(i: int, N_q: int, N_k: int, causal: bool) -> int:
    """Number of allowed keys for query row i (keys 0 .. count-1)."""
    if not causal:
        return N_k
    return int(min(N_k, max(0, i + (N_k - N_q) + 1)))


def attention_rows(q, k, v, scale, causal, rows, check_rows_sum=True):
    """O [n, d] and lse [n] for the (b, h, i) triples in rows.

    q: [B, N_q, H, d]; k, v: [B, N_k, H, d] (float64 arrays).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, N_q, H, d = q.shape
    N_k = k.shape[1]
    rows = np.asarray(rows, dtype=np.int64).reshape(-1, 3)
    O = np.zeros((len(rows), d))
    lse = np.full(len(rows), -np.inf)
    # group rows by (b, h) so each group is one matrix product
    order = np.lexsort((rows[:, 2], rows[:, 1], rows[:, 0]))
    for bh in np.unique(rows[:, 0] * H + rows[:, 1]):
        b, h = divmod(int(bh), H)
        sel = order[(rows[order, 0] == b) & (rows[order, 1] == h)]
        qi = q[b, rows[sel, 2], h, :]                    # [m, d]
        S = scale * (qi @ k[b, :, h, :].T)               # [m, N_k]
        cnt = np.array([allowed_keys(int(i), N_q, N_k, causal) for i in rows[sel, 2]])
        mask = np.arange(N_k)[None, :] < cnt[:, None]
        S = np.where(mask, S, -np.inf)
        M = S.max(axis=1, initial=-np.inf)
        Msafe = np.where(np.isfinite(M), M, 0.0)
        W = np.where(mask, np.exp(S - Msafe[:, None]), 0.0)
        L = W.sum(axis=1)
        Lsafe = np.where(L > 0, L, 1.0)
        P = W / Lsafe[:, None]
        if check_rows_sum:
            ok = cnt > 0
            if ok.any():
                err = np.abs(P[ok].sum(axis=1) - 1.0).max()
                assert err < 1e-12, f"softmax rows do not sum to 1 (err {err})"
        O[sel] = P @ v[b, :, h, :]
        lse[sel] = np.where(L > 0, M + np.log(Lsafe), -np.inf)
    return O, lse


def attention_full(q, k, v, scale, causal):
    """O [B, N_q, H, d] and lse [B, H, N_q] over every row."""
    B, N_q, H, d = np.shape(q)
    bb, hh, ii = np.meshgrid(np.arange(B), np.arange(H), np.arange(N_q), indexing="ij")
    rows = np.stack([bb.ravel(), hh.ravel(), ii.ravel()], axis=1)
    O_r, lse_r = attention_rows(q, k, v, scale, causal, rows)
    O = np.zeros((B, N_q, H, d))
    O[rows[:, 0], rows[:, 2], rows[:, 1], :] = O_r
    return O, lse_r.reshape(B, H, N_q)
