"""Exact causal GQA attention on selected rows of a long sequence (TEST
INFRASTRUCTURE ONLY; imported by tests/ alone).

The full oracle (``oracle.cpp``) computes attention in O(S^2 hd), out of reach
at 32K-512K tokens.  One query row, though, is an O(S hd) computation straight
from the definition of causal softmax attention (the decoder's attention
block, as in the pages' model description): for query i of head h, with kv
head g = h // (nh / nkv),

    s_j = q_i . k_j / sqrt(hd) for j <= i,  lse_i = log sum_j exp(s_j),
    p_j = exp(s_j - lse_i),  o_i = sum_j p_j v_j,

and its backward, with delta_i = dO_i . o_i and dP_ij = dO_i . v_j,

    dS_ij = p_ij (dP_ij - delta_i),  dq_i = sum_j dS_ij k_j / sqrt(hd),
    dv_j = sum_h sum_{i >= j} p_ij dO_i,  dk_j = sum_h sum_{i >= j} dS_ij q_i / sqrt(hd).

dv_j and dk_j need every query i >= j, so key rows are taken near the end of
the sequence.  Everything is float64 numpy; the rows are computed one head at
a time as small dense products.
"""
from __future__ import annotations

import numpy as np


def rows_needed(q_rows, k_rows, S):
    """The query rows attention_rows reads: q_rows and every row at or after
    the first of k_rows (sorted)."""
    k_rows = np.asarray(k_rows, dtype=np.int64)
    first_key = int(k_rows.min()) if k_rows.size else S
    return np.union1d(np.asarray(q_rows, dtype=np.int64), np.arange(first_key, S))


def attention_rows(q, k, v, dout, n_heads, n_kv, hd, q_rows, k_rows):
    """k, v: [S, nkv*hd] (one sequence, float64); q, dout: [S, nh*hd], or
    only the rows_needed(q_rows, k_rows, S) of them, in that order.
    Returns o, dq and the magnitude sums |.| of their summands for q_rows,
    lse (natural log) [len(q_rows), nh], and dk, dv with summand magnitudes
    for k_rows."""
    S = k.shape[0]
    scale = 1.0 / np.sqrt(hd)
    grp = n_heads // n_kv
    q_rows = np.asarray(q_rows, dtype=np.int64)
    k_rows = np.asarray(k_rows, dtype=np.int64)
    need = rows_needed(q_rows, k_rows, S)
    if q.shape[0] == S and need.size != S:  # full arrays given
        q, dout = q[need], dout[need]
    assert q.shape[0] == need.size and dout.shape[0] == need.size
    pos = {int(r): i for i, r in enumerate(need)}
    qi = np.array([pos[int(r)] for r in q_rows], dtype=np.int64)
    nq, nk = q_rows.size, k_rows.size
    out = {
        "o": np.zeros((nq, n_heads * hd)), "lse": np.zeros((nq, n_heads)),
        "dq": np.zeros((nq, n_heads * hd)), "dq_mag": np.zeros((nq, n_heads * hd)),
        "dk": np.zeros((nk, n_kv * hd)), "dk_mag": np.zeros((nk, n_kv * hd)),
        "dv": np.zeros((nk, n_kv * hd)), "dv_mag": np.zeros((nk, n_kv * hd)),
    }
    later = need[:, None] >= k_rows[None, :]  # query i attends to key j
    for h in range(n_heads):
        g = h // grp
        K = k[:, g * hd:(g + 1) * hd]
        V = v[:, g * hd:(g + 1) * hd]
        Q = q[:, h * hd:(h + 1) * hd]
        dO = dout[:, h * hd:(h + 1) * hd]
        s = (Q @ K.T) * scale
        s[np.arange(S)[None, :] > need[:, None]] = -np.inf
        m = s.max(axis=1)
        lse = m + np.log(np.exp(s - m[:, None]).sum(axis=1))
        P = np.exp(s - lse[:, None])
        o = P @ V
        delta = (dO * o).sum(axis=1)
        dP = dO @ V.T
        dS = P * (dP - delta[:, None])
        # magnitudes of the terms behind each dS entry: dP_ij and the summands
        # of delta_i (an implementation that forms delta from its own rounded o
        # errs in proportion to sum |dO| |o|, not to |delta|)
        dSmag = P * (np.abs(dP) + (np.abs(dO) * np.abs(o)).sum(axis=1)[:, None])
        cols = slice(h * hd, (h + 1) * hd)
        out["o"][:, cols] = o[qi]
        out["lse"][:, h] = lse[qi]
        out["dq"][:, cols] = scale * (dS[qi] @ K)
        out["dq_mag"][:, cols] = scale * (dSmag[qi] @ np.abs(K))
        gcols = slice(g * hd, (g + 1) * hd)
        Pk = P[:, k_rows] * later
        dSk = dS[:, k_rows] * later
        out["dv"][:, gcols] += Pk.T @ dO
        out["dv_mag"][:, gcols] += Pk.T @ np.abs(dO)
        out["dk"][:, gcols] += scale * (dSk.T @ Q)
        out["dk_mag"][:, gcols] += scale * ((dSmag[:, k_rows] * later).T @ np.abs(Q))
    return out
