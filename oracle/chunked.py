"""Chunked KDA algebra in fp64 numpy — TEST INFRASTRUCTURE ONLY.

A second formulation of the KDA forward, written step by step from
"在 TPU 上加速 Kimi K3 KDA" (junyi.dev tpu-kda report):

  * §6.1  the gate's inclusive prefix sum inside each chunk (``gate_cumsum``);
  * §3/§4 the decayed score matrices Aqk and Akk, both as the elementwise
          decay tensor (``decay_scores_direct``) and as the sub-block
          midpoint strip products (``decay_scores_strips``) whose exponent
          budget is (SB/2)*|lower_bound|/ln 2 (``exponent_budget``);
  * §4    the solve with (I+L), by the finite Neumann factor chain applied
          to the right-hand side (``neumann_apply``) and as 16x16 block
          forward substitution (``blocked_solve``);
  * §4/§6.3 the WY right-hand side [beta*v | beta*k*exp(G)];
  * §6.2  the chunk recurrence and output, reading the entry state;
  * §6.4/§6.5 the flat packed-chunk table with seq_id / start / end flags.

It exists only to pin the token recurrence in ``kda_oracle.c`` (the two
formulations must agree to rounding on small inputs) and to check the
algebra the kernels rely on. It imports nothing from the CUDA path. Library
primitives used as single steps: ``numpy.cumsum``, ``@`` (matmul) and
``numpy.linalg.solve``.
"""
from __future__ import annotations

import math

import numpy as np

SB = 16  # sub-block size (§1–§2)
BT = 64  # chunk size (§3, appendix A)


def exponent_budget(sb: int = SB, lower_bound: float = -5.0) -> float:
    """Worst base-2 exponent of a midpoint-rescaled strip factor, §4 and §13:
    (SB/2) * |lower_bound| / ln 2 (8*5/0.693 = 57.7 for the K3 setting)."""
    return (sb / 2) * abs(lower_bound) / math.log(2.0)


def chunk_table(cu_seqlens, bt: int = BT):
    """Flat packed-chunk table over varlen sequences (§6.4–§6.5).

    Each sequence is cut into ceil(len/bt) chunks that restart at the
    sequence start. Returns a dict of int64 arrays, one entry per chunk in
    sequence order: ``seq_id``, ``local_chunk``, ``start`` (first token in the
    unpadded packing), ``length`` (tokens in the chunk), ``aligned_start``
    (chunk_id*bt: the address the same chunk has once every sequence is
    padded to a multiple of bt), ``aligned_cu_seqlens`` (per sequence),
    ``start_flag`` and ``end_flag``.
    """
    cu = [int(x) for x in cu_seqlens]
    seq_id, local, start, length, sflag, eflag = [], [], [], [], [], []
    aligned_cu = [0]
    for n in range(len(cu) - 1):
        L = cu[n + 1] - cu[n]
        nc = (L + bt - 1) // bt
        aligned_cu.append(aligned_cu[-1] + nc * bt)
        for c in range(nc):
            seq_id.append(n)
            local.append(c)
            start.append(cu[n] + c * bt)
            length.append(min(bt, L - c * bt))
            sflag.append(1 if c == 0 else 0)
            eflag.append(1 if c == nc - 1 else 0)
    a = lambda x: np.asarray(x, dtype=np.int64)
    return {
        "seq_id": a(seq_id), "local_chunk": a(local), "start": a(start),
        "length": a(length), "aligned_start": a(np.arange(len(seq_id)) * bt),
        "aligned_cu_seqlens": a(aligned_cu), "start_flag": a(sflag), "end_flag": a(eflag),
    }


def gate_cumsum(g):
    """Inclusive prefix sum of the log-decay along the chunk's tokens (§6.1)."""
    return np.cumsum(np.asarray(g, dtype=np.float64), axis=0)


def decay_scores_direct(a, b, G, strict: bool):
    """Elementwise decay tensor (§3, the form the strips replace):
    A[t,s] = sum_c a[t,c] b[s,c] exp(G[t,c] - G[s,c]) for s <= t (s < t if strict)."""
    n = a.shape[0]
    A = np.zeros((n, n))
    for t in range(n):
        for s in range(t if strict else t + 1):
            A[t, s] = np.sum(a[t] * b[s] * np.exp(G[t] - G[s]))
    return A


def decay_scores_strips(a, b, G, strict: bool, sb: int = SB):
    """Sub-block midpoint strip products (§4).

    For the strip of columns in sub-block j, with reference m_j the
    sub-block's midpoint row (16j+7, clipped to the chunk), the factor
    exp(G_t - G_s) is split as exp(G_t - G_m) * exp(G_m - G_s):
    ``a~_t = a_t exp(G_t - G_m)`` for rows t >= 16j and
    ``b~_s = b_s exp(G_m - G_s)`` for the strip's columns; the strip is a~ @ b~^T.
    Returns (A, max_abs_exponent), the exponent in base 2, over every factor
    the strips form.
    """
    n = a.shape[0]
    A = np.zeros((n, n))
    worst = 0.0
    for j0 in range(0, n, sb):
        j1 = min(j0 + sb, n)
        m = min(j0 + sb // 2 - 1, n - 1)
        ea = G[j0:] - G[m]          # rows t >= j0
        eb = G[m] - G[j0:j1]        # columns of the strip
        worst = max(worst, float(np.max(np.abs(eb))) / math.log(2.0),
                    float(np.max(ea[: j1 - j0])) / math.log(2.0) if j1 > j0 else 0.0)
        at = a[j0:] * np.exp(ea)
        bs = b[j0:j1] * np.exp(eb)
        A[j0:, j0:j1] = at @ bs.T
    keep = np.tril(np.ones((n, n)), -1 if strict else 0)
    return A * keep, worst


def neumann_apply(L, R):
    """(I+L)^{-1} R by the finite factor chain (I-L)(I+L^2)(I+L^4)... applied
    to the right-hand side, never forming the inverse (§4). Exact for a
    strictly lower-triangular (nilpotent) L of size n once 2^f >= n."""
    n = L.shape[0]
    X = R - L @ R
    P = L @ L
    span = 2
    while span < n:
        X = X + P @ X
        P = P @ P
        span *= 2
    return X


def blocked_solve(L, R, sb: int = SB):
    """(I+L)^{-1} R by 16x16 block forward substitution: the diagonal blocks
    are inverted by their own 4-factor Neumann chain, then
    X_i = (I+L_ii)^{-1} (R_i - sum_{j<i} L_ij X_j)."""
    n = L.shape[0]
    X = np.zeros_like(R, dtype=np.float64)
    for i0 in range(0, n, sb):
        i1 = min(i0 + sb, n)
        acc = R[i0:i1] - L[i0:i1, :i0] @ X[:i0]
        X[i0:i1] = neumann_apply(L[i0:i1, i0:i1], acc)
    return X


def chunk_step(q, k, v, g, beta, S, scale, solver: str = "blocked"):
    """One chunk of one (sequence, head) chain: §4 intra-chunk work, then the
    §6.2 recurrence and output reading the entry state S ([K,V], key rows).

    Returns (o [n,V], S_next [K,V], parts) with the chunk intermediates in
    ``parts`` (G, Aqk, L, u, w, v_new, strip exponent)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    beta = np.asarray(beta, dtype=np.float64)
    G = gate_cumsum(g)                                  # step (1)
    Aqk, e1 = decay_scores_strips(q, k, G, strict=False)  # step (2)
    Akk, e2 = decay_scores_strips(k, k, G, strict=True)
    L = beta[:, None] * Akk
    R = np.concatenate([beta[:, None] * v, beta[:, None] * k * np.exp(G)], axis=1)
    if solver == "blocked":                             # step (3)
        X = blocked_solve(L, R)
    elif solver == "neumann":
        X = neumann_apply(L, R)
    else:
        X = np.linalg.solve(np.eye(L.shape[0]) + L, R)
    V = v.shape[1]
    u, w = X[:, :V], X[:, V:]                           # step (4)
    v_new = u - w @ S                                   # step (5): entry state
    o = scale * ((q * np.exp(G)) @ S) + scale * (Aqk @ v_new)
    G_last = G[-1]
    S_next = np.exp(G_last)[:, None] * S + (k * np.exp(G_last[None, :] - G)).T @ v_new
    parts = {"G": G, "Aqk": Aqk, "L": L, "u": u, "w": w, "v_new": v_new,
             "exponent": max(e1, e2)}
    return o, S_next, parts


def kda_chunked(q, k, v, g, beta, cu_seqlens, initial_state=None, scale=None,
                bt: int = BT, solver: str = "blocked"):
    """Chunked KDA forward over varlen sequences: the chunk table of §6.5,
    the entry state loaded at each start_flag and stored at each end_flag."""
    q = np.asarray(q, dtype=np.float64)
    T, H, K = q.shape
    V = np.asarray(v).shape[2]
    cu = [int(x) for x in cu_seqlens]
    N = len(cu) - 1
    if scale is None:
        scale = K ** -0.5
    o = np.zeros((T, H, V))
    sT = np.zeros((N, H, K, V))
    tab = chunk_table(cu, bt)
    for h in range(H):
        S = None
        for c in range(len(tab["seq_id"])):
            n = int(tab["seq_id"][c])
            if tab["start_flag"][c]:
                S = (np.zeros((K, V)) if initial_state is None
                     else np.asarray(initial_state, dtype=np.float64)[n, h].copy())
            t0 = int(tab["start"][c])
            t1 = t0 + int(tab["length"][c])
            oc, S, _ = chunk_step(q[t0:t1, h], np.asarray(k)[t0:t1, h], np.asarray(v)[t0:t1, h],
                                  np.asarray(g)[t0:t1, h], np.asarray(beta)[t0:t1, h], S,
                                  scale, solver)
            o[t0:t1, h] = oc
            if tab["end_flag"][c]:
                sT[n, h] = S
        for n in range(N):  # empty sequences carry the initial state through
            if cu[n + 1] == cu[n]:
                sT[n, h] = (0.0 if initial_state is None
                            else np.asarray(initial_state, dtype=np.float64)[n, h])
    return o, sT
