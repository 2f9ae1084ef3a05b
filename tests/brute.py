"""Brute-force restatement of the kept set K for tiny vocabularies.

Independent of the oracle's sort-based code: the order is established by
counting, for every token, how many tokens precede it (O(V^2)); prefix masses
are sums over those ranks.  Used only to pin the oracle on V <= 64.
"""
import numpy as np


def rank_of(y):
    """rank[t] = number of allowed tokens before t in (y desc, index asc)."""
    V = y.size
    allowed = y > -np.inf
    rank = np.full(V, -1, np.int64)
    for t in range(V):
        if not allowed[t]:
            continue
        before = 0
        for s in range(V):
            if allowed[s] and (y[s] > y[t] or (y[s] == y[t] and s < t)):
                before += 1
        rank[t] = before
    return rank


def kept_set(y, top_k=0, top_p=1.0, min_p=0.0):
    """Return (K as a boolean mask, probabilities over K) for processed logits y."""
    y = np.asarray(y, np.float32)
    rank = rank_of(y)
    n = int((rank >= 0).sum())
    by_rank = np.full(n, -1, np.int64)
    for t in range(y.size):
        if rank[t] >= 0:
            by_rank[rank[t]] = t
    ymax = float(y[by_rank[0]])
    w = np.array([np.exp(np.float64(y[t]) - ymax) for t in by_rank])
    Lk = top_k if 0 < top_k < n else n
    L = Lk
    if top_p < 1.0:
        Sk = w[:Lk].sum()
        for c in range(1, Lk + 1):
            if w[:c].sum() / Sk >= top_p:
                L = min(L, c)
                break
    if min_p > 0.0:
        L = min(L, int((w >= min_p).sum()))
    K = np.zeros(y.size, bool)
    K[by_rank[:L]] = True
    P = np.zeros(y.size)
    P[by_rank[:L]] = w[:L] / w[:L].sum()
    return K, P
