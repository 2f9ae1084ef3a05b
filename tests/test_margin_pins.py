"""Pins of the oracle's decision-margin machinery, by brute force.

The parity rule excuses decisions within 1e-5 relative ("rows whose decision
margin is below 1e-5 relative are counted and reported").  The oracle states
that margin as a perturbation model, and these tests enumerate the model's
extreme points on tiny rows instead of re-deriving its closed forms:

- top-p: every renormalised probability of the top-k prefix may move by
  1e-5 relative; min-p: every ratio w = exp(y - ymax) may (the maximum's own
  w = 1 is exact).  kept_lo / kept_hi must be the smallest / largest kept
  size over all such perturbations.
- draw: each processed logit y_t and each Gumbel value g_t may move by
  1e-5 * max(1, |value|); the draw's flag must fire exactly when some
  perturbation changes the winner.
- accept: P(x) may move by 1e-5 relative (u and q are inputs, exact).
- residual: each P_t may move by 1e-5 relative and each g_t as above.

Rows are built with the decision placed at chosen distances from its
threshold (inside and outside the margin), so both answers are exercised.
"""
import itertools

import numpy as np
import pytest

from oracle import oracle as O
from tests.helpers import sample_workload, verify_workload

DELTA = 1e-5


def _m(v):
    return DELTA * max(1.0, abs(v))


# ----------------------------------------------------------- kept sizes


def _brute_kept_range(y_sorted, top_k, top_p, min_p):
    """Smallest and largest kept size over the vertices of the perturbation
    box (the comparisons are monotone in every perturbed quantity, so the
    extremes are reached at vertices)."""
    n = len(y_sorted)
    w = np.exp(y_sorted.astype(np.float64) - float(y_sorted[0]))
    Lk = top_k if 0 < top_k < n else n
    Lp_set = {Lk}
    if top_p < 1.0:
        p = w[:Lk] / w[:Lk].sum()
        Lp_set = set()
        for signs in itertools.product((-1.0, 1.0), repeat=Lk):
            pp = p * (1.0 + DELTA * np.asarray(signs))
            c = np.cumsum(pp)
            hit = np.flatnonzero(c >= float(top_p))
            Lp_set.add(int(hit[0]) + 1 if hit.size else Lk)
    Lm_set = {n}
    if min_p > 0.0:
        Lm_set = set()
        free = [j for j in range(n) if w[j] != 1.0]
        for signs in itertools.product((-1.0, 1.0), repeat=len(free)):
            ww = w.copy()
            for j, s in zip(free, signs):
                ww[j] = w[j] * (1.0 + DELTA * s)
            L = 0
            while L < n and ww[L] >= float(min_p):
                L += 1
            Lm_set.add(L)
    lo = min(Lk, min(Lp_set), min(Lm_set))
    hi = min(Lk, max(Lp_set), max(Lm_set))
    return lo, hi


def _sorted_y(processed_row):
    y = processed_row[np.isfinite(processed_row)]
    idx = np.flatnonzero(np.isfinite(processed_row))
    order = np.lexsort((idx, -y))
    return y[order]


@pytest.mark.parametrize("eps", [-3e-5, -1.2e-5, -0.8e-5, -0.3e-5, 0.0, 0.3e-5, 0.8e-5, 1.2e-5, 3e-5])
def test_kept_range_top_p_equals_brute_force(eps):
    rng = np.random.default_rng(100)
    rows, top_ps, top_ks = [], [], []
    for r in range(24):
        y = np.sort(rng.normal(0.0, 1.0, 8).astype(np.float32))[::-1].copy()
        w = np.exp(y.astype(np.float64) - float(y[0]))
        top_k = int(rng.choice([0, 6]))
        Lk = top_k if top_k else 8
        c = np.cumsum(w[:Lk]) / w[:Lk].sum()
        i = int(rng.integers(0, Lk - 1))
        # a prefix mass placed eps (relative) from the threshold
        top_ps.append(np.float32(c[i] * (1.0 + eps)))
        rows.append(y)
        top_ks.append(top_k)
    z = np.stack(rows)
    w_ = sample_workload(z, temperature=1.0, top_k=np.array(top_ks), top_p=np.array(top_ps))
    res = O.process_sample(w_, want_processed=True)
    for r in range(len(rows)):
        lo, hi = _brute_kept_range(_sorted_y(res["processed"][r]), top_ks[r], float(top_ps[r]), 0.0)
        assert (res["kept_lo"][r], res["kept_hi"][r]) == (lo, hi), (r, eps, res["kept_lo"][r], res["kept_hi"][r], lo, hi)
        assert lo <= res["kept_own"][r] <= hi


@pytest.mark.parametrize("eps", [-3e-5, -1.2e-5, -0.8e-5, -0.3e-5, 0.3e-5, 0.8e-5, 1.2e-5, 3e-5])
def test_kept_range_min_p_equals_brute_force(eps):
    rng = np.random.default_rng(200)
    rows, min_ps = [], []
    for r in range(24):
        y = np.sort(rng.normal(0.0, 1.5, 8).astype(np.float32))[::-1].copy()
        if r % 4 == 0:
            y[1] = y[0]  # a second exact 1 ratio
        w = np.exp(y.astype(np.float64) - float(y[0]))
        i = int(rng.integers(1, 8))
        min_ps.append(np.float32(min(1.0, w[i] * (1.0 + eps))))
        rows.append(y)
    z = np.stack(rows)
    w_ = sample_workload(z, temperature=1.0, min_p=np.array(min_ps))
    res = O.process_sample(w_, want_processed=True)
    for r in range(len(rows)):
        lo, hi = _brute_kept_range(_sorted_y(res["processed"][r]), 0, 1.0, float(min_ps[r]))
        assert (res["kept_lo"][r], res["kept_hi"][r]) == (lo, hi), (r, eps, res["kept_lo"][r], res["kept_hi"][r], lo, hi)
        assert lo <= res["kept_own"][r] <= hi


def test_kept_range_joint_filters_equals_brute_force():
    rng = np.random.default_rng(300)
    n = 40
    z = rng.normal(0.0, 1.0, (n, 8)).astype(np.float32)
    top_k = rng.choice([0, 3, 6], n).astype(np.int32)
    top_p = np.empty(n, np.float32)
    min_p = np.empty(n, np.float32)
    for r in range(n):
        y = np.sort(z[r].astype(np.float64))[::-1]
        w = np.exp(y - y[0])
        Lk = top_k[r] if top_k[r] else 8
        c = np.cumsum(w[:Lk]) / w[:Lk].sum()
        top_p[r] = np.float32(c[rng.integers(0, Lk - 1)] * (1.0 + rng.choice([-2e-5, -0.5e-5, 0.5e-5, 2e-5])))
        min_p[r] = np.float32(w[rng.integers(1, 8)] * (1.0 + rng.choice([-2e-5, -0.5e-5, 0.5e-5, 2e-5])))
    w_ = sample_workload(z, temperature=1.0, top_k=top_k, top_p=top_p, min_p=min_p)
    res = O.process_sample(w_, want_processed=True)
    for r in range(n):
        lo, hi = _brute_kept_range(_sorted_y(res["processed"][r]), int(top_k[r]), float(top_p[r]), float(min_p[r]))
        assert (res["kept_lo"][r], res["kept_hi"][r]) == (lo, hi), r


# ------------------------------------------------------------ draw flag


def _winner(scores, tokens):
    best = None
    for s, t in zip(scores, tokens):
        if s is None:
            continue
        if best is None or s > best[0] or (s == best[0] and t < best[1]):
            best = (s, t)
    return None if best is None else best[1]


def _brute_draw_flag(y, g):
    """The winner of argmax(y + g) (lowest index on ties) is not the same at
    every vertex of the perturbation box of y and g."""
    n = len(y)
    winners = set()
    for sy in itertools.product((-1.0, 1.0), repeat=n):
        for sg in itertools.product((-1.0, 1.0), repeat=n):
            sc = [y[t] + sy[t] * _m(y[t]) + g[t] + sg[t] * _m(g[t]) for t in range(n)]
            winners.add(_winner(sc, range(n)))
    return len(winners) > 1


@pytest.mark.parametrize("k_gap", [-3.0, -1.5, -0.6, -0.2, 0.2, 0.6, 1.5, 3.0])
def test_draw_flag_fires_exactly_when_a_perturbation_flips(k_gap):
    seeds = range(6)
    V = 4
    for seed in seeds:
        pos = 17 + seed
        g = [O.gumbel(seed, 0, pos, t, 0) for t in range(V)]
        y0 = np.float32(2.0)
        scale = _m(float(y0)) + _m(g[0]) + _m(float(y0) + g[0] - g[1]) + _m(g[1])
        y1 = np.float32(float(y0) + g[0] - g[1] + k_gap * scale)
        z = np.array([[y0, y1, -30.0, -31.0]], np.float32)
        w_ = sample_workload(z, temperature=1.0, seed=seed, position=pos)
        res = O.process_sample(w_)
        want = _brute_draw_flag([float(v) for v in z[0]], g)
        assert bool(res["sub_margin"][0]) == want, (seed, k_gap, res["sub_margin"][0], want)
        assert res["token"][0] == _winner([float(z[0][t]) + g[t] for t in range(V)], range(V))


# ----------------------------------------------------- accept / residual


def _row_P(y):
    w = np.exp(np.asarray(y, np.float64) - float(np.max(y)))
    return w / w.sum()


def _brute_residual_flag(P, q, g):
    """Over the vertices of the box (P_t +- 1e-5 P_t, g_t +- margin): does the
    residual winner (argmax of log(P - q) + g over P > q) change?"""
    n = len(P)
    winners = set()
    for sp in itertools.product((-1.0, 1.0), repeat=n):
        for sg in itertools.product((-1.0, 1.0), repeat=n):
            sc = []
            for t in range(n):
                r = P[t] * (1.0 + DELTA * sp[t]) - q[t]
                sc.append(np.log(r) + g[t] + sg[t] * _m(g[t]) if r > 0 else None)
            winners.add(_winner(sc, range(n)))
    return len(winners) > 1


def _brute_bonus_flag(y, seed, pos):
    g = [O.gumbel(seed, 0, pos, t, 0) for t in range(len(y))]
    return _brute_draw_flag([float(v) for v in y], g)


@pytest.mark.parametrize("eps", [-3e-5, -1.1e-5, -0.9e-5, -0.4e-5, 0.4e-5, 0.9e-5, 1.1e-5, 3e-5])
def test_accept_flag_fires_exactly_when_a_perturbation_flips(eps):
    V = 4
    for seed in range(5):
        pos = 40 + seed
        y0 = np.array([1.0, 0.5, -0.25, -1.0], np.float32)
        y1 = np.array([-20.0, 25.0, -20.0, -21.0], np.float32)  # bonus row: a clear winner
        P = _row_P(y0)
        x = 1
        u = O.uniform(seed, 0, pos, 0, 1)
        qx = np.float32(P[x] / u * (1.0 + eps))
        if qx > 1.0:
            continue
        q = np.zeros(V, np.float32)
        q[x] = qx
        w_ = verify_workload(np.stack([y0, y1]), [1], [x], q[None, :], seed=seed, position=pos)
        res = O.spec_verify(w_)
        uq = float(u) * float(qx)
        accept_flip = (uq < P[x] * (1 - DELTA)) != (uq < P[x] * (1 + DELTA))
        accepted = uq < P[x]
        if accepted:
            other = _brute_bonus_flag(y1, seed, pos + 1)
        else:
            gr = [O.gumbel(seed, 0, pos, t, 2) for t in range(V)]
            other = _brute_residual_flag(P, q.astype(np.float64), gr)
        assert bool(res["sub_margin"][0]) == (accept_flip or other), (seed, eps, res["sub_margin"][0], accept_flip, other)
        assert res["num_accepted"][0] == int(accepted)


@pytest.mark.parametrize("k_gap", [-3.0, -1.3, -0.7, -0.2, 0.2, 0.7, 1.3, 3.0])
def test_residual_flag_fires_exactly_when_a_perturbation_flips(k_gap):
    V = 4
    done = 0
    for seed in range(40):
        pos = 60 + seed
        u = O.uniform(seed, 0, pos, 0, 1)
        if u < 0.5:
            continue  # keep the draft clearly rejected below
        y0 = np.array([0.2, 1.4, -0.3, -2.0], np.float32)  # P ~ (.19, .62, .12, .03)
        P = _row_P(y0)
        x, a, b = 2, 0, 1
        gr = [O.gumbel(seed, 0, pos, t, 2) for t in range(V)]
        # residuals: r_a = P_a (q_a = 0); r_b chosen so that log r_b + g_b
        # sits k_gap margins from log r_a + g_a
        scale = DELTA * P[a] / P[a] + _m(gr[a]) + DELTA * 2.0 + _m(gr[b])
        rb = P[a] * np.exp(gr[a] - gr[b] + k_gap * scale)
        if not (0.05 * P[b] < rb < 0.95 * P[b]):
            continue
        q = np.zeros(V, np.float64)
        q[b] = P[b] - rb
        q[x] = 0.95  # u * q >= 0.47 > P_x: rejected
        q[3] = 1.0   # token 3 leaves no residual
        q32 = q.astype(np.float32)
        w_ = verify_workload(np.stack([y0, np.array([-9.0, 30.0, -9.0, -9.0], np.float32)]), [1], [x],
                             q32[None, :], seed=seed, position=pos)
        res = O.spec_verify(w_)
        assert res["num_accepted"][0] == 0
        want = _brute_residual_flag(P, q32.astype(np.float64), gr)
        assert bool(res["sub_margin"][0]) == want, (seed, k_gap, res["sub_margin"][0], want)
        done += 1
        if done == 4:
            break
    assert done > 0


# ------------------------------------- logits known within a bound (LM head)


def _brute_interval_flag(z, b, T, g):
    """The winner of argmax((z_t + e_t) / T + g_t), e_t in [-b_t, b_t], with
    y_t and g_t each moving by their margin as well, differs between vertices
    of that box (greedy, T = 0: argmax of z_t + e_t, z_t's margin)."""
    n = len(z)
    inv_t = float(np.float32(1.0) / np.float32(T)) if T else None
    winners = set()
    for se in itertools.product((-1.0, 1.0), repeat=n):
        for sy in itertools.product((-1.0, 1.0), repeat=n):
            sgs = itertools.product((-1.0, 1.0), repeat=n) if T else [(0.0,) * n]
            for sg in sgs:
                sc = []
                for t in range(n):
                    if T:
                        y = float(np.float32(z[t]) * np.float32(inv_t))
                        sc.append(y + se[t] * b[t] * inv_t + sy[t] * _m(y) + g[t] + sg[t] * _m(g[t]))
                    else:
                        sc.append(z[t] + se[t] * b[t] + sy[t] * _m(z[t]))
                winners.add(_winner(sc, range(n)))
    return len(winners) > 1


@pytest.mark.parametrize("T", [0.0, 0.7, 1.3])
@pytest.mark.parametrize("k_gap", [-2.0, -1.2, -0.85, -0.2, 0.2, 0.85, 1.2, 2.0])
def test_interval_flag_fires_exactly_when_a_logit_in_its_bound_flips(T, k_gap):
    V = 4
    for seed in range(4):
        pos = 40 + seed
        b = np.array([0.01, 0.004, 0.02, 0.001]) * (1 + seed)
        g = O.gumbel_row(seed, 0, pos, V) if T else np.zeros(V)
        inv_t = float(np.float32(1.0) / np.float32(T)) if T else 1.0
        z0 = np.float32(1.5)
        # the total uncertainty of tokens 0 and 1 (the two leaders)
        y0 = float(np.float32(z0) * np.float32(inv_t)) if T else float(z0)
        unc = (b[0] + b[1]) * inv_t + 2 * _m(y0) + (_m(g[0]) + _m(g[1]) if T else 0.0)
        # token 1's score sits k_gap uncertainties below token 0's
        z1 = np.float32(float(z0) + (g[0] - g[1]) / inv_t + k_gap * unc / inv_t)
        z = np.array([[z0, z1, -30.0, -31.0]], np.float32)
        flags = O.interval_flags(z, b[None, :], np.array([T], np.float32), np.array([seed], np.uint64),
                                 np.array([pos], np.int64))
        want = _brute_interval_flag([float(v) for v in z[0]], b, T, g)
        assert bool(flags[0]) == want, (seed, T, k_gap, flags[0], want)


def test_interval_flags_reduce_to_the_draw_margin_at_zero_bound():
    # with exact logits the interval test is the oracle's own draw margin
    rng = np.random.default_rng(5)
    z = rng.normal(0, 2, (24, 7)).astype(np.float32)
    z[:, 2:] -= 30.0
    T = rng.uniform(0.5, 1.5, 24).astype(np.float32)
    seed = rng.integers(0, 2**63, 24, dtype=np.uint64)
    pos = rng.integers(0, 1000, 24).astype(np.int64)
    for r in range(0, 24, 2):  # even rows: tokens 0 and 1 tie to within the margin
        g = O.gumbel_row(int(seed[r]), r, int(pos[r]), 2)
        z[r, 1] = np.float32(float(z[r, 0]) + (g[0] - g[1]) * float(T[r]))
    w = sample_workload(z, temperature=T, seed=seed, position=pos)
    res = O.process_sample(w)
    flags = O.interval_flags(z, 0.0, T, seed, pos)
    assert np.array_equal(flags, res["sub_margin"]) and flags.any() and not flags.all()
    # caller row ids (the Philox counter's row word), above 2^31 too
    w["row_id"] = rng.integers(0, 2**32, 24, dtype=np.uint64).astype(np.uint32)
    res = O.process_sample(w)
    assert np.array_equal(O.interval_flags(z, 0.0, T, seed, pos, w["row_id"]), res["sub_margin"])
