"""Pins of the CPU oracle against things other than itself.

- Philox4x32-10 against triton's library implementation (interpreter, CPU).
- Gumbel noise against scipy's Gumbel distribution (KS test).
- Processed logits against hand-derived dyadic values (tests/golden).
- Kept sets and probabilities against an O(V^2) rank-counting brute force.
- Greedy against numpy's argmax (first occurrence).
- Gumbel-max draw: decomposability over vocabulary partitions (FlashSampling
  page), and its law against the kept distribution by chi-square on 1e6 draws.
- Speculative verification: exact enumeration on V <= 8 of the accept /
  residual composition, chi-square of the realised algorithm, greedy case.
"""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

from oracle import oracle as O
from speculative_verification_gb300 import workloads as W
from tests import brute
from tests.helpers import sample_workload, verify_workload
from tests.parity import subset_sample

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

# ------------------------------------------------------------------- Philox


def test_philox_matches_triton_library():
    pytest.importorskip("triton")
    rng = np.random.default_rng(7)
    ctrs = [[0, 0, 0, 0], [1, 0, 0, 0], [0xFFFFFFFF] * 4]
    ctrs += rng.integers(0, 2**32, size=(13, 4), dtype=np.uint64).tolist()
    seeds = [0, 0, 0x7FFFFFFF7FFFFFFF] + rng.integers(0, 2**62, size=13, dtype=np.int64).tolist()
    env = dict(os.environ, TRITON_INTERPRET="1")
    r = subprocess.run([sys.executable, os.path.join(HERE, "_triton_philox.py")],
                       input=json.dumps({"ctr": ctrs, "seed": [int(s) for s in seeds]}),
                       capture_output=True, text=True, env=env, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    ref = json.loads(r.stdout)
    for ctr, seed, want in zip(ctrs, seeds, ref):
        key = [int(seed) & 0xFFFFFFFF, int(seed) >> 32]
        got = O.philox4x32_10(ctr, key).tolist()
        assert got == want, (ctr, seed, got, want)


def test_uniform_structure_and_law():
    from scipy import stats
    u = np.array([O.uniform(123, 5, p, t, 0) for p in range(50) for t in range(400)], np.float64)
    n = u * 2.0**24
    assert np.all(n == np.round(n)) and np.all(n.astype(np.int64) % 2 == 1)  # odd multiples of 2^-24
    assert u.min() > 0.0 and u.max() < 1.0
    assert stats.kstest(u, "uniform").pvalue > 1e-3
    # the 4 lanes of one Philox block are 4 consecutive tokens
    out = O.philox4x32_10([10, 3, 5, 0], [123, 0])
    for lane in range(4):
        x = int(out[lane])
        assert O.uniform(123, 5, 3, 40 + lane, 0) == ((x >> 9) * 2 + 1) / 2.0**24


def test_gumbel_law():
    from scipy import stats
    g = np.array([O.gumbel(99, 1, p, t, 2) for p in range(100) for t in range(500)])
    assert stats.kstest(g, stats.gumbel_r.cdf).pvalue > 1e-3
    # bounded by the largest uniform: -log(-log(1 - 2^-24))
    assert g.max() < -np.log(-np.log1p(-(2.0**-24))) + 1e-12


# ------------------------------------------------------- processed logits


def _load_cases():
    with open(os.path.join(HERE, "golden", "processed_cases.json")) as f:
        return json.load(f)["cases"]


def _case_workload(c):
    mask = None
    if c["mask_words_hex"]:
        mask = np.array([[int(h, 16) for h in c["mask_words_hex"]]], np.uint32)
    return sample_workload(
        np.array([c["logits"]], np.float32), dtype=c["dtype"], temperature=c["temperature"],
        repetition=c["repetition"], frequency=c["frequency"], presence=c["presence"],
        history=[c["history"]], bias=[(c["bias_ids"], c["bias_vals"])], mask_words=mask)


@pytest.mark.parametrize("case", _load_cases(), ids=lambda c: c["name"])
def test_processed_logits_golden(case):
    w = _case_workload(case)
    r = O.process_sample(w, want_processed=True)
    want = np.array([-np.inf if v == "-inf" else v for v in case["expected"]], np.float32)
    got = r["processed"][0]
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), (got, want)
    assert r["status"][0] == 0
    if "expected_token" in case:
        assert r["token"][0] == case["expected_token"]


# ------------------------------------------------------------ kept sets


def _tiny_rows(rng, n, V):
    # small integers / 4 => many exact ties, as bf16 logits have in practice
    return (rng.integers(-12, 13, size=(n, V)) / 4.0).astype(np.float32)


@pytest.mark.parametrize("V", [5, 17, 33, 64])
def test_kept_set_matches_brute_force(V):
    rng = np.random.default_rng(V)
    n = 60
    z = _tiny_rows(rng, n, V)
    temp = rng.choice([0.5, 1.0, 1.7], size=n).astype(np.float32)
    top_k = rng.choice([0, 1, 2, 3, V // 2, V, V + 5], size=n).astype(np.int32)
    top_p = rng.choice([1.0, 0.3, 0.5, 0.9, 0.99], size=n).astype(np.float32)
    min_p = rng.choice([0.0, 0.01, 0.2, 0.7], size=n).astype(np.float32)
    mask = rng.integers(0, 2**32, size=(n, (V + 31) // 32), dtype=np.uint64).astype(np.uint32)
    mask[:, 0] |= 1  # keep at least token 0 allowed
    w = sample_workload(z, temperature=temp, top_k=top_k, top_p=top_p, min_p=min_p, mask_words=mask)
    res = O.process_sample(w, want_processed=True)
    for r in range(n):
        y = res["processed"][r]
        K, Pb = brute.kept_set(y, int(top_k[r]), float(top_p[r]), float(min_p[r]))
        st, P = O.row_probs(w, r)
        assert st == 0
        if res["kept_lo"][r] == res["kept_hi"][r]:  # cut not within margin
            assert res["kept"][r] == K.sum()
            assert np.array_equal(P > 0, K), r
            np.testing.assert_allclose(P, Pb, rtol=1e-12, atol=1e-15)
        assert res["token"][r] in np.flatnonzero(P > 0)


def test_top_k_ties_take_lowest_indices():
    z = np.array([[1.0, 3.0, 2.0, 3.0, 2.0, 2.0, 0.0, 2.0]], np.float32)
    w = sample_workload(z, temperature=1.0, top_k=4)
    st, P = O.row_probs(w, 0)
    assert np.flatnonzero(P > 0).tolist() == [1, 2, 3, 4]  # both 3.0s, then the first two 2.0s


def test_two_stage_top_k_union_contains_global_top_k():
    rng = np.random.default_rng(11)
    for _ in range(20):
        V = int(rng.integers(50, 400))
        k = int(rng.integers(1, 40))
        z = _tiny_rows(rng, 1, V)
        w = sample_workload(z, temperature=1.0, top_k=k)
        _, P = O.row_probs(w, 0)
        K = set(np.flatnonzero(P > 0).tolist())
        cuts = np.sort(rng.choice(np.arange(1, V), size=int(rng.integers(1, 8)), replace=False))
        union = set()
        for lo, hi in zip(np.r_[0, cuts], np.r_[cuts, V]):
            idx = np.arange(lo, hi)
            order = np.lexsort((idx, -z[0, lo:hi]))  # y desc, index asc
            union |= set(idx[order[:k]].tolist())
        assert K <= union


def test_greedy_is_first_argmax():
    rng = np.random.default_rng(3)
    z = _tiny_rows(rng, 40, 50)
    w = sample_workload(z, temperature=0.0)
    r = O.process_sample(w)
    assert np.array_equal(r["token"], np.argmax(z, axis=1))
    assert np.all(r["kept"] == 1)


# ------------------------------------------------------------------ draw


def test_draw_is_gumbel_argmax_and_decomposes_over_partitions():
    rng = np.random.default_rng(5)
    n, V = 30, 300
    z = rng.normal(0, 2, size=(n, V)).astype(np.float32)
    top_k = rng.choice([0, 10, 100], size=n).astype(np.int32)
    w = sample_workload(z, temperature=0.9, top_k=top_k, seed=77, position=np.arange(n) * 3)
    res = O.process_sample(w, want_processed=True)
    for r in range(n):
        _, P = O.row_probs(w, r)
        K = np.flatnonzero(P > 0)
        y = res["processed"][r].astype(np.float64)
        s = np.array([y[t] + O.gumbel(77, r, 3 * r, int(t), 0) for t in K])
        # argmax over random partitions of K, then over the partition winners
        cuts = np.sort(rng.choice(np.arange(1, len(K)), size=min(5, len(K) - 1), replace=False)) if len(K) > 1 else []
        winners = [max(zip(s[lo:hi], -K[lo:hi]))for lo, hi in zip(np.r_[0, cuts], np.r_[cuts, len(K)])]
        best = -max(winners)[1]
        assert best == res["token"][r]


@pytest.mark.parametrize("params", [
    dict(temperature=1.0),
    dict(temperature=0.7, top_k=5),
    dict(temperature=1.3, top_p=0.8),
    dict(temperature=1.0, min_p=0.1),
    dict(temperature=0.8, top_k=12, top_p=0.9, min_p=0.02),
])
def test_draw_law_chi_square(params):
    from scipy import stats
    rng = np.random.default_rng(sum(map(ord, str(params))))
    V = 24
    z = rng.normal(0, 1.5, size=(1, V)).astype(np.float32)
    N = 1_000_000
    w = sample_workload(np.repeat(z, 1, axis=0), row_stride=0, seed=12345, **params)
    w["num_rows"] = N
    for key in ("temperature", "top_k", "top_p", "min_p"):
        if w.get(key) is not None:
            w[key] = np.full(N, w[key][0], w[key].dtype)
    w["seed"] = np.full(N, 12345, np.uint64)
    w["position"] = np.arange(N, dtype=np.int64)
    res = O.process_sample(w)
    _, P = O.row_probs(dict(w, num_rows=1), 0)
    K = np.flatnonzero(P > 0)
    counts = np.bincount(res["token"], minlength=V)
    assert counts[P == 0].sum() == 0
    chi = stats.chisquare(counts[K], N * P[K])
    assert chi.pvalue > 1e-3, (chi, params)


# ------------------------------------------------------ verification


def _enumerate_first_token_law(w, q, draft_len):
    """Exact law of the first emitted token of a 1-request verify workload."""
    V = w["vocab"]
    sw = dict(kind="sample", num_rows=1, vocab=V, dtype=w["dtype"], logits=w["target_logits"][:1],
              row_stride=V, **{k: w.get(k) for k in ("temperature", "top_k", "top_p", "min_p",
                                                      "repetition", "frequency", "presence",
                                                      "hist_offsets", "hist_ids", "seed", "position")})
    _, P0 = O.row_probs(sw, 0)
    empty, r0 = O.residual_probs(P0, q[0])
    law = np.zeros(V)
    for x in range(V):
        if q[0][x] == 0:
            continue
        a = min(1.0, P0[x] / q[0][x])
        law[x] += q[0][x] * a
        law += q[0][x] * (1.0 - a) * (P0 if empty else r0)
    return P0, law


@pytest.mark.parametrize("V", [3, 5, 8])
def test_spec_verify_exact_enumeration(V):
    rng = np.random.default_rng(100 + V)
    for trial in range(8):
        k = int(rng.integers(1, 4))
        z = rng.normal(0, 1.2, size=(k + 1, V)).astype(np.float32)
        q = rng.dirichlet(np.ones(V) * 0.7, size=k).astype(np.float32)
        params = dict(temperature=float(rng.choice([0.6, 1.0, 1.4])), top_k=int(rng.choice([0, 2, V])),
                      top_p=float(rng.choice([1.0, 0.8])), repetition=1.2, frequency=0.3, presence=0.1,
                      history=[rng.integers(0, V, size=3).tolist()])
        w = verify_workload(z, [k], np.zeros(k, np.int32), q, **params)
        P0, law = _enumerate_first_token_law(w, q, k)
        # the identity is exact when sum(q) = 1; fp32 q misses 1 by ~1e-8
        tol = 4 * np.abs(1.0 - q.astype(np.float64).sum(axis=1)).max() + 1e-12
        np.testing.assert_allclose(law, P0, rtol=0, atol=tol)
        # conditional law of the second token given that draft x0 was accepted:
        # the target row 1 distribution with x0 appended to the history
        if k >= 2:
            for x0 in range(V):
                sw1 = dict(kind="sample", num_rows=1, vocab=V, dtype="f32", logits=z[1:2], row_stride=V,
                           temperature=w["temperature"], top_k=w["top_k"], top_p=w["top_p"], min_p=None,
                           repetition=w["repetition"], frequency=w["frequency"], presence=w["presence"],
                           hist_offsets=w["hist_offsets"], hist_ids=w["hist_ids"], seed=w["seed"],
                           position=w["position"])
                _, P1 = O.row_probs(sw1, 0, extra_hist=np.array([x0], np.int32))
                empty, r1 = O.residual_probs(P1, q[1])
                law1 = np.zeros(V)
                for x in range(V):
                    if q[1][x] == 0:
                        continue
                    a = min(1.0, P1[x] / q[1][x])
                    law1[x] += q[1][x] * a
                    law1 += q[1][x] * (1.0 - a) * (P1 if empty else r1)
                np.testing.assert_allclose(law1, P1, rtol=0, atol=tol)


def test_spec_verify_realised_law_chi_square():
    from scipy import stats
    rng = np.random.default_rng(9)
    V, N = 8, 1_000_000
    z = rng.normal(0, 1.0, size=(2, V)).astype(np.float32)
    q = rng.dirichlet(np.ones(V), size=1).astype(np.float32)
    drafts = rng.choice(V, size=N, p=q[0].astype(np.float64) / q[0].astype(np.float64).sum()).astype(np.int32)
    w = verify_workload(np.tile(z, (N, 1)), np.ones(N, np.int32), drafts, np.tile(q, (N, 1)),
                        temperature=1.0, top_p=0.9, seed=31, position=np.arange(N) * 2)
    res = O.spec_verify(w)
    assert np.all(res["status"] == 0)
    first = res["out_tokens"][:, 0]
    sw = sample_workload(z[:1], temperature=1.0, top_p=0.9)
    _, P0 = O.row_probs(sw, 0)
    K = np.flatnonzero(P0 > 0)
    counts = np.bincount(first, minlength=V)
    assert counts[P0 == 0].sum() == 0
    assert stats.chisquare(counts[K], N * P0[K]).pvalue > 1e-3
    # after an accepted draft the bonus token follows row 1 (x0 in its history
    # only matters with penalties, which are off here)
    acc = res["num_accepted"] == 1
    _, P1 = O.row_probs(sample_workload(z[1:2], temperature=1.0, top_p=0.9), 0)
    K1 = np.flatnonzero(P1 > 0)
    c1 = np.bincount(res["out_tokens"][acc, 1], minlength=V)
    assert stats.chisquare(c1[K1], acc.sum() * P1[K1]).pvalue > 1e-3


def test_spec_verify_greedy_special_case():
    rng = np.random.default_rng(4)
    V, R, k = 50, 40, 4
    z = rng.normal(0, 1, size=(R * (k + 1), V)).astype(np.float32)
    arg = np.argmax(z, axis=1).reshape(R, k + 1)
    drafts = arg[:, :k].copy()
    cut = rng.integers(0, k + 1, size=R)  # first mismatching draft position
    for i in range(R):
        if cut[i] < k:
            drafts[i, cut[i]] = (arg[i, cut[i]] + 1) % V
    q = rng.dirichlet(np.ones(V), size=R * k).astype(np.float32)
    w = verify_workload(z, np.full(R, k), drafts.reshape(-1), q, temperature=0.0)
    res = O.spec_verify(w)
    for i in range(R):
        c = int(cut[i])
        assert res["num_accepted"][i] == c
        want = list(drafts[i, :c]) + [arg[i, c]] + [-1] * (k - c)
        assert res["out_tokens"][i].tolist() == want


# ----------------------------------------------------------- statuses


def test_status_codes():
    V = 40
    z = np.zeros((8, V), np.float32)
    z[3, 7] = np.nan
    z[4, 9] = np.inf
    temp = np.array([1, -1, 1, 1, 1, 1, 1, 0], np.float32)
    top_p = np.array([1, 1, 0, 1, 1, 1, 1, 1], np.float32)
    mask = np.full((8, 2), 0xFFFFFFFF, np.uint32)
    mask[5] = 0
    hist = [[], [], [], [], [], [], [V], [1, 2]]
    bias = [([1, 1], [0.5, 0.5]), ([], []), ([], []), ([], []), ([], []), ([], []), ([], []), ([3], [1.0])]
    w = sample_workload(z, temperature=temp, top_p=top_p, mask_words=mask, history=hist, bias=bias)
    r = O.process_sample(w)
    assert r["status"].tolist() == [3, 4, 4, 2, 2, 1, 3, 0]
    assert r["token"][:7].tolist() == [-1] * 7


def test_masked_nan_is_ignored_and_bias_cannot_unmask():
    z = np.zeros((1, 40), np.float32)
    z[0, 5] = np.nan
    mask = np.array([[0xFFFFFFFF & ~(1 << 5) & ~(1 << 6), 0xFF]], np.uint32)
    w = sample_workload(z, temperature=1.0, mask_words=mask, bias=[([6], [50.0])])
    r = O.process_sample(w, want_processed=True)
    assert r["status"][0] == 0
    assert r["processed"][0, 5] == -np.inf and r["processed"][0, 6] == -np.inf


def test_workload_generators_are_seeded():
    a, b = W.make(2, rows=3, vocab=1000), W.make(2, rows=3, vocab=1000)
    for key in ("logits", "temperature", "hist_ids", "bias_vals", "position"):
        assert np.array_equal(a[key], b[key])
    m = W.make(3, rows=2, vocab=1000)
    assert m["bitmask"].shape == (2, 32)


def test_row_id_is_philox_counter_word_2():
    """The draw of a row depends on its own logits, parameters and row id
    only: reordering a batch while carrying each row's id along leaves every
    row's token unchanged, and an explicit id equal to the row's index is the
    default.  The token is the Gumbel argmax with the id in counter word 2."""
    w = W.make(2, rows=6, vocab=64)
    base = O.process_sample(w)
    ids = dict(w, row_id=np.arange(6, dtype=np.uint32))
    assert np.array_equal(O.process_sample(ids)["token"], base["token"])
    perm = np.array([4, 1, 5, 0, 3, 2])
    moved = subset_sample(w, perm)
    moved["row_id"] = perm.astype(np.uint32)
    assert np.array_equal(O.process_sample(moved)["token"], base["token"][perm])
    # brute force on an unfiltered row: argmax of y + g(seed, id, position, t)
    z = np.random.default_rng(5).normal(0, 1, (1, 64)).astype(np.float32)
    one = sample_workload(z, temperature=1.0, seed=77, position=[9])
    for rid in (0, 3, 4000000000):
        one["row_id"] = np.array([rid], np.uint32)
        g = np.array([O.gumbel(77, int(np.int32(np.uint32(rid))), 9, t, 0) for t in range(64)])
        assert O.process_sample(one)["token"][0] == int(np.argmax(z[0].astype(np.float64) + g))


def test_commit_accepted_hand_example():
    """The step after verification, on a hand-worked example: request 0
    accepted 2 drafts (emits 5, 6, 7 after 1 held token), request 1 none
    (emits 8 at slot 5), request 2 failed (status 3: unchanged), request 3
    would overflow its buffer, request 4 reports an impossible count."""
    out = np.array([[5, 6, 7], [8, -1, -1], [1, 2, 3], [4, 4, 4], [9, 9, 9]], np.int32)
    tokens = np.full((5, 6), -9, np.int32)
    t, n, p, nxt, st = O.commit_accepted(out, [2, 0, 2, 2, 3], [0, 0, 3, 0, 0], tokens, [1, 5, 0, 4, 0],
                                         [10, 20, 30, 40, 50])
    expect = np.full((5, 6), -9, np.int32)
    expect[0, 1:4] = [5, 6, 7]
    expect[1, 5] = 8
    assert np.array_equal(t, expect)
    assert list(n) == [4, 6, 0, 4, 0]
    assert list(p) == [13, 21, 30, 40, 50]
    assert list(nxt) == [7, 8, -1, -1, -1]
    assert list(st) == [0, 0, 3, 6, 6]
