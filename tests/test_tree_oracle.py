"""Pins of the oracle's tree verification (recursive rejection over each
node's children; a reading of "Accelerating Sonar through speculation",
section "EAGLE", which names tree drafts without an acceptance rule).

- A chain-shaped tree is the linear rule: identical outputs to the linear
  verification on the same inputs, penalties included (the path of a node is
  the linear position's preceding drafts).
- The law of the emitted tokens (chi-square over 3e5 requests, children drawn
  independently from q): the first token follows the root's filtered target
  distribution, and after an accepted child the next token follows that
  child's distribution.  A residual that is not renormalised between
  siblings, or taken against the wrong base, breaks the first law.
- The greedy special case, and the status of malformed trees.
"""
import numpy as np

from oracle import oracle as O
from tests.helpers import chain_from_linear, sample_workload, tree_workload, verify_workload


def test_chain_tree_is_the_linear_rule():
    rng = np.random.default_rng(21)
    R, V, kmax = 120, 96, 4
    ks = rng.integers(0, kmax + 1, size=R).astype(np.int32)
    z = rng.normal(0, 2.0, size=(int(ks.sum()) + R, V)).astype(np.float32)
    # each draft distribution: a noisy copy of the target row it proposes for
    rows = np.concatenate([np.arange(o, o + k) for o, k in zip(np.r_[0, np.cumsum(ks + 1)][:-1], ks)]).astype(int)
    x = z[rows].astype(np.float64) + rng.normal(0, 0.7, size=(rows.size, V))
    q = np.exp(x - x.max(axis=1, keepdims=True))
    q = (q / q.sum(axis=1, keepdims=True)).astype(np.float32)
    drafts = np.array([rng.choice(V, p=qq.astype(np.float64) / qq.astype(np.float64).sum()) for qq in q], np.int32)
    hist = [rng.integers(0, V, size=int(rng.integers(0, 12))) for _ in range(R)]
    w = verify_workload(z, ks, drafts, q, max_draft=kmax, temperature=rng.uniform(0.0, 1.5, R) * (rng.random(R) > 0.2),
                        top_k=rng.choice([0, 5, 40], R), top_p=rng.choice([1.0, 0.9], R),
                        min_p=rng.choice([0.0, 0.05], R), repetition=1.3, frequency=0.2, presence=0.1,
                        seed=np.arange(R) + 5, position=rng.integers(0, 1000, R), history=hist)
    lin = O.spec_verify(w)
    tr = O.tree_verify(chain_from_linear(w))
    assert np.array_equal(lin["status"], tr["status"])
    assert np.array_equal(lin["num_accepted"], tr["num_accepted"])
    assert np.array_equal(lin["out_tokens"], tr["out_tokens"])
    assert np.array_equal(lin["sub_margin"], tr["sub_margin"])
    ok = lin["status"] == 0
    for i in np.flatnonzero(ok):
        n = int(tr["num_accepted"][i])
        assert tr["out_path"][i, :n].tolist() == list(range(1, n + 1))
    assert ok.sum() > 100 and (lin["num_accepted"][ok] > 0).sum() > 20


def test_tree_law_of_emitted_tokens():
    from scipy import stats
    rng = np.random.default_rng(33)
    V, N = 6, 300_000
    par = np.array([-1, 0, 0, 0, 1, 1], np.int32)  # root: 3 children; node 1: 2 children
    n = par.size
    z = rng.normal(0, 1.0, size=(n, V)).astype(np.float32)
    q0 = rng.dirichlet(np.ones(V)).astype(np.float32)
    q1 = rng.dirichlet(np.ones(V)).astype(np.float32)
    qrows = np.zeros((n, V), np.float32)
    qrows[0], qrows[1] = q0, q1
    tok = np.zeros((N, n), np.int32)
    tok[:, 1:4] = rng.choice(V, size=(N, 3), p=q0.astype(np.float64) / q0.astype(np.float64).sum())
    tok[:, 4:6] = rng.choice(V, size=(N, 2), p=q1.astype(np.float64) / q1.astype(np.float64).sum())
    w = tree_workload(np.tile(z, (N, 1)), np.arange(N + 1) * n, np.tile(par, N), tok.reshape(-1),
                      np.tile(qrows, (N, 1)), temperature=1.0, top_p=0.9, seed=77, position=np.arange(N) * 3)
    res = O.tree_verify(w)
    assert np.all(res["status"] == 0)

    def law(row):
        return O.row_probs(sample_workload(z[row:row + 1], temperature=1.0, top_p=0.9), 0)[1]

    def check(tokens, P):
        K = np.flatnonzero(P > 0)
        c = np.bincount(tokens, minlength=V)
        assert c[P == 0].sum() == 0
        assert stats.chisquare(c[K], tokens.size * P[K]).pvalue > 1e-3

    check(res["out_tokens"][:, 0], law(0))
    for node in (1, 2, 3):  # the second token after accepting `node` follows node's row
        sel = res["out_path"][:, 0] == node
        assert sel.sum() > 5000
        check(res["out_tokens"][sel, 1], law(node))
    # every sibling position gets accepted sometimes
    assert set(np.unique(res["out_path"][:, 0])) == {-1, 1, 2, 3}


def test_tree_greedy_special_case():
    V = 8
    par = [-1, 0, 0, 0, 2, 2]
    z = np.zeros((6, V), np.float32)
    z[0, 5] = 3.0   # root argmax 5
    z[2, 1] = 2.0   # node 2 argmax 1
    z[5, 7] = 1.0
    tok = [0, 4, 5, 5, 3, 1]   # nodes 2 and 3 both carry the argmax: node 2 is tried first
    q = np.full((6, V), 1.0 / V, np.float32)
    w = tree_workload(z, [0, 6], par, tok, q, temperature=0.0)
    res = O.tree_verify(w)
    assert res["status"][0] == 0
    assert res["num_accepted"][0] == 2
    assert res["out_path"][0, :3].tolist() == [2, 5, -1]
    assert res["out_tokens"][0, :3].tolist() == [5, 1, 7]   # node 5 is a leaf: its argmax is the bonus


def test_tree_statuses():
    V = 10
    z = np.zeros((4, V), np.float32)
    q = np.full((4, V), 0.1, np.float32)
    base = dict(target_logits=z, node_offsets=[0, 4], draft_probs=q)
    ok = O.tree_verify(tree_workload(parents=[-1, 0, 1, 1], node_tokens=[0, 1, 2, 3], **base))
    assert ok["status"][0] == 0
    bad_parent = O.tree_verify(tree_workload(parents=[-1, 0, 3, 1], node_tokens=[0, 1, 2, 3], **base))
    assert bad_parent["status"][0] == 4 and bad_parent["out_tokens"][0].tolist() == [-1] * 4
    bad_token = O.tree_verify(tree_workload(parents=[-1, 0, 1, 1], node_tokens=[0, 1, V, 3], **base))
    assert bad_token["status"][0] == 3
    too_many = O.tree_verify(tree_workload(parents=[-1, 0, 1, 1], node_tokens=[0, 1, 2, 3], max_nodes=3, **base))
    assert too_many["status"][0] == 4
    root_only = O.tree_verify(tree_workload(z[:1], [0, 1], [-1], [0], q[:1], temperature=0.0))
    assert root_only["num_accepted"][0] == 0 and root_only["out_tokens"][0, 0] == 0
