"""Tree-draft verification on the GPU (ss_tree_verify) against the oracle.

Accepted counts, emitted tokens, accepted node paths and statuses must match
exactly; requests where some decision on the walk is within the oracle's
margin are checked for validity only.  A chain-shaped tree must reproduce the
GPU's own linear verification bit for bit.
"""
import numpy as np
import pytest

from speculative_verification_gb300 import workloads as W
from tests import parity
from tests.helpers import chain_from_linear, tree_workload

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def ss():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_verification_gb300 import build as ss_build
    ss_build.build()
    from speculative_verification_gb300 import ss as _ss
    _ss.load()
    return _ss


def run_gpu(ss, w):
    dw = ss.to_device(w)
    o = ss.alloc_outputs(dw)
    ss.run(dw, o)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in o.items() if k != "workspace"}


def _check(ss, w, min_checked):
    chk, sub = parity.check_tree(w, run_gpu(ss, w))
    print("tree: %d requests compared, %d within margin" % (chk, sub))
    assert chk >= min_checked


@pytest.mark.parametrize("dtype,vocab", [("bf16", 5003), ("f32", 4096)])
def test_tree_random_small(ss, dtype, vocab):
    _check(ss, W.tree(seed=11, requests=40, vocab=vocab, max_nodes=16, dtype=dtype), 30)


def test_tree_full_vocab(ss):
    _check(ss, W.tree(seed=12, requests=12, vocab=128256, max_nodes=12), 9)


def test_tree_bushy_many_rejections(ss):
    # stars and two-level fans with drafts far from the target: many siblings
    # rejected in a row, each rejection a residual normalisation
    shapes = [np.array([-1] + [0] * 15, np.int32), np.array([-1, 0, 0, 0, 1, 1, 1, 2, 2, 2, 3, 3, 3], np.int32),
              np.array([-1] + [0] * 7, np.int32)] * 6
    w = W.tree(seed=13, requests=len(shapes), vocab=32000, max_nodes=16, shapes=shapes, greedy_frac=0.0,
               draft_noise=3.0)
    _check(ss, w, 12)


def test_chain_tree_equals_linear_verification(ss):
    w = W.make(4, requests=12, vocab=32000)
    dw = ss.to_device(w)
    o = ss.alloc_outputs(dw)
    ss.run(dw, o)
    torch.cuda.synchronize()
    lin = {k: v.cpu().numpy() for k, v in o.items() if k != "workspace"}
    tr = run_gpu(ss, chain_from_linear(w))
    assert np.array_equal(lin["status"], tr["status"])
    assert np.array_equal(lin["num_accepted"], tr["num_accepted"])
    assert np.array_equal(lin["out_tokens"], tr["out_tokens"])
    parity.check_tree(chain_from_linear(w), tr)


def test_tree_greedy_and_statuses(ss):
    V = 300
    rng = np.random.default_rng(5)
    z = rng.normal(0, 1, size=(6, V)).astype(np.float32)
    arg = np.argmax(z, axis=1)
    par = [-1, 0, 0, 0, 2, 2]
    tok = [0, (arg[0] + 1) % V, arg[0], arg[0], (arg[2] + 3) % V, arg[2]]
    q = np.full((6, V), 1.0 / V, np.float32)
    greedy = tree_workload(z, [0, 6], par, tok, q, temperature=0.0)
    g = run_gpu(ss, greedy)
    parity.check_tree(greedy, g)
    assert g["out_path"][0, :2].tolist() == [2, 5]
    # malformed trees, one request each
    zz = np.tile(z[:4], (5, 1))
    qq = np.tile(q[:4], (5, 1))
    pars = [[-1, 0, 1, 1], [-1, 0, 3, 1], [-1, 0, 1, 1], [-1, 0, 0, 0], [-1, 0, 1, 2]]
    toks = [[0, 1, 2, 3], [0, 1, 2, 3], [0, 1, V, 3], [0, 5, 6, 7], [0, -1, 2, 3]]
    w = tree_workload(zz, [0, 4, 8, 12, 16, 20], np.concatenate(pars), np.concatenate(toks), qq,
                      temperature=[1.0, 1.0, 1.0, -1.0, 0.5], max_nodes=4)
    res = run_gpu(ss, w)
    parity.check_tree(w, res)
    assert res["status"].tolist() == [0, 4, 3, 4, 3]
    # a node count above max_nodes
    w2 = tree_workload(z[:4], [0, 4], [-1, 0, 1, 1], [0, 1, 2, 3], q[:4], max_nodes=3)
    res2 = run_gpu(ss, w2)
    parity.check_tree(w2, res2)
    assert res2["status"][0] == 4


def test_tree_graph_capture_and_repeat(ss):
    w = W.tree(seed=14, requests=20, vocab=32000, max_nodes=10)
    dw = ss.to_device(w)
    o1 = ss.alloc_outputs(dw)
    o2 = ss.alloc_outputs(dw)
    ss.run(dw, o1)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        ss.run(dw, o2, stream=s)  # warm-up on the capture stream
        torch.cuda.synchronize()
        o2["out_tokens"].fill_(-7)
        with torch.cuda.graph(graph, stream=s):
            ss.run(dw, o2, stream=s)
    for _ in range(3):  # the workspace counters return to zero after every call
        graph.replay()
    torch.cuda.synchronize()
    for key in ("out_tokens", "out_path", "num_accepted", "status", "kept"):
        assert torch.equal(o1[key], o2[key]), key


def test_tree_requests_split_with_row_ids(ss):
    # requests split over two calls (as over two GPUs), keyed by their ids,
    # give what the whole batch gives
    w = W.tree(seed=15, requests=18, vocab=20000, max_nodes=8)
    w["row_id"] = np.arange(18, dtype=np.uint32)
    whole = run_gpu(ss, w)
    a = run_gpu(ss, parity.subset_tree(w, list(range(0, 9))))
    b = run_gpu(ss, parity.subset_tree(w, list(range(9, 18))))
    for key in ("out_tokens", "out_path", "num_accepted", "status"):
        assert np.array_equal(np.concatenate([a[key], b[key]]), whole[key]), key


TREE_KEYS = ("out_tokens", "out_path", "num_accepted", "status", "kept")


def _tree_outputs(ss, dw, count, **kw):
    o = ss.alloc_outputs(dw)
    params = {k: dw.get(k) for k in ss.PARAM_FIELDS}
    params["bitmask_stride"] = dw.get("bitmask_stride", 0)
    ss.ss_tree_verify(dw["target_logits"], dw["node_offsets"], dw["parents"], dw["node_tokens"], dw["draft_probs"],
                      params, o["out_tokens"], o["num_accepted"], o["status"], o["workspace"], vocab=dw["vocab"],
                      max_nodes=dw["max_nodes"], dtype=dw["dtype"], row_stride=dw["row_stride"],
                      draft_stride=dw["draft_stride"], out_path=o["out_path"], out_kept=o["kept"],
                      num_nodes_total=count, **kw)
    torch.cuda.synchronize()
    return o


@pytest.mark.parametrize("requests,max_nodes", [(32, 16), (3, 4)])  # ordered launch; one without the ordering
def test_tree_node_count_keeps_the_outputs(ss, requests, max_nodes):
    w = W.tree(seed=40 + requests, requests=requests, vocab=9001, max_nodes=max_nodes)
    dw = ss.to_device(w)
    nodes = int(w["node_offsets"][-1])
    full = _tree_outputs(ss, dw, 0)
    counted = _tree_outputs(ss, dw, nodes)
    for key in TREE_KEYS:
        assert torch.equal(full[key], counted[key]), key
    assert (full["status"].cpu().numpy() == 0).all()


@pytest.mark.parametrize("requests,max_nodes", [(32, 16), (3, 4)])
@pytest.mark.parametrize("delta", [-1, 1])
def test_tree_wrong_node_count_reports_bad_param(ss, requests, max_nodes, delta):
    w = W.tree(seed=50 + requests, requests=requests, vocab=5003, max_nodes=max_nodes)
    dw = ss.to_device(w)
    nodes = int(w["node_offsets"][-1])
    if not (requests <= nodes + delta <= requests * max_nodes):
        pytest.skip("count outside the accepted range")
    ref = _tree_outputs(ss, dw, 0)
    o = _tree_outputs(ss, dw, nodes + delta)
    assert (o["status"].cpu().numpy() == 4).all()  # SS_ROW_BAD_PARAM
    assert (o["num_accepted"].cpu().numpy() == 0).all()
    assert (o["out_tokens"].cpu().numpy() == -1).all() and (o["out_path"].cpu().numpy() == -1).all()
    # the workspace is untouched: a correct call on it gives the reference
    params = {k: dw.get(k) for k in ss.PARAM_FIELDS}
    params["bitmask_stride"] = dw.get("bitmask_stride", 0)
    ss.ss_tree_verify(dw["target_logits"], dw["node_offsets"], dw["parents"], dw["node_tokens"], dw["draft_probs"],
                      params, o["out_tokens"], o["num_accepted"], o["status"], o["workspace"], vocab=dw["vocab"],
                      max_nodes=dw["max_nodes"], dtype=dw["dtype"], row_stride=dw["row_stride"],
                      draft_stride=dw["draft_stride"], out_path=o["out_path"], out_kept=o["kept"],
                      num_nodes_total=nodes)
    torch.cuda.synchronize()
    for key in TREE_KEYS:
        assert torch.equal(ref[key], o[key]), key


def test_tree_node_count_overlapped_in_a_graph(ss):
    sets = [ss.to_device(W.tree(seed=70 + i, requests=24, vocab=128256, max_nodes=16)) for i in range(3)]
    ref = [_tree_outputs(ss, dw, 0) for dw in sets]
    outs = [ss.alloc_outputs(dw) for dw in sets]
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            for dw, o in zip(sets, outs):
                ss.run(dw, o, stream=stream, overlap_previous=True, target_rows=True)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    for r, o in zip(ref, outs):
        for key in TREE_KEYS:
            assert torch.equal(r[key], o[key]), key
