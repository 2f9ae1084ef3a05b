"""Vocabulary-sharded sampling (tensor-parallel logits) through the C ABI.

Each shard's records come from ss_sample_shard on a slice of the
vocabulary; ss_merge_shards must return exactly what ss_process_sample
returns on the whole rows (token, status and kept-set size), for any
number of shards and any order of the records, and agree with the oracle.
"""
import numpy as np
import pytest

from speculative_verification_gb300 import workloads as W
from tests import parity

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

CAP = 1024


@pytest.fixture(scope="module")
def ss():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_verification_gb300 import build as ss_build
    ss_build.build()
    from speculative_verification_gb300 import ss as _ss
    _ss.load()
    return _ss


def _whole(ss, w):
    dw = ss.to_device(w)
    o = ss.alloc_outputs(dw)
    ss.run(dw, o)
    torch.cuda.synchronize()
    return dw, {k: o[k].cpu().numpy() for k in ("token", "status", "kept")}


def _sharded(ss, dw, bounds, order=None):
    V = int(dw["vocab"])
    n = int(dw["num_rows"])
    params = {k: dw.get(k) for k in ss.PARAM_FIELDS}
    params["bitmask_stride"] = dw.get("bitmask_stride", 0)
    rec_bytes = ss.ss_shard_record_bytes(CAP)
    recs = []
    for off, length in bounds:
        rec = torch.empty(n * rec_bytes, dtype=torch.uint8, device="cuda")
        ss.ss_sample_shard(dw["logits"][:, off:], params, rec, vocab=V, vocab_offset=off, shard_len=length,
                           list_cap=CAP, num_rows=n, dtype=dw["dtype"], row_stride=int(dw["row_stride"]))
        recs.append(rec)
    if order is not None:
        recs = [recs[i] for i in order]
    tok = torch.empty(n, dtype=torch.int32, device="cuda")
    st = torch.empty(n, dtype=torch.int32, device="cuda")
    kept = torch.empty(n, dtype=torch.int32, device="cuda")
    ss.ss_merge_shards(recs, params, tok, st, vocab=V, list_cap=CAP, out_kept=kept)
    torch.cuda.synchronize()
    return {"token": tok.cpu().numpy(), "status": st.cpu().numpy(), "kept": kept.cpu().numpy()}


@pytest.mark.parametrize("P", [1, 2, 4, 8])
def test_sharded_equals_whole_decode(ss, P):
    w = W.shardable(W.make(2, rows=16))
    dw, whole = _whole(ss, w)
    got = _sharded(ss, dw, W.even_shards(int(w["vocab"]), P))
    for k in ("token", "status", "kept"):
        assert np.array_equal(got[k], whole[k]), (k, got[k], whole[k])
    parity.check_sample(w, got)


def test_sharded_uneven_shards_any_order_with_mask(ss):
    w = W.shardable(W.make(3, rows=12, vocab=20011), k=64)  # grammar mask, ragged vocabulary
    dw, whole = _whole(ss, w)
    bounds = [(0, 4000), (4000, 96), (4096, 9600), (13696, 6315)]
    got = _sharded(ss, dw, bounds, order=[2, 0, 3, 1])
    for k in ("token", "status", "kept"):
        assert np.array_equal(got[k], whole[k]), (k, got[k], whole[k])
    parity.check_sample(w, got)


def test_sharded_unsupported_rows(ss):
    w = W.make(2, rows=8, vocab=5003)
    w["temperature"] = np.full(8, 1.0, np.float32)
    w["top_k"] = np.array([0, 0, 0, 50, 2000, 0, 10, 0], np.int32)
    w["top_p"] = np.array([0.9, 1.0, 1.0, 0.9, 1.0, 1.0, 1.0, 1.0], np.float32)
    w["min_p"] = np.array([0.0, 0.05, 0.0, 0.0, 0.0, 0.0, 0.0, 0.0], np.float32)
    dw, whole = _whole(ss, w)
    got = _sharded(ss, dw, W.even_shards(5003, 3))
    # top-p or min-p without top-k, and top_k above the list capacity
    assert list(got["status"][[0, 1, 4]]) == [7, 7, 7]
    ok = np.array([2, 3, 5, 6, 7])
    for k in ("token", "status", "kept"):
        assert np.array_equal(got[k][ok], whole[k][ok]), (k, got[k][ok], whole[k][ok])


def _rounds(ss, dw, bounds, order=None):
    """The four-round protocol over the given shards (records of every shard
    reused by every round; the merge sees them in `order`)."""
    V = int(dw["vocab"])
    n = int(dw["num_rows"])
    params = {k: dw.get(k) for k in ss.PARAM_FIELDS}
    params["bitmask_stride"] = dw.get("bitmask_stride", 0)
    rec_bytes = ss.ss_shard_round_record_bytes()
    recs = [torch.zeros(n * rec_bytes, dtype=torch.uint8, device="cuda") for _ in bounds]
    state = torch.zeros(ss.ss_shard_round_state_bytes(n), dtype=torch.uint8, device="cuda")
    tok = torch.full((n,), -7, dtype=torch.int32, device="cuda")
    st = torch.full((n,), -7, dtype=torch.int32, device="cuda")
    kept = torch.full((n,), -7, dtype=torch.int32, device="cuda")
    merged = recs if order is None else [recs[i] for i in order]
    for rnd in range(4):
        for (off, length), rec in zip(bounds, recs):
            ss.ss_shard_round(dw["logits"][:, off:], params, state, rec, round=rnd, vocab=V, vocab_offset=off,
                              shard_len=length, num_rows=n, dtype=dw["dtype"], row_stride=int(dw["row_stride"]))
        ss.ss_merge_round(merged, params, state, tok, st, round=rnd, vocab=V, out_kept=kept)
    torch.cuda.synchronize()
    return {"token": tok.cpu().numpy(), "status": st.cpu().numpy(), "kept": kept.cpu().numpy()}


def _no_top_k(w):
    """The workload with every top-k switched off: top-p / min-p / plain /
    greedy rows, the ones the rounds serve."""
    w = dict(w)
    w["top_k"] = np.zeros(int(w["num_rows"]), np.int32)
    return w


@pytest.mark.parametrize("P", [1, 2, 3, 8])
def test_rounds_equal_whole_decode(ss, P):
    """Top-p and min-p rows without top-k (the heterogeneous decode rows with
    their top-k removed): the rounds reproduce the single call exactly."""
    w = _no_top_k(W.make(2, rows=24))
    dw, whole = _whole(ss, w)
    got = _rounds(ss, dw, W.even_shards(int(w["vocab"]), P))
    for k in ("token", "status", "kept"):
        assert np.array_equal(got[k], whole[k]), (k, got[k], whole[k])
    parity.check_sample(w, got)


def test_rounds_uneven_shards_any_order_with_mask_and_flat_rows(ss):
    w = _no_top_k(W.make(3, rows=12, vocab=20011))  # grammar mask, ragged vocabulary, top-p 0.95
    w["temperature"] = np.linspace(0.5, 1.6, 12).astype(np.float32)
    w["min_p"] = np.tile(np.array([0.0, 0.02, 0.3], np.float32), 4)
    dw, whole = _whole(ss, w)
    bounds = [(0, 4000), (4000, 96), (4096, 9600), (13696, 6315)]
    got = _rounds(ss, dw, bounds, order=[2, 0, 3, 1])
    for k in ("token", "status", "kept"):
        assert np.array_equal(got[k], whole[k]), (k, got[k], whole[k])
    parity.check_sample(w, got)


def test_rounds_statuses_and_top_k_rows(ss):
    w = W.make(2, rows=6, vocab=5003)
    w["temperature"] = np.array([1.0, 1.0, 0.0, -1.0, 1.0, 1.0], np.float32)
    w["top_k"] = np.array([50, 0, 0, 0, 0, 0], np.int32)
    w["top_p"] = np.array([1.0, 0.9, 1.0, 0.9, 1.0, 0.5], np.float32)
    w["min_p"] = np.array([0.0, 0.0, 0.0, 0.0, 0.1, 0.1], np.float32)
    dw, whole = _whole(ss, w)
    got = _rounds(ss, dw, W.even_shards(5003, 3))
    assert (got["token"][0], got["status"][0], got["kept"][0]) == (-7, -7, -7)  # a top-k row: left to the list path
    ok = np.arange(1, 6)
    for k in ("token", "status", "kept"):
        assert np.array_equal(got[k][ok], whole[k][ok]), (k, got[k][ok], whole[k][ok])


def test_list_path_then_rounds_cover_the_headline_rows(ss):
    """Workload 2 as it is (top-k rows and top-p / min-p rows without one):
    the list path's merge, then the four rounds, give every row exactly what
    the single call gives."""
    w = W.make(2, rows=24)
    dw, whole = _whole(ss, w)
    bounds = W.even_shards(int(w["vocab"]), 4)
    first = _sharded(ss, dw, bounds)
    assert np.all(first["status"][(w["top_k"] == 0) & (w["temperature"] > 0) &
                                  ((w["top_p"] < 1) | (w["min_p"] > 0))] == 7)
    got = _rounds(ss, dw, bounds)
    topk = (w["top_k"] > 0) & (w["temperature"] > 0)
    for k in ("token", "status", "kept"):
        merged = np.where(topk, first[k], got[k])
        assert np.array_equal(merged, whole[k]), (k, merged, whole[k])
