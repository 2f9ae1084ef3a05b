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
