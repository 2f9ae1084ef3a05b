"""Linear verification with the caller's count of target rows
(ss_verify_args.num_target_rows): the launch with one cluster per target row
gives the outputs of the full launch bit for bit, and the oracle's; a count
that is not the offsets' sum makes every request report SS_ROW_BAD_PARAM and
leaves the workspace fit for the next call."""
import numpy as np
import pytest

from speculative_verification_gb300 import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

KEYS = ("out_tokens", "num_accepted", "status", "kept")
BAD_PARAM = 4  # SS_ROW_BAD_PARAM


@pytest.fixture(scope="module")
def ss():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_verification_gb300 import build as ss_build
    ss_build.build()
    from speculative_verification_gb300 import ss as _ss
    _ss.load()
    return _ss


def _call(ss, dw, o, rows, **kw):
    params = {k: dw.get(k) for k in ss.PARAM_FIELDS}
    params["bitmask_stride"] = dw.get("bitmask_stride", 0)
    ss.ss_spec_verify(dw["target_logits"], dw["draft_offsets"], dw["draft_tokens"], dw["draft_probs"], params,
                      o["out_tokens"], o["num_accepted"], o["status"], o["workspace"], vocab=dw["vocab"],
                      max_draft=dw["max_draft"], dtype=dw["dtype"], row_stride=dw["row_stride"],
                      draft_stride=dw["draft_stride"], out_kept=o["kept"], num_target_rows=rows, **kw)


def _outputs(ss, dw, rows, **kw):
    o = ss.alloc_outputs(dw)
    _call(ss, dw, o, rows, **kw)
    torch.cuda.synchronize()
    return {k: o[k].cpu().numpy() for k in KEYS}


def _rows(w):
    return int(w["draft_offsets"][-1]) + int(w["num_requests"])


def _same(a, b):
    for k in KEYS:
        assert np.array_equal(a[k], b[k]), k


@pytest.mark.parametrize("vocab", [5003, 128256, 262144])
def test_compact_launch_equals_full_launch(ss, vocab):
    # half the requests without drafts, the others with 1..7: the compact
    # launch is taken (idle clusters outnumber the rows past position 0)
    w = W.make(5, requests=48, vocab=vocab, seed=21)
    dw = ss.to_device(w)
    full = _outputs(ss, dw, 0)
    compact = _outputs(ss, dw, _rows(w))
    _same(full, compact)
    assert (full["status"] == 0).all()


def test_compact_launch_against_the_oracle(ss):
    from tests import parity
    w = W.make(5, requests=40, vocab=9001, seed=5)
    dw = ss.to_device(w)
    o = ss.alloc_outputs(dw)
    ss.run(dw, o, target_rows=True)
    torch.cuda.synchronize()
    gpu = {k: v.cpu().numpy() for k, v in o.items() if k != "workspace"}
    c = parity.check_verify(w, gpu)
    print("compact launch: %d requests OK, %d compared exactly" % (c.total, c.exact))
    assert c.exact > 0 and c.sub <= 0.01 * c.total + 1


def test_compact_launch_long_and_uneven_drafts(ss):
    # a few long drafts among many requests without any: the position search
    # runs over 60 positions and 300 requests
    w = W.make(5, requests=300, vocab=4099, max_draft=60, seed=8, plain_top_k_max=500)
    k = np.diff(w["draft_offsets"])
    assert k.max() > 30 and (k == 0).sum() >= 150
    dw = ss.to_device(w)
    _same(_outputs(ss, dw, 0), _outputs(ss, dw, _rows(w)))


def test_count_without_idle_clusters_keeps_the_full_launch(ss):
    # every request has max_draft drafts: the count equals the full launch
    w = W.make(4, requests=16, k=4, vocab=7001, seed=4)
    dw = ss.to_device(w)
    assert _rows(w) == 16 * 5
    _same(_outputs(ss, dw, 0), _outputs(ss, dw, _rows(w)))


@pytest.mark.parametrize("delta", [-1, 1])
@pytest.mark.parametrize("compact", [True, False])
def test_wrong_count_reports_bad_param(ss, delta, compact):
    if compact:
        w = W.make(5, requests=32, vocab=6007, seed=13)
    else:
        w = W.make(4, requests=16, k=3, vocab=6007, seed=13)
        w["max_draft"] = 4  # one idle position per request: the full launch stays
    dw = ss.to_device(w)
    ref = _outputs(ss, dw, 0)
    o = ss.alloc_outputs(dw)
    for key in ("out_tokens", "num_accepted", "status"):
        o[key].fill_(77)
    _call(ss, dw, o, _rows(w) + delta)
    torch.cuda.synchronize()
    assert (o["status"].cpu().numpy() == BAD_PARAM).all()
    assert (o["num_accepted"].cpu().numpy() == 0).all()
    assert (o["out_tokens"].cpu().numpy() == -1).all()
    # the same workspace then serves a correct call
    _call(ss, dw, o, _rows(w))
    torch.cuda.synchronize()
    _same(ref, {k: o[k].cpu().numpy() for k in KEYS})


def test_bad_draft_count_counts_as_no_drafts(ss):
    w = W.make(5, requests=24, vocab=3001, seed=17)
    off = w["draft_offsets"].copy()
    # request 20 claims max_draft + 3 drafts (invalid): every later offset moves
    bad = 20
    extra = int(w["max_draft"]) + 3 - int(off[bad + 1] - off[bad])
    off[bad + 1:] += extra
    w = dict(w, draft_offsets=off)
    n = int(w["num_requests"])
    rows = sum((int(off[i + 1] - off[i]) if 0 <= off[i + 1] - off[i] <= w["max_draft"] else 0) + 1 for i in range(n))
    # the target rows and drafts of the later requests are never read past the
    # arrays: pad both so every stated row exists
    pad_rows = int(off[-1]) + n - int(w["target_logits"].shape[0])
    if pad_rows > 0:
        w["target_logits"] = np.concatenate([w["target_logits"], w["target_logits"][:pad_rows]])
        w["draft_probs"] = np.concatenate([w["draft_probs"], w["draft_probs"][:pad_rows]])
        w["draft_tokens"] = np.concatenate([w["draft_tokens"], w["draft_tokens"][:pad_rows]])
    dw = ss.to_device(w)
    full = _outputs(ss, dw, 0)
    assert full["status"][bad] == BAD_PARAM
    _same(full, _outputs(ss, dw, rows))


def test_compact_launch_overlapped_in_a_graph(ss):
    sets = [W.make(5, requests=32, vocab=128256, seed=60 + i) for i in range(3)]
    dws = [ss.to_device(w) for w in sets]
    ref = [_outputs(ss, dw, 0) for dw in dws]
    outs = [ss.alloc_outputs(dw) for dw in dws]
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            for dw, o in zip(dws, outs):
                ss.run(dw, o, stream=stream, overlap_previous=True, target_rows=True)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    for r, o in zip(ref, outs):
        _same(r, {k: o[k].cpu().numpy() for k in KEYS})


def test_noalloc_with_a_count(ss):
    w = W.make(5, requests=20, vocab=9001, max_draft=7, seed=23, plain_top_k_max=500)
    dw = ss.to_device(w)
    ref = _outputs(ss, dw, 0)
    o = ss.alloc_outputs(dw)
    params = {k: dw.get(k) for k in ss.PARAM_FIELDS}
    params["bitmask_stride"] = dw.get("bitmask_stride", 0)
    ss.ss_spec_verify_noalloc(dw["target_logits"], dw["draft_offsets"], dw["draft_tokens"], dw["draft_probs"], params,
                              o["out_tokens"], o["num_accepted"], o["status"], vocab=dw["vocab"],
                              max_draft=dw["max_draft"], dtype=dw["dtype"], row_stride=dw["row_stride"],
                              draft_stride=dw["draft_stride"], out_kept=o["kept"], num_target_rows=_rows(w))
    torch.cuda.synchronize()
    _same(ref, {k: o[k].cpu().numpy() for k in KEYS})


def test_compact_launch_debug_rows_and_row_ids(ss):
    # the processed rows written by the compact launch and caller-given row
    # ids: equal to the full launch's, row for row
    w = W.make(5, requests=36, vocab=7001, seed=31, plain_top_k_max=800)
    w["row_id"] = np.random.default_rng(5).integers(0, 2**32, 36, dtype=np.uint64).astype(np.uint32)
    dw = ss.to_device(w)
    res = []
    for rows in (0, _rows(w)):
        o = ss.alloc_outputs(dw, debug=True)
        o["processed"].fill_(-123.0)
        params = {k: dw.get(k) for k in ss.PARAM_FIELDS}
        params["bitmask_stride"] = dw.get("bitmask_stride", 0)
        ss.ss_spec_verify(dw["target_logits"], dw["draft_offsets"], dw["draft_tokens"], dw["draft_probs"], params,
                          o["out_tokens"], o["num_accepted"], o["status"], o["workspace"], vocab=dw["vocab"],
                          max_draft=dw["max_draft"], dtype=dw["dtype"], row_stride=dw["row_stride"],
                          draft_stride=dw["draft_stride"], out_kept=o["kept"], debug_processed=o["processed"],
                          num_target_rows=rows)
        torch.cuda.synchronize()
        res.append({k: o[k].cpu().numpy() for k in KEYS + ("processed",)})
    for k in KEYS:
        assert np.array_equal(res[0][k], res[1][k]), k
    assert np.array_equal(res[0]["processed"].view(np.uint32), res[1]["processed"].view(np.uint32))
    assert not (res[1]["processed"] == -123.0).all(axis=1).any()  # every target row written
