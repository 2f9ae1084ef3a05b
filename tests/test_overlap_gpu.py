"""Back-to-back calls that overlap (SS_SAMPLE_OVERLAP_PREVIOUS,
SS_VERIFY_OVERLAP_PREVIOUS, SS_TREE_OVERLAP_PREVIOUS: programmatic dependent
launch): every call's
results equal those of the same call made alone, including when consecutive
calls write the same output buffers (the later call's writes land last), when
verification calls share one workspace, and inside a CUDA graph."""
import numpy as np
import pytest

from speculative_verification_gb300 import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

KEYS = ("token", "status", "kept")


@pytest.fixture(scope="module")
def ss():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_verification_gb300 import build as ss_build
    ss_build.build()
    from speculative_verification_gb300 import ss as _ss
    _ss.load()
    return _ss


def _sets(ss, n, rows=32, vocab=128256):
    return [ss.to_device(W.make(2, rows=rows, vocab=vocab, seed=50 + i)) for i in range(n)]


def _alone(ss, sets):
    ref = []
    for dw in sets:
        o = ss.alloc_outputs(dw)
        ss.run(dw, o)
        torch.cuda.synchronize()
        ref.append({k: o[k].clone() for k in KEYS})
    return ref


def test_overlapped_calls_equal_calls_alone(ss):
    sets = _sets(ss, 6)
    ref = _alone(ss, sets)
    outs = [ss.alloc_outputs(dw) for dw in sets]
    for dw, o in zip(sets, outs):
        ss.run(dw, o, overlap_previous=True)
    torch.cuda.synchronize()
    for r, o in zip(ref, outs):
        for k in KEYS:
            assert torch.equal(r[k], o[k]), k


def test_overlapped_calls_into_the_same_outputs_keep_the_last(ss):
    sets = _sets(ss, 5)
    ref = _alone(ss, sets)
    o = ss.alloc_outputs(sets[0])
    dbg = torch.empty((int(sets[0]["num_rows"]), int(sets[0]["vocab"])), dtype=torch.float32, device="cuda")
    o["processed"] = dbg
    for rep in range(3):
        for dw in sets:
            ss.run(dw, o, debug=True, overlap_previous=True)
        torch.cuda.synchronize()
        for k in KEYS:
            assert torch.equal(ref[-1][k], o[k]), (rep, k)
    # the debug rows of the last call too
    last = ss.alloc_outputs(sets[-1], debug=True)
    ss.run(sets[-1], last, debug=True)
    torch.cuda.synchronize()
    assert torch.equal(last["processed"], dbg)


def test_overlapped_calls_in_a_graph(ss):
    sets = _sets(ss, 4)
    ref = _alone(ss, sets)
    outs = [ss.alloc_outputs(dw) for dw in sets]
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for dw, o in zip(sets, outs):  # warm-up outside the capture
            ss.run(dw, o, stream=stream, overlap_previous=True)
    stream.synchronize()
    for o in outs:
        for k in KEYS:
            o[k].fill_(-7)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            for dw, o in zip(sets, outs):
                ss.run(dw, o, stream=stream, overlap_previous=True)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    for r, o in zip(ref, outs):
        for k in KEYS:
            assert torch.equal(r[k], o[k]), k


def test_overlap_flag_on_fp32_and_verification_is_harmless(ss):
    # the flag is honoured by bf16 sampling only; fp32 calls run as usual
    w = W.make(2, rows=8, vocab=5003, seed=3)
    w32 = dict(w, dtype="f32", logits=W.bf16_bits_to_f32(w["logits"]))
    dw = ss.to_device(w32)
    a, b = ss.alloc_outputs(dw), ss.alloc_outputs(dw)
    ss.run(dw, a)
    ss.run(dw, b, overlap_previous=True)
    torch.cuda.synchronize()
    for k in KEYS:
        assert torch.equal(a[k], b[k]), k
    assert np.all(a["status"].cpu().numpy() == 0)


VKEYS = ("out_tokens", "num_accepted", "status", "kept")


def _vsets(ss, n):
    return [ss.to_device(W.make(4, requests=16, k=4, vocab=128256, seed=70 + i)) for i in range(n)]


def test_overlapped_verification_with_one_workspace(ss):
    # consecutive verification calls share the outputs and the workspace: a
    # call may start early but uses the workspace only after the one before
    sets = _vsets(ss, 4)
    ref = []
    for dw in sets:
        o = ss.alloc_outputs(dw)
        ss.run(dw, o)
        torch.cuda.synchronize()
        ref.append({k: o[k].clone() for k in VKEYS})
    o = ss.alloc_outputs(sets[0])
    for rep in range(3):
        for dw in sets:
            ss.run(dw, o, overlap_previous=True)
        torch.cuda.synchronize()
        for k in VKEYS:
            assert torch.equal(ref[-1][k], o[k]), (rep, k)
    # each call's own outputs, overlapped, into separate buffers (one workspace each)
    sep = [ss.alloc_outputs(dw) for dw in sets]
    for dw, oo in zip(sets, sep):
        ss.run(dw, oo, overlap_previous=True)
    torch.cuda.synchronize()
    for r, oo in zip(ref, sep):
        for k in VKEYS:
            assert torch.equal(r[k], oo[k]), k


def test_overlapped_sampling_after_verification(ss):
    # a sampling call overlapping the verification call before it
    v = _vsets(ss, 1)[0]
    s_sets = _sets(ss, 2)
    ref_s = _alone(ss, s_sets)
    ov = ss.alloc_outputs(v)
    ss.run(v, ov)
    torch.cuda.synchronize()
    ref_v = {k: ov[k].clone() for k in VKEYS}
    o2 = ss.alloc_outputs(v)
    so = [ss.alloc_outputs(dw) for dw in s_sets]
    ss.run(v, o2, overlap_previous=True)
    for dw, oo in zip(s_sets, so):
        ss.run(dw, oo, overlap_previous=True)
    torch.cuda.synchronize()
    for k in VKEYS:
        assert torch.equal(ref_v[k], o2[k]), k
    for r, oo in zip(ref_s, so):
        for k in KEYS:
            assert torch.equal(r[k], oo[k]), k


TKEYS = ("out_tokens", "out_path", "num_accepted", "status")


def test_overlapped_tree_verification_with_one_workspace(ss):
    # draft trees of different shapes, back to back, into shared outputs and
    # one workspace, then each into its own, alone and in a graph
    hosts = [W.tree(seed=300 + i, requests=24, vocab=128256, max_nodes=16) for i in range(4)]
    sets = [ss.to_device(w) for w in hosts]
    rows = [int(w["node_offsets"][-1]) for w in hosts]
    ref = []
    for dw in sets:
        o = ss.alloc_outputs(dw)
        ss.run(dw, o)
        torch.cuda.synchronize()
        ref.append({k: o[k].clone() for k in TKEYS + ("kept",)})
    big = max(range(len(sets)), key=lambda i: rows[i])
    o = ss.alloc_outputs(sets[big])
    for rep in range(3):
        for dw in sets:
            ss.run(dw, o, overlap_previous=True)
        torch.cuda.synchronize()
        for k in TKEYS:
            assert torch.equal(ref[-1][k], o[k]), (rep, k)
        assert torch.equal(ref[-1]["kept"], o["kept"][:rows[-1]]), rep
    sep = [ss.alloc_outputs(dw) for dw in sets]
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            for dw, oo in zip(sets, sep):
                ss.run(dw, oo, stream=stream, overlap_previous=True)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    for r, oo in zip(ref, sep):
        for k in TKEYS + ("kept",):
            assert torch.equal(r[k], oo[k]), k
    assert any(int(r["num_accepted"].sum()) > 0 for r in ref)
