"""The LM head fused with the draw (tcgen05 tensor cores), through the C ABI:
its logits agree with an fp64 matrix multiply of the same bf16 inputs within
an accumulation bound, and its tokens are the oracle's draw on those logits.
A row is compared exactly unless its draw can change with the logits anywhere
inside that bound (plus the oracle's 1e-5 margin): such rows are counted."""
import numpy as np
import pytest

from oracle import oracle as O
from speculative_verification_gb300 import workloads as W

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


def _run(ss, w, debug):
    dev = torch.device("cuda")
    h = torch.from_numpy(w["hidden_states"].view(np.int16)).to(dev).view(torch.bfloat16)
    wt = torch.from_numpy(w["weight"].view(np.int16)).to(dev).view(torch.bfloat16)
    B, V = w["batch"], w["vocab"]
    temp = torch.from_numpy(w["temperature"]).to(dev)
    seed = torch.from_numpy(w["seed"].view(np.int64)).to(dev)
    pos = torch.from_numpy(w["position"]).to(dev)
    rid = torch.from_numpy(w["row_id"].view(np.int32)).to(dev) if w.get("row_id") is not None else None
    scratch = torch.empty(ss.ss_fused_scratch_bytes(B), dtype=torch.uint8, device=dev)
    tok = torch.empty(B, dtype=torch.int32, device=dev)
    st = torch.empty(B, dtype=torch.int32, device=dev)
    dbg = torch.empty((B, V), dtype=torch.float32, device=dev) if debug else None
    ss.ss_fused_lmhead_sample(h, wt, temp, seed, pos, scratch, tok, st, row_id=rid, debug_logits=dbg)
    torch.cuda.synchronize()
    return tok.cpu().numpy(), st.cpu().numpy(), (dbg.cpu().numpy() if debug else None)


def _check(w, tok, st, logits):
    ref = O.lmhead_sample(w)
    assert np.array_equal(st, ref["status"])
    # the fp32 sums of the tensor cores against the fp64 product: within
    # 1e-5 of sum |h_i w_i| (+ 1e-6), checked here on every logit
    h = (w["hidden_states"].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    wt = (w["weight"].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    bound = 1e-5 * (np.abs(h) @ np.abs(wt).T) + 1e-6
    err = np.abs(logits.astype(np.float64) - ref["logits"].astype(np.float64))
    assert np.all(err <= bound), float(np.max(err / bound))
    # so a draw that no logit inside its bound can change must match exactly
    sub = O.interval_flags(ref["logits"], bound, w["temperature"], w["seed"], w["position"],
                           w.get("row_id")) != 0
    assert np.all(sub[ref["sub_margin"] != 0])  # the wider test contains the oracle's own
    mism = np.flatnonzero(~sub & (tok != ref["token"]))
    assert mism.size == 0, (mism, tok[mism], ref["token"][mism])
    assert sub.sum() <= 0.1 * len(sub) + 1, int(sub.sum())
    return int((~sub).sum()), int(sub.sum())


def test_fused_small_ragged_vocab(ss):
    w = W.lmhead(batch=8, hidden=256, vocab=1000, seed=3)
    tok, st, logits = _run(ss, w, debug=True)
    print("fused small", _check(w, tok, st, logits))


def test_fused_batch_not_multiple_of_32_with_row_ids(ss):
    w = W.lmhead(batch=45, hidden=512, vocab=40111, seed=4)
    w["row_id"] = np.random.default_rng(1).integers(0, 2**32, 45, dtype=np.uint64).astype(np.uint32)
    tok, st, logits = _run(ss, w, debug=True)
    print("fused B=45", _check(w, tok, st, logits))


def test_fused_full_vocabulary(ss):
    w = W.lmhead(batch=16, hidden=1024, vocab=128256, seed=5)
    tok, st, logits = _run(ss, w, debug=True)
    print("fused V=128256 (exact, within the bound)", _check(w, tok, st, logits))
    tok2, st2, _ = _run(ss, w, debug=False)  # the same draw without the debug output
    assert np.array_equal(tok2, tok) and np.array_equal(st2, st)


def test_fused_bad_parameters(ss):
    w = W.lmhead(batch=4, hidden=128, vocab=300, seed=6)
    w["temperature"] = np.array([1.0, -1.0, np.inf, 0.0], np.float32)
    tok, st, _ = _run(ss, w, debug=False)
    assert list(st) == [0, 4, 4, 0] and tok[1] == -1 and tok[2] == -1
