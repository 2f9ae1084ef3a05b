"""ss_spec_verify_noalloc, the verification entry point that allocates nothing.

It serves callers that cannot allocate device memory (a serving engine that
gives all GPU memory to its own pool at start-up, a plugin without an
allocator) and therefore cannot pass a workspace: its scratch is a static
device array inside the library.  Its results must equal those of
ss_spec_verify with a caller workspace, call after call -- the static array
keeps the previous call's contents, so a second call is the one that would
show a missing reset.  This file sorts last so that a stop-at-first-failure
run has already run every other test.
"""
import ctypes as C

import numpy as np
import pytest

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


def _call_noalloc(ss, dw, o):
    params = {k: dw.get(k) for k in ss.PARAM_FIELDS}
    params["bitmask_stride"] = dw.get("bitmask_stride", 0)
    ss.ss_spec_verify_noalloc(dw["target_logits"], dw["draft_offsets"], dw["draft_tokens"], dw["draft_probs"], params,
                              o["out_tokens"], o["num_accepted"], o["status"], vocab=dw["vocab"],
                              max_draft=dw["max_draft"], dtype=dw["dtype"], row_stride=dw["row_stride"],
                              draft_stride=dw["draft_stride"], out_kept=o["kept"])


def _outputs(o):
    return {k: o[k].cpu().numpy() for k in ("out_tokens", "num_accepted", "status", "kept")}


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls(ss):
    # the larger batch first: the smaller batch's counters then fall on the
    # bytes where the larger one left its per-position results, which a
    # missing reset would show; then both shapes again
    large = W.make(5, requests=20, vocab=9001, max_draft=7, plain_top_k_max=500)
    small = W.make(4, requests=12, k=4, vocab=7001)
    for w in (large, small, large, small):
        dw = ss.to_device(w)
        ref = ss.alloc_outputs(dw)
        ss.run(dw, ref)
        got = ss.alloc_outputs(dw)
        for key in ("out_tokens", "num_accepted", "status", "kept"):
            got[key].fill_(-99)
        _call_noalloc(ss, dw, got)
        torch.cuda.synchronize()
        a, b = _outputs(ref), _outputs(got)
        for key in a:
            assert np.array_equal(a[key], b[key]), key
        assert np.all(b["status"] == 0)


def test_noalloc_rejects_batches_beyond_its_scratch(ss):
    lib = ss.load()
    a = ss.ss_verify_args()
    a.num_requests = 1 << 20  # 1M requests x 8 positions x 16 B: far beyond 1 MiB
    a.vocab = 1000
    a.max_draft = 7
    assert lib.ss_spec_verify_noalloc(C.byref(a), None) == ss.SS_ERR_SCRATCH_LIMIT
