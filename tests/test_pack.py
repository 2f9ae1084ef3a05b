"""The packed input layout the end-to-end benchmark copies in one piece:
every array of a workload must come back bit for bit from its view."""
import numpy as np
import pytest

from speculative_verification_gb300 import ss
from speculative_verification_gb300 import workloads as W


@pytest.mark.parametrize("make", [lambda: W.make(2, rows=6, vocab=1000), lambda: W.make(4, requests=3, vocab=777),
                                  lambda: W.tree(seed=2, requests=3, vocab=500, max_nodes=5)])
def test_packed_views_reproduce_every_array(make):
    torch = pytest.importorskip("torch")
    w = make()
    lay, total = ss.pack_layout(w)
    assert total % 256 == 0
    offs = sorted((off, n) for off, n, _, _ in lay.values())
    for (o1, n1), (o2, _) in zip(offs, offs[1:]):
        assert o1 % 256 == 0 and o1 + n1 <= o2  # aligned, no overlap
    buf = torch.zeros(total, dtype=torch.uint8)
    view = buf.numpy()
    for key, (off, nbytes, _, _) in lay.items():
        arr = np.ascontiguousarray(w[key])
        view[off:off + nbytes] = arr.reshape(-1).view(np.uint8)
    v = ss.views(buf, lay, w)
    for key, val in w.items():
        if isinstance(val, np.ndarray):
            got = v[key]
            if got.dtype == torch.bfloat16:
                got = got.view(torch.int16)
            assert got.numpy().tobytes() == np.ascontiguousarray(val).tobytes(), key
        else:
            assert v[key] == val
