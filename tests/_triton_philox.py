"""Philox4x32-10 from triton's own library routine (tl.philox), run by the
triton interpreter on the CPU.  Reads JSON {"ctr": [[c0,c1,c2,c3],...],
"seed": [...]} on stdin and prints the four output words per counter."""
import json
import os
import sys

os.environ["TRITON_INTERPRET"] = "1"
import numpy as np  # noqa: E402
import torch  # noqa: E402
import triton  # noqa: E402
import triton.language as tl  # noqa: E402


@triton.jit
def _philox_kernel(out, c0p, c1p, c2p, c3p, seed, N: tl.constexpr):
    i = tl.arange(0, N)
    a, b, c, d = tl.philox(seed, tl.load(c0p + i), tl.load(c1p + i), tl.load(c2p + i), tl.load(c3p + i))
    tl.store(out + 4 * i + 0, a)
    tl.store(out + 4 * i + 1, b)
    tl.store(out + 4 * i + 2, c)
    tl.store(out + 4 * i + 3, d)


def main():
    req = json.load(sys.stdin)
    res = []
    for ctr, seed in zip(req["ctr"], req["seed"]):
        cols = [torch.tensor(np.array([ctr[j]], np.uint32).view(np.int32)) for j in range(4)]
        out = torch.zeros(4, dtype=torch.int32)
        _philox_kernel[(1,)](out, *cols, int(seed), N=1)
        res.append([int(x) & 0xFFFFFFFF for x in out.tolist()])
    json.dump(res, sys.stdout)


if __name__ == "__main__":
    main()
