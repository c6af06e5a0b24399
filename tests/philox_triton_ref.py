"""Philox-4x32-10 words from Triton's own generator (tl.philox), run on the CPU by
Triton's interpreter: an implementation independent of the oracle, used as a pin.

Reads JSON [[c0, c1, c2, c3, seed], ...] on stdin and prints [[w0, w1, w2, w3], ...].
Triton keys the generator with (seed mod 2^32, seed div 2^32)."""
import json
import os
import sys

os.environ["TRITON_INTERPRET"] = "1"

import torch  # noqa: E402
import triton  # noqa: E402
import triton.language as tl  # noqa: E402


@triton.jit
def _philox_kernel(ctr, out, seed):
    off = tl.arange(0, 4)
    c = tl.load(ctr + off)
    c0 = tl.sum(tl.where(off == 0, c, 0)).to(tl.uint32)
    c1 = tl.sum(tl.where(off == 1, c, 0)).to(tl.uint32)
    c2 = tl.sum(tl.where(off == 2, c, 0)).to(tl.uint32)
    c3 = tl.sum(tl.where(off == 3, c, 0)).to(tl.uint32)
    w0, w1, w2, w3 = tl.philox(seed, c0, c1, c2, c3)
    tl.store(out + 0, w0.to(tl.int64))
    tl.store(out + 1, w1.to(tl.int64))
    tl.store(out + 2, w2.to(tl.int64))
    tl.store(out + 3, w3.to(tl.int64))


def main():
    items = json.load(sys.stdin)
    res = []
    for c0, c1, c2, c3, seed in items:
        ctr = torch.tensor([c0, c1, c2, c3], dtype=torch.int64)
        out = torch.zeros(4, dtype=torch.int64)
        _philox_kernel[(1,)](ctr, out, seed)
        res.append([int(x) & 0xFFFFFFFF for x in out.tolist()])
    print(json.dumps(res))


if __name__ == "__main__":
    main()
