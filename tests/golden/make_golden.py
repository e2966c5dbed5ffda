"""Writes the stored oracle outputs under tests/golden/ (run from the repo root:
python tests/golden/make_golden.py).  Every value comes from the float64
oracle alone (oracle.forward) on seeded inputs; the pages print no worked
example of the block, so none of these numbers is theirs.  The files let the
CPU tests notice any later change to the oracle's arithmetic, and give the GPU
tests a parity case that needs no oracle run.

Cases (page "Swin Transformer" (shifted window attention; relative position
bias) and page "Swin Transformer V2" (scaled cosine attention)):
  v1: B = 1, 8 x 8 tokens, C = 32, 1 head, M = 4, shift 2, V1 logits
  v2: the same grid, V2 cosine logits, tau = 0.1
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import oracle  # noqa: E402

HERE = os.path.dirname(os.path.abspath(__file__))
CASES = {"v1": dict(mode=0), "v2": dict(mode=1)}
B, H, W, C, HEADS, M, SHIFT = 1, 8, 8, 32, 1, 4, 2


def _bf16(a):
    """Round to the nearest bfloat16 (8 significant bits, ties to even), so
    that a GPU run consumes exactly these values."""
    u = np.asarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def inputs(seed=2024):
    r = np.random.default_rng(seed)
    q = lambda *shape, s=1.0: _bf16(r.uniform(-1, 1, shape) * s)  # noqa: E731
    return dict(x=q(B, H, W, C, s=2.0), Wqkv=q(3 * C, C, s=0.5), bqkv=q(3 * C, s=0.1),
                table=q((2 * M - 1) ** 2, HEADS), tau=np.full(HEADS, 0.1),
                Wproj=q(C, C, s=0.03), bproj=q(C, s=0.1))


def compute(mode):
    p = inputs()
    return p, oracle.forward(p["x"], p["Wqkv"], p["bqkv"], p["table"], p["tau"] if mode else None, p["Wproj"],
                             p["bproj"], heads=HEADS, M=M, shift=SHIFT, mode=mode)


def path(name):
    return os.path.join(HERE, "oracle_tiny_%s.txt" % name)


def main():
    oracle.build()
    for name, kw in CASES.items():
        _, out = compute(kw["mode"])
        with open(path(name), "w") as f:
            f.write("# oracle.forward, case %s: B=%d H=%d W=%d C=%d heads=%d M=%d shift=%d mode=%d\n"
                    % (name, B, H, W, C, HEADS, M, SHIFT, kw["mode"]))
            f.write("# written by tests/golden/make_golden.py (float64 oracle; no page prints these values)\n")
            np.savetxt(f, out.reshape(-1, C), fmt="%.17g")


if __name__ == "__main__":
    main()
