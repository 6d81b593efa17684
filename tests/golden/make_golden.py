"""Writes the golden fixtures of this folder from the fp64 oracle (and nothing else).

Soft-DTW value and input gradients of the plain definition (Cuturi & Blondel,
ICML 2017, the method the SoftDTW-CUDA (PyTorch + Numba) README's
"Acknowledgments" credit; squared Euclidean cost, R[0,0] = 0, borders +inf,
softmin_g(a) = -g log sum exp(-a/g)), for seeded synthetic inputs:

  small_config.txt   the small configuration: B=4, N=M=64, D=4, x, y ~ N(0,1),
                     gamma = 1, upstream weights 1/B (batch-mean loss)
  ragged_tiny.txt    B=3, N=5, M=4, D=2, gamma = 0.7, upstream weights (0.5, -1.25, 2.0)

Each file: '#' header lines (what, inputs, a checksum of the inputs so a change of
the generator shows), then one 'name shape' line per array followed by its values,
17 significant digits. Run from the repository root:
    python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from differentiable_series_alignment_gb300 import synth  # noqa: E402

CASES = {
    "small_config": dict(B=4, N=64, M=64, D=4, gamma=1.0, seed=0, repeat=0, weights=None),
    "ragged_tiny": dict(B=3, N=5, M=4, D=2, gamma=0.7, seed=90, repeat=5004, weights=[0.5, -1.25, 2.0]),
}


def inputs(c):
    return synth.iid_normal_pair(c["B"], c["N"], c["M"], c["D"], c["seed"], repeat=c["repeat"])


def weights(c):
    return np.full(c["B"], 1.0 / c["B"]) if c["weights"] is None else np.asarray(c["weights"], np.float64)


def checksum(x, y):
    return float(np.sum(x.astype(np.float64)) + 2.0 * np.sum(y.astype(np.float64) ** 2))


def write(name, c):
    x, y = inputs(c)
    loss, gx, gy = oracle.batch(x, y, c["gamma"], grad_loss=weights(c))
    path = os.path.join(HERE, name + ".txt")
    with open(path, "w") as f:
        f.write(f"# Soft-DTW loss and input gradients by the fp64 oracle (tests/golden/make_golden.py)\n")
        f.write(f"# inputs: synth.iid_normal_pair(B={c['B']}, N={c['N']}, M={c['M']}, D={c['D']}, "
                f"seed={c['seed']}, repeat={c['repeat']}); gamma={c['gamma']}; "
                f"weights={'1/B' if c['weights'] is None else c['weights']}\n")
        f.write(f"# input checksum {checksum(x, y):.17g}\n")
        for an, a in (("loss", loss), ("grad_x", gx), ("grad_y", gy)):
            a = np.asarray(a, np.float64)
            f.write(f"{an} {' '.join(str(d) for d in a.shape)}\n")
            flat = a.reshape(-1)
            for i in range(0, flat.size, 8):
                f.write(" ".join(f"{v:.17g}" for v in flat[i:i + 8]) + "\n")
    return path


def read(name):
    """(header dict, arrays dict) of a fixture."""
    arrays, cur, shape, vals, hdr = {}, None, None, [], {}
    with open(os.path.join(HERE, name + ".txt")) as f:
        for line in f:
            line = line.strip()
            if line.startswith("# input checksum"):
                hdr["checksum"] = float(line.split()[-1])
                continue
            if not line or line.startswith("#"):
                continue
            head = line.split()
            if head[0].isidentifier():
                if cur is not None:
                    arrays[cur] = np.asarray(vals, np.float64).reshape(shape)
                cur, shape, vals = head[0], tuple(int(v) for v in head[1:]), []
            else:
                vals.extend(float(v) for v in head)
    if cur is not None:
        arrays[cur] = np.asarray(vals, np.float64).reshape(shape)
    return hdr, arrays


if __name__ == "__main__":
    for n, c in CASES.items():
        print(write(n, c))
