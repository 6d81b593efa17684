"""Derives the exp2 polynomial used by the DP kernels (common.cuh, `exp2_neg`).

Method (Cody & Waite range reduction, then a polynomial): for x <= 0 write
x = n + f with n = rint(x) and f in [-1/2, 1/2], so 2^x = 2^n * 2^f. 2^f is
approximated by p(f) = 1 + c1 f + ... + c7 f^7, fitted here by least squares in
relative error on Chebyshev nodes of [-1/2, 1/2] (near-minimax), with p(0) = 1
exactly. The fitted relative error (~1e-9) is far below one fp32 ulp, so the
fp32 evaluation error is dominated by round-to-nearest rounding, which carries
no systematic bias: the recursions sum ~N+M such terms along each path, and a
biased exponential would accumulate into the alignment matrix.

    python fit_exp2.py     # prints the coefficients and the fit error
"""
import numpy as np


def fit(degree=7, nodes=4000):
    k = np.arange(nodes)
    f = 0.5 * np.cos((2 * k + 1) * np.pi / (2 * nodes))
    target = np.exp2(f)
    A = np.stack([f ** j for j in range(1, degree + 1)], axis=1)
    # minimise sum ((1 + A c) / target - 1)^2
    W = 1.0 / target
    c, *_ = np.linalg.lstsq(A * W[:, None], (target - 1.0) * W, rcond=None)
    return c


def main():
    c = fit()
    c32 = c.astype(np.float32)
    f = np.linspace(-0.5, 0.5, 200001)
    p = 1.0 + sum(float(c32[j]) * f ** (j + 1) for j in range(len(c32)))
    err = p / np.exp2(f) - 1
    print("relative fit error (fp32 coefficients): max %.3e mean %.3e" % (np.abs(err).max(), err.mean()))
    for j, v in enumerate(c32, start=1):
        print(f"c{j} = {float(v)!r}f")


if __name__ == "__main__":
    main()
