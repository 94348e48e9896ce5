"""Writes the stored fixtures under tests/golden/ by calling only the oracle.

Run from the repository root:  python tests/golden/make_golden.py

u_zero_diag_weights.txt: with P1 = 0 every evidence entry is 0, so the Self
entry is sigmoid(0) = 0.5 and every Exchange entry is SiLU(0) = 0 minus the
count correction ("Ask Self, Ask Others", Sec. 3.1 eq.(2); Appendix A.1.1).
Feeding V = identity (d = T) makes Y equal the flow matrix F, whose diagonal
the file lists.  The test checks these numbers against the closed form of
Appendix A.1.3, F_ii = e^0.5 / (e^0.5 + (i-1) i^-lambda), and the oracle
against the file.
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402

ROWS = [1, 2, 3, 10, 64, 128]


def main() -> None:
    T = 128
    P = np.zeros((1, 1, T, T))
    V = np.eye(T).reshape(1, 1, T, T)
    rng = np.random.default_rng(7)
    P2 = rng.standard_normal((1, 1, T, T))
    lines = ["# lambda  i(one-based)  F_ii   (oracle, P1 = 0, V = identity, T = 128, tau_S = 1, causal)"]
    for lam in (0.0, 0.5):
        Y, _ = oracle.fwd(P, P2, V, 1.0, lam, True)
        for i in ROWS:
            lines.append(f"{lam:.1f} {i:d} {Y[0, 0, i - 1, i - 1]:.17g}")
    with open(os.path.join(HERE, "u_zero_diag_weights.txt"), "w") as f:
        f.write("\n".join(lines) + "\n")


if __name__ == "__main__":
    main()
