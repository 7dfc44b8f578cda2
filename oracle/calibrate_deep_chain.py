"""Calibrate the draft-noise sigma of the deep-chain workload with the oracle.

TEST INFRASTRUCTURE.  The deep-chain workload (one sequence, gamma = 48, V = 152064 bf16,
target T = 0.6, sharpened draft T_d = 0.2) asks for a mean per-token acceptance of about
0.56, the per-token rate SubSpec's report derives from tau = 27.08 at a draft depth of 48
("SubSpec: the target model's own low-bit shadow as the draft model", section 3.7).  The
per-token acceptance of draft position i is the overlap sum_x min(p_i(x), q_i(x))
("How speculative decoding makes LLMs go brrr", module 3: the mass accepted drafts cover).

The noise draws are fixed by the data seed, so the mean overlap is a function of sigma
alone; this script bisects sigma on [0, 4] and prints the value that
``workloads.DEEP_CHAIN_SIGMA`` holds.  It calls only the oracle and the input generator.

    python -m oracle.calibrate_deep_chain
"""
from __future__ import annotations

import sys
import os

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import numpy as np  # noqa: E402

import oracle  # noqa: E402
import workloads  # noqa: E402

TARGET = 0.56


def mean_overlap(sigma: float, orc: "oracle.Oracle") -> float:
    w = workloads.deep_chain_with_sigma(sigma)
    ov = orc.row_overlap(w.target[0, :w.gamma], w.draft[0], w.T[0], w.Td[0])
    return float(np.mean(ov))


def calibrate(tol: float = 1e-4) -> float:
    orc = oracle.get()
    lo, hi = 0.0, 4.0
    f_lo, f_hi = mean_overlap(lo, orc), mean_overlap(hi, orc)
    print(f"sigma={lo}: {f_lo:.5f}   sigma={hi}: {f_hi:.5f}")
    assert f_lo > TARGET > f_hi
    while hi - lo > tol:
        mid = 0.5 * (lo + hi)
        f = mean_overlap(mid, orc)
        print(f"sigma={mid:.10f}: {f:.6f}")
        if f > TARGET:
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


if __name__ == "__main__":
    s = calibrate()
    print(f"DEEP_CHAIN_SIGMA = {s!r}   mean overlap {mean_overlap(s, oracle.get()):.6f}")
