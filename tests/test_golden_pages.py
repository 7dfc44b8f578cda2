"""Values the pages print, pinned against the oracle and the workload recipes (CPU).

tests/golden/subspec_deep_chain.txt holds SubSpec's printed draft depth, tokens per verify
and per-token acceptance.  The deep-chain workload (one sequence, gamma = 48, V = 152064,
T = 0.6, T_d = 0.2) takes its draft noise from a calibration against that per-token rate:
its mean overlap sum_x min(p_i, q_i) -- the probability that the draft token at position i
is accepted ("How speculative decoding makes LLMs go brrr", module 3) -- must match it.
"""
import os

import numpy as np
import pytest

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_golden(name: str) -> dict:
    vals = {}
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.strip()
            if line and not line.startswith("#"):
                k, v = line.split()
                vals[k] = float(v)
    return vals


def test_subspec_numbers_are_consistent():
    g = read_golden("subspec_deep_chain.txt")
    assert g["depth"] == 48
    assert g["tau"] / g["depth"] == pytest.approx(g["per_token_acceptance"], abs=5e-4)


def test_deep_chain_overlap_matches_the_printed_per_token_rate():
    g = read_golden("subspec_deep_chain.txt")
    w = workloads.config(2)
    assert w.gamma == g["depth"]
    ov = oracle.get().row_overlap(w.target[0, :w.gamma], w.draft[0], w.T[0], w.Td[0])
    assert float(np.mean(ov)) == pytest.approx(g["per_token_acceptance"], abs=5e-3)
