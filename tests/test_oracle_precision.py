"""The oracle takes each float-to-integer decision (the accept test, the race argmax) on the
fp32 rounding of its fp64 value -- the precision the kernels decide in.  These tests count
the decisions that pure fp64 would take the other way, and check that every one of them
lies inside the near-tie bands the parity rules flag (|u - p/q| < 1e-5 at a tested
position, top two race scores within 1e-6), so the fp32 reading can never turn an
unflagged comparison.

Accept test: u is exact in fp32 (24 random bits), so (float)u < (float)a and u < a differ
only when a rounds across u: |u - a| <= ulp(a) / 2 < 6e-8 for a < 1, and never for a >= 1
(u < 1 <= both).  Race: the oracle's winner changes on a strictly larger fp32 score, so the
fp64 argmax differs exactly when another token's fp64 score exceeds the winner's, which the
oracle records as second > best (then best - second < 0 < 1e-6: flagged).
"""
import numpy as np
import pytest

import oracle
import workloads


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


def fp32_fp64_differences(r: "oracle.OracleResult", gamma: int):
    """(accept decisions that differ, race decisions that differ, decisions) of one
    oracle result."""
    bad = (r.flags & oracle.FLAG_BAD_TOKEN) != 0
    tested = np.minimum(np.where(bad, -1, r.n_accepted) + 1, gamma)
    acc_diff = 0
    if gamma:
        mask = (np.arange(gamma)[None, :] < tested[:, None]) & ~bad[:, None]
        a = r.a
        with np.errstate(invalid="ignore", over="ignore"):
            d64 = r.u < a
            d32 = r.u.astype(np.float32) < a.astype(np.float32)
        diff = mask & (d64 != d32)
        acc_diff = int(diff.sum())
        # every differing accept decision sits within the near-tie band
        assert np.all(np.abs(r.u - a)[diff] < 1e-5)
        assert np.all((r.flags[np.any(diff, axis=1)] & oracle.FLAG_ACCEPT_NEAR_TIE) != 0)
    race_diff_mask = ~bad & np.isfinite(r.race[:, 1]) & (r.race[:, 1] > r.race[:, 0])
    assert np.all((r.flags[race_diff_mask] & oracle.FLAG_RACE_NEAR_TIE) != 0)
    decisions = int(np.sum(np.where(bad, 0, tested + 1)))
    return acc_diff, int(race_diff_mask.sum()), decisions


def test_fp32_decisions_equal_fp64_outside_the_flagged_bands(orc):
    counts = np.zeros(3, dtype=np.int64)
    w0 = workloads.config(0)
    for seed in range(400):
        counts += fp32_fp64_differences(orc.verify(w0.target, w0.draft, w0.tokens, w0.T, w0.Td, seed), w0.gamma)
    w = workloads.generic(B=64, gamma=8, V=3000, dtype="bf16", seed=11, sigma=0.6, T=0.9, Td=0.4)
    for seed in range(40):
        counts += fp32_fp64_differences(orc.verify(w.target, w.draft, w.tokens, w.T, w.Td, seed), w.gamma)
    assert counts[2] > 5000
    # the counts themselves are a property of these inputs; none occurred when written
    assert counts[0] + counts[1] == 0, counts


def test_a_planted_rounding_case_is_caught():
    """A synthetic oracle result where a rounds across u in fp32: counted and flagged."""
    u = np.float64(np.float32(0.75))
    a = u + 2.0 ** -27                     # (float)a == u: fp32 rejects, fp64 accepts
    assert np.float32(a) == np.float32(u)
    r = oracle.OracleResult(
        tokens=np.zeros((1, 2), np.int32), n_accepted=np.array([0], np.int32),
        logp=np.zeros((1, 1)), logq=np.zeros((1, 1)), u=np.array([[u]]), a=np.array([[a]]),
        logZp=np.zeros((1, 2)), logZq=np.zeros((1, 1)), race=np.array([[1.0, 0.5, 0.0]]),
        flags=np.array([oracle.FLAG_ACCEPT_NEAR_TIE], np.int32))
    acc, race, dec = fp32_fp64_differences(r, 1)
    assert (acc, race, dec) == (1, 0, 2)
