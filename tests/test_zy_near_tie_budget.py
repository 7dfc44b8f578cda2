"""Near-tie budget (marked gpu): over every sampling comparison with the oracle in the
session, the decisions the oracle flags as near-ties -- a tested position with
|u - p/q| < 1e-5, or a race whose top two scores are within 1e-6 -- stay under 1e-4 of the
decisions compared.  Collected after the other GPU modules (and before the allocation-free
entry point's file), so it sees their totals; run alone it has nothing to count and skips.
"""
import pytest

from _parity import TOTALS

pytestmark = pytest.mark.gpu


def test_near_tie_decisions_under_budget():
    if TOTALS["decisions"] == 0:
        pytest.skip("no sampling comparisons ran in this session")
    assert TOTALS["flagged"] < 1e-4 * TOTALS["decisions"], TOTALS
