"""Helpers shared by the GPU parity tests: move a workload to the device, run the library
through its C ABI, run the oracle on the same inputs, and compare under the stated rules.

Parity rules (the method is an exact sampler, so the particular draw is pinned by the
random-number contract):
  * greedy mode: tokens and accepted counts bit-exact;
  * sampling mode: tokens and accepted counts bit-exact, except sequences the oracle flags
    as near-ties (|u - p/q| < 1e-5 at a tested position, or top-two race scores within
    1e-6); flagged decisions (positions and races) must stay under 1e-4 of all decisions
    compared in the session (tests/test_zy_near_tie_budget.py);
  * p(d_i) and q(d_i) within 1e-5 relative; u_i bit-exact; ln Z within 1e-6 relative.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads

NEAR_TIE = oracle.FLAG_ACCEPT_NEAR_TIE | oracle.FLAG_RACE_NEAR_TIE | oracle.FLAG_RESIDUAL_EMPTY

# The accept-test band: a tested position whose |u - p/q| is below this is a near-tie.
ACCEPT_BAND = 1e-5

# Running totals over the session (every module that compares sampling results with the
# oracle adds to them): decisions compared (each tested position and each race), decisions
# flagged as near-ties, sequences, and flagged sequences whose outputs differed.
TOTALS = {"decisions": 0, "flagged": 0, "sequences": 0, "mismatch_flagged": 0}


def decision_counts(r: "oracle.OracleResult", gamma: int):
    """(decisions, flagged decisions) of oracle results `r`: the tested positions of each
    sequence (0..min(j, gamma - 1) for first rejection j) and its race; a tested position is
    flagged when |u - p/q| < ACCEPT_BAND, a race when the oracle flags its top two scores as
    within 1e-6 (or its residual as empty).  Sequences with a bad draft token decide
    nothing."""
    bad = (r.flags & oracle.FLAG_BAD_TOKEN) != 0
    n = np.where(bad, -1, r.n_accepted)
    tested = np.minimum(n + 1, gamma)                      # positions whose test ran
    decisions = int(np.sum(np.where(bad, 0, tested + 1)))
    flagged = 0
    if gamma:
        pos = np.arange(gamma)[None, :]
        mask = (pos < tested[:, None]) & ~bad[:, None]
        near = np.abs(r.u - r.a) < ACCEPT_BAND
        flagged += int(np.sum(mask & near))
    race_flag = (r.flags & (oracle.FLAG_RACE_NEAR_TIE | oracle.FLAG_RESIDUAL_EMPTY)) != 0
    flagged += int(np.sum(race_flag & ~bad))
    return decisions, flagged


def to_device(a: np.ndarray, dtype: str, dev) -> torch.Tensor:
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev)


class DeviceWorkload:
    def __init__(self, w: workloads.Workload, dev="cuda:0"):
        self.w = w
        self.dev = torch.device(dev)
        self.target = to_device(w.target, w.dtype, self.dev)
        self.draft = to_device(w.draft, w.dtype, self.dev)
        self.tokens = torch.from_numpy(np.ascontiguousarray(w.tokens)).to(self.dev)
        self.T = torch.from_numpy(w.T.astype(np.float32)).to(self.dev)
        self.Td = torch.from_numpy(w.Td.astype(np.float32)).to(self.dev)


def run_gpu(sv, dw: DeviceWorkload, seed: int, per_seq_temps: bool = True, seq_index_base=0,
            diagnostics=True, flags=0):
    w = dw.w
    kw = {}
    if per_seq_temps:
        kw = dict(T_per_seq=dw.T, Td_per_seq=dw.Td)
    out_t, out_n, diag = sv.spec_verify_ex(dw.target, dw.draft, dw.tokens, float(w.T[0]),
                                           float(w.Td[0]), seed, seq_index_base=seq_index_base,
                                           diagnostics=diagnostics, flags=flags, **kw)
    torch.cuda.synchronize()
    res = {"tokens": out_t.cpu().numpy(), "n": out_n.cpu().numpy()}
    if diag:
        res.update({k: v.cpu().numpy() for k, v in diag.items()})
    return res


def compare_sampling(w: workloads.Workload, g: dict, r: "oracle.OracleResult",
                     check_values: bool = True, idx=None, count: bool = True):
    """Assert parity of GPU results `g` with oracle results `r` (same sequences).
    `idx` selects GPU rows when the oracle ran on a subset.  `count` adds the comparison's
    decisions to TOTALS (False when the same oracle result is compared a second time)."""
    if idx is not None:
        g = {k: v[idx] for k, v in g.items()}
    B, gamma = w.B if idx is None else len(idx), w.gamma
    flagged = (r.flags & NEAR_TIE) != 0
    bad = (r.flags & oracle.FLAG_BAD_TOKEN) != 0
    if count:
        decisions, flagged_decisions = decision_counts(r, gamma)
        TOTALS["decisions"] += decisions
        TOTALS["flagged"] += flagged_decisions
        TOTALS["sequences"] += B
    for b in range(B):
        if flagged[b]:
            TOTALS["mismatch_flagged"] += int(g["n"][b] != r.n_accepted[b] or
                                               not np.array_equal(g["tokens"][b], r.tokens[b]))
            # still a valid cycle
            j = g["n"][b]
            assert 0 <= j <= gamma
            assert np.all(g["tokens"][b, j + 1:] == -1) and 0 <= g["tokens"][b, j] < w.V
            continue
        assert g["n"][b] == r.n_accepted[b], (b, g["n"][b], r.n_accepted[b], r.flags[b])
        np.testing.assert_array_equal(g["tokens"][b], r.tokens[b], err_msg=f"sequence {b}")
    if not check_values or "u" not in g:
        return
    ok = ~bad
    np.testing.assert_array_equal(g["u"].astype(np.float64), r.u)
    if gamma:
        for name, ref in (("logp", r.logp), ("logq", r.logq)):
            got = g[name][ok].astype(np.float64)
            want = ref[ok]
            fin = np.isfinite(want)
            assert np.array_equal(np.isfinite(got), fin), name
            # p and q within 1e-5 relative  <=>  |ln p_gpu - ln p_oracle| < ~1e-5; a probability
            # so small that |ln p| * 2^-24 (fp32's own resolution of the logarithm the kernels
            # keep) approaches that is allowed four such units more
            err = np.abs(np.expm1(got[fin] - want[fin]))
            allow = 1e-5 + 4.0 * 2.0 ** -24 * np.abs(want[fin])
            assert err.size == 0 or np.all(err < allow), (name, float(err.max()))
        zq = g["logZq"].astype(np.float64)
        np.testing.assert_allclose(zq, r.logZq, rtol=1e-6, atol=1e-6)
    zp = g["logZp"].astype(np.float64)
    np.testing.assert_allclose(zp, r.logZp, rtol=1e-6, atol=1e-6)
    # the winning race score ln w(y) - ln E_y (a check of the device Philox and E mapping).
    # For a residual, ln(p - q) at the winner inherits the errors of ln p and ln q (fp32, a few
    # 1e-6) amplified by (q/p) / (1 - q/p): the allowance grows with that factor.
    sel = ok & ~flagged
    for b in np.flatnonzero(sel):
        j, y = int(r.n_accepted[b]), int(r.tokens[b, r.n_accepted[b]])
        cond = 0.0
        if j < gamma:
            lp = float(workloads.as_f32(w.target[b, j, y:y + 1], w.dtype)[0]) / float(w.T[b]) - r.logZp[b, j]
            lq = float(workloads.as_f32(w.draft[b, j, y:y + 1], w.dtype)[0]) / float(w.Td[b]) - r.logZq[b, j]
            ratio = np.exp(min(0.0, lq - lp))
            cond = ratio / max(1.0 - ratio, 1e-12)
        tol = 2e-5 + 1e-5 * abs(r.race[b, 0]) + 1e-5 * cond
        assert abs(float(g["race"][b, 0]) - r.race[b, 0]) <= tol, (b, float(g["race"][b, 0]), r.race[b, 0], cond)


def gpu_near_ties(g: dict, gamma: int) -> np.ndarray:
    """Sequences whose decisions are near-ties by the GPU's own diagnostics (the same rules
    as the oracle's flags, applied to a full-read call's outputs): used where the oracle
    does not run on every sequence."""
    B = len(g["n"])
    flagged = np.zeros(B, dtype=bool)
    for b in range(B):
        j = int(g["n"][b])
        if j < 0:
            continue
        for i in range(min(j + 1, gamma)):
            a = np.exp(min(0.0, float(g["logp"][b, i]) - float(g["logq"][b, i])))
            if abs(float(g["u"][b, i]) - a) < 1e-5:
                flagged[b] = True
        best, second = float(g["race"][b, 0]), float(g["race"][b, 1])
        if np.isfinite(second) and abs(best - second) <= 1e-6 * max(1.0, abs(best)):
            flagged[b] = True
    return flagged


def compare_greedy(g_tokens, g_n, r_tokens, r_n):
    np.testing.assert_array_equal(g_n, r_n)
    np.testing.assert_array_equal(g_tokens, r_tokens)
