"""The LM head on the tensor cores (marked gpu): logits against an fp64 product of the
same bf16 inputs, and the statistics epilogue (ln Z, ln p(token)) against the oracle's fp64
softmax of those logits.

Tolerance: bf16 x bf16 products are exact in fp32; the tensor cores add d of them in fp32,
so a logit carries an absolute error of a few times 2^-24 * sum |h_k w_k| (the tests allow
2e-5 * that sum + 1e-5); ln Z and ln p inherit the logits' error divided by T, plus the fp32
softmax sum's own (allowed: 1e-4 absolute at these sizes).
"""
import os

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_31_gb300 as m
    m.load_library()
    return m


def bf16_pair(rows, V, d, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    h = workloads.to_bf16_bits((rng.standard_normal((rows, d)) * scale).astype(np.float32))
    w = workloads.to_bf16_bits((rng.standard_normal((V, d)) / np.sqrt(d) * 4).astype(np.float32))
    return h, w


def to_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


@pytest.mark.parametrize("rows,V,d", [(128, 256, 64), (256, 1024, 128), (200, 1000, 192), (37, 5003, 256)])
def test_lmhead_logits_match_fp64(sv, rows, V, d):
    h, w = bf16_pair(rows, V, d, rows + V + d)
    got = sv.spec_lmhead_logits(to_dev(h), to_dev(w))
    torch.cuda.synchronize()
    assert sv.spec_verify_check() == sv.SPEC_OK
    hf = workloads.bf16_bits_to_f32(h).astype(np.float64)
    wf = workloads.bf16_bits_to_f32(w).astype(np.float64)
    want = hf @ wf.T
    bound = 2e-5 * (np.abs(hf) @ np.abs(wf).T) + 1e-5
    err = np.abs(got.cpu().numpy().astype(np.float64) - want)
    assert np.all(err <= bound), float((err - bound).max())


@pytest.mark.parametrize("rows,V,d,T", [(256, 1024, 128, 1.0), (300, 8191, 256, 0.6), (129, 152064, 128, 1.3)])
def test_lmhead_row_stats_match_oracle(sv, rows, V, d, T):
    h, w = bf16_pair(rows, V, d, rows * 7 + V)
    rng = np.random.default_rng(1)
    tok = rng.integers(0, V, size=rows).astype(np.int32)
    tok[::5] = -1
    temps = np.full(rows, T, np.float32)
    temps[1::3] = T * 0.5
    logz, logp = sv.spec_lmhead_row_stats(to_dev(h), to_dev(w), torch.from_numpy(temps).cuda(),
                                          torch.from_numpy(tok).cuda())
    torch.cuda.synchronize()
    assert sv.spec_verify_check() == sv.SPEC_OK
    hf = workloads.bf16_bits_to_f32(h).astype(np.float64)
    wf = workloads.bf16_bits_to_f32(w).astype(np.float64)
    logits = (hf @ wf.T).astype(np.float32)  # the rows as the oracle reads them
    orc = oracle.get()
    want_z = np.array([orc.row_log_normalisers(logits[r:r + 1], temps[r])[0] for r in range(rows)])
    np.testing.assert_allclose(logz.cpu().numpy(), want_z, rtol=0, atol=1e-4)
    lp = logp.cpu().numpy()
    for r in range(rows):
        if tok[r] < 0:
            assert np.isnan(lp[r])
        else:
            assert abs(lp[r] - (logits[r, tok[r]] / temps[r] - want_z[r])) < 1e-4


def test_lmhead_argument_checks(sv):
    dev = torch.device("cuda")
    h = torch.zeros((4, 100), dtype=torch.bfloat16, device=dev)   # d not a multiple of 64
    w = torch.zeros((10, 100), dtype=torch.bfloat16, device=dev)
    with pytest.raises(sv.SpecVerifyError) as e:
        sv.spec_lmhead_logits(h, w)
    assert e.value.code == sv.SPEC_EINVAL


def lmhead_workload(B, gamma, V, d, seed, sigma=0.3, scale=1.0):
    """Hidden states and heads for a verify from hidden states: draft states are the
    target's plus noise, the draft head the target's plus noise; draft tokens drawn from
    the draft logits (computed here in fp64 from the bf16 inputs) at T_d."""
    rng = np.random.default_rng(seed)
    ht32 = (rng.standard_normal((B, gamma + 1, d)) * scale).astype(np.float32)
    wt32 = (rng.standard_normal((V, d)) / np.sqrt(d) * 6).astype(np.float32)
    hd32 = (ht32[:, :gamma] + rng.standard_normal((B, gamma, d)) * sigma).astype(np.float32)
    wd32 = (wt32 + rng.standard_normal((V, d)) / np.sqrt(d) * sigma).astype(np.float32)
    ht, wt, hd, wd = (workloads.to_bf16_bits(a) for a in (ht32, wt32, hd32, wd32))
    return ht, wt, hd, wd


def host_logits(h_bits, w_bits):
    """Logits H W^T from the bf16 inputs, products and sums in fp64, and the per-logit bound
    on how far the tensor cores' fp32 accumulation may lie from them (the bound
    test_lmhead_logits_match_fp64 checks: 2e-5 sum_k |h_k w_k| + 1e-5), widened by the
    fp32 rounding of the exact value that the oracle is given."""
    hf = workloads.bf16_bits_to_f32(h_bits).astype(np.float64)
    wf = workloads.bf16_bits_to_f32(w_bits).astype(np.float64)
    exact = hf @ wf.T
    bound = 2e-5 * (np.abs(hf) @ np.abs(wf).T) + 1e-5 + 2.0 ** -24 * np.abs(exact)
    return exact.astype(np.float32), bound


def gemm_sensitive(orc, lt, et, ld, ed, tok, T, Td, seed, r):
    """Sequences whose oracle decisions a logit error within the bounds (et, ed) could
    change: a tested position whose accept ratio a = p(d)/q(d) may move across u (or lies
    within the usual 1e-5 band), or a race whose winner's score interval meets another
    token's (widened by the usual 1e-6).  ln Z moves by at most the row's largest logit
    error / T; each token's score ln w - ln E moves within the interval its weight takes
    over the perturbed p and q."""
    B, G1, V = lt.shape
    g = G1 - 1
    flagged = np.zeros(B, dtype=bool)
    for b in range(B):
        j = int(r.n_accepted[b])
        emax_t = et[b].max(axis=1) / T
        emax_d = ed[b].max(axis=1) / Td if g else None
        for i in range(min(j + 1, g)):
            x = int(tok[b, i])
            dp = et[b, i, x] / T + emax_t[i]
            dq = ed[b, i, x] / Td + emax_d[i]
            la = np.log(r.a[b, i]) if r.a[b, i] > 0 else -np.inf
            lo, hi = np.exp(la - dp - dq), np.exp(la + dp + dq)
            if lo - 1e-5 <= r.u[b, i] <= hi + 1e-5:
                flagged[b] = True
        if r.flags[b] & oracle.FLAG_RESIDUAL_EMPTY:  # the race fell back to p_j
            flagged[b] = True
            continue
        row = j
        lp = lt[b, row].astype(np.float64) / T - r.logZp[b, row]
        dp = et[b, row] / T + emax_t[row]
        lnE = np.log(orc.race_exponentials(seed, b, row, V))
        p_lo, p_hi = np.exp(lp - dp), np.exp(lp + dp)
        if j < g:
            lq = ld[b, row].astype(np.float64) / Td - r.logZq[b, row]
            dq = ed[b, row] / Td + emax_d[row]
            w_lo = np.maximum(0.0, p_lo - np.exp(lq + dq))
            w_hi = np.maximum(0.0, p_hi - np.exp(lq - dq))
        else:
            w_lo, w_hi = p_lo, p_hi
        with np.errstate(divide="ignore"):
            s_lo, s_hi = np.log(w_lo) - lnE, np.log(w_hi) - lnE
        y = int(r.tokens[b, j])
        others = np.delete(s_hi, y)
        if others.size and others.max() >= s_lo[y] - 1e-6:
            flagged[b] = True
    return flagged


@pytest.mark.parametrize("B,gamma,V,d,T,Td", [(4, 3, 4096, 128, 1.0, 0.5), (8, 5, 10000, 256, 0.8, 0.4),
                                               (3, 0, 2048, 64, 1.0, 1.0), (64, 8, 32000, 256, 1.0, 0.5),
                                               (8, 4, 50257, 1024, 1.0, 0.6),
                                               # the race's hidden states need 64 KB of shared memory
                                               (4, 2, 3001, 16384, 1.0, 0.8)])
def test_verify_from_hidden_states_matches_oracle(sv, B, gamma, V, d, T, Td):
    """The verify from hidden states against the oracle run on logits computed on the host
    (fp64 products of the same bf16 inputs, rounded to fp32), independent of the library's
    GEMM.  Tokens and counts must match except in sequences where the GEMM's error bound
    could move a decision (those must still be valid cycles); and the logits path run on the
    tensor cores' logits must give the fused path's tokens outside those sequences (the fused
    race scores its candidates with logits recomputed by dot products, equal to the GEMM's
    within the same error bound)."""
    ht, wt, hd, wd = lmhead_workload(B, gamma, V, d, seed=B * 100 + V)
    dev = torch.device("cuda")
    Ht, Wt, Hd, Wd = (to_dev(a) for a in (ht, wt, hd, wd))
    lt, et = host_logits(ht.reshape(B * (gamma + 1), d), wt)
    lt, et = lt.reshape(B, gamma + 1, V), et.reshape(B, gamma + 1, V)
    if gamma:
        ld, ed = host_logits(hd.reshape(B * gamma, d), wd)
        ld, ed = ld.reshape(B, gamma, V), ed.reshape(B, gamma, V)
    else:
        ld, ed = np.zeros((B, 0, V), np.float32), np.zeros((B, 0, V))
    rng = np.random.default_rng(7)
    tok = np.zeros((B, gamma), np.int32)
    for b in range(B):
        if gamma:
            tok[b] = workloads.draw_drafts(rng, ld[b], Td)
    dtok = torch.from_numpy(tok).to(dev)
    Tv, Tdv = np.full(B, T, np.float32), np.full(B, Td, np.float32)
    orc = oracle.get()
    # the logits path on the tensor cores' own logits (consistency of the fused path)
    lt_gpu = sv.spec_lmhead_logits(Ht.reshape(B * (gamma + 1), d), Wt).reshape(B, gamma + 1, V)
    ld_gpu = (sv.spec_lmhead_logits(Hd.reshape(B * gamma, d), Wd).reshape(B, gamma, V) if gamma
              else torch.empty((B, 0, V), dtype=torch.float32, device=dev))
    n_flagged = n_seq = 0
    for seed in range(3):
        t, n = sv.spec_verify_lmhead(Ht, Wt, Hd if gamma else None, Wd if gamma else None, dtok, T, Td, seed)
        torch.cuda.synchronize()
        assert sv.spec_verify_check() == sv.SPEC_OK
        gt, gn = t.cpu().numpy(), n.cpu().numpy()
        r = orc.verify(lt, ld, tok, Tv, Tdv, seed)
        flagged = gemm_sensitive(orc, lt, et, ld, ed, tok, T, Td, seed, r)
        n_flagged += int(flagged.sum())
        n_seq += B
        for b in range(B):
            j = int(gn[b])
            assert 0 <= j <= gamma and 0 <= gt[b, j] < V and np.all(gt[b, j + 1:] == -1)
            if flagged[b]:
                continue
            assert j == r.n_accepted[b], (seed, b, j, r.n_accepted[b])
            np.testing.assert_array_equal(gt[b], r.tokens[b], err_msg=f"seed {seed} sequence {b}")
        tl, nl, _ = sv.spec_verify_ex(lt_gpu, ld_gpu, dtok, T, Td, seed)
        torch.cuda.synchronize()
        ok = ~flagged
        np.testing.assert_array_equal(nl.cpu().numpy()[ok], gn[ok])
        np.testing.assert_array_equal(tl.cpu().numpy()[ok], gt[ok])
    # the bound is loose (worst-case accumulation error): most decisions still compare
    assert n_flagged <= max(2, 0.1 * n_seq), (n_flagged, n_seq)


@pytest.mark.parametrize("B,gamma,V,d,T,Td", [(64, 8, 32000, 256, 1.0, 0.5), (8, 4, 50257, 1024, 1.0, 0.6)])
def test_race_again_gives_the_same_tokens(sv, B, gamma, V, d, T, Td):
    """The race's starting score is a guess the winner almost always beats; when it does
    not, the sequence is raced again from the best score found.  With the guess forced above
    every winner, every sequence takes that path: the tokens must not change."""
    ht, wt, hd, wd = lmhead_workload(B, gamma, V, d, seed=B * 100 + V + 1)
    Ht, Wt, Hd, Wd = (to_dev(a) for a in (ht, wt, hd, wd))
    ld = host_logits(hd.reshape(B * gamma, d), wd)[0].reshape(B, gamma, V)
    rng = np.random.default_rng(11)
    tok = torch.from_numpy(np.stack([workloads.draw_drafts(rng, ld[b], Td) for b in range(B)])
                           .astype(np.int32)).to(Ht.device)
    for seed in range(3):
        t0, n0 = sv.spec_verify_lmhead(Ht, Wt, Hd, Wd, tok, T, Td, seed)
        t1, n1 = sv.spec_verify_lmhead(Ht, Wt, Hd, Wd, tok, T, Td, seed, flags=sv.SPEC_DEBUG_RACE_AGAIN)
        torch.cuda.synchronize()
        assert sv.spec_verify_check() == sv.SPEC_OK
        np.testing.assert_array_equal(n1.cpu().numpy(), n0.cpu().numpy())
        np.testing.assert_array_equal(t1.cpu().numpy(), t0.cpu().numpy())


N_LM_CASES = int(os.environ.get("SPECVERIFY_LM_FUZZ_CASES", "6"))


@pytest.mark.parametrize("case", range(N_LM_CASES))
def test_random_lmhead_shapes(sv, case):
    """Seeded random shapes of the verify from hidden states (batch, draft length, odd and
    even vocabularies, hidden sizes, temperatures) against the oracle on host fp64 logits,
    outside the sequences the GEMM's error bound could move."""
    rng = np.random.default_rng(31_000 + case)
    B = int(rng.integers(1, 13))
    gamma = int(rng.choice([0, 1, 3, 6]))
    V = int(rng.integers(64, 40_000))
    d = int(rng.choice([64, 128, 256, 512]))
    T = float(rng.uniform(0.6, 1.5))
    Td = float(T * rng.uniform(0.5, 1.0))
    ht, wt, hd, wd = lmhead_workload(B, gamma, V, d, seed=case)
    Ht, Wt, Hd, Wd = (to_dev(a) for a in (ht, wt, hd, wd))
    lt, et = host_logits(ht.reshape(B * (gamma + 1), d), wt)
    lt, et = lt.reshape(B, gamma + 1, V), et.reshape(B, gamma + 1, V)
    if gamma:
        ld, ed = host_logits(hd.reshape(B * gamma, d), wd)
        ld, ed = ld.reshape(B, gamma, V), ed.reshape(B, gamma, V)
    else:
        ld, ed = np.zeros((B, 0, V), np.float32), np.zeros((B, 0, V))
    tok = np.zeros((B, gamma), np.int32)
    for b in range(B):
        if gamma:
            tok[b] = workloads.draw_drafts(rng, ld[b], Td)
    orc = oracle.get()
    seed = int(rng.integers(0, 1 << 31))
    t, n = sv.spec_verify_lmhead(Ht, Wt, Hd if gamma else None, Wd if gamma else None,
                                 torch.from_numpy(tok).to(Ht.device), T, Td, seed)
    torch.cuda.synchronize()
    assert sv.spec_verify_check() == sv.SPEC_OK
    gt, gn = t.cpu().numpy(), n.cpu().numpy()
    r = orc.verify(lt, ld, tok, np.full(B, T, np.float32), np.full(B, Td, np.float32), seed)
    flagged = gemm_sensitive(orc, lt, et, ld, ed, tok, T, Td, seed, r)
    for b in range(B):
        j = int(gn[b])
        assert 0 <= j <= gamma and 0 <= gt[b, j] < V and np.all(gt[b, j + 1:] == -1)
        if flagged[b]:
            continue
        assert j == r.n_accepted[b], (case, b, j, r.n_accepted[b])
        np.testing.assert_array_equal(gt[b], r.tokens[b], err_msg=f"case {case} sequence {b}")
