"""The LM head on the tensor cores (marked gpu): logits against an fp64 product of the
same bf16 inputs, and the statistics epilogue (ln Z, ln p(token)) against the oracle's fp64
softmax of those logits.

Tolerance: bf16 x bf16 products are exact in fp32; the tensor cores add d of them in fp32,
so a logit carries an absolute error of a few times 2^-24 * sum |h_k w_k| (the tests allow
2e-5 * that sum + 1e-5); ln Z and ln p inherit the logits' error divided by T, plus the fp32
softmax sum's own (allowed: 1e-4 absolute at these sizes).
"""
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


@pytest.mark.parametrize("B,gamma,V,d,T,Td", [(4, 3, 4096, 128, 1.0, 0.5), (8, 5, 10000, 256, 0.8, 0.4),
                                               (3, 0, 2048, 64, 1.0, 1.0), (64, 8, 32000, 256, 1.0, 0.5)])
def test_verify_from_hidden_states_matches_oracle(sv, B, gamma, V, d, T, Td):
    """The fused verify equals the oracle run on the logits the tensor cores compute (the
    same GEMM: spec_lmhead_logits) under the usual parity rules, and the logits path on
    those logits."""
    from _parity import compare_sampling
    ht, wt, hd, wd = lmhead_workload(B, gamma, V, d, seed=B * 100 + V)
    dev = torch.device("cuda")
    Ht, Wt, Hd, Wd = (to_dev(a) for a in (ht, wt, hd, wd))
    lt = sv.spec_lmhead_logits(Ht.reshape(B * (gamma + 1), d), Wt).reshape(B, gamma + 1, V)
    ld = (sv.spec_lmhead_logits(Hd.reshape(B * gamma, d), Wd).reshape(B, gamma, V) if gamma
          else torch.empty((B, 0, V), dtype=torch.float32, device=dev))
    torch.cuda.synchronize()
    lt_np, ld_np = lt.cpu().numpy(), ld.cpu().numpy()
    rng = np.random.default_rng(7)
    tok = np.zeros((B, gamma), np.int32)
    for b in range(B):
        if gamma:
            tok[b] = workloads.draw_drafts(rng, ld_np[b], Td)
    dtok = torch.from_numpy(tok).to(dev)
    w = workloads.Workload("lmhead", B, gamma, V, "f32", lt_np, ld_np, tok,
                           np.full(B, T, np.float32), np.full(B, Td, np.float32))
    orc = oracle.get()
    for seed in range(3):
        t, n = sv.spec_verify_lmhead(Ht, Wt, Hd if gamma else None, Wd if gamma else None, dtok, T, Td, seed)
        torch.cuda.synchronize()
        assert sv.spec_verify_check() == sv.SPEC_OK
        g = {"tokens": t.cpu().numpy(), "n": n.cpu().numpy()}
        compare_sampling(w, g, orc.verify(lt_np, ld_np, tok, w.T, w.Td, seed))
