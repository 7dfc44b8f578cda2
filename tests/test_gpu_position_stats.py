"""GPU parity of the per-position statistics and the adaptive draft length (marked gpu).

H(p_i), H(q_i) and KL(p_i || q_i) from the paired streaming pass are compared with the
oracle's fp64 values within a tolerance derived from the fp32 arithmetic (below); the
class-centre update and the k* rule are compared bit for bit with the oracle run on the
same fp32 entropies (both sides compute them in fp64, each operation rounded on its own,
in the same order).  The verify outputs of a call that also asks for the statistics follow
the usual parity rules.

Tolerance: an entropy is ln 2 (log2 s - A / s) with s and A summed in fp32 over V terms in
a tree (per lane, then across lanes and pieces): the relative error of each sum is a few
times 1e-7, so log2 s and A / s carry absolute errors of about 1e-6 times their size plus
a few 1e-7; KL adds the draft terms.  The tests allow 3e-5 + 2e-5 |value|.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from _parity import DeviceWorkload, compare_sampling

pytestmark = pytest.mark.gpu

ATOL, RTOL = 3e-5, 2e-5


@pytest.fixture(scope="module")
def sv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_31_gb300 as m
    m.load_library()
    return m


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


def close(got, want, what):
    got = np.asarray(got, np.float64)
    fin = np.isfinite(want)
    assert np.array_equal(np.isfinite(got), fin), what
    assert np.array_equal(got[~fin], want[~fin]), what
    err = np.abs(got[fin] - want[fin]) - (ATOL + RTOL * np.abs(want[fin]))
    assert err.size == 0 or err.max() <= 0, (what, float(err.max()))


SHAPES = [
    # B, gamma, V, dtype, T, Td
    (2, 4, 5003, "bf16", 1.0, 1.0),
    (3, 3, 9000, "f32", 0.6, 0.2),
    (4, 0, 777, "bf16", 0.8, 0.8),
    (2, 6, 20000, "bf16", 1.3, 0.4),
    (5, 2, 7, "f32", 1.0, 0.5),
]


@pytest.mark.parametrize("B,gamma,V,dtype,T,Td", SHAPES)
def test_position_stats_match_oracle(sv, orc, B, gamma, V, dtype, T, Td):
    w = workloads.generic(B=B, gamma=gamma, V=V, dtype=dtype, seed=V + gamma, sigma=0.8, T=T, Td=Td)
    dw = DeviceWorkload(w)
    for seed in range(2):
        t, n, d = sv.spec_verify_ex(dw.target, dw.draft, dw.tokens, T, Td, seed,
                                    diagnostics=True, position_stats=True)
        torch.cuda.synchronize()
        hp, hq, kl = orc.position_stats(w.target, w.draft, w.T, w.Td)
        close(d["Hp"].cpu().numpy(), hp, "H_p")
        if gamma:
            close(d["Hq"].cpu().numpy(), hq, "H_q")
            close(d["KL"].cpu().numpy(), kl, "KL")
        g = {k: v.cpu().numpy() for k, v in d.items()}
        g.update(tokens=t.cpu().numpy(), n=n.cpu().numpy())
        compare_sampling(w, g, orc.verify(w.target, w.draft, w.tokens, w.T, w.Td, seed))
    assert sv.spec_verify_check() == sv.SPEC_OK


def test_position_stats_per_sequence_temperatures_and_centres(sv, orc):
    """Per-sequence temperatures; the class centres move exactly as the oracle's update
    moves them with the same entropies and accepted counts."""
    w = workloads.generic(B=6, gamma=5, V=6001, dtype="bf16", seed=3, sigma=0.5)
    rng = np.random.default_rng(2)
    w.T[:] = rng.uniform(0.3, 1.2, size=w.B)
    w.Td[:] = 0.5 * w.T
    dw = DeviceWorkload(w)
    c0 = np.stack([rng.uniform(0, 2, w.B), rng.uniform(2, 4, w.B)], axis=1)
    centres = torch.from_numpy(c0.copy()).cuda()
    want_c = c0.copy()
    for seed in range(4):
        t, n, d = sv.spec_verify_ex(dw.target, dw.draft, dw.tokens, 1.0, 1.0, seed,
                                    T_per_seq=dw.T, Td_per_seq=dw.Td, position_stats=True,
                                    ctrl_centres=centres, ctrl_beta=0.25)
        torch.cuda.synchronize()
        hq_gpu = d["Hq"].cpu().numpy().astype(np.float64)
        want_c = orc.entropy_centres_update(hq_gpu, n.cpu().numpy(), 0.25, want_c)
        np.testing.assert_array_equal(centres.cpu().numpy(), want_c)
        hp, hq, kl = orc.position_stats(w.target, w.draft, w.T, w.Td)
        close(hq_gpu, hq, "H_q")
        close(d["KL"].cpu().numpy(), kl, "KL")
        r = orc.verify(w.target, w.draft, w.tokens, w.T, w.Td, seed)
        compare_sampling(w, {"tokens": t.cpu().numpy(), "n": n.cpu().numpy()}, r)


def test_position_stats_degenerate_rows(sv, orc):
    """One-hot draft rows (entropy 0, KL = -ln p(d)); draft = target at the same temperature
    (KL 0, equal entropies); a draft row that misses part of p's support (KL = +inf)."""
    V, g = 3000, 3
    w = workloads.generic(B=3, gamma=g, V=V, dtype="f32", seed=8, T=0.9, Td=0.9)
    draft = w.draft.copy()
    draft[0] = -np.inf
    for i in range(g):
        draft[0, i, w.tokens[0, i]] = 0.0
    draft[1] = w.target[1, :g]
    draft[2, :, :10] = -np.inf
    w2 = workloads.Workload("degenerate", 3, g, V, "f32", w.target, draft, w.tokens, w.T, w.Td)
    dw = DeviceWorkload(w2)
    _, _, d = sv.spec_verify_ex(dw.target, dw.draft, dw.tokens, 0.9, 0.9, 0, position_stats=True)
    torch.cuda.synchronize()
    hp, hq, kl = orc.position_stats(w2.target, w2.draft, w2.T, w2.Td)
    close(d["Hq"].cpu().numpy(), hq, "H_q")
    close(d["KL"].cpu().numpy(), kl, "KL")
    close(d["Hp"].cpu().numpy(), hp, "H_p")
    assert np.all(d["Hq"].cpu().numpy()[0] == 0.0)
    assert np.all(np.isinf(d["KL"].cpu().numpy()[2]))


def test_position_stats_throughput_workload_sampled(sv, orc):
    """B=256, gamma=12, V=152064: every position of 16 sampled sequences."""
    w = workloads.config(4)
    dw = DeviceWorkload(w)
    _, _, d = sv.spec_verify_ex(dw.target, dw.draft, dw.tokens, float(w.T[0]), float(w.Td[0]), 0,
                                position_stats=True)
    torch.cuda.synchronize()
    idx = np.sort(np.random.default_rng(4).choice(w.B, size=16, replace=False))
    sub = w.subset(idx)
    hp, hq, kl = orc.position_stats(sub.target, sub.draft, sub.T, sub.Td)
    close(d["Hp"].cpu().numpy()[idx], hp, "H_p")
    close(d["Hq"].cpu().numpy()[idx], hq, "H_q")
    close(d["KL"].cpu().numpy()[idx], kl, "KL")


@pytest.mark.parametrize("dtype,V,T", [("bf16", 128256, 1.0), ("f32", 5003, 0.3), ("bf16", 9, 2.0)])
def test_row_entropy_matches_oracle(sv, orc, dtype, V, T):
    rng = np.random.default_rng(V)
    x = (rng.standard_normal((7, V)) * 3).astype(np.float32)
    rows = workloads.to_bf16_bits(x) if dtype == "bf16" else x
    dev = torch.device("cuda")
    if dtype == "bf16":
        t = torch.from_numpy(rows.view(np.int16)).to(dev).view(torch.bfloat16)
    else:
        t = torch.from_numpy(rows).to(dev)
    h = sv.spec_row_entropy(t, T)
    torch.cuda.synchronize()
    close(h.cpu().numpy(), orc.row_entropies(rows, T), "row entropy")


def test_adaptive_k_bit_exact(sv, orc):
    rng = np.random.default_rng(9)
    B, K = 300, 24
    H = rng.uniform(0.0, 4.0, size=(B, K)).astype(np.float32)
    H[:50] = np.sort(H[:50], axis=1)              # confidence falling along the draft
    H[50:60] = 1.5                                # equal distances for some
    centres = np.stack([rng.uniform(0.2, 1.5, B), rng.uniform(1.5, 3.5, B)], axis=1)
    centres[60:70] = 1.5                          # coinciding centres
    cand = [1, 2, 3, 4, 6, 8, 11, 12, 16, 20, 24]
    for Cd, Cv in ((0.2, 1.0), (0.7, 1.0), (0.05, 0.5)):
        k, eff = sv.spec_adaptive_k(torch.from_numpy(H).cuda(), torch.from_numpy(centres).cuda(),
                                    cand, Cd, Cv)
        torch.cuda.synchronize()
        wk, weff = orc.adaptive_k(H.astype(np.float64), centres, np.array(cand, np.int32), Cd, Cv)
        np.testing.assert_array_equal(k.cpu().numpy(), wk)
        np.testing.assert_array_equal(eff.cpu().numpy(), weff)


def test_controller_argument_checks(sv):
    dev = torch.device("cuda")
    H = torch.zeros((2, 4), dtype=torch.float32, device=dev)
    c = torch.zeros((2, 2), dtype=torch.float64, device=dev)
    for cand, Cd, Cv in (([0, 2], 0.1, 1.0), ([5], 0.1, 1.0), ([2], float("nan"), 1.0),
                         ([2], -1.0, 1.0), (list(range(1, 5)) * 17, 0.1, 1.0)):
        with pytest.raises(sv.SpecVerifyError) as e:
            sv.spec_adaptive_k(H, c, cand, Cd, Cv)
        assert e.value.code == sv.SPEC_EINVAL
    w = workloads.generic(B=2, gamma=3, V=64, dtype="bf16", seed=1)
    dw = DeviceWorkload(w)
    for beta in (0.0, 1.5, float("nan")):
        with pytest.raises(sv.SpecVerifyError) as e:
            sv.spec_verify_ex(dw.target, dw.draft, dw.tokens, 1.0, 1.0, 0, ctrl_centres=c,
                              ctrl_beta=beta)
        assert e.value.code == sv.SPEC_EINVAL
    with pytest.raises(sv.SpecVerifyError) as e:
        sv.spec_row_entropy(torch.zeros((3, 10), dtype=torch.bfloat16, device=dev), 0.0)
    assert e.value.code == sv.SPEC_EINVAL
