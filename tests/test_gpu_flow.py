"""The flow schedule (SPEC_FLAG_FUSED; marked gpu): one persistent launch whose scans and
races run while later sequences are still being streamed.  It computes what the default
two-kernel schedule computes with the same arithmetic in the same order, so its outputs are
compared with the default path's bit for bit, and with the oracle.

Shapes cover several race units per raced row, gamma above 32 (the scan merges and decides
positions 32 at a time), gamma = 0, unaligned fp32 rows, tiny vocabularies, bad draft
tokens, a caller workspace full of garbage, and calls of different shapes back to back (the
flow region must be clean at every call).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from _parity import DeviceWorkload, compare_sampling, run_gpu

pytestmark = pytest.mark.gpu


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


DIAG = ("logp", "logq", "logZp", "logZq", "u")


def assert_same(flow: dict, base: dict, diag=True):
    np.testing.assert_array_equal(flow["n"], base["n"])
    np.testing.assert_array_equal(flow["tokens"], base["tokens"])
    if diag:
        for k in DIAG:
            np.testing.assert_array_equal(flow[k], base[k], err_msg=k)
        np.testing.assert_array_equal(flow["race"][:, 0], base["race"][:, 0])


SHAPES = [
    # B, gamma, V, dtype
    (3, 4, 5003, "bf16"),     # unaligned bf16 rows
    (2, 7, 9000, "f32"),
    (4, 0, 777, "bf16"),      # bonus token only
    (5, 2, 7, "bf16"),        # V below one vector
    (2, 3, 1, "f32"),         # V = 1
    (2, 40, 3001, "f32"),     # gamma > 32: two scan chunks; unaligned fp32 rows
    (3, 33, 8192, "bf16"),    # gamma = 33, one race unit exactly
    (40, 3, 20000, "bf16"),   # many sequences, three race units each
    (2, 5, 40000, "f32"),     # five race units, fp32
]


@pytest.mark.parametrize("B,gamma,V,dtype", SHAPES)
def test_flow_matches_default_bitwise_and_oracle(sv, orc, B, gamma, V, dtype):
    w = workloads.generic(B=B, gamma=gamma, V=V, dtype=dtype, seed=B * 77 + gamma * 13 + V,
                          sigma=0.8, T=0.9, Td=0.45)
    dw = DeviceWorkload(w)
    for seed in (0, 5):
        base = run_gpu(sv, dw, seed)
        flow = run_gpu(sv, dw, seed, flags=sv.SPEC_FLAG_FUSED)
        assert_same(flow, base)
        compare_sampling(w, flow, orc.verify(w.target, w.draft, w.tokens, w.T, w.Td, seed))
        # without diagnostics the scan stops merging rows after the first rejection
        bare = run_gpu(sv, dw, seed, diagnostics=False, flags=sv.SPEC_FLAG_FUSED)
        assert_same(bare, base, diag=False)
    assert sv.spec_verify_check() == sv.SPEC_OK


@pytest.mark.parametrize("cfg,B", [(3, 16), (4, 6), (2, 1), (1, 1), (0, 1)])
def test_flow_on_named_workloads(sv, orc, cfg, B):
    """The named workloads' shapes (their first B sequences): per-sequence temperatures,
    heavy-tailed rows, deep chains, 16 to 19 race units per raced row."""
    w = workloads.config(cfg, B=B)
    dw = DeviceWorkload(w)
    seed = 1234
    base = run_gpu(sv, dw, seed)
    flow = run_gpu(sv, dw, seed, flags=sv.SPEC_FLAG_FUSED)
    assert_same(flow, base)
    compare_sampling(w, flow, orc.verify(w.target, w.draft, w.tokens, w.T, w.Td, seed))
    assert sv.spec_verify_check() == sv.SPEC_OK


def test_flow_full_throughput_workload_matches_default(sv):
    """The throughput workload at full size (B=256, gamma=12, V=152064) in the launch
    configuration the benchmark times: flow and default outputs agree bit for bit."""
    w = workloads.config(4)
    dw = DeviceWorkload(w)
    for seed in (0, 99):
        base = run_gpu(sv, dw, seed)
        flow = run_gpu(sv, dw, seed, flags=sv.SPEC_FLAG_FUSED)
        assert_same(flow, base)
    assert sv.spec_verify_check() == sv.SPEC_OK


def test_flow_calls_of_different_shapes_back_to_back(sv, orc):
    """The flow region is zeroed for every call: alternating shapes (whose regions overlap
    differently) and the default path in between leave no trace."""
    ws = [workloads.generic(B=6, gamma=5, V=12000, dtype="bf16", seed=1, sigma=0.7),
          workloads.generic(B=2, gamma=20, V=30001, dtype="bf16", seed=2, sigma=0.7),
          workloads.generic(B=9, gamma=1, V=5000, dtype="f32", seed=3, sigma=0.7)]
    dws = [DeviceWorkload(w) for w in ws]
    for rep in range(3):
        for k, (w, dw) in enumerate(zip(ws, dws)):
            seed = rep * 10 + k
            flow = run_gpu(sv, dw, seed, flags=sv.SPEC_FLAG_FUSED)
            base = run_gpu(sv, dw, seed)
            assert_same(flow, base)
            if rep == 0:
                compare_sampling(w, flow, orc.verify(w.target, w.draft, w.tokens, w.T, w.Td, seed))
    assert sv.spec_verify_check() == sv.SPEC_OK


def test_flow_with_a_garbage_caller_workspace(sv):
    w = workloads.generic(B=7, gamma=6, V=10007, dtype="bf16", seed=11, sigma=0.9)
    dw = DeviceWorkload(w)
    need = sv.spec_verify_workspace_bytes(w.B, w.gamma, w.V, sv.SPEC_BF16)
    ws = torch.full((need,), 0xAB, dtype=torch.uint8, device="cuda")
    base = run_gpu(sv, dw, 3)
    for _ in range(2):
        t, n, d = sv.spec_verify_ex(dw.target, dw.draft, dw.tokens, float(w.T[0]), float(w.Td[0]), 3,
                                    T_per_seq=dw.T, Td_per_seq=dw.Td, workspace=ws,
                                    diagnostics=True, flags=sv.SPEC_FLAG_FUSED)
        torch.cuda.synchronize()
        flow = {k: v.cpu().numpy() for k, v in d.items()}
        flow.update(tokens=t.cpu().numpy(), n=n.cpu().numpy())
        assert_same(flow, base)
    assert sv.spec_verify_check() == sv.SPEC_OK


def test_flow_bad_draft_tokens(sv, orc):
    w = workloads.generic(B=4, gamma=5, V=3000, dtype="bf16", seed=12)
    tok = w.tokens.copy()
    tok[1, 3] = w.V        # out of range
    tok[3, 0] = -1
    dw = DeviceWorkload(w)
    dw.tokens = torch.from_numpy(tok).cuda()
    flow = run_gpu(sv, dw, 0, flags=sv.SPEC_FLAG_FUSED)
    assert sv.spec_verify_check() == sv.SPEC_EBADTOKEN
    base = run_gpu(sv, dw, 0)
    assert sv.spec_verify_check() == sv.SPEC_EBADTOKEN
    assert_same(flow, base)
    assert flow["n"][1] == -1 and flow["n"][3] == -1
    assert np.all(flow["tokens"][1] == -1) and np.all(flow["tokens"][3] == -1)
    r = orc.verify(w.target, w.draft, tok, w.T, w.Td, 0)
    for b in (0, 2):
        if not (r.flags[b] & (oracle.FLAG_ACCEPT_NEAR_TIE | oracle.FLAG_RACE_NEAR_TIE)):
            assert flow["n"][b] == r.n_accepted[b]
            np.testing.assert_array_equal(flow["tokens"][b], r.tokens[b])
