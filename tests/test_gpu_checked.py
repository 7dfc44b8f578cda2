"""The index-checked build, libspecverify_checked.so (marked gpu).

It is the library compiled with SPECVERIFY_CHECKED: the sampling (default and early-exit)
and greedy kernels test every computed index into the logits, tokens, outputs and workspace
regions before the access, and record SPEC_EINDEX instead of making it.  Here the small
ragged shapes of the parity and early-exit suites run through it: every call must finish
with the status word clear (no index left its buffer) and give the oracle's results.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from _parity import DeviceWorkload, compare_greedy, compare_sampling, run_gpu

pytestmark = pytest.mark.gpu

SHAPES = [
    # B, gamma, V, dtype, draft noise
    (1, 5, 1024, "f32", 0.5),
    (3, 4, 5003, "bf16", 0.3),
    (2, 7, 9000, "f32", 0.2),
    (4, 0, 777, "bf16", 1.0),
    (2, 3, 1, "f32", 1.0),
    (5, 2, 7, "bf16", 0.5),
    (2, 6, 20000, "bf16", 0.7),
    (1, 1, 4100, "f32", 0.7),
    (8, 8, 20000, "bf16", 0.1),
    (3, 48, 2500, "bf16", 0.01),
    (33, 6, 12000, "bf16", 1.2),
    (24, 8, 128257, "bf16", 0.8),
]


@pytest.fixture(scope="module")
def sv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_31_gb300 as m
    m.specverify.use_library(m.specverify.CHECKED_LIB_PATH)
    yield m
    m.specverify.use_library(m.specverify.LIB_PATH)


@pytest.mark.parametrize("B,gamma,V,dtype,sigma", SHAPES)
def test_checked_build_sampling_early_exit_and_greedy(sv, B, gamma, V, dtype, sigma):
    orc = oracle.get()
    w = workloads.generic(B=B, gamma=gamma, V=V, dtype=dtype, seed=B * 13 + V + gamma,
                          sigma=sigma, T=0.9, Td=0.45)
    dw = DeviceWorkload(w)
    for seed in range(2):
        r = orc.verify(w.target, w.draft, w.tokens, w.T, w.Td, seed)
        for flags in (0, sv.SPEC_FLAG_EARLY_EXIT):
            g = run_gpu(sv, dw, seed, per_seq_temps=(seed == 1), diagnostics=(flags == 0),
                        flags=flags)
            assert sv.spec_verify_check() == sv.SPEC_OK, (seed, flags)
            compare_sampling(w, g, r, check_values=(flags == 0), count=False)
    wg = workloads.generic(B=B, gamma=gamma, V=V, dtype=dtype, seed=B + V, greedy=True)
    dg = DeviceWorkload(wg)
    t, n = sv.spec_verify_greedy_ex(dg.target, dg.tokens)
    assert sv.spec_verify_check() == sv.SPEC_OK
    rt, rn, _ = orc.verify_greedy(wg.target, wg.tokens)
    compare_greedy(t.cpu().numpy(), n.cpu().numpy(), rt, rn)


def test_checked_build_bad_tokens_still_reported(sv):
    """A draft token outside [0, V) is the input error it always was (SPEC_EBADTOKEN), found
    before any gather at that index is made."""
    w = workloads.generic(B=4, gamma=3, V=500, dtype="bf16", seed=6)
    tok = w.tokens.copy()
    tok[1, 1] = 500
    tok[3, 0] = -1
    dw = DeviceWorkload(w)
    dtok = torch.from_numpy(tok).cuda()
    for flags in (0, sv.SPEC_FLAG_EARLY_EXIT):
        t, n, _ = sv.spec_verify_ex(dw.target, dw.draft, dtok, 1.0, 1.0, 3, flags=flags)
        assert sv.spec_verify_check() == sv.SPEC_EBADTOKEN
        got = n.cpu().numpy()
        assert got[1] == -1 and got[3] == -1


@pytest.mark.parametrize("cfg", [3, 4])
def test_checked_build_named_batched_workloads_full_size(sv, cfg):
    """The batched-serving and throughput workloads at full size through the checked build:
    no index leaves its buffer, and the tokens are the normal build's, on the full read,
    the early-exit path and in greedy mode."""
    w = workloads.config(cfg)
    dw = DeviceWorkload(w)
    results = {}
    for lib in (sv.specverify.CHECKED_LIB_PATH, sv.specverify.LIB_PATH):
        sv.specverify.use_library(lib)
        for flags in (0, sv.SPEC_FLAG_EARLY_EXIT):
            g = run_gpu(sv, dw, 7, per_seq_temps=(cfg == 3), diagnostics=False, flags=flags)
            assert sv.spec_verify_check() == sv.SPEC_OK, (lib, flags)
            results[(lib, flags)] = g
    sv.specverify.use_library(sv.specverify.CHECKED_LIB_PATH)
    for flags in (0, sv.SPEC_FLAG_EARLY_EXIT):
        a = results[(sv.specverify.CHECKED_LIB_PATH, flags)]
        b = results[(sv.specverify.LIB_PATH, flags)]
        np.testing.assert_array_equal(a["tokens"], b["tokens"])
        np.testing.assert_array_equal(a["n"], b["n"])
    wg = workloads.config(cfg, greedy=True)
    dg = DeviceWorkload(wg)
    t, n = sv.spec_verify_greedy_ex(dg.target, dg.tokens)
    assert sv.spec_verify_check() == sv.SPEC_OK
    rt, rn, _ = oracle.get().verify_greedy(wg.target, wg.tokens)
    compare_greedy(t.cpu().numpy(), n.cpu().numpy(), rt, rn)


def test_checked_build_token_trees(sv):
    """Token-tree verifies (random trees with ragged rows, and SubSpec's depth-48 tree at
    V = 152064) through the checked build: status clear, and the normal build's tokens."""
    from _parity import to_device
    rng = np.random.default_rng(4)
    cases = [workloads.tree(workloads.random_tree(rng, 20, 4), B=5, V=4099, dtype="bf16", seed=8,
                            scale=3.0, sigma=0.6, T=0.9, Td=0.45),
             workloads.tree(workloads.deep_narrow_tree(48, 6), B=2, V=152064, dtype="bf16",
                            seed=1005, scale=5.0, sigma=workloads.DEEP_CHAIN_SIGMA, T=0.6, Td=0.2)]
    dev = torch.device("cuda")
    for w in cases:
        t = to_device(w.target, w.dtype, dev)
        d = to_device(w.draft, w.dtype, dev)
        tok = torch.from_numpy(np.ascontiguousarray(w.tokens)).to(dev)
        outs = []
        for lib in (sv.specverify.CHECKED_LIB_PATH, sv.specverify.LIB_PATH):
            sv.specverify.use_library(lib)
            for seed in range(2):
                o = sv.spec_verify_tree(t, d, tok, w.parent, float(w.T[0]), float(w.Td[0]), seed)
                assert sv.spec_verify_check() == sv.SPEC_OK
                outs.append([x.cpu().numpy() for x in o])
        sv.specverify.use_library(sv.specverify.CHECKED_LIB_PATH)
        for a, b in zip(outs[:2], outs[2:]):
            for x, y in zip(a, b):
                np.testing.assert_array_equal(x, y)



def test_checked_build_verify_from_hidden_states(sv):
    """The verify from hidden states through the index-checked build (its race publishes
    each block's winner through the checked slot index): the status word stays clear and
    the tokens equal the normal build's, including the forced second race."""
    from test_gpu_lmhead import host_logits, lmhead_workload, to_dev
    B, gamma, V, d = 6, 4, 10001, 256
    ht, wt, hd, wd = lmhead_workload(B, gamma, V, d, seed=5)
    Ht, Wt, Hd, Wd = (to_dev(a) for a in (ht, wt, hd, wd))
    ld = host_logits(hd.reshape(B * gamma, d), wd)[0].reshape(B, gamma, V)
    rng = np.random.default_rng(3)
    tok = torch.from_numpy(np.stack([workloads.draw_drafts(rng, ld[b], 0.6) for b in range(B)])
                           .astype(np.int32)).to(Ht.device)
    got = []
    for path in (sv.specverify.CHECKED_LIB_PATH, sv.specverify.LIB_PATH):
        sv.specverify.use_library(path)
        for flags in (0, sv.SPEC_DEBUG_RACE_AGAIN):
            t, n = sv.spec_verify_lmhead(Ht, Wt, Hd, Wd, tok, 0.9, 0.6, 17, flags=flags)
            torch.cuda.synchronize()
            assert sv.spec_verify_check() == sv.SPEC_OK, (path, flags)
            got.append((t.cpu().numpy(), n.cpu().numpy()))
    sv.specverify.use_library(sv.specverify.CHECKED_LIB_PATH)
    for t, n in got[1:]:
        np.testing.assert_array_equal(n, got[0][1])
        np.testing.assert_array_equal(t, got[0][0])
