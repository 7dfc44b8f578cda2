"""GPU parity of token-tree verification (spec_verify_tree) against the oracle (marked gpu).

Tokens, accepted counts and accepted nodes must equal the oracle's, except for sequences
the oracle flags as near-ties (an accept test within 1e-5 of its threshold, or top-two race
scores within 1e-6); those must still be a valid walk of the tree.  Shapes: chain-shaped
trees (which must also agree with the chain verify), random trees with up to four children
per node, a single-node tree, fp32 and bf16, ragged V, per-sequence temperatures, and the
deep and narrow static tree of SubSpec's configuration (depth 48, six children per node,
V = 152064).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from _parity import TOTALS, DeviceWorkload, to_device

pytestmark = pytest.mark.gpu

NEAR = oracle.FLAG_ACCEPT_NEAR_TIE | oracle.FLAG_RACE_NEAR_TIE | oracle.FLAG_RESIDUAL_EMPTY


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


def run_tree(sv, w, seed, per_seq=False, seq_index_base=0):
    dev = torch.device("cuda")
    t = to_device(w.target, w.dtype, dev)
    d = to_device(w.draft, w.dtype, dev) if w.draft.shape[1] else None
    tok = torch.from_numpy(np.ascontiguousarray(w.tokens)).to(dev)
    kw = {}
    if per_seq:
        kw = dict(T_per_seq=torch.from_numpy(w.T).to(dev), Td_per_seq=torch.from_numpy(w.Td).to(dev))
    out_t, nodes, n = sv.spec_verify_tree(t, d, tok, w.parent, float(w.T[0]), float(w.Td[0]), seed,
                                          seq_index_base=seq_index_base, **kw)
    torch.cuda.synchronize()
    return out_t.cpu().numpy(), nodes.cpu().numpy(), n.cpu().numpy()


def compare_tree(w, g, r):
    gt, gn, gc = g
    rt, rn, rc, flags = r
    children = {u: [v for v in range(1, w.N) if w.parent[v] == u] for u in range(w.N)}
    TOTALS["sequences"] += w.B
    for b in range(w.B):
        if flags[b] & NEAR:
            TOTALS["flagged"] += 1
            # still a valid walk: each accepted node a child of the previous, tokens match
            u = 0
            for k in range(gc[b]):
                v = gn[b, k]
                assert v in children[u] and gt[b, k] == w.tokens[b, v]
                u = v
            assert 0 <= gt[b, gc[b]] < w.V
            continue
        assert gc[b] == rc[b], (b, gc[b], rc[b])
        np.testing.assert_array_equal(gt[b], rt[b], err_msg=f"sequence {b}")
        np.testing.assert_array_equal(gn[b], rn[b], err_msg=f"nodes {b}")
    TOTALS["decisions"] += int(np.sum(np.maximum(rc, 0) + 1))


@pytest.mark.parametrize("B,gamma,V,dtype", [(3, 5, 3000, "bf16"), (2, 8, 1001, "f32"), (4, 1, 777, "bf16")])
def test_chain_tree_matches_chain_verify(sv, orc, B, gamma, V, dtype):
    w = workloads.generic(B=B, gamma=gamma, V=V, dtype=dtype, seed=V, sigma=0.5, T=0.8, Td=0.5)
    parent = np.arange(-1, gamma, dtype=np.int32)
    tok = np.concatenate([np.zeros((B, 1), np.int32), w.tokens], axis=1)
    tw = workloads.TreeWorkload("chain", B, V, dtype, parent, w.target, w.draft, tok, w.T, w.Td)
    dw = DeviceWorkload(w)
    for seed in range(4):
        g = run_tree(sv, tw, seed)
        r = orc.verify_tree(tw.target, tw.draft, tw.tokens, parent, tw.T, tw.Td, seed)
        compare_tree(tw, g, r)
        ct, cn, _ = sv.spec_verify_ex(dw.target, dw.draft, dw.tokens, float(w.T[0]), float(w.Td[0]), seed)
        torch.cuda.synchronize()
        ok = (r[3] & NEAR) == 0
        np.testing.assert_array_equal(g[0][ok], ct.cpu().numpy()[ok])
        np.testing.assert_array_equal(g[2][ok], cn.cpu().numpy()[ok])


@pytest.mark.parametrize("N,width,V,dtype,sigma", [(12, 3, 4099, "bf16", 0.6), (20, 4, 2000, "f32", 1.2),
                                                   (30, 2, 9000, "bf16", 0.3), (9, 4, 17, "f32", 2.0)])
def test_random_trees(sv, orc, N, width, V, dtype, sigma):
    rng = np.random.default_rng(N * 100 + V)
    for rep in range(2):
        parent = workloads.random_tree(rng, N, width)
        w = workloads.tree(parent, B=5, V=V, dtype=dtype, seed=rep + V, scale=3.0, sigma=sigma,
                           T=0.9, Td=0.45)
        for seed in range(3):
            compare_tree(w, run_tree(sv, w, seed),
                         orc.verify_tree(w.target, w.draft, w.tokens, w.parent, w.T, w.Td, seed))


def test_per_sequence_temperatures_and_index_base(sv, orc):
    parent = workloads.deep_narrow_tree(4, 3)
    w = workloads.tree(parent, B=6, V=5000, dtype="bf16", seed=4, scale=3.0, sigma=0.7)
    rng = np.random.default_rng(1)
    w.T[:] = rng.uniform(0.3, 1.2, size=w.B)
    w.Td[:] = 0.5 * w.T
    for seed in range(3):
        compare_tree(w, run_tree(sv, w, seed, per_seq=True),
                     orc.verify_tree(w.target, w.draft, w.tokens, w.parent, w.T, w.Td, seed))
    # two halves with seq_index_base give the one-call result
    full = run_tree(sv, w, 7, per_seq=True)
    halves = [run_tree(sv, w.subset(range(lo, lo + 3)), 7, per_seq=True, seq_index_base=lo) for lo in (0, 3)]
    np.testing.assert_array_equal(full[0], np.concatenate([h[0] for h in halves]))
    np.testing.assert_array_equal(full[2], np.concatenate([h[2] for h in halves]))


def test_single_node_tree_and_bad_tokens(sv, orc):
    w = workloads.tree(np.array([-1], np.int32), B=3, V=1000, dtype="f32", seed=2)
    g = run_tree(sv, w, 5)
    r = orc.verify_tree(w.target, w.draft, w.tokens, w.parent, w.T, w.Td, 5)
    compare_tree(w, g, r)
    assert np.all(g[2] == 0)
    parent = workloads.deep_narrow_tree(3, 2)
    w = workloads.tree(parent, B=3, V=500, dtype="bf16", seed=3)
    w.tokens[1, 5] = 500
    w.tokens[2, 1] = -7
    g = run_tree(sv, w, 1)
    assert sv.spec_verify_check() == sv.SPEC_EBADTOKEN
    assert sv.spec_verify_check() == sv.SPEC_OK
    r = orc.verify_tree(w.target, w.draft, w.tokens, w.parent, w.T, w.Td, 1)
    np.testing.assert_array_equal(g[2], r[2])
    np.testing.assert_array_equal(g[0], r[0])


def test_invalid_trees(sv):
    dev = torch.device("cuda")
    t = torch.zeros((1, 3, 64), dtype=torch.bfloat16, device=dev)
    d = torch.zeros((1, 1, 64), dtype=torch.bfloat16, device=dev)
    tok = torch.zeros((1, 3), dtype=torch.int32, device=dev)
    for parent in ([0, 0, 1], [-1, 1, 0], [-1, 0, 2]):
        with pytest.raises(sv.SpecVerifyError) as e:
            sv.spec_verify_tree(t, d, tok, parent, 1.0, 1.0, 0)
        assert e.value.code == sv.SPEC_EINVAL
    big = torch.zeros((1, 600, 8), dtype=torch.bfloat16, device=dev)
    with pytest.raises(sv.SpecVerifyError):
        sv.spec_verify_tree(big, torch.zeros((1, 599, 8), dtype=torch.bfloat16, device=dev),
                            torch.zeros((1, 600), dtype=torch.int32, device=dev),
                            list(range(-1, 599)), 1.0, 1.0, 0)


def test_deep_narrow_subspec_tree(sv, orc):
    """SubSpec's static tree: depth 48, six children per main-path node (289 nodes, 48 draft
    rows), V = 152064 bf16, T = 0.6, T_d = 0.2; two sequences against the oracle."""
    parent = workloads.deep_narrow_tree(48, 6)
    w = workloads.tree(parent, B=2, V=152064, dtype="bf16", seed=1005, scale=5.0,
                       sigma=workloads.DEEP_CHAIN_SIGMA, T=0.6, Td=0.2)
    for seed in range(2):
        g = run_tree(sv, w, seed)
        r = orc.verify_tree(w.target, w.draft, w.tokens, w.parent, w.T, w.Td, seed)
        compare_tree(w, g, r)
