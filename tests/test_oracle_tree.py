"""Pins of the oracle's token-tree verification (the multi-draft rule; see the oracle's
header for the reading taken).

* A chain-shaped tree is the chain verify: bit-exact tokens and counts on random inputs.
* Losslessness, exactly: on small trees with a synthetic target model p(. | path) and draft
  model q(. | path), an exact evaluation of the rule (independent of the C code: it
  enumerates every draft assignment, weighted by the drafts' probability, and follows the
  rule's accept probabilities and residuals in closed form) gives an output whose
  extension by target draws has the target model's joint law, within 1e-12.
* The oracle samples from that law: 3*10^4 seeded cycles, chi-square against the exact
  law of the emitted sequence (p > 1e-3).
"""
import itertools

import numpy as np
import pytest
from scipy.stats import chisquare

import oracle
import workloads


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


def chain_parent(n):
    return np.arange(-1, n - 1, dtype=np.int32)


@pytest.mark.parametrize("B,gamma,V,dtype,sigma", [(4, 5, 300, "bf16", 0.6), (3, 8, 1000, "f32", 0.2),
                                                   (5, 1, 50, "bf16", 1.0), (2, 0, 64, "f32", 0.5)])
def test_chain_tree_is_the_chain_verify(orc, B, gamma, V, dtype, sigma):
    w = workloads.generic(B=B, gamma=gamma, V=V, dtype=dtype, seed=V + gamma, sigma=sigma, T=0.9, Td=0.6)
    tok = np.concatenate([np.zeros((B, 1), np.int32), w.tokens], axis=1)
    for seed in range(8):
        r = orc.verify(w.target, w.draft, w.tokens, w.T, w.Td, seed)
        t, nodes, n, f = orc.verify_tree(w.target, w.draft, tok, chain_parent(gamma + 1), w.T, w.Td, seed)
        np.testing.assert_array_equal(t, r.tokens)
        np.testing.assert_array_equal(n, r.n_accepted)
        for b in range(B):
            assert list(nodes[b, :n[b]]) == list(range(1, n[b] + 1))


# --- exact evaluation of the rule on small trees ---------------------------------------

def softmax64(l):
    l = np.asarray(l, np.float64)
    m = l.max()
    e = np.exp(l - m)
    return e / e.sum()


class Model:
    """p(. | prefix) and q(. | prefix) for prefixes up to `depth` tokens, as fp32 logits."""

    def __init__(self, V, depth, seed, T=1.0, Td=1.0, sharp=2.0, noise=0.8):
        rng = np.random.default_rng(seed)
        self.V, self.T, self.Td = V, T, Td
        self.lp, self.lq = {}, {}
        for k in range(depth + 1):
            for pre in itertools.product(range(V), repeat=k):
                lt = (rng.standard_normal(V) * sharp).astype(np.float32)
                self.lp[pre] = lt
                self.lq[pre] = (lt + rng.standard_normal(V) * noise).astype(np.float32)

    def p(self, pre):
        return softmax64(self.lp[pre].astype(np.float64) / self.T)

    def q(self, pre):
        return softmax64(self.lq[pre].astype(np.float64) / self.Td)


def children_of(parent):
    ch = {u: [] for u in range(len(parent))}
    for v in range(1, len(parent)):
        ch[int(parent[v])].append(v)
    return ch


def rule_law(model, parent, tokens):
    """Exact law {emitted tuple: prob} of the multi-draft rule for one draft assignment."""
    ch = children_of(parent)
    paths = {0: ()}
    for v in range(1, len(parent)):
        paths[v] = paths[int(parent[v])] + (int(tokens[v]),)

    def law(u):
        pre = paths[u]
        p = model.p(pre)
        out = {}
        if not ch[u]:
            for y in range(model.V):
                out[(y,)] = out.get((y,), 0.0) + p[y]
            return out
        q = model.q(pre)
        c, N, still = 0.0, 1.0, 1.0
        for v in ch[u]:
            x = int(tokens[v])
            pp = max(0.0, p[x] - c * q[x]) / N
            a = min(1.0, pp / q[x]) if q[x] > 0 else (1.0 if pp > 0 else 0.0)
            if a > 0:
                for seq, pr in law(v).items():
                    out[(x,) + seq] = out.get((x,) + seq, 0.0) + still * a * pr
            still *= 1.0 - a
            c += N
            N = float(np.maximum(0.0, p - c * q).sum())
        r = np.maximum(0.0, p - c * q)
        r = r / r.sum() if r.sum() > 0 else p
        for y in range(model.V):
            out[(y,)] = out.get((y,), 0.0) + still * r[y]
        return out

    return law(0)


def assignments(model, parent):
    """Every draft assignment with its probability (children drawn i.i.d. from q_parent)."""
    N = len(parent)
    for toks in itertools.product(range(model.V), repeat=N - 1):
        tokens = (0,) + toks
        paths = {0: ()}
        prob = 1.0
        for v in range(1, N):
            u = int(parent[v])
            prob *= model.q(paths[u])[tokens[v]]
            paths[v] = paths[u] + (tokens[v],)
        yield tokens, prob


def emitted_law(model, parent):
    law = {}
    for tokens, prob in assignments(model, parent):
        for seq, pr in rule_law(model, parent, tokens).items():
            law[seq] = law.get(seq, 0.0) + prob * pr
    return law


TREES = {
    "fork-then-chain": np.array([-1, 0, 0, 1], np.int32),         # root: 2 children; first has 1
    "wide": np.array([-1, 0, 0, 0], np.int32),                    # root: 3 children
    "two-level": np.array([-1, 0, 0, 1, 1, 2, 2], np.int32),      # binary, depth 2
    "deep-narrow": np.array([-1, 0, 0, 1, 1, 3, 3], np.int32),    # main path with side leaves
    "four-wide": np.array([-1, 0, 0, 0, 0], np.int32),            # root: 4 children
}


@pytest.mark.parametrize("name", sorted(TREES))
@pytest.mark.parametrize("T,Td", [(1.0, 1.0), (1.0, 0.4)])
def test_rule_is_lossless_exactly(name, T, Td):
    parent = TREES[name]
    d = np.zeros(len(parent), int)
    for v in range(1, len(parent)):
        d[v] = d[parent[v]] + 1
    depth = int(d.max())
    V = 3
    model = Model(V, depth + 1, seed=len(parent) * 7 + int(T * 10) + int(Td * 100), T=T, Td=Td)
    law = emitted_law(model, parent)
    assert abs(sum(law.values()) - 1.0) < 1e-12
    L = depth + 1
    joint = {}
    for seq, pr in law.items():  # extend each emitted sequence with target draws to length L
        stack = [(seq, pr)]
        while stack:
            s, w = stack.pop()
            if len(s) == L:
                joint[s] = joint.get(s, 0.0) + w
                continue
            p = model.p(s)
            for y in range(V):
                stack.append((s + (y,), w * p[y]))
    for s in itertools.product(range(V), repeat=L):
        want = 1.0
        for k in range(L):
            want *= model.p(s[:k])[s[k]]
        assert abs(joint.get(s, 0.0) - want) < 1e-12, (name, s)


def sampler_pvalue(orc, name, noise=0.8):
    parent = TREES[name]
    N = len(parent)
    d = np.zeros(N, int)
    for v in range(1, N):
        d[v] = d[parent[v]] + 1
    depth = int(d.max())
    V, B = 3, 30000
    model = Model(V, depth + 1, seed=99 + N, T=1.0, Td=0.5, noise=noise)
    law = emitted_law(model, parent)
    internal = [u for u in range(N) if any(parent[v] == u for v in range(1, N))]
    rng = np.random.default_rng(123)
    tokens = np.zeros((B, N), np.int32)
    target = np.zeros((B, N, V), np.float32)
    draft = np.zeros((B, len(internal), V), np.float32)
    for b in range(B):
        paths = {0: ()}
        for v in range(1, N):
            u = int(parent[v])
            tokens[b, v] = rng.choice(V, p=model.q(paths[u]))
            paths[v] = paths[u] + (int(tokens[b, v]),)
        for u in range(N):
            target[b, u] = model.lp[paths[u]]
        for m, u in enumerate(internal):
            draft[b, m] = model.lq[paths[u]]
    out_t, nodes, n, flags = orc.verify_tree(target, draft, tokens, parent, 1.0, 0.5, seed=5)
    counts = {}
    for b in range(B):
        seq = tuple(int(x) for x in out_t[b, :n[b] + 1])
        counts[seq] = counts.get(seq, 0) + 1
    keys = sorted(law)
    assert set(counts) <= set(keys)
    obs = np.array([counts.get(k, 0) for k in keys], float)
    exp = np.array([law[k] for k in keys]) * B
    keep = exp > 5
    obs_k = np.append(obs[keep], obs[~keep].sum())
    exp_k = np.append(exp[keep], exp[~keep].sum())
    if exp_k[-1] == 0:
        obs_k, exp_k = obs_k[:-1], exp_k[:-1]
    return chisquare(obs_k, exp_k * obs_k.sum() / exp_k.sum()).pvalue


@pytest.mark.parametrize("name", ["fork-then-chain", "two-level", "four-wide"])
def test_oracle_samples_the_rule(orc, name):
    assert sampler_pvalue(orc, name) > 1e-3


@pytest.mark.parametrize("mutation", [10, 11])
def test_planted_tree_mistakes_fail_the_sampler_pin(mutation, tmp_path):
    """A residual coefficient stuck at 1, or a residual left unnormalised, in a rebuilt
    oracle fails the chi-square against the rule's exact law."""
    path = str(tmp_path / f"liboracle_m{mutation}.so")
    oracle.build(path, mutation=mutation)
    bad = oracle.Oracle(path)
    assert min(sampler_pvalue(bad, n, noise=2.0)
               for n in ("four-wide", "two-level", "wide", "fork-then-chain")) < 1e-6


def test_tree_bad_tokens_and_arguments(orc):
    parent = np.array([-1, 0, 0, 1], np.int32)
    target = np.zeros((2, 4, 5), np.float32)
    draft = np.zeros((2, 2, 5), np.float32)
    tok = np.array([[0, 1, 2, 3], [0, 1, 5, 3]], np.int32)
    t, nodes, n, f = orc.verify_tree(target, draft, tok, parent, 1.0, 1.0, 0)
    assert n[1] == -1 and np.all(t[1] == -1) and (f[1] & oracle.FLAG_BAD_TOKEN)
    assert n[0] >= 0
    with pytest.raises(ValueError):
        orc.verify_tree(target, draft, tok, np.array([-1, 0, 3, 1], np.int32), 1.0, 1.0, 0)
