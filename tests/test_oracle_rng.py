"""Pins of the oracle's random numbers (CPU only).

* Philox4x32-10 against an independent library implementation: Triton's Philox
  (``triton.language.philox_impl``), run by Triton's CPU interpreter in a child process.
* Uniformity of the acceptance uniforms (chi-square over 2^16 buckets) and their 24-bit
  grid; the race exponentials against Exp(1) (Kolmogorov-Smirnov) and their mean.
* The race's winning score minus the log of the total weight against the standard Gumbel law.
"""
import json
import os
import subprocess
import sys

import numpy as np
import pytest
from scipy import stats

import oracle

_TRITON_PHILOX = r"""
import os, sys, json
os.environ["TRITON_INTERPRET"] = "1"
import numpy as np, torch, triton, triton.language as tl

@triton.jit
def kern(c_ptr, k_ptr, o_ptr, n, BLOCK: tl.constexpr):
    offs = tl.program_id(0) * BLOCK + tl.arange(0, BLOCK)
    m = offs < n
    c0 = tl.load(c_ptr + offs * 4 + 0, mask=m).to(tl.uint32)
    c1 = tl.load(c_ptr + offs * 4 + 1, mask=m).to(tl.uint32)
    c2 = tl.load(c_ptr + offs * 4 + 2, mask=m).to(tl.uint32)
    c3 = tl.load(c_ptr + offs * 4 + 3, mask=m).to(tl.uint32)
    k0 = tl.load(k_ptr + offs * 2 + 0, mask=m).to(tl.uint32)
    k1 = tl.load(k_ptr + offs * 2 + 1, mask=m).to(tl.uint32)
    a, b, c, d = tl.philox_impl(c0, c1, c2, c3, k0, k1, 10)
    tl.store(o_ptr + offs * 4 + 0, a.to(tl.int64), mask=m)
    tl.store(o_ptr + offs * 4 + 1, b.to(tl.int64), mask=m)
    tl.store(o_ptr + offs * 4 + 2, c.to(tl.int64), mask=m)
    tl.store(o_ptr + offs * 4 + 3, d.to(tl.int64), mask=m)

data = json.loads(sys.stdin.read())
C = np.array(data["C"], dtype=np.int64); K = np.array(data["K"], dtype=np.int64)
n = C.shape[0]
out = torch.zeros(n * 4, dtype=torch.int64)
kern[(triton.cdiv(n, 64),)](torch.from_numpy(C.copy()), torch.from_numpy(K.copy()), out, n,
                            BLOCK=64)
print(json.dumps((out.numpy() & 0xffffffff).tolist()))
"""


def _counters_and_keys(n, seed=7):
    rng = np.random.default_rng(seed)
    C = rng.integers(0, 2**32, size=(n, 4), dtype=np.uint64)
    K = rng.integers(0, 2**32, size=(n, 2), dtype=np.uint64)
    # corner cases: all-zero, all-ones, and the counters the verify contract uses
    C[0], K[0] = 0, 0
    C[1], K[1] = 0xFFFFFFFF, 0xFFFFFFFF
    C[2], K[2] = [0, 3, 17, 0], [12345, 0]
    C[3], K[3] = [38015, 48, 255, 1], [0xDEADBEEF, 0x01234567]
    return C, K


def test_philox_matches_triton():
    pytest.importorskip("triton")
    pytest.importorskip("torch")
    C, K = _counters_and_keys(256)
    env = dict(os.environ, TRITON_INTERPRET="1")
    res = subprocess.run([sys.executable, "-c", _TRITON_PHILOX],
                         input=json.dumps({"C": C.astype(np.int64).tolist(),
                                           "K": K.astype(np.int64).tolist()}),
                         capture_output=True, text=True, env=env, timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    ref = np.array(json.loads(res.stdout.strip().splitlines()[-1]), dtype=np.uint64).reshape(-1, 4)
    got = oracle.get().philox_bulk(C.astype(np.uint32), K.astype(np.uint32)).astype(np.uint64)
    np.testing.assert_array_equal(got, ref)


def test_philox_key_and_counter_sensitivity():
    """Every input word changes every output word (a dropped or swapped word fails)."""
    orc = oracle.get()
    base_c, base_k = np.array([5, 6, 7, 8], np.uint32), np.array([9, 10], np.uint32)
    base = orc.philox(base_c, base_k)
    for w in range(4):
        c = base_c.copy(); c[w] ^= 1
        assert np.all(orc.philox(c, base_k) != base)
    for w in range(2):
        k = base_k.copy(); k[w] ^= 1
        assert np.all(orc.philox(base_c, k) != base)


def test_accept_uniforms_grid_and_uniformity():
    orc = oracle.get()
    u = orc.accept_uniforms(seed=20260807, B=1 << 18, gamma=16).ravel()  # 4.2M values
    assert u.min() >= 0.0 and u.max() < 1.0
    # 24-bit grid: u * 2^24 is an integer, so u is exact in fp32
    np.testing.assert_array_equal(u * 16777216.0, np.floor(u * 16777216.0))
    np.testing.assert_array_equal(u.astype(np.float32).astype(np.float64), u)
    counts = np.bincount((u * 65536).astype(np.int64), minlength=65536)
    chi2, p = stats.chisquare(counts)
    assert p > 1e-4, (chi2, p)
    # independence of neighbouring positions (lag-1 correlation ~ 0)
    uu = u.reshape(-1, 16)
    r = np.corrcoef(uu[:, :-1].ravel(), uu[:, 1:].ravel())[0, 1]
    assert abs(r) < 5.0 / np.sqrt(uu[:, 1:].size)


def test_accept_uniform_depends_on_sequence_position_and_seed():
    orc = oracle.get()
    a = orc.accept_uniforms(seed=1, B=64, gamma=8)
    b = orc.accept_uniforms(seed=2, B=64, gamma=8)
    c = orc.accept_uniforms(seed=1, B=64, gamma=8, b_base=64)
    assert np.mean(a == b) < 0.01 and np.mean(a == c) < 0.01
    assert len(np.unique(a)) > 0.99 * a.size
    # b_base shifts the global sequence index
    np.testing.assert_array_equal(orc.accept_uniforms(seed=1, B=32, gamma=8, b_base=32), a[32:])


def test_race_exponentials_are_exp1():
    orc = oracle.get()
    e = np.concatenate([orc.race_exponentials(seed=3, b=b, pos=p, n=200_000)
                        for b, p in [(0, 0), (1, 5), (77, 12)]])
    assert e.min() > 0.0
    ks = stats.kstest(e, "expon")
    assert ks.pvalue > 1e-4, ks
    assert abs(e.mean() - 1.0) < 5.0 / np.sqrt(e.size)
    # the smallest possible value is -log1p(-2^-33) > 0, the largest -log(2^-33) ~ 22.9
    assert e.max() < 23.0


def test_race_exponential_word_layout():
    """Token x uses word (x & 3) of counter (x >> 2, pos, b, 1)."""
    orc = oracle.get()
    seed, b, pos = 0x1234_5678_9ABC_DEF0, 11, 3
    key = np.array([seed & 0xFFFFFFFF, seed >> 32], np.uint32)
    for x in [0, 1, 2, 3, 4, 7, 1001, 152063]:
        w = orc.philox(np.array([x >> 2, pos, b, 1], np.uint32), key)[x & 3]
        U = (float(w) + 0.5) / 2**32
        assert orc.race_exponential(seed, b, pos, x) == pytest.approx(-np.log1p(-U), rel=1e-15)
    # acceptance: word 0 of counter (0, i, b, 0), top 24 bits
    for i in [0, 1, 47]:
        w = orc.philox(np.array([0, i, b, 0], np.uint32), key)[0]
        assert orc.accept_uniform(seed, b, i) == (int(w) >> 8) / 2**24


def test_race_winner_score_is_gumbel_shifted_by_the_log_total_weight():
    """The verify from hidden states starts each race from ln N - 2 (N the total weight) and
    races again when the winner falls below it; that start is cheap only if the winning
    score max_x ln w(x) - ln E_x is ln N plus a standard Gumbel variable, as the race's
    exponentials make it.  Over many independent races of one weight vector: the winning
    scores minus ln N follow the standard Gumbel law (Kolmogorov-Smirnov), and the share
    below -2 is exp(-e^2) < 7e-4 within binomial error."""
    orc = oracle.get()
    rng = np.random.default_rng(0)
    V = 512
    w = rng.gamma(0.3, size=V)
    w[rng.random(V) < 0.2] = 0.0  # zero weights take no part
    lnN = np.log(w.sum())
    with np.errstate(divide="ignore"):
        lw = np.log(w)
    n = 20_000
    g = np.empty(n)
    for k in range(n):  # race k: sequence k of seed 11, row 3
        g[k] = np.max(lw - np.log(orc.race_exponentials(11, k, 3, V))) - lnN
    assert stats.kstest(g, stats.gumbel_r.cdf).pvalue > 1e-3
    p = np.exp(-np.exp(2.0))
    low = int((g < -2.0).sum())
    assert abs(low - n * p) < 5 * np.sqrt(n * p * (1 - p)) + 1, (low, n * p)
