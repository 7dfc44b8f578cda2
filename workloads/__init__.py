"""Seeded synthetic inputs for the speculative-decoding verify step.

This module only makes inputs: logits, draft tokens and temperatures.  It holds none of
the verify step's arithmetic, and both the CPU oracle and the CUDA path take their inputs
from it.  Everything is drawn from ``numpy.random.default_rng`` streams spawned per
sequence from one data seed, so any subset of sequences can be regenerated alone and the
result does not depend on the number of worker threads.

The five named workloads follow the shapes the pages' systems run at (one sequence with a
deep draft chain as in SubSpec's offloaded decoding, and batched serving shapes), with the
logit distributions stated for each below.  Draft tokens play the drafter's part: they are
drawn from the draft distribution q = softmax(L_d / T_d) by the Gumbel-max trick on numpy's
generator (greedy workloads take the argmax of the draft row instead).  bf16 logits are
stored as uint16 bit patterns, rounded to nearest-even from float32.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field
from typing import Callable, Optional, Sequence

import numpy as np

# Draft-noise sigma of the deep-chain workload (B=1, gamma=48, V=152064, T=0.6, T_d=0.2),
# found by oracle/calibrate_deep_chain.py: with data seed 1002 the mean over the 48 draft
# positions of sum_x min(p, q) is 0.5597 (bf16 rounding makes it a step function of sigma).
DEEP_CHAIN_SIGMA = 1.020355224609375


@dataclass
class Workload:
    name: str
    B: int
    gamma: int
    V: int
    dtype: str                 # "f32" or "bf16"
    target: np.ndarray         # [B, gamma+1, V] float32, or uint16 bf16 bits
    draft: np.ndarray          # [B, gamma, V]
    tokens: np.ndarray         # [B, gamma] int32, drawn from q (sampling) or argmax (greedy)
    T: np.ndarray              # [B] float32 target temperature
    Td: np.ndarray             # [B] float32 draft temperature
    greedy: bool = False       # tokens are draft argmaxes (greedy workload)
    info: dict = field(default_factory=dict)

    @property
    def rows(self) -> int:
        """Verified logit rows per call: B * (gamma + 1)."""
        return self.B * (self.gamma + 1)

    def bytes_sampling(self) -> int:
        """Bytes of one read of every target and draft logit."""
        s = 2 if self.dtype == "bf16" else 4
        return s * self.V * self.B * (2 * self.gamma + 1)

    def bytes_greedy(self) -> int:
        s = 2 if self.dtype == "bf16" else 4
        return s * self.V * self.B * (self.gamma + 1)

    def subset(self, idx: Sequence[int]) -> "Workload":
        idx = np.asarray(idx, dtype=np.int64)
        return Workload(self.name, len(idx), self.gamma, self.V, self.dtype,
                        np.ascontiguousarray(self.target[idx]),
                        np.ascontiguousarray(self.draft[idx]),
                        np.ascontiguousarray(self.tokens[idx]), self.T[idx].copy(),
                        self.Td[idx].copy(), self.greedy, dict(self.info))


# ---------------------------------------------------------------------------------------
# encoding helpers
# ---------------------------------------------------------------------------------------

def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest, ties to even."""
    bits = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = np.uint32(0x7FFF) + ((bits >> np.uint32(16)) & np.uint32(1))
    return ((bits + rounding) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float32 (exact)."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(
        np.float32)


def as_f32(a: np.ndarray, dtype: str) -> np.ndarray:
    return bf16_bits_to_f32(a) if dtype == "bf16" else np.asarray(a, dtype=np.float32)


def _encode(x: np.ndarray, dtype: str) -> np.ndarray:
    return to_bf16_bits(x) if dtype == "bf16" else np.ascontiguousarray(x, dtype=np.float32)


def _gumbel(rng: np.random.Generator, shape) -> np.ndarray:
    e = rng.standard_exponential(shape, dtype=np.float32)
    return -np.log(np.maximum(e, np.float32(1e-30)))


def draw_drafts(rng: np.random.Generator, draft_f32: np.ndarray, Td: float) -> np.ndarray:
    """The drafter's draw: one token per row from softmax(row / Td) (Gumbel-max)."""
    z = draft_f32 / np.float32(Td) + _gumbel(rng, draft_f32.shape)
    return np.argmax(z, axis=-1).astype(np.int32)


# ---------------------------------------------------------------------------------------
# logit shapes
# ---------------------------------------------------------------------------------------

def normal_rows(rng, rows, V, scale):
    return (rng.standard_normal((rows, V), dtype=np.float32) * np.float32(scale))


def zipf_shaped_rows(rng, rows, V, scale):
    """Sorted N(0, 1) scaled by `scale`, then randomly permuted, one draw per row."""
    out = np.empty((rows, V), dtype=np.float32)
    for r in range(rows):
        s = np.sort(rng.standard_normal(V, dtype=np.float32)) * np.float32(scale)
        out[r] = s[rng.permutation(V)]
    return out


def heavy_tailed_rows(rng, rows, V, gumbel_scale=2.0, spike=8.0, n_spikes=16):
    """Gumbel(0, 1) * gumbel_scale plus +spike on n_spikes random tokens per row."""
    out = _gumbel(rng, (rows, V)) * np.float32(gumbel_scale)
    for r in range(rows):
        out[r, rng.choice(V, size=n_spikes, replace=False)] += np.float32(spike)
    return out


# ---------------------------------------------------------------------------------------
# generic builder
# ---------------------------------------------------------------------------------------

def _one_sequence(rng, gamma, V, dtype, target_fn, sigma, T, Td, greedy):
    """Draw one sequence: target rows, draft rows = target + N(0, sigma^2), draft tokens."""
    t32 = target_fn(rng, gamma + 1, V)
    noise = rng.standard_normal((gamma, V), dtype=np.float32)
    d32 = t32[:gamma] + noise * np.float32(sigma)
    t_enc, d_enc = _encode(t32, dtype), _encode(d32, dtype)
    d_used = as_f32(d_enc, dtype)
    if greedy:
        tok = np.argmax(d_used, axis=-1).astype(np.int32) if gamma else np.zeros(0, np.int32)
    else:
        tok = draw_drafts(rng, d_used, Td) if gamma else np.zeros(0, np.int32)
    return t_enc, d_enc, tok


def make_workload(name: str, B: int, gamma: int, V: int, dtype: str, seed: int,
                  target_fn: Callable, sigma, T, Td_ratio: Optional[float] = None, Td=None,
                  greedy: bool = False, threads: Optional[int] = None,
                  per_seq_params: Optional[Callable] = None) -> Workload:
    """Build a workload.  Each sequence b uses its own generator spawned from `seed`.
    per_seq_params(rng) -> (T, Td, sigma) overrides the scalars for that sequence
    (drawn first from the sequence's generator)."""
    children = np.random.SeedSequence(seed).spawn(B)
    tshape, dshape = (B, gamma + 1, V), (B, gamma, V)
    edt = np.uint16 if dtype == "bf16" else np.float32
    target = np.empty(tshape, dtype=edt)
    draft = np.empty(dshape, dtype=edt)
    tokens = np.empty((B, gamma), dtype=np.int32)
    Tb = np.empty(B, dtype=np.float32)
    Tdb = np.empty(B, dtype=np.float32)
    sig = np.empty(B, dtype=np.float64)

    def work(b):
        rng = np.random.default_rng(children[b])
        if per_seq_params is not None:
            t_b, td_b, s_b = per_seq_params(rng)
        else:
            t_b = T
            td_b = Td if Td is not None else (T * Td_ratio)
            s_b = sigma
        t_b, td_b = np.float32(t_b), np.float32(td_b)
        te, de, tok = _one_sequence(rng, gamma, V, dtype, target_fn, s_b, t_b, td_b, greedy)
        target[b], draft[b], tokens[b] = te, de, tok
        Tb[b], Tdb[b], sig[b] = t_b, td_b, s_b

    nthreads = threads or min(B, os.cpu_count() or 1, 32)
    if nthreads <= 1 or B == 1:
        for b in range(B):
            work(b)
    else:
        with ThreadPoolExecutor(nthreads) as ex:
            list(ex.map(work, range(B)))
    return Workload(name, B, gamma, V, dtype, target, draft, tokens, Tb, Tdb, greedy,
                    {"seed": seed, "sigma": sig})


# ---------------------------------------------------------------------------------------
# the five named workloads
# ---------------------------------------------------------------------------------------

CONFIG_NAMES = {
    0: "small: B=1, gamma=5, V=1024 fp32, N(0,2^2) target, draft noise 0.5, T=T_d=1",
    1: "single sequence: B=1, gamma=16, V=128256 bf16, Zipf-shaped target x3, draft noise 0.7",
    2: "deep chain: B=1, gamma=48, V=152064 bf16, Zipf-shaped target x5, T=0.6, T_d=0.2",
    3: "batched serving: B=64, gamma=8, V=128256 bf16, T_b~U[0.3,1.2], T_d=T_b/2, sigma_b~U[0.3,1.5]",
    4: "throughput stress: B=256, gamma=12, V=152064 bf16, 2*Gumbel + 8 on 16 tokens, noise 1, T=1, T_d=0.2",
}

CONFIG_SHAPES = {0: (1, 5, 1024, "f32"), 1: (1, 16, 128256, "bf16"), 2: (1, 48, 152064, "bf16"),
                 3: (64, 8, 128256, "bf16"), 4: (256, 12, 152064, "bf16")}


def config(cfg: int, greedy: bool = False, seed: Optional[int] = None,
           threads: Optional[int] = None, B: Optional[int] = None) -> Workload:
    """Named workload `cfg` (0..4).  Data seed defaults to 1000 + cfg.  `B` may shrink the
    batch (the first B sequences of the full workload, identical values)."""
    seed = 1000 + cfg if seed is None else seed
    Bf, g, V, dt = CONFIG_SHAPES[cfg]
    B = Bf if B is None else B
    name = f"cfg{cfg}" + ("-greedy" if greedy else "")
    if cfg == 0:
        return make_workload(name, B, g, V, dt, seed, lambda r, n, v: normal_rows(r, n, v, 2.0),
                             0.5, 1.0, Td=1.0, greedy=greedy, threads=threads)
    if cfg == 1:
        return make_workload(name, B, g, V, dt, seed,
                             lambda r, n, v: zipf_shaped_rows(r, n, v, 3.0), 0.7, 1.0, Td=1.0,
                             greedy=greedy, threads=threads)
    if cfg == 2:
        return make_workload(name, B, g, V, dt, seed,
                             lambda r, n, v: zipf_shaped_rows(r, n, v, 5.0), DEEP_CHAIN_SIGMA,
                             0.6, Td=0.2, greedy=greedy, threads=threads)
    if cfg == 3:
        def params(rng):
            t = rng.uniform(0.3, 1.2)
            return t, 0.5 * t, rng.uniform(0.3, 1.5)
        return make_workload(name, B, g, V, dt, seed,
                             lambda r, n, v: zipf_shaped_rows(r, n, v, 3.0), None, None,
                             greedy=greedy, threads=threads, per_seq_params=params)
    if cfg == 4:
        return make_workload(name, B, g, V, dt, seed, heavy_tailed_rows, 1.0, 1.0, Td=0.2,
                             greedy=greedy, threads=threads)
    raise ValueError(f"unknown workload {cfg}")


def deep_chain_with_sigma(sigma: float, seed: int = 1002) -> Workload:
    """The deep-chain workload at an explicit draft-noise sigma (for its calibration)."""
    Bf, g, V, dt = CONFIG_SHAPES[2]
    return make_workload(f"cfg2-sigma{sigma}", 1, g, V, dt, seed,
                         lambda r, n, v: zipf_shaped_rows(r, n, v, 5.0), sigma, 0.6, Td=0.2)


def generic(B: int, gamma: int, V: int, dtype: str = "bf16", seed: int = 0, scale: float = 2.0,
            sigma: float = 0.5, T: float = 1.0, Td: float = 1.0, greedy: bool = False,
            kind: str = "normal") -> Workload:
    """Small ad-hoc workload for parity and edge-case tests."""
    fns = {
        "normal": lambda r, n, v: normal_rows(r, n, v, scale),
        "zipf": lambda r, n, v: zipf_shaped_rows(r, n, v, scale),
        "heavy": heavy_tailed_rows if V >= 16 else (lambda r, n, v: normal_rows(r, n, v, scale)),
    }
    return make_workload(f"generic-{B}x{gamma}x{V}-{dtype}-{kind}", B, gamma, V, dtype, seed,
                         fns[kind], sigma, T, Td=Td, greedy=greedy)


# ---------------------------------------------------------------------------------------
# token trees
# ---------------------------------------------------------------------------------------

@dataclass
class TreeWorkload:
    """A static draft token tree per sequence.  parent[n] < n (parent[0] = -1); target row
    n is p at node n; draft row m is q at the m-th internal node (in node order); node n's
    token (n >= 1) is drawn from q at its parent; siblings are independent draws."""
    name: str
    B: int
    V: int
    dtype: str
    parent: np.ndarray         # [N] int32
    target: np.ndarray         # [B, N, V]
    draft: np.ndarray          # [B, M, V]
    tokens: np.ndarray         # [B, N] int32 (column 0 unused: 0)
    T: np.ndarray              # [B] float32
    Td: np.ndarray             # [B] float32
    info: dict = field(default_factory=dict)

    @property
    def N(self) -> int:
        return len(self.parent)

    @property
    def internal(self) -> np.ndarray:
        has = np.zeros(self.N, bool)
        has[self.parent[1:]] = True
        return np.nonzero(has)[0]

    @property
    def depth(self) -> int:
        d = np.zeros(self.N, np.int64)
        for n in range(1, self.N):
            d[n] = d[self.parent[n]] + 1
        return int(d.max()) if self.N > 1 else 0

    def rows(self) -> int:
        """Logit rows per call: every node's target row and every internal node's draft row."""
        return self.B * (self.N + len(self.internal))

    def bytes(self) -> int:
        return (2 if self.dtype == "bf16" else 4) * self.V * self.rows()

    def subset(self, idx: Sequence[int]) -> "TreeWorkload":
        idx = np.asarray(idx)
        return TreeWorkload(self.name, len(idx), self.V, self.dtype, self.parent, self.target[idx],
                            self.draft[idx], self.tokens[idx], self.T[idx], self.Td[idx], self.info)


def deep_narrow_tree(depth: int, k: int) -> np.ndarray:
    """SubSpec-style static tree, deep and narrow: a main path of `depth` draft levels whose
    nodes each have k children, the first continuing the path and the others leaves."""
    parent = [-1]
    main = 0
    for _ in range(depth):
        first = len(parent)
        parent.extend([main] * k)
        main = first
    return np.asarray(parent, np.int32)


def random_tree(rng: np.random.Generator, N: int, max_children: int = 4) -> np.ndarray:
    """A random tree of N nodes in node order (each node's parent is an earlier node with
    fewer than max_children children)."""
    parent = [-1]
    nchild = [0]
    for n in range(1, N):
        cand = [u for u in range(n) if nchild[u] < max_children]
        u = int(rng.choice(cand))
        parent.append(u)
        nchild[u] += 1
        nchild.append(0)
    return np.asarray(parent, np.int32)


def tree(parent, B: int, V: int, dtype: str = "bf16", seed: int = 0, scale: float = 5.0,
         sigma: float = 1.0, T: float = 0.6, Td: float = 0.2, name: str = "tree") -> TreeWorkload:
    """Per sequence: Zipf-shaped target rows (one per node), draft rows = target + N(0, sigma^2)
    at internal nodes, children drawn from q at their parent (independently)."""
    parent = np.asarray(parent, np.int32)
    N = len(parent)
    has = np.zeros(N, bool)
    has[parent[1:]] = True
    internal = np.nonzero(has)[0]
    drow = -np.ones(N, np.int64)
    drow[internal] = np.arange(len(internal))
    rngs = [np.random.default_rng(s) for s in np.random.SeedSequence(seed).spawn(B)]
    tgt, drf, tok = [], [], np.zeros((B, N), np.int32)
    for b, rng in enumerate(rngs):
        t32 = zipf_shaped_rows(rng, N, V, scale)
        d32 = t32[internal] + rng.standard_normal((len(internal), V), dtype=np.float32) * np.float32(sigma)
        t_enc, d_enc = _encode(t32, dtype), _encode(d32, dtype)
        d_used = as_f32(d_enc, dtype)
        for n in range(1, N):
            tok[b, n] = draw_drafts(rng, d_used[drow[parent[n]]][None, :], Td)[0]
        tgt.append(t_enc)
        drf.append(d_enc)
    shape_d = (B, len(internal), V)
    draft = np.stack(drf) if len(internal) else np.zeros(shape_d, tgt[0].dtype)
    return TreeWorkload(name, B, V, dtype, parent, np.stack(tgt), draft, tok,
                        np.full(B, T, np.float32), np.full(B, Td, np.float32))
