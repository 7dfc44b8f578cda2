"""CPU oracle of the speculative-decoding verify step (ctypes binding).

TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.  Only ``tests/``, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import this package.
The CUDA library never imports, links or calls it, and the two share no source.

The arithmetic lives in ``specverify_oracle.c`` (plain single-threaded C, fp64); this
module compiles it with gcc and wraps its entry points for numpy arrays.  See the C file's
header for the pages and sections each step follows and for the random-number contract.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "specverify_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

F32, BF16 = 0, 1

FLAG_ACCEPT_NEAR_TIE = 1
FLAG_RACE_NEAR_TIE = 2
FLAG_BAD_TOKEN = 4
FLAG_RESIDUAL_EMPTY = 8


def build(out_path: str = _LIB_PATH, mutation: int = 0) -> str:
    """Compile the oracle with gcc.  ``mutation`` > 0 plants a known mistake (tests only)."""
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
           f"-DORACLE_MUTATION={int(mutation)}", "-o", out_path, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    return out_path


def _needs_build(path: str) -> bool:
    return (not os.path.exists(path)) or os.path.getmtime(path) < os.path.getmtime(_SRC)


_P = ctypes.c_void_p


class Oracle:
    """Handle on one compiled copy of the oracle."""

    def __init__(self, path: str = _LIB_PATH):
        if path == _LIB_PATH and _needs_build(path):
            build(path)
        self.path = path
        lib = ctypes.CDLL(path)
        lib.oracle_philox4x32_10.argtypes = [_P, _P, _P]
        lib.oracle_philox4x32_10.restype = None
        lib.oracle_accept_uniform.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32]
        lib.oracle_accept_uniform.restype = ctypes.c_double
        lib.oracle_race_exponential.argtypes = [ctypes.c_uint64, ctypes.c_uint32,
                                                ctypes.c_uint32, ctypes.c_uint32]
        lib.oracle_race_exponential.restype = ctypes.c_double
        lib.oracle_philox_bulk.argtypes = [_P, _P, ctypes.c_int64, _P]
        lib.oracle_philox_bulk.restype = None
        lib.oracle_accept_uniforms.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int,
                                               ctypes.c_int, _P]
        lib.oracle_accept_uniforms.restype = None
        lib.oracle_race_exponentials.argtypes = [ctypes.c_uint64, ctypes.c_uint32,
                                                 ctypes.c_uint32, ctypes.c_uint32,
                                                 ctypes.c_int64, _P]
        lib.oracle_race_exponentials.restype = None
        lib.oracle_row_log_normalisers.argtypes = [ctypes.c_int, _P, ctypes.c_int, ctypes.c_int,
                                                   _P, _P]
        lib.oracle_row_log_normalisers.restype = None
        lib.oracle_row_overlap.argtypes = [ctypes.c_int, _P, _P, ctypes.c_int, ctypes.c_int,
                                           _P, _P, _P]
        lib.oracle_row_overlap.restype = None
        lib.oracle_position_stats.argtypes = [ctypes.c_int, _P, _P, ctypes.c_int, ctypes.c_int,
                                              ctypes.c_int, _P, _P, _P, _P, _P]
        lib.oracle_position_stats.restype = None
        lib.oracle_row_kl.argtypes = [ctypes.c_int, _P, _P, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_double, ctypes.c_double, _P]
        lib.oracle_row_kl.restype = None
        lib.oracle_row_entropies.argtypes = [ctypes.c_int, _P, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_double, _P]
        lib.oracle_row_entropies.restype = None
        lib.oracle_entropy_centres_update.argtypes = [ctypes.c_int, ctypes.c_int, _P, _P,
                                                      ctypes.c_double, _P]
        lib.oracle_entropy_centres_update.restype = None
        lib.oracle_soft_accept.argtypes = [ctypes.c_double, ctypes.c_double, ctypes.c_double]
        lib.oracle_soft_accept.restype = ctypes.c_double
        lib.oracle_adaptive_k.argtypes = [ctypes.c_int, ctypes.c_int, _P, _P, _P, ctypes.c_int,
                                          ctypes.c_double, ctypes.c_double, _P, _P]
        lib.oracle_adaptive_k.restype = ctypes.c_int
        lib.oracle_verify_tree.argtypes = [ctypes.c_int, _P, _P, _P, _P, ctypes.c_int,
                                           ctypes.c_int, ctypes.c_int, _P, _P, ctypes.c_uint64,
                                           ctypes.c_uint32, _P, _P, _P, _P]
        lib.oracle_verify_tree.restype = ctypes.c_int
        lib.oracle_verify.argtypes = [ctypes.c_int, _P, _P, _P, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_int, _P, _P, ctypes.c_uint64, ctypes.c_uint32,
                                      _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]
        lib.oracle_verify.restype = ctypes.c_int
        lib.oracle_verify_greedy.argtypes = [ctypes.c_int, _P, _P, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int, _P, _P, _P]
        lib.oracle_verify_greedy.restype = ctypes.c_int
        self.lib = lib

    # -- random numbers --------------------------------------------------------------
    def philox(self, counter, key) -> np.ndarray:
        c = np.ascontiguousarray(counter, dtype=np.uint32)
        k = np.ascontiguousarray(key, dtype=np.uint32)
        out = np.zeros(4, dtype=np.uint32)
        self.lib.oracle_philox4x32_10(c.ctypes.data, k.ctypes.data, out.ctypes.data)
        return out

    def philox_bulk(self, counters, keys) -> np.ndarray:
        c = np.ascontiguousarray(counters, dtype=np.uint32).reshape(-1, 4)
        k = np.ascontiguousarray(keys, dtype=np.uint32).reshape(-1, 2)
        assert c.shape[0] == k.shape[0]
        out = np.zeros_like(c)
        self.lib.oracle_philox_bulk(c.ctypes.data, k.ctypes.data, c.shape[0], out.ctypes.data)
        return out

    def accept_uniforms(self, seed: int, B: int, gamma: int, b_base: int = 0) -> np.ndarray:
        out = np.zeros((B, gamma), np.float64)
        self.lib.oracle_accept_uniforms(seed, b_base, B, gamma, out.ctypes.data)
        return out

    def race_exponentials(self, seed: int, b: int, pos: int, n: int, x0: int = 0) -> np.ndarray:
        out = np.zeros(n, np.float64)
        self.lib.oracle_race_exponentials(seed, b, pos, x0, n, out.ctypes.data)
        return out

    def accept_uniform(self, seed: int, b: int, i: int) -> float:
        return self.lib.oracle_accept_uniform(seed, b, i)

    def race_exponential(self, seed: int, b: int, pos: int, x: int) -> float:
        return self.lib.oracle_race_exponential(seed, b, pos, x)

    # -- row statistics --------------------------------------------------------------
    def row_log_normalisers(self, rows: np.ndarray, temps) -> np.ndarray:
        dtype, a = _logits(rows)
        R, V = a.shape[0], a.shape[1]
        t = np.ascontiguousarray(np.broadcast_to(np.asarray(temps, np.float64), (R,)))
        out = np.zeros(R, dtype=np.float64)
        self.lib.oracle_row_log_normalisers(dtype, a.ctypes.data, R, V, t.ctypes.data,
                                            out.ctypes.data)
        return out

    def row_overlap(self, target_rows, draft_rows, T, Td) -> np.ndarray:
        dtype, a = _logits(target_rows)
        dtype2, d = _logits(draft_rows)
        assert dtype == dtype2 and a.shape == d.shape
        R, V = a.shape
        t = np.ascontiguousarray(np.broadcast_to(np.asarray(T, np.float64), (R,)))
        td = np.ascontiguousarray(np.broadcast_to(np.asarray(Td, np.float64), (R,)))
        out = np.zeros(R, dtype=np.float64)
        self.lib.oracle_row_overlap(dtype, a.ctypes.data, d.ctypes.data, R, V, t.ctypes.data,
                                    td.ctypes.data, out.ctypes.data)
        return out

    # -- per-position statistics and the adaptive draft length ([SPARSESPEC] section 3.3)
    def position_stats(self, target, draft, T, Td):
        """(H(p_i) [B, g+1], H(q_i) [B, g], KL(p_i || q_i) [B, g]) in nats, fp64."""
        dtype, t = _logits(target)
        dtype2, d = _logits(draft)
        assert dtype == dtype2
        B, G1, V = t.shape
        g = G1 - 1
        assert d.shape == (B, g, V)
        Tb = np.ascontiguousarray(np.broadcast_to(np.asarray(T, np.float64), (B,)))
        Tdb = np.ascontiguousarray(np.broadcast_to(np.asarray(Td, np.float64), (B,)))
        hp, hq, kl = np.zeros((B, g + 1)), np.zeros((B, g)), np.zeros((B, g))
        self.lib.oracle_position_stats(dtype, t.ctypes.data, d.ctypes.data, B, g, V,
                                       Tb.ctypes.data, Tdb.ctypes.data, hp.ctypes.data,
                                       hq.ctypes.data, kl.ctypes.data)
        return hp, hq, kl

    def row_entropies(self, rows, temp: float) -> np.ndarray:
        dtype, a = _logits(rows)
        R, V = a.shape
        out = np.zeros(R)
        self.lib.oracle_row_entropies(dtype, a.ctypes.data, R, V, float(temp), out.ctypes.data)
        return out

    def row_kl(self, target_rows, draft_rows, T: float, Td: float) -> np.ndarray:
        dtype, a = _logits(target_rows)
        dtype2, d = _logits(draft_rows)
        assert dtype == dtype2 and a.shape == d.shape
        R, V = a.shape
        out = np.zeros(R)
        self.lib.oracle_row_kl(dtype, a.ctypes.data, d.ctypes.data, R, V, float(T), float(Td),
                               out.ctypes.data)
        return out

    def entropy_centres_update(self, Hq, n_accepted, beta: float, centres) -> np.ndarray:
        """New class centres [B, 2] (accepted, rejected) after one verify."""
        h = np.ascontiguousarray(Hq, dtype=np.float64)
        B, g = h.shape
        n = np.ascontiguousarray(n_accepted, dtype=np.int32).reshape(B)
        c = np.array(centres, dtype=np.float64, copy=True).reshape(B, 2)
        self.lib.oracle_entropy_centres_update(B, g, h.ctypes.data, n.ctypes.data,
                                               float(beta), c.ctypes.data)
        return c

    def soft_accept(self, H: float, c_acc: float, c_rej: float) -> float:
        return self.lib.oracle_soft_accept(float(H), float(c_acc), float(c_rej))

    def adaptive_k(self, H, centres, candidates, Cd: float, Cv: float):
        """(k* [B] int32, best efficiency [B]) from the next K draft entropies H [B, K]."""
        h = np.ascontiguousarray(H, dtype=np.float64)
        B, K = h.shape
        c = np.ascontiguousarray(centres, dtype=np.float64).reshape(B, 2)
        cand = np.ascontiguousarray(candidates, dtype=np.int32)
        k = np.zeros(B, np.int32)
        eff = np.zeros(B)
        rc = self.lib.oracle_adaptive_k(B, K, h.ctypes.data, c.ctypes.data, cand.ctypes.data,
                                        len(cand), float(Cd), float(Cv), k.ctypes.data,
                                        eff.ctypes.data)
        if rc != 0:
            raise ValueError("oracle_adaptive_k: candidates must lie in 1..K")
        return k, eff

    # -- the verify step ---------------------------------------------------------------
    def verify(self, target, draft, tokens, T, Td, seed: int, b_base: int = 0) -> "OracleResult":
        """Sampling-mode verify.  target [B, g+1, V], draft [B, g, V] as float32 arrays or
        uint16 arrays holding bf16 bits; tokens [B, g]; T, Td scalars or [B]."""
        dtype, t = _logits(target)
        dtype2, d = _logits(draft)
        assert dtype == dtype2
        B, G1, V = t.shape
        g = G1 - 1
        assert d.shape == (B, g, V), (d.shape, (B, g, V))
        tok = np.ascontiguousarray(tokens, dtype=np.int32).reshape(B, g)
        Tb = np.ascontiguousarray(np.broadcast_to(np.asarray(T, np.float64), (B,)))
        Tdb = np.ascontiguousarray(np.broadcast_to(np.asarray(Td, np.float64), (B,)))
        r = OracleResult(
            tokens=np.zeros((B, g + 1), np.int32), n_accepted=np.zeros(B, np.int32),
            logp=np.zeros((B, g)), logq=np.zeros((B, g)), u=np.zeros((B, g)),
            a=np.zeros((B, g)), logZp=np.zeros((B, g + 1)), logZq=np.zeros((B, g)),
            race=np.zeros((B, 3)), flags=np.zeros(B, np.int32))
        rc = self.lib.oracle_verify(
            dtype, t.ctypes.data, d.ctypes.data, tok.ctypes.data, B, g, V, Tb.ctypes.data,
            Tdb.ctypes.data, seed, b_base, r.tokens.ctypes.data, r.n_accepted.ctypes.data,
            r.logp.ctypes.data, r.logq.ctypes.data, r.u.ctypes.data, r.a.ctypes.data,
            r.logZp.ctypes.data, r.logZq.ctypes.data, r.race.ctypes.data, r.flags.ctypes.data)
        if rc != 0:
            raise ValueError("oracle_verify rejected its arguments")
        return r

    def verify_tree(self, target, draft, tokens, parent, T, Td, seed: int, b_base: int = 0):
        """Token-tree verify.  target [B, N, V], draft [B, M, V] (M internal nodes), tokens
        [B, N], parent [N].  Returns (tokens [B, D+1], nodes [B, D], n [B], flags [B])."""
        dtype, t = _logits(target)
        dtype2, d = _logits(draft)
        assert dtype == dtype2
        B, N, V = t.shape
        par = np.ascontiguousarray(parent, dtype=np.int32)
        assert par.shape == (N,)
        depth = np.zeros(N, np.int64)
        for n in range(1, N):
            depth[n] = depth[par[n]] + 1
        D = int(depth.max()) if N > 1 else 0
        tok = np.ascontiguousarray(tokens, dtype=np.int32).reshape(B, N)
        Tb = np.ascontiguousarray(np.broadcast_to(np.asarray(T, np.float64), (B,)))
        Tdb = np.ascontiguousarray(np.broadcast_to(np.asarray(Td, np.float64), (B,)))
        out_t = np.zeros((B, D + 1), np.int32)
        out_nodes = np.zeros((B, max(D, 1)), np.int32)
        out_n = np.zeros(B, np.int32)
        flags = np.zeros(B, np.int32)
        rc = self.lib.oracle_verify_tree(dtype, t.ctypes.data, d.ctypes.data, tok.ctypes.data,
                                         par.ctypes.data, B, N, V, Tb.ctypes.data, Tdb.ctypes.data,
                                         seed, b_base, out_t.ctypes.data, out_nodes.ctypes.data,
                                         out_n.ctypes.data, flags.ctypes.data)
        if rc != 0:
            raise ValueError("oracle_verify_tree rejected its arguments")
        return out_t, out_nodes[:, :D], out_n, flags

    def verify_greedy(self, target, tokens):
        dtype, t = _logits(target)
        B, G1, V = t.shape
        g = G1 - 1
        tok = np.ascontiguousarray(tokens, dtype=np.int32).reshape(B, g)
        out_t = np.zeros((B, g + 1), np.int32)
        out_n = np.zeros(B, np.int32)
        argmax = np.zeros((B, g + 1), np.int32)
        rc = self.lib.oracle_verify_greedy(dtype, t.ctypes.data, tok.ctypes.data, B, g, V,
                                           out_t.ctypes.data, out_n.ctypes.data,
                                           argmax.ctypes.data)
        if rc != 0:
            raise ValueError("oracle_verify_greedy rejected its arguments")
        return out_t, out_n, argmax


@dataclass
class OracleResult:
    tokens: np.ndarray      # [B, g+1] int32, -1 padded
    n_accepted: np.ndarray  # [B] int32 (-1 = bad draft token)
    logp: np.ndarray        # [B, g] ln p_i(d_i)
    logq: np.ndarray        # [B, g] ln q_i(d_i)
    u: np.ndarray           # [B, g] acceptance uniforms
    a: np.ndarray           # [B, g] p/q at the draft tokens
    logZp: np.ndarray       # [B, g+1] ln of the target normalisers at T
    logZq: np.ndarray       # [B, g] ln of the draft normalisers at T_d
    race: np.ndarray        # [B, 3] best score, second score, row raced
    flags: np.ndarray       # [B] FLAG_* bits


def _logits(a):
    """(dtype code, contiguous array) for float32 logits or uint16 bf16 bit patterns."""
    a = np.asarray(a)
    if a.dtype == np.float32:
        return F32, np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return BF16, np.ascontiguousarray(a)
    raise TypeError(f"oracle logits must be float32 or uint16 (bf16 bits), got {a.dtype}")


_default = None


def get() -> Oracle:
    """The default compiled oracle (built on first use)."""
    global _default
    if _default is None:
        _default = Oracle()
    return _default
