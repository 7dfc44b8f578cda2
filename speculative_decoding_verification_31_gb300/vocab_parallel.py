"""Vocabulary-parallel sampling verify: the logits split by vocabulary column over ranks.

Rank w holds columns [x_w, x_w + V_w) of every target and draft row (as a tensor-parallel LM
head leaves them).  One verify is four library calls on every rank around two collectives:

    stats, gathered = spec_vp_partials(shard)        # per-row (max, sum) of the shard's
                                                     # columns; logits at owned draft tokens
    all_gather(stats); all_reduce(gathered, MAX)     # O(B gamma) floats
    tokens, n, state = spec_vp_decide(...)           # merge rows in rank order, accept/reject
    keys = spec_vp_race(shard, state)                # race over the shard's columns
    all_reduce(keys, MAX)                            # O(B) int64
    spec_vp_finish(keys, state, tokens)              # the drawn token

The functions here only marshal arguments (the library computes every step) and run the two
collectives through ``torch.distributed``; ``verify_vocab_parallel`` takes a backend object so
that the same orchestration can be exercised with ranks on CPU.
"""
from __future__ import annotations

import ctypes

import torch
import torch.distributed as dist

from .specverify import (SpecVerifyError, SPEC_OK, _call, _check_temps, _dtype_code, _make_opts, _ptr,
                         _stream_handle, load_library)


def vocab_range(V: int, world: int, rank: int) -> tuple[int, int]:
    """[lo, hi) of the vocabulary columns held by `rank` of `world`: contiguous, starting on
    multiples of 8 (the race's random-number blocks and 16-byte vectors stay whole), in blocks
    of 8 columns whose counts differ by at most one (the last block may be short)."""
    if world < 1 or not 0 <= rank < world or V < 1:
        raise ValueError(f"bad vocabulary split: V={V} world={world} rank={rank}")
    n8 = -(-V // 8)
    if n8 < world:
        raise ValueError(f"V={V} is too small to give each of {world} ranks a column block of 8")
    base, extra = divmod(n8, world)
    lo = 8 * (rank * base + min(rank, extra))
    hi = min(V, 8 * ((rank + 1) * base + min(rank + 1, extra)))
    return lo, hi


def _shapes(target_shard, draft_shard, draft_tokens=None, need_tokens=True):
    if target_shard.dim() != 3 or not target_shard.is_cuda or not target_shard.is_contiguous():
        raise ValueError("target_shard must be a contiguous CUDA tensor [B, gamma+1, V_shard]")
    B, g1, Vs = target_shard.shape
    g = g1 - 1
    if g > 0:
        if draft_shard is None or tuple(draft_shard.shape) != (B, g, Vs) or \
                draft_shard.dtype != target_shard.dtype or not draft_shard.is_contiguous():
            raise ValueError(f"draft_shard must be contiguous [B, gamma, V_shard] = {(B, g, Vs)}")
        if need_tokens and (draft_tokens is None or tuple(draft_tokens.shape) != (B, g)
                            or draft_tokens.dtype != torch.int32):
            raise ValueError(f"draft_tokens must be int32 [B, gamma] = {(B, g)}")
    return B, g, Vs


def spec_vp_partials(target_shard, draft_shard, draft_tokens, x_offset: int, T: float, T_d: float, *,
                     T_per_seq=None, Td_per_seq=None, seq_index_base: int = 0, workspace=None,
                     d_status=None, stream=None):
    """(stats [B, 2 gamma + 1, 2], gathered [B, gamma, 2]) of this rank's shard (fp32)."""
    B, g, Vs = _shapes(target_shard, draft_shard, draft_tokens)
    dev = target_shard.device
    stats = torch.empty((B, 2 * g + 1, 2), dtype=torch.float32, device=dev)
    gathered = torch.empty((B, g, 2), dtype=torch.float32, device=dev)
    T_per_seq = _check_temps(T_per_seq, B, dev, "T_per_seq")
    Td_per_seq = _check_temps(Td_per_seq, B, dev, "Td_per_seq")
    o = _make_opts(_dtype_code(target_shard), T_per_seq, Td_per_seq, seq_index_base, workspace,
                   d_status, None, None)
    rc = _call(dev, "spec_vp_partials",
        _ptr(target_shard), _ptr(draft_shard) if g else None, _ptr(draft_tokens) if g else None,
        B, g, Vs, int(x_offset), float(T), float(T_d), _ptr(stats), _ptr(gathered) if g else None,
        ctypes.byref(o), _stream_handle(stream, dev))
    if rc != SPEC_OK:
        raise SpecVerifyError(rc, "spec_vp_partials")
    return stats, gathered


def spec_vp_decide(stats_all, gathered, draft_tokens, V: int, T: float, T_d: float, seed: int, *,
                   dtype_code: int, T_per_seq=None, Td_per_seq=None, seq_index_base: int = 0,
                   d_status=None, stream=None):
    """(out_tokens [B, gamma+1], out_n_accepted [B], state) from every rank's statistics
    stats_all [W, B, 2 gamma + 1, 2] and the max-reduced gathered logits."""
    W, B, R, _ = stats_all.shape
    g = (R - 1) // 2
    dev = stats_all.device
    if not stats_all.is_contiguous() or stats_all.dtype != torch.float32:
        raise ValueError("stats_all must be a contiguous float32 [W, B, 2 gamma + 1, 2] tensor")
    out_t = torch.empty((B, g + 1), dtype=torch.int32, device=dev)
    out_n = torch.empty((B,), dtype=torch.int32, device=dev)
    lib = load_library()
    state = torch.empty((max(1, int(lib.spec_vp_state_bytes(B))),), dtype=torch.uint8, device=dev)
    T_per_seq = _check_temps(T_per_seq, B, dev, "T_per_seq")
    Td_per_seq = _check_temps(Td_per_seq, B, dev, "Td_per_seq")
    o = _make_opts(dtype_code, T_per_seq, Td_per_seq, seq_index_base, None, d_status, None, None)
    rc = _call(dev, "spec_vp_decide", _ptr(stats_all), W, _ptr(gathered) if g else None,
                            _ptr(draft_tokens) if g else None, B, g, int(V), float(T), float(T_d),
                            int(seed) & (2**64 - 1), _ptr(out_t), _ptr(out_n), _ptr(state),
                            ctypes.byref(o), _stream_handle(stream, dev))
    if rc != SPEC_OK:
        raise SpecVerifyError(rc, "spec_vp_decide")
    return out_t, out_n, state


def spec_vp_race(target_shard, draft_shard, x_offset: int, seed: int, state, *,
                 seq_index_base: int = 0, d_status=None, stream=None):
    """keys [B, 2] int64: this rank's race winners (residual, and the p_j fallback)."""
    B, g, Vs = _shapes(target_shard, draft_shard, need_tokens=False)
    dev = target_shard.device
    keys = torch.empty((B, 2), dtype=torch.int64, device=dev)
    o = _make_opts(_dtype_code(target_shard), None, None, seq_index_base, None, d_status, None, None)
    rc = _call(dev, "spec_vp_race", _ptr(target_shard), _ptr(draft_shard) if g else None, B, g, Vs,
                                     int(x_offset), int(seed) & (2**64 - 1), _ptr(state), _ptr(keys),
                                     ctypes.byref(o), _stream_handle(stream, dev))
    if rc != SPEC_OK:
        raise SpecVerifyError(rc, "spec_vp_race")
    return keys


def spec_vp_finish(keys, state, out_tokens, stream=None):
    """Write the drawn tokens (from the max-reduced keys) into out_tokens [B, gamma+1]."""
    B, g1 = out_tokens.shape
    rc = _call(out_tokens.device, "spec_vp_finish", _ptr(keys), _ptr(state), B, g1 - 1, _ptr(out_tokens),
                                       _stream_handle(stream, out_tokens.device))
    if rc != SPEC_OK:
        raise SpecVerifyError(rc, "spec_vp_finish")
    return out_tokens


class LibraryBackend:
    """The four per-rank steps on this rank's GPU (libspecverify)."""

    def partials(self, shard):
        return spec_vp_partials(shard.target, shard.draft, shard.tokens, shard.x_offset, shard.T,
                                shard.T_d, T_per_seq=shard.T_per_seq, Td_per_seq=shard.Td_per_seq,
                                seq_index_base=shard.seq_index_base)

    def decide(self, stats_all, gathered, shard, seed):
        return spec_vp_decide(stats_all, gathered, shard.tokens, shard.V, shard.T, shard.T_d, seed,
                              dtype_code=_dtype_code(shard.target), T_per_seq=shard.T_per_seq,
                              Td_per_seq=shard.Td_per_seq, seq_index_base=shard.seq_index_base)

    def race(self, shard, state, seed):
        return spec_vp_race(shard.target, shard.draft, shard.x_offset, seed, state,
                            seq_index_base=shard.seq_index_base)

    def finish(self, keys, state, tokens):
        return spec_vp_finish(keys, state, tokens)


class VocabShard:
    """This rank's columns [x_offset, x_offset + V_shard) of the target [B, gamma+1, .] and
    draft [B, gamma, .] logits, the draft tokens (global indices), the whole vocabulary size
    V, and the temperatures (scalars, or [B] tensors on the shard's device)."""

    def __init__(self, target, draft, tokens, x_offset: int, V: int, T: float, T_d: float,
                 T_per_seq=None, Td_per_seq=None, seq_index_base: int = 0):
        self.target, self.draft, self.tokens = target, draft, tokens
        self.x_offset, self.V, self.T, self.T_d = int(x_offset), int(V), float(T), float(T_d)
        self.T_per_seq, self.Td_per_seq = T_per_seq, Td_per_seq
        self.seq_index_base = int(seq_index_base)


def _host_staged(group) -> bool:
    """Whether the group's collectives take host tensors (gloo): the exchanged statistics
    and keys (O(B gamma) bytes) then travel through host memory."""
    return dist.get_backend(group) == "gloo"


def _all_gather(t, world, group, staged):
    src = t.cpu() if staged else t.contiguous()
    parts = [torch.empty_like(src) for _ in range(world)]
    dist.all_gather(parts, src, group=group)
    return torch.stack(parts).to(t.device)


def _all_reduce_max(t, group, staged):
    if not staged:
        dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
        return t
    h = t.cpu()
    dist.all_reduce(h, op=dist.ReduceOp.MAX, group=group)
    t.copy_(h)
    return t


def verify_vocab_parallel(shard: VocabShard, seed: int, group=None, backend=None):
    """One sampling verify with the vocabulary split over the ranks of `group` (every rank
    calls this with its own shard; without an initialised process group, one rank holding the
    whole vocabulary).  Returns (out_tokens [B, gamma+1], out_n_accepted [B]), the same on
    every rank."""
    backend = backend or LibraryBackend()
    distributed = dist.is_available() and dist.is_initialized()
    world = dist.get_world_size(group) if distributed else 1
    stats, gathered = backend.partials(shard)
    staged = world > 1 and stats.is_cuda and _host_staged(group)
    if world > 1:
        stats_all = _all_gather(stats, world, group, staged)
        if gathered.numel():
            _all_reduce_max(gathered, group, staged)
    else:
        stats_all = stats.unsqueeze(0)
    tokens, n, state = backend.decide(stats_all.contiguous(), gathered, shard, seed)
    keys = backend.race(shard, state, seed)
    if world > 1:
        _all_reduce_max(keys, group, staged)
    backend.finish(keys, state, tokens)
    return tokens, n
