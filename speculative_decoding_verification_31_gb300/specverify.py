"""Python binding of libspecverify (ctypes): argument marshalling only.

Every step of the verify path runs in the CUDA library; this module checks tensor shapes,
allocates outputs with PyTorch when the caller gives none, and passes raw device pointers
and the CUDA stream handle through the C ABI declared in ``include/specverify.h``.  There
is no fallback: if the compiled library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libspecverify.so")
CHECKED_LIB_PATH = os.path.join(_HERE, "libspecverify_checked.so")  # index-checked build (tests)

SPEC_OK, SPEC_EINVAL, SPEC_ECUDA, SPEC_EBADTOKEN, SPEC_ETIMEOUT, SPEC_ENOMEM = range(6)
SPEC_ESCRATCH = 6
SPEC_EINDEX = 7
SPEC_NOALLOC_SCRATCH_BYTES = 8 << 20
SPEC_DEBUG_NEVER_READY, SPEC_FLAG_EARLY_EXIT, SPEC_FLAG_FULL_READ, SPEC_DEBUG_RACE_AGAIN = 2, 4, 8, 16
SPEC_F32, SPEC_BF16 = 0, 1

EXPORTED = ("spec_verify", "spec_verify_greedy", "spec_verify_ex", "spec_verify_greedy_ex",
            "spec_verify_workspace_bytes", "spec_verify_check", "spec_verify_strerror",
            "spec_verify_opts_init", "spec_verify_noalloc", "spec_row_entropy",
            "spec_adaptive_k", "spec_verify_tree", "spec_verify_host", "spec_lmhead_logits",
            "spec_lmhead_row_stats", "spec_verify_lmhead", "spec_vp_state_bytes",
            "spec_vp_partials", "spec_vp_decide", "spec_vp_race", "spec_vp_finish",
            "spec_philox4x32_10")


class SpecVerifyError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {spec_verify_strerror(code)} (status {code})")
        self.code = code


class SpecVerifyOpts(ctypes.Structure):
    """Mirror of ``spec_verify_opts``."""
    _fields_ = [
        ("dtype", ctypes.c_int32),
        ("seq_index_base", ctypes.c_uint32),
        ("T_per_seq", ctypes.c_void_p),
        ("Td_per_seq", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t),
        ("d_status", ctypes.c_void_p),
        ("out_logp_draft", ctypes.c_void_p),
        ("out_logq_draft", ctypes.c_void_p),
        ("out_logZ_p", ctypes.c_void_p),
        ("out_logZ_q", ctypes.c_void_p),
        ("out_u", ctypes.c_void_p),
        ("out_race", ctypes.c_void_p),
        ("prof_events", ctypes.c_void_p * 4),
        ("flags", ctypes.c_uint32),
        ("out_H_p", ctypes.c_void_p),
        ("out_H_q", ctypes.c_void_p),
        ("out_KL", ctypes.c_void_p),
        ("ctrl_centres", ctypes.c_void_p),
        ("ctrl_beta", ctypes.c_double),
    ]


_lib = None


def use_library(path: str) -> ctypes.CDLL:
    """Make every entry point of this module call the library at `path` from now on (the
    index-checked build, for tests); returns it."""
    global _lib
    _lib = None
    return load_library(path)


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libspecverify.so (built by ``build.build()``); raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libspecverify.so is not built ({path}); run "
                           "`python -m speculative_decoding_verification_31_gb300.build`")
    lib = ctypes.CDLL(path)
    P, I, U64, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64, ctypes.c_float
    OP = ctypes.POINTER(SpecVerifyOpts)
    lib.spec_verify.argtypes = [P, P, P, I, I, I, F, F, U64, P, P, P]
    lib.spec_verify_greedy.argtypes = [P, P, I, I, I, P, P, P]
    lib.spec_verify_ex.argtypes = [P, P, P, I, I, I, F, F, U64, P, P, OP, P]
    lib.spec_verify_greedy_ex.argtypes = [P, P, I, I, I, P, P, OP, P]
    lib.spec_verify_noalloc.argtypes = [P, P, P, I, I, I, F, F, U64, P, P, OP, P]
    for f in ("spec_verify", "spec_verify_greedy", "spec_verify_ex", "spec_verify_greedy_ex",
              "spec_verify_noalloc"):
        getattr(lib, f).restype = ctypes.c_int
    lib.spec_verify_workspace_bytes.argtypes = [I, I, I, I]
    lib.spec_verify_workspace_bytes.restype = ctypes.c_size_t
    lib.spec_verify_check.argtypes = [P, P]
    lib.spec_verify_check.restype = ctypes.c_int
    lib.spec_verify_strerror.argtypes = [I]
    lib.spec_verify_strerror.restype = ctypes.c_char_p
    lib.spec_verify_opts_init.argtypes = [OP]
    lib.spec_verify_opts_init.restype = None
    lib.spec_verify_lmhead.argtypes = [P, P, P, P, P, I, I, I, I, F, F, U64, P, P, OP, P]
    lib.spec_verify_lmhead.restype = ctypes.c_int
    lib.spec_lmhead_logits.argtypes = [P, P, I, I, I, P, P]
    lib.spec_lmhead_logits.restype = ctypes.c_int
    lib.spec_lmhead_row_stats.argtypes = [P, P, I, I, I, P, P, P, P, P]
    lib.spec_lmhead_row_stats.restype = ctypes.c_int
    lib.spec_verify_host.argtypes = [P, P, P, I, I, I, F, F, U64, P, P, OP, P]
    lib.spec_verify_host.restype = ctypes.c_int
    lib.spec_verify_tree.argtypes = [P, P, P, P, I, I, I, F, F, U64, P, P, P, OP, P]
    lib.spec_verify_tree.restype = ctypes.c_int
    lib.spec_row_entropy.argtypes = [P, I, I, F, I, P, P]
    lib.spec_row_entropy.restype = ctypes.c_int
    D = ctypes.c_double
    lib.spec_adaptive_k.argtypes = [P, I, I, P, P, I, D, D, P, P, P]
    lib.spec_adaptive_k.restype = ctypes.c_int
    lib.spec_vp_state_bytes.argtypes = [I]
    lib.spec_vp_state_bytes.restype = ctypes.c_size_t
    lib.spec_vp_partials.argtypes = [P, P, P, I, I, I, I, F, F, P, P, OP, P]
    lib.spec_vp_decide.argtypes = [P, I, P, P, I, I, I, F, F, U64, P, P, P, OP, P]
    lib.spec_vp_race.argtypes = [P, P, I, I, I, I, U64, P, P, OP, P]
    lib.spec_vp_finish.argtypes = [P, P, I, I, P, P]
    for f in ("spec_vp_partials", "spec_vp_decide", "spec_vp_race", "spec_vp_finish"):
        getattr(lib, f).restype = ctypes.c_int
    lib.spec_philox4x32_10.argtypes = [P, P, ctypes.c_int64, I, P, P]
    lib.spec_philox4x32_10.restype = ctypes.c_int
    _lib = lib
    return lib


def _call(device, name: str, *args) -> int:
    """Call entry point `name` with `device` current: the library finds its per-device state
    (workspace, status word, SM count) through the current device, which must be the device
    of the tensors and of the stream the call is given.  The device is switched (and
    switched back) only when it is not current already."""
    fn = getattr(load_library(), name)
    idx = device.index if isinstance(device, torch.device) else device
    if idx is None or idx == torch.cuda.current_device():
        return fn(*args)
    with torch.cuda.device(device):
        return fn(*args)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


# The current stream's raw handle without building a torch.cuda.Stream object (which costs
# about 2 us of host time per call); torch.cuda.current_stream where torch lacks the accessor.
_current_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream_handle(stream, device) -> ctypes.c_void_p:
    if stream is None and _current_raw_stream is not None:
        idx = device.index if isinstance(device, torch.device) else device
        if idx is None:
            idx = torch.cuda.current_device()
        return ctypes.c_void_p(_current_raw_stream(idx))
    if stream is None:
        stream = torch.cuda.current_stream(device)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return SPEC_BF16
    if t.dtype == torch.float32:
        return SPEC_F32
    raise TypeError(f"logits must be bfloat16 or float32, got {t.dtype}")


def _check_shapes(target, draft, tokens, greedy=False):
    if target.dim() != 3 or not target.is_cuda or not target.is_contiguous():
        raise ValueError("target_logits must be a contiguous CUDA tensor [B, gamma+1, V]")
    B, G1, V = target.shape
    g = G1 - 1
    if not greedy and g > 0:
        if draft is None or tuple(draft.shape) != (B, g, V) or not draft.is_contiguous():
            raise ValueError(f"draft_logits must be contiguous [B, gamma, V] = {(B, g, V)}")
        if draft.dtype != target.dtype:
            raise TypeError("target and draft logits must have the same dtype")
    if g > 0:
        if tokens is None or tuple(tokens.shape) != (B, g) or tokens.dtype != torch.int32 \
                or not tokens.is_contiguous():
            raise ValueError(f"draft_tokens must be contiguous int32 [B, gamma] = {(B, g)}")
    return B, g, V


def _outputs(target, B, g, out_tokens, out_n):
    dev = target.device
    if out_tokens is None:
        out_tokens = torch.empty((B, g + 1), dtype=torch.int32, device=dev)
    if out_n is None:
        out_n = torch.empty((B,), dtype=torch.int32, device=dev)
    return out_tokens, out_n


def spec_verify(target_logits, draft_logits, draft_tokens, T: float, T_d: float, seed: int,
                out_tokens=None, out_n_accepted=None, stream=None):
    """Sampling-mode verify on bf16 logits (see ``spec_verify`` in the C header).
    Returns (out_tokens [B, gamma+1] int32, out_n_accepted [B] int32), both on the device."""
    B, g, V = _check_shapes(target_logits, draft_logits, draft_tokens)
    if target_logits.dtype != torch.bfloat16:
        raise TypeError("spec_verify takes bf16 logits; use spec_verify_ex for float32")
    out_tokens, out_n_accepted = _outputs(target_logits, B, g, out_tokens, out_n_accepted)
    rc = _call(target_logits.device, "spec_verify",
        _ptr(target_logits), _ptr(draft_logits), _ptr(draft_tokens), B, g, V, T, T_d,
        int(seed) & (2**64 - 1), _ptr(out_tokens), _ptr(out_n_accepted),
        _stream_handle(stream, target_logits.device))
    if rc != SPEC_OK:
        raise SpecVerifyError(rc, "spec_verify")
    return out_tokens, out_n_accepted


def spec_verify_greedy(target_logits, draft_tokens, out_tokens=None, out_n_accepted=None,
                       stream=None):
    """Greedy (argmax-match) verify on bf16 target logits."""
    B, g, V = _check_shapes(target_logits, None, draft_tokens, greedy=True)
    if target_logits.dtype != torch.bfloat16:
        raise TypeError("spec_verify_greedy takes bf16 logits; use spec_verify_greedy_ex")
    out_tokens, out_n_accepted = _outputs(target_logits, B, g, out_tokens, out_n_accepted)
    rc = _call(target_logits.device, "spec_verify_greedy",
        _ptr(target_logits), _ptr(draft_tokens), B, g, V, _ptr(out_tokens),
        _ptr(out_n_accepted), _stream_handle(stream, target_logits.device))
    if rc != SPEC_OK:
        raise SpecVerifyError(rc, "spec_verify_greedy")
    return out_tokens, out_n_accepted


def _make_opts(dtype, T_per_seq, Td_per_seq, seq_index_base, workspace, d_status, diag,
               prof_events: Optional[Sequence], flags: int = 0):
    o = SpecVerifyOpts()  # zero-initialised, as spec_verify_opts_init leaves it
    o.dtype = dtype
    o.flags = int(flags)
    o.seq_index_base = int(seq_index_base)
    o.T_per_seq = T_per_seq.data_ptr() if T_per_seq is not None else None
    o.Td_per_seq = Td_per_seq.data_ptr() if Td_per_seq is not None else None
    if workspace is not None:
        o.workspace = workspace.data_ptr()
        o.workspace_bytes = workspace.numel() * workspace.element_size()
    o.d_status = d_status.data_ptr() if d_status is not None else None
    if diag:
        o.out_logp_draft = diag["logp"].data_ptr()
        o.out_logq_draft = diag["logq"].data_ptr()
        o.out_logZ_p = diag["logZp"].data_ptr()
        o.out_logZ_q = diag["logZq"].data_ptr()
        o.out_u = diag["u"].data_ptr()
        o.out_race = diag["race"].data_ptr()
    if prof_events:
        for k, ev in enumerate(prof_events[:4]):
            if ev is not None and not ev.cuda_event:
                raise ValueError("torch creates a CUDA event on its first record(); record "
                                 "each profiling event once before passing it")
            o.prof_events[k] = ev.cuda_event if ev is not None else None
    return o


def _check_temps(t, B, dev, name):
    if t is None:
        return None
    if tuple(t.shape) != (B,) or t.dtype != torch.float32 or t.device != dev \
            or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous float32 [B] tensor on {dev}")
    return t


def spec_verify_ex(target_logits, draft_logits, draft_tokens, T: float, T_d: float, seed: int,
                   out_tokens=None, out_n_accepted=None, *, T_per_seq=None, Td_per_seq=None,
                   seq_index_base: int = 0, workspace=None, d_status=None,
                   diagnostics: bool = False, position_stats=False,
                   ctrl_centres=None, ctrl_beta: float = 0.0, prof_events=None, flags: int = 0,
                   stream=None):
    """Full form (see ``spec_verify_ex`` in the C header).  Returns
    (out_tokens, out_n_accepted, diag) where diag holds the diagnostic outputs when
    ``diagnostics`` is set (ln p(d_i), ln q(d_i), ln Z_p, ln Z_q, u, race scores) and the
    per-position statistics when ``position_stats`` is set (H_p, H_q, KL; a dict of those
    three float32 tensors is written in place of new ones).  ``ctrl_centres``
    (float64 [B, 2] on the device) is updated in place with rate ``ctrl_beta``."""
    B, g, V = _check_shapes(target_logits, draft_logits, draft_tokens)
    dev = target_logits.device
    out_tokens, out_n_accepted = _outputs(target_logits, B, g, out_tokens, out_n_accepted)
    T_per_seq = _check_temps(T_per_seq, B, dev, "T_per_seq")
    Td_per_seq = _check_temps(Td_per_seq, B, dev, "Td_per_seq")
    diag = None
    if diagnostics:
        f = dict(dtype=torch.float32, device=dev)
        diag = {"logp": torch.full((B, g), float("nan"), **f),
                "logq": torch.full((B, g), float("nan"), **f),
                "logZp": torch.full((B, g + 1), float("nan"), **f),
                "logZq": torch.full((B, g), float("nan"), **f),
                "u": torch.full((B, g), float("nan"), **f),
                "race": torch.full((B, 2), float("nan"), **f)}
    o = _make_opts(_dtype_code(target_logits), T_per_seq, Td_per_seq, seq_index_base, workspace,
                   d_status, diag, prof_events, flags)
    if position_stats:
        diag = dict(diag or {})
        if isinstance(position_stats, dict):  # caller-allocated outputs
            for k, shape in (("Hp", (B, g + 1)), ("Hq", (B, g)), ("KL", (B, g))):
                t = position_stats[k]
                if tuple(t.shape) != shape or t.dtype != torch.float32 or not t.is_contiguous():
                    raise ValueError(f"position_stats[{k!r}] must be contiguous float32 {shape}")
                diag[k] = t
        else:
            f = dict(dtype=torch.float32, device=dev)
            diag.update(Hp=torch.full((B, g + 1), float("nan"), **f),
                        Hq=torch.full((B, g), float("nan"), **f),
                        KL=torch.full((B, g), float("nan"), **f))
        o.out_H_p, o.out_H_q, o.out_KL = (diag[k].data_ptr() for k in ("Hp", "Hq", "KL"))
    if ctrl_centres is not None:
        if tuple(ctrl_centres.shape) != (B, 2) or ctrl_centres.dtype != torch.float64 \
                or ctrl_centres.device != dev or not ctrl_centres.is_contiguous():
            raise ValueError(f"ctrl_centres must be a contiguous float64 [B, 2] tensor on {dev}")
        o.ctrl_centres = ctrl_centres.data_ptr()
        o.ctrl_beta = float(ctrl_beta)
    rc = _call(dev, "spec_verify_ex",
        _ptr(target_logits), _ptr(draft_logits), _ptr(draft_tokens), B, g, V, float(T),
        float(T_d), int(seed) & (2**64 - 1), _ptr(out_tokens), _ptr(out_n_accepted),
        ctypes.byref(o), _stream_handle(stream, dev))
    if rc != SPEC_OK:
        raise SpecVerifyError(rc, "spec_verify_ex")
    return out_tokens, out_n_accepted, diag


def spec_verify_greedy_ex(target_logits, draft_tokens, out_tokens=None, out_n_accepted=None, *,
                          workspace=None, d_status=None, prof_events=None, stream=None):
    B, g, V = _check_shapes(target_logits, None, draft_tokens, greedy=True)
    dev = target_logits.device
    out_tokens, out_n_accepted = _outputs(target_logits, B, g, out_tokens, out_n_accepted)
    o = _make_opts(_dtype_code(target_logits), None, None, 0, workspace, d_status, None,
                   prof_events)
    rc = _call(dev, "spec_verify_greedy_ex",
        _ptr(target_logits), _ptr(draft_tokens), B, g, V, _ptr(out_tokens), _ptr(out_n_accepted),
        ctypes.byref(o), _stream_handle(stream, dev))
    if rc != SPEC_OK:
        raise SpecVerifyError(rc, "spec_verify_greedy_ex")
    return out_tokens, out_n_accepted


def spec_verify_noalloc(target_logits, draft_logits, draft_tokens, T: float, T_d: float,
                        seed: int, out_tokens, out_n_accepted, *, T_per_seq=None,
                        Td_per_seq=None, seq_index_base: int = 0, d_status=None, diag=None,
                        flags: int = 0, stream=None):
    """Allocation-free sampling verify (see ``spec_verify_noalloc`` in the C header): the
    library's scratch is a static device array, so nothing is allocated by the library.  The
    caller passes every output, including the optional diagnostic tensors in ``diag`` (a dict
    with the keys of ``spec_verify_ex``'s diagnostics)."""
    B, g, V = _check_shapes(target_logits, draft_logits, draft_tokens)
    dev = target_logits.device
    if out_tokens is None or out_n_accepted is None:
        raise ValueError("spec_verify_noalloc needs caller-allocated outputs")
    T_per_seq = _check_temps(T_per_seq, B, dev, "T_per_seq")
    Td_per_seq = _check_temps(Td_per_seq, B, dev, "Td_per_seq")
    o = _make_opts(_dtype_code(target_logits), T_per_seq, Td_per_seq, seq_index_base, None,
                   d_status, diag, None, flags)
    rc = _call(dev, "spec_verify_noalloc",
        _ptr(target_logits), _ptr(draft_logits), _ptr(draft_tokens), B, g, V, float(T),
        float(T_d), int(seed) & (2**64 - 1), _ptr(out_tokens), _ptr(out_n_accepted),
        ctypes.byref(o), _stream_handle(stream, dev))
    if rc != SPEC_OK:
        raise SpecVerifyError(rc, "spec_verify_noalloc")
    return out_tokens, out_n_accepted


def spec_verify_host(target_logits, draft_logits, draft_tokens, T: float, T_d: float, seed: int,
                     out_tokens, out_n_accepted, *, T_per_seq=None, Td_per_seq=None,
                     seq_index_base: int = 0, full_read: bool = False, stream=None):
    """Sampling verify on pinned host tensors (see ``spec_verify_host`` in the C header): the
    kernels read the logits and write the outputs in place over the host link.  Every
    tensor is a contiguous pinned CPU tensor (or a CUDA tensor); the outputs are valid once
    the stream has finished."""
    for name, t in (("target_logits", target_logits), ("draft_logits", draft_logits),
                    ("draft_tokens", draft_tokens), ("out_tokens", out_tokens),
                    ("out_n_accepted", out_n_accepted)):
        if t is not None and t.numel() and not t.is_cuda and not t.is_pinned():
            raise ValueError(f"{name} must be pinned host memory or a CUDA tensor")
        if t is not None and not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    B, G1, V = target_logits.shape
    g = G1 - 1
    dev = torch.device("cuda", torch.cuda.current_device())
    o = _make_opts(_dtype_code(target_logits), T_per_seq, Td_per_seq, seq_index_base, None,
                   None, None, None, SPEC_FLAG_FULL_READ if full_read else 0)
    if g == 0:  # nothing to read: no draft rows or tokens
        draft_logits = draft_tokens = None
    rc = _call(dev, "spec_verify_host",
        _ptr(target_logits), _ptr(draft_logits), _ptr(draft_tokens), B, g, V, float(T),
        float(T_d), int(seed) & (2**64 - 1), _ptr(out_tokens), _ptr(out_n_accepted),
        ctypes.byref(o), _stream_handle(stream, dev))
    if rc != SPEC_OK:
        raise SpecVerifyError(rc, "spec_verify_host")
    return out_tokens, out_n_accepted


def _check_lmhead(hidden, weight):
    for name, t in (("hidden", hidden), ("weight", weight)):
        if t.dim() != 2 or t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bf16 CUDA matrix")
    if hidden.shape[1] != weight.shape[1]:
        raise ValueError("hidden [rows, d] and weight [V, d] must share d")
    return hidden.shape[0], weight.shape[0], hidden.shape[1]


def spec_lmhead_logits(hidden, weight, out_logits=None, stream=None):
    """Logits hidden @ weight^T (fp32) on the tensor cores."""
    rows, V, d = _check_lmhead(hidden, weight)
    if out_logits is None:
        out_logits = torch.empty((rows, V), dtype=torch.float32, device=hidden.device)
    rc = _call(hidden.device, "spec_lmhead_logits", _ptr(hidden), _ptr(weight), rows, V, d, _ptr(out_logits),
                                           _stream_handle(stream, hidden.device))
    if rc != SPEC_OK:
        raise SpecVerifyError(rc, "spec_lmhead_logits")
    return out_logits


def spec_lmhead_row_stats(hidden, weight, T_row, token_row=None, stream=None):
    """(ln Z [rows], ln p(token) [rows] or None) of softmax(hidden @ weight^T / T_row)
    without writing the logits."""
    rows, V, d = _check_lmhead(hidden, weight)
    dev = hidden.device
    logz = torch.empty((rows,), dtype=torch.float32, device=dev)
    logp = torch.empty((rows,), dtype=torch.float32, device=dev) if token_row is not None else None
    rc = _call(dev, "spec_lmhead_row_stats", _ptr(hidden), _ptr(weight), rows, V, d, _ptr(T_row),
                                              _ptr(token_row), _ptr(logz), _ptr(logp),
                                              _stream_handle(stream, dev))
    if rc != SPEC_OK:
        raise SpecVerifyError(rc, "spec_lmhead_row_stats")
    return logz, logp


def spec_verify_lmhead(h_target, w_target, h_draft, w_draft, draft_tokens, T: float, T_d: float,
                       seed: int, out_tokens=None, out_n_accepted=None, *, T_per_seq=None,
                       Td_per_seq=None, seq_index_base: int = 0, prof_events=None, flags: int = 0,
                       stream=None):
    """Sampling verify from hidden states (see ``spec_verify_lmhead`` in the C header):
    h_target bf16 [B, gamma+1, d], w_target [V, d], h_draft [B, gamma, d], w_draft [V, d]."""
    if h_target.dim() != 3 or h_target.dtype != torch.bfloat16 or not h_target.is_contiguous():
        raise ValueError("h_target must be a contiguous bf16 tensor [B, gamma+1, d]")
    B, G1, d = h_target.shape
    g = G1 - 1
    V = w_target.shape[0]
    for name, t, shape in (("w_target", w_target, (V, d)), ("h_draft", h_draft, (B, g, d)),
                           ("w_draft", w_draft, (V, d))):
        if g == 0 and name != "w_target":
            continue
        if tuple(t.shape) != shape or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bf16 tensor {shape}")
    dev = h_target.device
    out_tokens, out_n_accepted = _outputs(h_target, B, g, out_tokens, out_n_accepted)
    T_per_seq = _check_temps(T_per_seq, B, dev, "T_per_seq")
    Td_per_seq = _check_temps(Td_per_seq, B, dev, "Td_per_seq")
    o = _make_opts(SPEC_BF16, T_per_seq, Td_per_seq, seq_index_base, None, None, None, prof_events, flags)
    rc = _call(dev, "spec_verify_lmhead",
        _ptr(h_target), _ptr(w_target), _ptr(h_draft) if g else None, _ptr(w_draft) if g else None,
        _ptr(draft_tokens) if g else None, B, g, V, d, float(T), float(T_d), int(seed) & (2**64 - 1),
        _ptr(out_tokens), _ptr(out_n_accepted), ctypes.byref(o), _stream_handle(stream, dev))
    if rc != SPEC_OK:
        raise SpecVerifyError(rc, "spec_verify_lmhead")
    return out_tokens, out_n_accepted


class Tree:
    """A static token tree prepared once for spec_verify_tree: the parent array as the C
    call takes it, and its node, internal-node and depth counts."""

    def __init__(self, parent: Sequence[int]):
        par = [int(x) for x in parent]
        self.N = len(par)
        self.valid = self.N >= 1 and par[0] == -1 and all(0 <= par[n] < n for n in range(1, self.N))
        self.M = len({par[v] for v in range(1, self.N)}) if self.valid else 0
        depth = [0] * self.N
        if self.valid:
            for n in range(1, self.N):
                depth[n] = depth[par[n]] + 1
        self.D = max(depth) if depth else 0
        self.c_parent = (ctypes.c_int32 * self.N)(*par)


def spec_verify_tree(target_logits, draft_logits, draft_tokens, tree, T: float, T_d: float,
                     seed: int, *, out_tokens=None, out_nodes=None, out_n_accepted=None,
                     T_per_seq=None, Td_per_seq=None, seq_index_base: int = 0, workspace=None,
                     d_status=None, prof_events=None, stream=None):
    """Token-tree verify (see ``spec_verify_tree`` in the C header).  target [B, N, V],
    draft [B, M, V] (M internal nodes), draft_tokens int32 [B, N]; ``tree``: a Tree or the
    N parent indices.  Returns (out_tokens [B, D+1], out_nodes [B, D], out_n_accepted [B])
    on the device (new tensors unless given).  An invalid tree is passed through: the
    library answers SPEC_EINVAL."""
    if not isinstance(tree, Tree):
        tree = Tree(tree)
    if target_logits.dim() != 3 or not target_logits.is_cuda or not target_logits.is_contiguous():
        raise ValueError("target_logits must be a contiguous CUDA tensor [B, N, V]")
    B, N, V = target_logits.shape
    if tree.N != N:
        raise ValueError(f"the tree must have N = {N} nodes")
    M, D = tree.M, tree.D
    if M and (draft_logits is None or tuple(draft_logits.shape) != (B, M, V)
              or draft_logits.dtype != target_logits.dtype or not draft_logits.is_contiguous()):
        raise ValueError(f"draft_logits must be contiguous [B, M, V] = {(B, M, V)}")
    if tuple(draft_tokens.shape) != (B, N) or draft_tokens.dtype != torch.int32:
        raise ValueError(f"draft_tokens must be int32 [B, N] = {(B, N)}")
    dev = target_logits.device
    if out_tokens is None:
        out_tokens = torch.empty((B, D + 1), dtype=torch.int32, device=dev)
    if out_nodes is None:
        out_nodes = torch.empty((B, max(D, 1)), dtype=torch.int32, device=dev)
    if out_n_accepted is None:
        out_n_accepted = torch.empty((B,), dtype=torch.int32, device=dev)
    T_per_seq = _check_temps(T_per_seq, B, dev, "T_per_seq")
    Td_per_seq = _check_temps(Td_per_seq, B, dev, "Td_per_seq")
    o = _make_opts(_dtype_code(target_logits), T_per_seq, Td_per_seq, seq_index_base, workspace,
                   d_status, None, prof_events)
    rc = _call(dev, "spec_verify_tree",
        _ptr(target_logits), _ptr(draft_logits) if (M or not tree.valid) else None,
        _ptr(draft_tokens), tree.c_parent, B, N, V, float(T), float(T_d), int(seed) & (2**64 - 1),
        _ptr(out_tokens), _ptr(out_nodes), _ptr(out_n_accepted), ctypes.byref(o),
        _stream_handle(stream, dev))
    if rc != SPEC_OK:
        raise SpecVerifyError(rc, "spec_verify_tree")
    return out_tokens, out_nodes[:, :D], out_n_accepted


def spec_row_entropy(logits, T: float, out_H=None, stream=None):
    """Entropy (nats) of softmax(row / T) of every row of a contiguous [rows, V] bf16 or
    float32 CUDA tensor (see ``spec_row_entropy`` in the C header)."""
    if logits.dim() != 2 or not logits.is_cuda or not logits.is_contiguous():
        raise ValueError("logits must be a contiguous CUDA tensor [rows, V]")
    rows, V = logits.shape
    if out_H is None:
        out_H = torch.empty((rows,), dtype=torch.float32, device=logits.device)
    rc = _call(logits.device, "spec_row_entropy", _ptr(logits), rows, V, float(T), _dtype_code(logits),
                                         _ptr(out_H), _stream_handle(stream, logits.device))
    if rc != SPEC_OK:
        raise SpecVerifyError(rc, "spec_row_entropy")
    return out_H


def spec_adaptive_k(H_next, centres, candidates: Sequence[int], C_d: float, C_v: float,
                    out_k=None, out_eff=None, stream=None):
    """Adaptive draft length per sequence (see ``spec_adaptive_k`` in the C header):
    H_next float32 [B, K] and centres float64 [B, 2] on the device; returns (k [B] int32,
    best efficiency [B] float64)."""
    if H_next.dim() != 2 or H_next.dtype != torch.float32 or not H_next.is_contiguous():
        raise ValueError("H_next must be a contiguous float32 [B, K] tensor")
    B, K = H_next.shape
    dev = H_next.device
    if tuple(centres.shape) != (B, 2) or centres.dtype != torch.float64 or not centres.is_contiguous():
        raise ValueError("centres must be a contiguous float64 [B, 2] tensor")
    cand = (ctypes.c_int32 * len(candidates))(*[int(c) for c in candidates])
    if out_k is None:
        out_k = torch.empty((B,), dtype=torch.int32, device=dev)
    if out_eff is None:
        out_eff = torch.empty((B,), dtype=torch.float64, device=dev)
    rc = _call(dev, "spec_adaptive_k", _ptr(H_next), B, K, _ptr(centres), cand, len(candidates),
                                        float(C_d), float(C_v), _ptr(out_k), _ptr(out_eff),
                                        _stream_handle(stream, dev))
    if rc != SPEC_OK:
        raise SpecVerifyError(rc, "spec_adaptive_k")
    return out_k, out_eff


def spec_philox4x32_10(counters, keys, form: int = 0, out=None, stream=None):
    """Diagnostic: the device Philox4x32-10 of counters [n, 4] under keys [n, 2] (int32 CUDA
    tensors holding the uint32 bits), as the verify kernels evaluate it (form 0: plain; form
    1: the race's evaluation, counter word 3 taken as 1).  Returns out [n, 4] (int32 bits)."""
    n = counters.shape[0]
    for name, t, cols in (("counters", counters, 4), ("keys", keys, 2)):
        if tuple(t.shape) != (n, cols) or t.dtype != torch.int32 or not t.is_cuda \
                or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous int32 CUDA tensor [n, {cols}]")
    if out is None:
        out = torch.empty((n, 4), dtype=torch.int32, device=counters.device)
    rc = _call(counters.device, "spec_philox4x32_10", _ptr(counters), _ptr(keys), n, int(form), _ptr(out),
                                           _stream_handle(stream, counters.device))
    if rc != SPEC_OK:
        raise SpecVerifyError(rc, "spec_philox4x32_10")
    return out


def spec_verify_workspace_bytes(B: int, gamma: int, V: int, dtype: int = SPEC_BF16) -> int:
    return int(load_library().spec_verify_workspace_bytes(B, gamma, V, dtype))


def spec_verify_check(stream=None, d_status=None, device=None) -> int:
    """Synchronise the stream and return (and clear) the device status word."""
    if device is None and d_status is not None:
        device = d_status.device
    if device is None:
        return int(load_library().spec_verify_check(_stream_handle(stream, device), _ptr(d_status)))
    return int(_call(device, "spec_verify_check", _stream_handle(stream, device), _ptr(d_status)))


def spec_verify_strerror(code: int) -> str:
    return load_library().spec_verify_strerror(int(code)).decode()
