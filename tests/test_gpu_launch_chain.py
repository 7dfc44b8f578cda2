"""Back-to-back calls of every schedule on one stream (marked gpu).

The streaming kernels are launched as programmatic dependents of whatever kernel precedes
them, and the last kernel of each schedule lets the next launch be set up early; every
schedule shares the per-device workspace.  Calls issued back to back without a host
synchronisation, alternating schedules, shapes and the streaming pass's two launch shapes
(a claiming block per SM for large calls, a warp per piece for small ones), must give the
same bits as the same calls run one at a time, and inputs written by a torch kernel just
before a call must be the ones it reads.
"""
import numpy as np
import pytest
import torch

import workloads
from _parity import DeviceWorkload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_31_gb300 as m
    m.load_library()
    return m


def _calls(sv, dws):
    """(name, thunk) pairs; each thunk enqueues one call and returns its output tensors."""
    out = []
    for k, dw in enumerate(dws):
        w = dw.w
        kw = dict(T_per_seq=dw.T, Td_per_seq=dw.Td)

        def default(dw=dw, w=w, kw=kw, k=k):
            t, n, _ = sv.spec_verify_ex(dw.target, dw.draft, dw.tokens, float(w.T[0]), float(w.Td[0]),
                                        17 + k, **kw)
            return [t, n]

        def early(dw=dw, w=w, kw=kw, k=k):
            t, n, _ = sv.spec_verify_ex(dw.target, dw.draft, dw.tokens, float(w.T[0]), float(w.Td[0]),
                                        17 + k, flags=sv.SPEC_FLAG_EARLY_EXIT, **kw)
            return [t, n]

        def stats(dw=dw, w=w, kw=kw, k=k):
            t, n, d = sv.spec_verify_ex(dw.target, dw.draft, dw.tokens, float(w.T[0]), float(w.Td[0]),
                                        17 + k, position_stats=True, **kw)
            return [t, n, d["Hp"], d["Hq"], d["KL"]]

        def greedy(dw=dw):
            t, n = sv.spec_verify_greedy_ex(dw.target, dw.tokens)
            return [t, n]

        out += [(f"default{k}", default), (f"early{k}", early), (f"stats{k}", stats),
                (f"greedy{k}", greedy)]
    return out


def _host(ts):
    return [t.cpu().numpy().copy() for t in ts]


def test_interleaved_schedules_match_isolated_calls(sv):
    # 24 x 17 rows of 13 pieces: more pieces than the streaming grid has warps (the claiming
    # launch); 3 x 9 rows: one warp per piece
    ws = [workloads.generic(B=24, gamma=8, V=128256, dtype="bf16", seed=5, sigma=0.8, T=0.9, Td=0.45),
          workloads.generic(B=3, gamma=4, V=30011, dtype="bf16", seed=6, sigma=0.8, T=0.9, Td=0.45),
          workloads.generic(B=5, gamma=3, V=4099, dtype="f32", seed=7, sigma=0.8, T=0.9, Td=0.45)]
    dws = [DeviceWorkload(w) for w in ws]
    calls = _calls(sv, dws)
    alone = {}
    for name, f in calls:
        r = f()
        torch.cuda.synchronize()
        alone[name] = _host(r)
    assert sv.spec_verify_check() == sv.SPEC_OK
    rng = np.random.default_rng(0)
    for rep in range(3):
        order = rng.permutation(len(calls))
        pending = [(calls[i][0], calls[i][1]()) for i in order]  # no synchronisation in between
        torch.cuda.synchronize()
        assert sv.spec_verify_check() == sv.SPEC_OK
        for name, r in pending:
            for a, b in zip(_host(r), alone[name]):
                np.testing.assert_array_equal(a, b, err_msg=f"{name}, repetition {rep}")


def test_inputs_written_just_before_a_call_are_read(sv):
    """A torch kernel overwrites the logits on the stream right before each call."""
    w1 = workloads.generic(B=24, gamma=8, V=128256, dtype="bf16", seed=8, sigma=0.8, T=0.9, Td=0.45)
    w2 = workloads.generic(B=24, gamma=8, V=128256, dtype="bf16", seed=9, sigma=0.8, T=0.9, Td=0.45)
    w2.tokens = w1.tokens  # the same draft tokens, other logits
    d1, d2 = DeviceWorkload(w1), DeviceWorkload(w2)
    expect = []
    for dw in (d1, d2):
        t, n, _ = sv.spec_verify_ex(dw.target, dw.draft, dw.tokens, float(w1.T[0]), float(w1.Td[0]), 3,
                                    T_per_seq=dw.T, Td_per_seq=dw.Td)
        g, gn = sv.spec_verify_greedy_ex(dw.target, dw.tokens)
        torch.cuda.synchronize()
        expect.append(_host([t, n, g, gn]))
    buf_t, buf_d = d1.target.clone(), d1.draft.clone()
    outs = []
    for src in (d2, d1, d2, d1):
        buf_t.copy_(src.target)
        buf_d.copy_(src.draft)
        t, n, _ = sv.spec_verify_ex(buf_t, buf_d, d1.tokens, float(w1.T[0]), float(w1.Td[0]), 3,
                                    T_per_seq=src.T, Td_per_seq=src.Td)
        buf_t.copy_(src.target)  # a kernel between the two calls, as between two verifies
        g, gn = sv.spec_verify_greedy_ex(buf_t, d1.tokens)
        outs.append((src is d2, [t, n, g, gn]))
    torch.cuda.synchronize()
    assert sv.spec_verify_check() == sv.SPEC_OK
    for second, r in outs:
        for a, b in zip(_host(r), expect[1 if second else 0]):
            np.testing.assert_array_equal(a, b)
