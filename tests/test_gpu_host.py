"""spec_verify_host: verification on pinned host buffers read in place over the host link
(marked gpu).  Its outputs must equal the device-buffer call's (the same kernels run on the
same values) and follow the usual parity rules against the oracle; pageable host memory is
refused."""
import ctypes

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


def host_tensors(w):
    if w.dtype == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(w.target).view(np.int16)).view(torch.bfloat16)
        d = torch.from_numpy(np.ascontiguousarray(w.draft).view(np.int16)).view(torch.bfloat16)
    else:
        t, d = torch.from_numpy(np.ascontiguousarray(w.target)), torch.from_numpy(np.ascontiguousarray(w.draft))
    return (t.pin_memory(), d.pin_memory(), torch.from_numpy(np.ascontiguousarray(w.tokens)).pin_memory())


@pytest.mark.parametrize("full_read", [False, True])
@pytest.mark.parametrize("B,gamma,V,dtype", [(3, 4, 5003, "bf16"), (2, 7, 9000, "f32"), (4, 0, 777, "bf16")])
def test_host_buffers_match_device_and_oracle(sv, orc, B, gamma, V, dtype, full_read):
    w = workloads.generic(B=B, gamma=gamma, V=V, dtype=dtype, seed=B * 13 + V, sigma=0.7, T=0.8, Td=0.4)
    ht, hd, htok = host_tensors(w)
    out_t = torch.empty((B, gamma + 1), dtype=torch.int32).pin_memory()
    out_n = torch.empty((B,), dtype=torch.int32).pin_memory()
    dw = DeviceWorkload(w)
    for seed in range(3):
        sv.spec_verify_host(ht, hd, htok, float(w.T[0]), float(w.Td[0]), seed, out_t, out_n,
                            full_read=full_read)
        torch.cuda.synchronize()
        g = run_gpu(sv, dw, seed, per_seq_temps=False, diagnostics=False,
                    flags=0 if full_read else sv.SPEC_FLAG_EARLY_EXIT)
        np.testing.assert_array_equal(out_t.numpy(), g["tokens"])
        np.testing.assert_array_equal(out_n.numpy(), g["n"])
        compare_sampling(w, {"tokens": out_t.numpy().copy(), "n": out_n.numpy().copy()},
                         orc.verify(w.target, w.draft, w.tokens, w.T, w.Td, seed))
    assert sv.spec_verify_check() == sv.SPEC_OK


def test_host_buffers_batched_workload_with_host_temperatures(sv, orc):
    """B=64, gamma=8, V=128256 bf16 with per-sequence temperatures, all in pinned host memory."""
    w = workloads.config(3)
    ht, hd, htok = host_tensors(w)
    T = torch.from_numpy(w.T).pin_memory()
    Td = torch.from_numpy(w.Td).pin_memory()
    out_t = torch.empty((w.B, w.gamma + 1), dtype=torch.int32).pin_memory()
    out_n = torch.empty((w.B,), dtype=torch.int32).pin_memory()
    for seed in range(2):
        sv.spec_verify_host(ht, hd, htok, 1.0, 1.0, seed, out_t, out_n, T_per_seq=T, Td_per_seq=Td)
        torch.cuda.synchronize()
        compare_sampling(w, {"tokens": out_t.numpy().copy(), "n": out_n.numpy().copy()},
                         orc.verify(w.target, w.draft, w.tokens, w.T, w.Td, seed))


def test_pageable_host_memory_is_refused(sv):
    w = workloads.generic(B=2, gamma=3, V=100, dtype="f32", seed=1)
    t = torch.from_numpy(np.ascontiguousarray(w.target))        # pageable
    d = torch.from_numpy(np.ascontiguousarray(w.draft))
    tok = torch.from_numpy(np.ascontiguousarray(w.tokens))
    out_t = torch.empty((2, 4), dtype=torch.int32)
    out_n = torch.empty((2,), dtype=torch.int32)
    with pytest.raises(ValueError):
        sv.spec_verify_host(t, d, tok, 1.0, 1.0, 0, out_t, out_n)
    o = sv.SpecVerifyOpts()
    lib = sv.load_library()
    lib.spec_verify_opts_init(ctypes.byref(o))
    o.dtype = sv.SPEC_F32
    P = ctypes.c_void_p
    rc = lib.spec_verify_host(P(t.data_ptr()), P(d.data_ptr()), P(tok.data_ptr()), 2, 3, 100, 1.0,
                              1.0, 0, P(out_t.data_ptr()), P(out_n.data_ptr()), ctypes.byref(o),
                              P(torch.cuda.current_stream().cuda_stream))
    assert rc == sv.SPEC_EINVAL
