"""The allocation-free entry point, spec_verify_noalloc (marked gpu).

Some callers cannot let a library call cudaMalloc: a server whose own pool already holds
nearly all device memory, or a caller that may not block on the device synchronisation an
allocation can imply.  spec_verify_noalloc keeps its scratch in a static device array
instead.  These tests call it through the C ABI and check that two calls in a row give the
same tokens, accepted counts and diagnostic values as the workspace-using spec_verify_ex,
that, in a fresh process, calls after the first change nothing in the device's free memory,
and that a problem too large for the static array is refused before anything runs.  The
file is named to be collected last; it also passes alone in a fresh process.
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


def _diag(B, g, dev):
    f = dict(dtype=torch.float32, device=dev)
    return {"logp": torch.full((B, g), float("nan"), **f),
            "logq": torch.full((B, g), float("nan"), **f),
            "logZp": torch.full((B, g + 1), float("nan"), **f),
            "logZq": torch.full((B, g), float("nan"), **f),
            "u": torch.full((B, g), float("nan"), **f),
            "race": torch.full((B, 2), float("nan"), **f)}


CASES = [
    ("batched bf16, per-sequence temperatures", lambda: workloads.config(3, B=12), True),
    ("fp32, unaligned rows", lambda: workloads.generic(B=3, gamma=5, V=5003, dtype="f32",
                                                       seed=21, T=0.8, Td=0.4), False),
    ("bf16, gamma = 0", lambda: workloads.generic(B=4, gamma=0, V=4099, dtype="bf16", seed=22),
     False),
]


@pytest.mark.parametrize("name,make,per_seq", CASES, ids=[c[0] for c in CASES])
def test_noalloc_matches_the_workspace_entry_point(sv, name, make, per_seq):
    w = make()
    dw = DeviceWorkload(w)
    B, g = w.B, w.gamma
    kw = dict(T_per_seq=dw.T, Td_per_seq=dw.Td) if per_seq else {}
    seed = 31337
    ref_t, ref_n, ref_d = sv.spec_verify_ex(dw.target, dw.draft, dw.tokens, float(w.T[0]),
                                            float(w.Td[0]), seed, diagnostics=True, **kw)
    torch.cuda.synchronize()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call in range(2):  # the static scratch keeps the previous call's contents
        out_t = torch.full((B, g + 1), -7, dtype=torch.int32, device="cuda")
        out_n = torch.full((B,), -7, dtype=torch.int32, device="cuda")
        diag = _diag(B, g, dw.target.device)
        sv.spec_verify_noalloc(dw.target, dw.draft, dw.tokens, float(w.T[0]), float(w.Td[0]),
                               seed, out_t, out_n, d_status=status, diag=diag, **kw)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(out_t.cpu().numpy(), ref_t.cpu().numpy(),
                                      err_msg=f"call {call}")
        np.testing.assert_array_equal(out_n.cpu().numpy(), ref_n.cpu().numpy())
        for k in ("logp", "logq", "logZp", "logZq", "u"):
            np.testing.assert_allclose(diag[k].cpu().numpy(), ref_d[k].cpu().numpy(),
                                       rtol=1e-6, atol=1e-6, equal_nan=True, err_msg=k)
        # the winning race score (the runner-up column is approximate and may vary by call)
        np.testing.assert_allclose(diag["race"][:, 0].cpu().numpy(), ref_d["race"][:, 0].cpu().numpy(),
                                   rtol=1e-6, atol=1e-6, equal_nan=True, err_msg="race")
        assert int(status.item()) == sv.SPEC_OK


_ALLOC_PROBE = r"""
import sys
import numpy as np
import torch
sys.path.insert(0, "tests")
import workloads
from _parity import DeviceWorkload
import speculative_decoding_verification_31_gb300 as sv
w = workloads.config(3, B=12)
dw = DeviceWorkload(w)
B, g = w.B, w.gamma
out_t = torch.empty((B, g + 1), dtype=torch.int32, device="cuda")
out_n = torch.empty((B,), dtype=torch.int32, device="cuda")
status = torch.zeros(1, dtype=torch.int32, device="cuda")
toks = []
def call():
    sv.spec_verify_noalloc(dw.target, dw.draft, dw.tokens, 1.0, 0.5, 7, out_t, out_n,
                           T_per_seq=dw.T, Td_per_seq=dw.Td, d_status=status)
    torch.cuda.synchronize()
    toks.append(out_t.cpu().numpy().copy())
call()  # the first call loads the library's kernels and looks up the static array
free0 = torch.cuda.mem_get_info()[0]
for _ in range(3):
    call()
free1 = torch.cuda.mem_get_info()[0]
assert all(np.array_equal(t, toks[0]) for t in toks), "calls disagree"
assert int(status.item()) == 0, int(status.item())
print("FREE", free0, free1)
"""


def test_noalloc_allocates_nothing():
    """In a fresh process where spec_verify_noalloc is the library's only entry point called,
    calls after the first (which loads the kernels and the static array's module) leave the
    device's free memory unchanged: the library allocates nothing on this path, not even its
    own status word (any cudaMalloc shows at the allocator's granularity)."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    r = subprocess.run([sys.executable, "-c", _ALLOC_PROBE], cwd=root, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    line = [ln for ln in r.stdout.splitlines() if ln.startswith("FREE")][-1]
    _, free0, free1 = line.split()
    assert int(free0) == int(free1), line


def test_noalloc_refuses_oversized_problems(sv):
    # B=4096, gamma=12, V=152064 bf16 needs far more than the static scratch
    need = sv.spec_verify_workspace_bytes(4096, 12, 152064, sv.SPEC_BF16)
    assert need > sv.SPEC_NOALLOC_SCRATCH_BYTES
    lib = sv.load_library()
    fake = 1 << 20  # 16-byte aligned, never dereferenced: the size check fails first
    opts = sv.SpecVerifyOpts()
    lib.spec_verify_opts_init(opts)
    rc = lib.spec_verify_noalloc(fake, fake, fake, 4096, 12, 152064, 1.0, 1.0, 0, fake, fake,
                                 opts, None)
    assert rc == sv.SPEC_ESCRATCH
    assert "scratch" in sv.spec_verify_strerror(rc)
    # a caller workspace makes no sense here
    opts.workspace = fake
    opts.workspace_bytes = 1 << 20
    rc = lib.spec_verify_noalloc(fake, fake, fake, 1, 2, 100, 1.0, 1.0, 0, fake, fake, opts,
                                 None)
    assert rc == sv.SPEC_EINVAL
