"""The device Philox4x32-10 word for word against the oracle's (marked gpu).

Both generators restate Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as
1, 2, 3" (SC'11), section 4, independently; the oracle's is pinned against Triton's Philox in
tests/test_oracle_rng.py.  Here the library's diagnostic entry point evaluates the device
generator exactly as the verify kernels do -- the plain ten rounds (acceptance uniforms) and
the race's evaluation with the per-row rounds precomputed -- and all four output words must
equal the oracle's on over a million counters: random counters and keys, the counters the
verify step actually uses, and corner values.
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_31_gb300 as m
    m.load_library()
    return m


def _counters(n, race_form):
    rng = np.random.default_rng(2024 + race_form)
    c = rng.integers(0, 2**32, size=(n, 4), dtype=np.uint64).astype(np.uint32)
    k = rng.integers(0, 2**32, size=(n, 2), dtype=np.uint64).astype(np.uint32)
    m = n // 4
    # counters the verify step uses: acceptance (0, i, b, 0) and race (x >> 2, r, b, 1)
    c[:m, 0] = 0
    c[:m, 1] = rng.integers(0, 2049, size=m)
    c[:m, 3] = 0
    c[m:2 * m, 0] = rng.integers(0, 152064 // 4, size=m)
    c[m:2 * m, 1] = rng.integers(0, 2049, size=m)
    c[m:2 * m, 2] = rng.integers(0, 1 << 16, size=m)
    c[m:2 * m, 3] = 1
    # corners: all-zero and all-ones words and keys
    corners = np.array([[0, 0, 0, 0], [0xFFFFFFFF] * 4, [1, 0, 0, 0], [0, 0, 0, 1],
                        [0xFFFFFFFF, 0, 0xFFFFFFFF, 0]], dtype=np.uint32)
    nc = min(len(corners), n - 2 * m)
    c[2 * m:2 * m + nc] = corners[:nc]
    k[2 * m:2 * m + nc] = np.array([[0, 0], [0xFFFFFFFF, 0xFFFFFFFF], [0, 0xFFFFFFFF],
                                    [0xFFFFFFFF, 0], [12345, 678]], dtype=np.uint32)[:nc]
    if race_form:
        c[:, 3] = 1  # the race's evaluation fixes word 3
    return c, k


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int32)).cuda()


@pytest.mark.parametrize("form", [0, 1])
def test_device_philox_all_four_words_equal_the_oracle(sv, form):
    n = (1 << 20) + 77
    c, k = _counters(n, form)
    got = sv.spec_philox4x32_10(_dev(c), _dev(k), form=form)
    torch.cuda.synchronize()
    got = got.cpu().numpy().view(np.uint32)
    want = oracle.get().philox_bulk(c, k)
    bad = np.nonzero(np.any(got != want, axis=1))[0]
    assert bad.size == 0, (bad[:5], c[bad[:5]], k[bad[:5]], got[bad[:5]], want[bad[:5]])


def test_device_philox_empty_and_tiny(sv):
    empty = torch.empty((0, 4), dtype=torch.int32, device="cuda")
    out = sv.spec_philox4x32_10(empty, torch.empty((0, 2), dtype=torch.int32, device="cuda"))
    assert out.shape == (0, 4)
    c, k = _counters(8, 0)
    got = sv.spec_philox4x32_10(_dev(c), _dev(k)).cpu().numpy().view(np.uint32)
    np.testing.assert_array_equal(got, oracle.get().philox_bulk(c, k))
