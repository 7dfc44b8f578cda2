"""The C ABI without a GPU: the library builds, loads, exports every entry point the header
declares, the binding's struct matches the C layout, and host-side argument checks return
SPEC_EINVAL before any CUDA call."""
import ctypes
import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "specverify.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(spec_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    if not shutil.which("nvcc") and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    from speculative_decoding_verification_31_gb300 import build
    build.build()
    import speculative_decoding_verification_31_gb300 as sv
    return sv.load_library()


def test_header_declares_the_boundary():
    names = declared_functions()
    for f in ("spec_verify", "spec_verify_greedy", "spec_verify_ex", "spec_verify_greedy_ex",
              "spec_verify_workspace_bytes", "spec_verify_check", "spec_verify_strerror",
              "spec_verify_opts_init", "spec_verify_noalloc", "spec_row_entropy", "spec_adaptive_k",
              "spec_verify_tree", "spec_verify_host", "spec_lmhead_logits",
              "spec_lmhead_row_stats", "spec_verify_lmhead", "spec_vp_state_bytes",
              "spec_vp_partials", "spec_vp_decide", "spec_vp_race", "spec_vp_finish",
              "spec_philox4x32_10"):
        assert f in names


def test_every_declared_symbol_is_exported(lib):
    import speculative_decoding_verification_31_gb300 as sv
    names = declared_functions()
    for f in names:
        assert hasattr(lib, f), f
    assert set(names) == set(sv.EXPORTED)
    nm = shutil.which("nm")
    if nm:
        out = subprocess.run([nm, "-D", "--defined-only", sv.specverify.LIB_PATH],
                             capture_output=True, text=True, check=True).stdout
        exported = set(re.findall(r"\bT (spec_\w+)", out))
        assert set(names) <= exported


def test_checked_library_exports_the_same_entry_points(lib):
    """The index-checked variant is the same ABI (built beside the library)."""
    import speculative_decoding_verification_31_gb300 as sv
    path = sv.specverify.CHECKED_LIB_PATH
    assert os.path.exists(path)
    checked = ctypes.CDLL(path)
    for f in declared_functions():
        assert hasattr(checked, f), f
    assert checked.spec_verify_strerror  # loads and resolves
    checked.spec_verify_strerror.restype = ctypes.c_char_p
    assert b"index" in checked.spec_verify_strerror(7)


def test_opts_struct_layout_matches_c(lib, tmp_path):
    from speculative_decoding_verification_31_gb300.specverify import SpecVerifyOpts
    src = tmp_path / "layout.c"
    src.write_text(
        '#include <stdio.h>\n#include <stddef.h>\n#include "specverify.h"\n'
        "int main(void){printf(\"%zu %zu %zu %zu\\n\", sizeof(spec_verify_opts),"
        " offsetof(spec_verify_opts, workspace_bytes), offsetof(spec_verify_opts, out_race),"
        " offsetof(spec_verify_opts, prof_events)); printf(\"%zu %zu %zu\\n\", offsetof(spec_verify_opts,"
        " flags), offsetof(spec_verify_opts, out_H_p), offsetof(spec_verify_opts, ctrl_beta));"
        " return 0;}\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True)
    size, ws, race, prof, dbg, hp, beta = map(int, subprocess.run(
        [str(exe)], capture_output=True, text=True, check=True).stdout.split())
    assert ctypes.sizeof(SpecVerifyOpts) == size
    assert SpecVerifyOpts.workspace_bytes.offset == ws
    assert SpecVerifyOpts.out_race.offset == race
    assert SpecVerifyOpts.prof_events.offset == prof
    assert SpecVerifyOpts.flags.offset == dbg
    assert SpecVerifyOpts.out_H_p.offset == hp
    assert SpecVerifyOpts.ctrl_beta.offset == beta


def test_strerror_and_workspace_size(lib):
    import speculative_decoding_verification_31_gb300 as sv
    for code in range(8):
        assert sv.spec_verify_strerror(code) != "unknown status"
    assert sv.spec_verify_strerror(99) == "unknown status"
    small = sv.spec_verify_workspace_bytes(1, 5, 1024, sv.SPEC_F32)
    big = sv.spec_verify_workspace_bytes(256, 12, 152064, sv.SPEC_BF16)
    assert 0 < small < big
    assert sv.spec_verify_workspace_bytes(-1, 5, 1024, sv.SPEC_F32) == 0
    assert sv.spec_verify_workspace_bytes(1, 5, 0, sv.SPEC_F32) == 0
    assert sv.spec_verify_workspace_bytes(1, 5, 10, 7) == 0
    assert big % 256 == 0


def test_host_validation_rejects_bad_sizes_without_a_device(lib):
    import speculative_decoding_verification_31_gb300 as sv
    P = ctypes.c_void_p
    fake = P(256)  # never dereferenced: validation fails first
    EINVAL = sv.SPEC_EINVAL
    assert lib.spec_verify(fake, fake, fake, -1, 3, 10, 1.0, 1.0, 0, fake, fake, None) == EINVAL
    assert lib.spec_verify(fake, fake, fake, 1, -1, 10, 1.0, 1.0, 0, fake, fake, None) == EINVAL
    assert lib.spec_verify(fake, fake, fake, 1, 3, 0, 1.0, 1.0, 0, fake, fake, None) == EINVAL
    assert lib.spec_verify(fake, fake, fake, 1, 3000, 10, 1.0, 1.0, 0, fake, fake, None) == EINVAL
    assert lib.spec_verify(None, fake, fake, 1, 3, 10, 1.0, 1.0, 0, fake, fake, None) == EINVAL
    assert lib.spec_verify(P(258), fake, fake, 1, 3, 10, 1.0, 1.0, 0, fake, fake, None) == EINVAL
    assert lib.spec_verify(fake, fake, fake, 1, 3, 10, 0.0, 1.0, 0, fake, fake, None) == EINVAL
    assert lib.spec_verify(fake, fake, fake, 1, 3, 10, 1.0, float("nan"), 0, fake, fake,
                           None) == EINVAL
    assert lib.spec_verify(fake, None, fake, 1, 3, 10, 1.0, 1.0, 0, fake, fake, None) == EINVAL
    assert lib.spec_verify_greedy(fake, None, 1, 3, 10, fake, fake, None) == EINVAL
    assert lib.spec_verify_greedy(fake, fake, 1, 3, 10, None, fake, None) == EINVAL
    # empty batch: nothing to do, no device touched
    assert lib.spec_verify(None, None, None, 0, 3, 10, 1.0, 1.0, 0, None, None, None) == 0
    opts = sv.SpecVerifyOpts()
    lib.spec_verify_opts_init(ctypes.byref(opts))
    assert opts.dtype == sv.SPEC_BF16 and opts.workspace is None
    opts.dtype = 5
    assert lib.spec_verify_ex(fake, fake, fake, 1, 3, 10, 1.0, 1.0, 0, fake, fake,
                              ctypes.byref(opts), None) == EINVAL
    # unknown flag bits (bit 0, once a schedule that was removed, included; SPEC_DEBUG_RACE_AGAIN
    # belongs to spec_verify_lmhead alone)
    for bad in (1, sv.SPEC_DEBUG_RACE_AGAIN, 32, 1 << 31):
        opts.dtype = sv.SPEC_BF16
        opts.flags = bad
        assert lib.spec_verify_ex(fake, fake, fake, 1, 3, 10, 1.0, 1.0, 0, fake, fake,
                                  ctypes.byref(opts), None) == EINVAL
        assert lib.spec_verify_noalloc(fake, fake, fake, 1, 3, 10, 1.0, 1.0, 0, fake, fake,
                                       ctypes.byref(opts), None) == EINVAL
    # the Philox diagnostic: sizes, forms and alignment are checked on the host
    assert lib.spec_philox4x32_10(fake, fake, -1, 0, fake, None) == EINVAL
    assert lib.spec_philox4x32_10(fake, fake, 4, 2, fake, None) == EINVAL
    assert lib.spec_philox4x32_10(P(264), fake, 4, 0, fake, None) == EINVAL
    assert lib.spec_philox4x32_10(fake, P(260), 4, 1, fake, None) == EINVAL
    assert lib.spec_philox4x32_10(fake, fake, 4, 0, None, None) == EINVAL
    assert lib.spec_philox4x32_10(None, None, 0, 0, None, None) == 0


def test_vocab_parallel_validation_without_a_device(lib):
    """The vocabulary-parallel steps reject bad sizes, offsets and pointers on the host."""
    import speculative_decoding_verification_31_gb300 as sv
    P = ctypes.c_void_p
    fake = P(256)
    EINVAL = sv.SPEC_EINVAL
    # x_offset must be a multiple of 8; B, gamma, V in range; pointers present and aligned
    assert lib.spec_vp_partials(fake, fake, fake, 2, 3, 100, 4, 1.0, 1.0, fake, fake, None, None) == EINVAL
    assert lib.spec_vp_partials(fake, fake, fake, 2, 3, 0, 0, 1.0, 1.0, fake, fake, None, None) == EINVAL
    assert lib.spec_vp_partials(P(258), fake, fake, 2, 3, 100, 0, 1.0, 1.0, fake, fake, None, None) == EINVAL
    assert lib.spec_vp_partials(fake, fake, fake, 2, 3, 100, 8, 0.0, 1.0, fake, fake, None, None) == EINVAL
    assert lib.spec_vp_partials(fake, None, fake, 2, 3, 100, 8, 1.0, 1.0, fake, fake, None, None) == EINVAL
    assert lib.spec_vp_decide(fake, 0, fake, fake, 2, 3, 100, 1.0, 1.0, 0, fake, fake, fake, None, None) == EINVAL
    assert lib.spec_vp_decide(fake, 2, fake, fake, 2, 3, 100, 1.0, 1.0, 0, fake, fake, None, None, None) == EINVAL
    assert lib.spec_vp_race(fake, fake, 2, 3, 100, 12, 0, fake, fake, None, None) == EINVAL
    assert lib.spec_vp_race(fake, fake, 2, 3, 100, 8, 0, None, fake, None, None) == EINVAL
    assert lib.spec_vp_finish(None, fake, 2, 3, fake, None) == EINVAL
    # empty batch: nothing to do
    assert lib.spec_vp_partials(None, None, None, 0, 3, 100, 0, 1.0, 1.0, None, None, None, None) == 0
    assert lib.spec_vp_finish(None, None, 0, 3, None, None) == 0
    assert lib.spec_vp_state_bytes(0) == 0 and lib.spec_vp_state_bytes(5) == 5 * 32


def test_vocab_range_partitions():
    from speculative_decoding_verification_31_gb300.vocab_parallel import vocab_range
    for V in (8, 17, 1001, 128256, 152064):
        for world in (1, 2, 3, 8):
            if -(-V // 8) < world:
                with pytest.raises(ValueError):
                    vocab_range(V, world, 0)
                continue
            ranges = [vocab_range(V, world, r) for r in range(world)]
            assert ranges[0][0] == 0 and ranges[-1][1] == V
            for (a, b), (c, d) in zip(ranges, ranges[1:]):
                assert b == c and a % 8 == 0 and c % 8 == 0 and b > a
            blocks = [-(-(b - a) // 8) for a, b in ranges]
            assert max(blocks) - min(blocks) <= 1


def test_product_path_does_not_import_the_oracle():
    """The package and the CUDA sources never name the oracle."""
    pkg = os.path.join(ROOT, "speculative_decoding_verification_31_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "specverify_oracle" not in text, f
