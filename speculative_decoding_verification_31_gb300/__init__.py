"""Speculative-decoding verify step on NVIDIA GB300 (sm_103a).

The hot path lives in ``libspecverify.so`` (hand-written CUDA, C ABI in
``include/specverify.h``); this package only builds it and binds it.
"""
from .specverify import (  # noqa: F401
    EXPORTED, SPEC_BF16, SPEC_DEBUG_NEVER_READY, SPEC_FLAG_EARLY_EXIT, SPEC_EBADTOKEN, SPEC_ECUDA, SPEC_EINVAL, SPEC_ENOMEM, SPEC_ESCRATCH, SPEC_EINDEX,
    SPEC_ETIMEOUT, SPEC_F32, SPEC_NOALLOC_SCRATCH_BYTES, SPEC_OK, SpecVerifyError,
    SpecVerifyOpts, load_library, spec_verify, spec_verify_check, spec_verify_ex,
    spec_verify_greedy, spec_verify_greedy_ex, spec_verify_noalloc, spec_verify_strerror,
    spec_verify_workspace_bytes, spec_row_entropy, spec_adaptive_k, spec_verify_tree, Tree,
    spec_verify_host, SPEC_FLAG_FULL_READ, SPEC_DEBUG_RACE_AGAIN, spec_lmhead_logits, spec_lmhead_row_stats,
    spec_verify_lmhead, spec_philox4x32_10)
from .vocab_parallel import (  # noqa: F401
    LibraryBackend, VocabShard, spec_vp_decide, spec_vp_finish, spec_vp_partials, spec_vp_race,
    verify_vocab_parallel, vocab_range)
