"""GB300-native batched speculative-decoding verification.

The verification step of speculative decoding (rejection sampling of K draft
tokens against target and draft logits, truncation at the first rejection,
residual or bonus sampling; and the greedy variant) as hand-written CUDA for
sm_103a behind the C ABI in include/spec_verify.h. This package is the thin
Python binding: ``spec_verify`` and friends take torch tensors and call the
library; there is no CPU or eager fallback.
"""
from .api import (  # noqa: F401
    SV_BF16,
    SV_F32,
    SV_GREEDY,
    SV_SAMPLE,
    SV_SEQ_BAD_TOKEN,
    SV_SEQ_INDEX,
    SV_SEQ_NONFINITE,
    SV_SEQ_TIMEOUT,
    SpecVerifyError,
    launches,
    spec_verify,
    spec_verify_debug,
    spec_verify_early_exit,
    spec_verify_filtered,
    spec_verify_filtered_debug,
    spec_verify_filtered_timed,
    spec_verify_gated,
    spec_verify_host,
    spec_verify_lmhead,
    spec_verify_lmhead_debug,
    spec_verify_lmhead_gated,
    spec_verify_lmhead_timed,
    spec_verify_sharded,
    spec_verify_static,
    spec_verify_timed,
    sv_device_checks,
    sv_early_exit_workspace_bytes,
    sv_filtered_workspace_bytes,
    sv_host_staging_bytes,
    sv_lmhead_logits,
    sv_lmhead_workspace_bytes,
    sv_sharded_workspace_bytes,
    sv_philox,
    sv_workspace_bytes,
    version,
)
from ._lib import LIB_PATH, LibraryMissing, load  # noqa: F401
