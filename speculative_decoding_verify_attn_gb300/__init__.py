"""GB300-native speculative-decoding hot path: verify attention, draft-window attention and the
speculative-sampling step, as hand-written sm_103a CUDA kernels behind a C ABI
(include/spec_verify.h).  This package holds the in-tree build script and a thin ctypes
binding whose functions carry the C names."""

from .binding import (  # noqa: F401
    SPEC_BF16, SPEC_ERR_CUDA, SPEC_ERR_INVALID_ARG, SPEC_ERR_UNSUPPORTED, SPEC_ERR_WORKSPACE, SPEC_F32, SPEC_OK,
    SPEC_SAMPLE_CHAIN, SPEC_SAMPLE_CHAIN_GREEDY, SPEC_SAMPLE_TREE, SPEC_SAMPLE_TREE_GREEDY, SPEC_STATUS_BAD_KV_LEN,
    SPEC_STATUS_BAD_POS, SPEC_STATUS_BAD_TOKEN, SPEC_STATUS_TIMEOUT, SpecAttnArgs, SpecError, SpecSampleArgs,
    SpecWindowArgs, lib, read_status, spec_abi_version, spec_draft_window_attn, spec_draft_window_attn_workspace,
    spec_sample, spec_sample_workspace, spec_status_string, spec_verify_attn, spec_verify_attn_workspace,
)
from .binding import SPEC_ERR_SCRATCH_LIMIT, spec_verify_attn_noalloc  # noqa: F401,E402
from .binding import SPEC_DEBUG_NO_LOADS  # noqa: F401,E402
from .binding import SPEC_COMMIT_CHAIN, SPEC_COMMIT_TREE, SpecCommitArgs, spec_commit  # noqa: F401,E402
from .binding import SpecLmheadArgs, spec_lmhead_sample, spec_lmhead_sample_workspace  # noqa: F401,E402
