"""GB300-native batched speculative-decoding verify/commit (CUDA kernels for sm_103a).

The compute path is libspecverify.so (C ABI in include/spec_verify.h); this package
only builds it and marshals torch tensors into it.
"""
from . import _build, binding  # noqa: F401
from .api import (markov_draft, markov_draft_topk, schedule_threshold, schedule_verify_len, schedule_verify_len_stale,  # noqa: F401
                  verify_greedy, verify_greedy_early_exit, verify_greedy_flat, verify_sample,
                  verify_sample_early_exit, verify_sample_flat,
                  verify_sample_host, workspace)
from .binding import (SpecError, spec_markov_draft, spec_markov_draft_topk, spec_markov_topk_workspace_size,
                      spec_schedule_threshold, spec_schedule_verify_len,  # noqa: F401
                      spec_schedule_verify_len_stale, spec_verify_greedy, spec_verify_greedy_early_exit,
                      spec_verify_greedy_flat, spec_verify_sample, spec_verify_sample_early_exit,
                      spec_verify_sample_flat, spec_verify_sample_noalloc,
                      spec_verify_workspace_size)


def build(force: bool = False) -> str:
    return _build.build(force=force)
