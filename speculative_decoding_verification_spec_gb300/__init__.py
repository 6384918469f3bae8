"""GB300 (sm_103a) speculative-decoding verify step: exact speculative sampling, its top-k, top-p
and grammar-mask variants, greedy and typical-acceptance tree verify, stochastic tree verify and the verify side of an SMC-SD round, as hand-written CUDA behind a C ABI (include/spec_verify.h).

The binding functions load the compiled library on first use and raise if it is missing: there is
no CPU fallback.
"""
from .binding import (  # noqa: F401
    EXPORTS,
    NOALLOC_SCRATCH_BYTES,
    SpecVerifyError,
    Workspace,
    load,
    set_kernel_events,
    set_tree_sample_cluster,
    set_wait_limit,
    smc_verify,
    spec_verify,
    spec_verify_greedy,
    spec_verify_masked,
    spec_verify_noalloc,
    spec_verify_topk,
    spec_verify_topp,
    tree_verify_greedy,
    tree_verify_sample,
    tree_verify_typical,
    workspace_bytes,
)
