"""CPU oracle for the P-EAGLE draft + verify step.

TEST INFRASTRUCTURE ONLY. This package is a plain, slow, float64 restatement
of what the method computes. It exists so that tests can check the CUDA path
against it. Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU-baseline / reference legs may import it. The product path (the CUDA
library and its Python binding) never imports, calls or links anything here,
and nothing here imports the product package.
"""

from .drafter import (  # noqa: F401
    rms_norm,
    rope_neox,
    silu,
    linear,
    gather_prefix_kv,
    causal_paged_attention,
    build_rows,
    run_layers,
    lm_head_logits,
    draft_pass,
    draft_sequential,
    draft_pass_refeed,
    argmax_lowest,
    top2_gap,
)
from .fp8 import e4m3_decode, dequant_rows, dequant_weights, E4M3_MAX  # noqa: F401
from .sampling import softmax_t, sample_inverse_cdf, sample_drafts, verify_stochastic  # noqa: F401
from .verify import (  # noqa: F401
    accept_length,
    verify,
    rebuild_metadata,
    rebuild_metadata_refeed,
    emitted_tokens,
    expected_tokens_iid,
    tokens_per_pass_linear,
    speedup_linear,
    breakeven_alpha,
    REQ_OK,
    REQ_CAPACITY,
    REQ_BAD_PAGE,
    REQ_BAD_INPUT,
)
