"""CPU fp64 oracle (test infrastructure only; see ``vocab_stats``).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU baseline
legs use this package.  The CUDA library never imports it.
"""

from .vocab_stats import (  # noqa: F401
    decode_bf16_bits,
    entropy_bwd,
    entropy_fwd,
    is_valid_id,
    kl_bwd,
    kl_fwd,
    linear_logits,
    linear_logp_bwd,
    linear_logp_fwd,
    logp_bwd,
    logp_fwd,
    row_log_softmax,
    row_stats,
    softcap,
    softcap_grad,
)
