"""fp64 CPU oracle (test infrastructure only; see fa_oracle.py's header)."""

from .fa_oracle import (  # noqa: F401
    backward,
    bwd_preprocess,
    forward,
    kv_head,
    storage_round,
    unit_backward,
    unit_backward_parts,
    unit_forward,
    unit_probs,
    unit_scores,
)
