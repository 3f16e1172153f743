"""fp64 CPU oracle (test infrastructure only; see moe_oracle's header)."""
from .moe_oracle import (  # noqa: F401
    widen_bf16, latent_projection, head_scores, softmax, topk_select,
    renormalised_gates, route, dispatch, gather, silu, expert_ffn, combine,
    forward, forward_bits, forward_ext, modality_mask, swiglu_ffn, forward_headlocal,
)
