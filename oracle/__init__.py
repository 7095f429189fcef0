"""CPU oracle for large-beam GDN decoding (float64 FullState).

TEST INFRASTRUCTURE: imported only by the tests, the package smoke check and
the bench's CPU-baseline / reference leg. The CUDA product path never imports
it, and it imports nothing from the product.
"""
from .fullstate import (  # noqa: F401
    EPS, l2_normalize, rms_normalize, decay_gate, write_gate, gdn_inputs, per_value_head,
    gdn_transition, state_from_records, step_from_records, prefill_scan,
    codebook_logits, log_normalizer, layer_feature, scores_f32, select_top,
    kept_scores_f32, ancestry_slots, token_paths, prefill, decode_request,
    chain_decode, chain_trace, CallTrace, RequestTrace,
)
