"""fp64 CPU oracle of the per-token recurrent form (test infrastructure only)."""
from .kvb_oracle import (PLAIN, GATED, GATED_DELTA, expand_qk, recurrent_step, recurrent_scan,
                         decode_sequence, verify, accept, short_context, prefill_state,
                         gated_prefill_closed_form, tree_path, verify_tree, accept_tree)

__all__ = ["PLAIN", "GATED", "GATED_DELTA", "expand_qk", "recurrent_step", "recurrent_scan",
           "decode_sequence", "verify", "accept", "short_context", "prefill_state",
           "gated_prefill_closed_form", "tree_path", "verify_tree", "accept_tree"]
