"""CPU oracle (float64) for filtering-first constrained SID beam decoding.

Test infrastructure: imported only by the tests, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py``.  It shares no code with the CUDA library.
"""
from .zerogr_oracle import (DENSE, SPARSE, DecodeResult, StepTable, Trie, brute_force, causal_attention,
                            choose_format, compact_layout, deco_forward, deco_hidden, decode,
                            filtered_log_softmax, rms_norm,
                            keys_to_sids, padded_slot_layout, path_score, score_first_log_probs,
                            serialize_index, sid_keys, table_row_tokens)

__all__ = [
    "DENSE", "SPARSE", "DecodeResult", "StepTable", "Trie", "brute_force", "causal_attention",
    "choose_format", "compact_layout", "deco_forward", "deco_hidden", "decode", "filtered_log_softmax",
    "rms_norm", "keys_to_sids", "padded_slot_layout",
    "path_score", "score_first_log_probs", "serialize_index", "sid_keys", "table_row_tokens",
]
