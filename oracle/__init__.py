"""fp64 CPU oracle (test infrastructure only; never called by the library)."""
from .tsel_oracle import (bf16_bits_to_f64, e4m3_bits_to_f64, decode_inputs, attention_probabilities,
                          importance, keep_count, select_topk, score_quanta, dynamic_budget,
                          gather_compact, prune)

__all__ = ["bf16_bits_to_f64", "e4m3_bits_to_f64", "decode_inputs", "attention_probabilities",
           "importance", "keep_count", "select_topk", "score_quanta", "dynamic_budget",
           "gather_compact", "prune"]
