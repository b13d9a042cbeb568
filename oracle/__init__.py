"""CPU oracle of the H2O eviction policy (test infrastructure; see h2o_oracle)."""
from . import kv_fp8
from .h2o_oracle import (NEAR_TIE, PrefillResult, RowCache, RowTrace, StepLog, decode_step,
                         default_scale, prefill, prefill_attention, prefill_select, run_row)

__all__ = ["kv_fp8", "NEAR_TIE", "PrefillResult", "RowCache", "RowTrace", "StepLog", "decode_step",
           "default_scale", "prefill", "prefill_attention", "prefill_select", "run_row"]
