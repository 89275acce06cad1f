"""CPU oracle of the multi-LoRA segmented linear (float64) -- test infrastructure.

Only tests, the smoke check and the benchmark's CPU-baseline leg may use it; the
CUDA product path never imports it.
"""
from .lora_oracle import (  # noqa: F401
    EIDX, OK, OraclePool, OracleError, lora_linear, lora_linear_case, pad_pool, pool_of_case,
    segments, validate_idx, within_tolerance,
)
