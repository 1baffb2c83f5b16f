"""CPU oracle of the sparse-KV reuse step -- test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It shares no code with the CUDA path.
"""
from .avsg_oracle import (EMPTY, EMPTY_BUCKET, MAX_AGE_BUCKET, OracleError, OracleRun,  # noqa: F401
                          StepResult, UnitBuffer, attention_from_host,
                          attention_through_buffer, sparse_attention, widen_bf16)
