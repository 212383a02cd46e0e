"""Float64 CPU oracle of the differential-attention forward.

Test infrastructure: only the tests, the smoke check and the benchmark's CPU
baseline use it.  It shares no code with the CUDA library.
"""
from .diffattn_oracle import (  # noqa: F401
    branch_logsumexp,
    differential_attention,
    differential_attention_backward,
    differential_attention_kv,
    differential_lambda,
    differential_lambda_backward,
    head_norm,
    lambda_init_schedule,
    signed_map,
    softmax_maps,
)
