"""CPU oracle for grouped-query attention (test infrastructure only).

This package is the plain, slow, obviously-correct statement of what the GPU
library computes. Only the test-suite, the smoke check and the benchmark's CPU
baseline may import it; the product path never does.
"""

from .gqa_oracle import (  # noqa: F401
    APPEND_OK,
    APPEND_CACHE_FULL,
    bf16_bits_to_f64,
    f32_to_bf16_bits,
    head_map,
    attention_probs,
    prefill,
    prefill_cached,
    decode,
    append,
    gather_paged,
    decode_paged,
    append_paged,
    rope,
    rope_f32,
    append_rope,
    append_paged_rope,
)
