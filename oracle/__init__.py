"""CPU oracle for the paged KV attention step: TEST INFRASTRUCTURE ONLY.

Only the test-suite, the package smoke check and the benchmark's CPU-baseline arm
may import this package. The CUDA library never imports it, and it imports nothing
from the library.
"""
from .paged_kv_oracle import (  # noqa: F401
    BLOCK_SIZE, attention_step, causal_softmax_attention, copy_blocks, decode_bits, gather_context,
    kv_head_of, paged_attention, query_positions, reshape_and_cache, rope, rope_reshape_and_cache,
    slot_mapping, slot_of,
)
from .spec_oracle import spec_accept  # noqa: F401,E402
