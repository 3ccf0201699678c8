"""fp64 CPU oracle for grouped-query attention (decode and causal prefill).

TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.  Only the test suite, the
package smoke check and the bench's CPU-baseline leg may import or run this
package.  The CUDA library never calls it and shares no code with it; the two
meet only through the seeded inputs of ``gqa_synth``.

Every function is a plain, unblocked-by-design restatement of what the design
record "ADR-0060: AHBM GQA Fused Attention Kernel (Llama3-70B)" says the kernels
compute (FlashAttention's scaled softmax(Q K^T) V with GQA head sharing and
causal masking).  See ``oracle.attention`` for the per-function citations and
``tests/test_oracle_pins.py`` for what pins each function to the pages and to
the mathematics rather than to itself.
"""
from .attention import (  # noqa: F401
    attend_rows,
    decode,
    decode_pairs,
    decode_multi,
    prefill_causal,
    prefill_causal_rows,
    partial_triplet,
    merge_triplets,
    finalize_triplet,
    merge_states,
    online_softmax_tiles,
)
