"""GB300 (sm_103a) grouped-query attention: split-KV decode and causal prefill.

The computation lives in ``libgqa_attn.so`` (CUDA kernels behind the C ABI of
``include/gqa_attn.h``).  This package is the thin Python binding: it checks
and marshals torch tensors into the C calls and raises on any non-zero status.
There is no CPU fallback: if the library is missing, every call raises.
"""
from ._binding import (  # noqa: F401
    GQAError,
    GQA_OK,
    GQA_ERR_INVALID_ARG,
    GQA_ERR_UNSUPPORTED,
    GQA_ERR_CUDA,
    GQA_ERR_WORKSPACE,
    GQA_ERR_TIMEOUT,
    GQA_ERR_OUT_OF_BOUNDS,
    lib_path,
    load_library,
    gqa_status_string,
    gqa_attn_abi_version,
    gqa_attn_decode_plan,
    gqa_attn_decode_workspace_size,
    gqa_attn_decode,
    gqa_attn_decode_kernel_count,
    gqa_attn_decode_paged,
    gqa_attn_decode_multi,
    gqa_attn_decode_paged_multi,
    gqa_attn_decode_multi_workspace_size,
    gqa_attn_decode_split,
    gqa_attn_decode_merge,
    gqa_attn_decode_noalloc,
    GQA_NOALLOC_SCRATCH_BYTES,
    gqa_attn_prefill_causal,
    gqa_attn_prefill_causal_paged,
    gqa_attn_merge_states,
    gqa_attn_prefill_causal_workspace_size,
    gqa_attn_prefill_causal_kernel_count,
    gqa_attn_prefill_causal_plan,
    gqa_attn_decode_from_host_arena_size,
    gqa_attn_decode_from_host,
    gqa_attn_prefill_causal_from_host_arena_size,
    gqa_attn_prefill_causal_from_host,
    gqa_attn_device_status,
    gqa_attn_selftest_bounded_wait,
    gqa_attn_bounds_checked,
    gqa_attn_selftest_bounds,
    gqa_attn_debug_s_tile_count,
)
from .sequence_parallel import (  # noqa: F401
    block_seqlens,
    decode_sequence_parallel,
    gather_states,
    ring_pass,
    ring_prefill_causal,
    ring_schedule,
)
