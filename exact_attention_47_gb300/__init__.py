"""GB300 (sm_103a) exact attention: tiled online-softmax prefill, its backward,
paged-KV decode, chunked prefill over the paged cache, and the residual
add + RMSNorm and SwiGLU fusions of the same layer.

The compute lives in ``lib/libattn47_sm103.so`` (hand-written CUDA, C-ABI
declared in ``include/attn47.h``); this package is its Python binding.
Importing the package does not load the library; the first call does, and
raises if it is not built.  Build with ``exact_attention_47_gb300.build_lib``.
"""

from ._binding import (  # noqa: F401
    ATTN_DEV_BAD_BLOCK,
    ATTN_DEV_BAD_SEQLEN,
    ATTN_DEV_TIMEOUT,
    BLOCK_SIZE,
    AttnError,
    abi_version,
    attn_bwd,
    attn_bwd_workspace_size,
    attn_decode_paged,
    attn_decode_paged_noalloc,
    attn_decode_paged_workspace_size,
    attn_fwd,
    attn_prefill_paged,
    device_status,
    fused_add_rmsnorm,
    fused_swiglu,
    library_path,
    load_library,
    selftest_exp2_poly,
    selftest_wait_timeout,
    set_decode_early_plan,
    set_decode_max_ctas,
    set_wait_timeout_ns,
    ssd_chunked_fwd,
    ssd_workspace_size,
    status_string,
    swiglu_projection,
)
