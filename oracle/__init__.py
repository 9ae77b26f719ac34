"""fp64 CPU oracle for exact attention — TEST INFRASTRUCTURE ONLY.

This package is the slow, obviously-correct statement of what the GPU path
computes.  Only the test-suite, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU-baseline / reference arm may import it.  The CUDA library never calls it,
and it imports nothing from the CUDA package: the two share no code.

Sources (web pages, cited by title and section):
  * "Advanced attention mechanisms – II" (Aryan Das): sections "Why?",
    "Flash Attention", "Tiling" (steps 1–3), "Softmax stabiliser",
    "Incremental / online softmax".
  * "Fast attention kernels and operator fusion accelerate AI models":
    sections "FlashAttention-style attention and Paged Attention" and
    "Operator fusion" (``fusions.py``: residual add + RMSNorm, SwiGLU).
  * "Accelerating Mamba-2 with high-performance forward kernels in NVIDIA
    CUDA Tile" (``ssd.py``: the SSD recurrence and its chunked form).

Every function here is pinned against brute force, closed forms, a library
routine and invariants the mathematics fixes: the forward and decode by
``tests/test_oracle_pins.py``, the backward by
``tests/test_oracle_backward_pins.py``, the chunked prefill over a paged
cache by ``tests/test_oracle_paged_prefill_pins.py``, the fusions by
``tests/test_oracle_fusion_pins.py``, the SSD by ``tests/test_oracle_ssd_pins.py``.  No function is
"parity unpinned".
"""

from .definitions import (  # noqa: F401
    attention,
    attention_backward,
    attention_online,
    combine_partials,
    decode_paged,
    gather_paged_keys,
    prefill_paged,
    score_matrix,
    softmax_probs,
    split_partials,
)
from .fusions import add_rmsnorm, round_bf16, swiglu, swiglu_projection  # noqa: F401
from .ssd import (  # noqa: F401
    ssd_chunk_cumsum,
    ssd_chunk_output,
    ssd_chunked,
    ssd_fwd_pass_state,
    ssd_recurrence,
)
