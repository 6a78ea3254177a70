"""Float64 CPU oracle of the decoder-only forward pass over a KV cache.

TEST INFRASTRUCTURE ONLY.  This package is the checker, not the product: only
``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import it.  It shares no code, table or helper with the CUDA library
(``decoder_only_forward_gb300``), and nothing in it imports that package.

Parity status of each function is stated in ``oracle/decoder_ref.py``'s
module docstring.
"""

from .decoder_ref import (  # noqa: F401
    OracleConfig,
    DictWeights,
    Session,
    rmsnorm,
    rope_inv_freq,
    llama3_scale_inv_freq,
    rope_rotate,
    attend_ref,
    silu,
    swiglu,
    route_topk,
    moe_ffn,
    kv_head_of,
    window_start,
)
