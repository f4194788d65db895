"""Plain, slow CPU oracle for the paged-KV attention path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product package imports this
module; only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline / reference arm may call it.  It shares no code with the CUDA path.

Everything is numpy float64 computed straight from the definition of
attention over a paged cache: gather K/V in logical order through the block
table, then softmax(q k^T * scale + mask) v.  See ``paged_attention.py``;
the per-head RMSNorm and rotary embedding fused into the append are in
``rope.py``.
"""
from .paged_attention import (  # noqa: F401
    bf16_bits_to_f64,
    kv_append,
    gather_sequence,
    attend_rows,
    paged_decode,
    paged_varlen,
)
from .rope import (  # noqa: F401
    f64_to_bf16_bits,
    kv_append_rope,
    norm_rope_rows,
    q_norm_rope,
    rms_norm_heads,
    rope_angles,
    rope_rotate,
)
