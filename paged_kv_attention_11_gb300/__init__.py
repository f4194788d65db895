"""Paged-KV attention for GB300 (sm_103a): Python binding of libpkv.so.

Three calls, same names as the C ABI (include/pkv.h):

* ``paged_kv_append``   scatter new K/V rows into the page pools
* ``paged_attn_decode`` one query per sequence over its paged prefix
* ``paged_attn_varlen`` packed variable-length (prefill) attention

plus ``paged_attn_decode_append`` (the decode step with its append in the
same launch), ``paged_attn_mixed`` (a step's decode rows and prefill chunks
in one launch), ``paged_attn_mixed_append`` (the same with the step's append
fused in), ``paged_attn_decode_shared_prefix`` (decode that reads a prefix
shared by a group of sequences once per group), ``paged_kv_append_rope`` (the
append with q/k RMSNorm and the rotary embedding fused in),
``rope_table`` (its cos/sin table) and ``pkv_copy`` (a step's host transfers
done by the SMs).

This module only marshals arguments (device pointers, sizes, the current
CUDA stream) into the library; every step of the computation runs in the
library's CUDA kernels.  There is no fallback: if libpkv.so is missing the
calls raise.
"""
from ._binding import (  # noqa: F401
    PKVError,
    DEVERR_LEN,
    DEVERR_PAGE,
    DEVERR_POS,
    DEVERR_SLOT,
    DEVERR_TIMEOUT,
    decode_workspace,
    decode_workspace_size,
    lib,
    lib_path,
    paged_attn_decode,
    paged_attn_decode_append,
    paged_attn_decode_shared_prefix,
    paged_attn_decode_static,
    paged_attn_mixed,
    paged_attn_mixed_append,
    paged_attn_varlen,
    paged_kv_append,
    paged_kv_append_rope,
    pkv_copy,
    rope_table,
    shared_prefix_workspace_size,
)
