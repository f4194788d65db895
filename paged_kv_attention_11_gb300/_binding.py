"""ctypes marshalling for libpkv.so (argument packing only)."""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "_build", "libpkv.so")
_lib: Optional[ctypes.CDLL] = None

DEVERR_SLOT = 1
DEVERR_PAGE = 2
DEVERR_LEN = 4
DEVERR_TIMEOUT = 8
DEVERR_POS = 16

_c_i32, _c_i64, _c_p, _c_f = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_float
_SIGS = {
    "paged_kv_append": [_c_p, _c_p, _c_p, _c_p, _c_p, _c_i32, _c_i32, _c_i32, _c_i32, _c_i64,
                        _c_p, _c_p],
    "paged_attn_decode_workspace_size": [_c_i32, _c_i32, _c_i32, _c_i32],
    "paged_attn_decode": [_c_p, _c_p, _c_p, _c_p, _c_p, _c_i32, _c_p, _c_i32, _c_i32, _c_i32,
                          _c_i32, _c_i32, _c_i64, _c_i32, _c_f, _c_i32, _c_p, ctypes.c_size_t,
                          _c_p, _c_p],
    "paged_attn_decode_append": [_c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_i32, _c_p, _c_i32,
                                 _c_i32, _c_i32, _c_i32, _c_i32, _c_i64, _c_i32, _c_f, _c_i32,
                                 _c_p, ctypes.c_size_t, _c_p, _c_p],
    "paged_attn_varlen": [_c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_i32, _c_i32, _c_i32,
                          _c_i32, _c_i32, _c_i32, _c_i32, _c_i32, _c_i32, _c_i64, _c_f, _c_i32,
                          _c_i32, _c_p, _c_p],
    "paged_attn_decode_static": [_c_p, _c_p, _c_p, _c_p, _c_p, _c_i32, _c_p, _c_i32, _c_i32,
                                 _c_i32, _c_i32, _c_i32, _c_i64, _c_i32, _c_f, _c_i32, _c_p,
                                 _c_p],
    "paged_attn_decode_shared_prefix_workspace_size": [_c_i32, _c_i32, _c_i32, _c_i32],
    "paged_attn_decode_shared_prefix": [_c_p, _c_p, _c_p, _c_p, _c_p, _c_i32, _c_p, _c_i32,
                                        _c_i32, _c_p, _c_i32, _c_i32, _c_i32, _c_i32, _c_i64,
                                        _c_i32, _c_f, _c_p, ctypes.c_size_t, _c_p, _c_p],
    "paged_attn_mixed": [_c_p, _c_p, _c_p, _c_i32, _c_p, _c_i32, _c_i32, _c_p, _c_p, _c_p, _c_p,
                         _c_p, _c_i32, _c_i32, _c_i32, _c_i32, _c_i32, _c_p, _c_p, _c_i32,
                         _c_i32, _c_i32, _c_i32, _c_i64, _c_f, _c_i32, _c_i32, _c_p,
                         ctypes.c_size_t, _c_p, _c_p],
    "paged_attn_mixed_append": [_c_p, _c_p, _c_p, _c_i32, _c_p, _c_i32, _c_i32, _c_p, _c_p, _c_p,
                                _c_p, _c_p, _c_i32, _c_i32, _c_i32, _c_i32, _c_i32, _c_p, _c_p,
                                _c_p, _c_i32, _c_p, _c_p, _c_i32, _c_i32, _c_i32, _c_i32, _c_i64,
                                _c_f, _c_i32, _c_i32, _c_p, ctypes.c_size_t, _c_p, _c_p],
    "pkv_rope_table": [_c_p, _c_i32, _c_i32, ctypes.c_double, _c_p],
    "paged_kv_append_rope": [_c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_i32, _c_p, _c_p,
                             _c_f, _c_i32, _c_i32, _c_i32, _c_i32, _c_i32, _c_i64, _c_p, _c_p],
    "pkv_copy": [_c_p, _c_p, ctypes.c_size_t, _c_p],
    "pkv_status_string": [_c_i32],
    "pkv_last_cuda_error": [],
}
_RES = {"paged_attn_decode_workspace_size": ctypes.c_size_t,
        "paged_attn_decode_shared_prefix_workspace_size": ctypes.c_size_t,
        "pkv_status_string": ctypes.c_char_p, "pkv_last_cuda_error": ctypes.c_char_p}


class PKVError(RuntimeError):
    def __init__(self, fn: str, status: int):
        L = lib()
        msg = L.pkv_status_string(status).decode()
        if status == 3:
            msg += ": " + L.pkv_last_cuda_error().decode()
        super().__init__(f"{fn} -> {msg}")
        self.status = status


def lib_path() -> str:
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    """Load libpkv.so (built by paged_kv_attention_11_gb300.build)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"{_LIB_PATH} is missing: build it with "
                "`python -m paged_kv_attention_11_gb300.build` (needs nvcc)")
        L = ctypes.CDLL(_LIB_PATH)
        for name, args in _SIGS.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = _RES.get(name, ctypes.c_int)
        _lib = L
    return _lib


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(fn: str, status: int):
    if status != 0:
        raise PKVError(fn, status)


def _bf16(t: torch.Tensor, name: str):
    if t.dtype != torch.bfloat16 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous bfloat16 tensor")


def paged_kv_append(k_new: torch.Tensor, v_new: torch.Tensor, k_cache: torch.Tensor,
                    v_cache: torch.Tensor, slot_mapping: torch.Tensor,
                    err_flag: Optional[torch.Tensor] = None, stream=None) -> None:
    """k_new/v_new [T, H_kv, D]; caches [num_pages, H_kv, P, D]; slots [T] int64."""
    for n, t in (("k_new", k_new), ("v_new", v_new), ("k_cache", k_cache), ("v_cache", v_cache)):
        _bf16(t, n)
    if slot_mapping.dtype != torch.int64:
        raise ValueError("slot_mapping must be int64")
    num_pages, H_kv, P, D = k_cache.shape
    _check("paged_kv_append", lib().paged_kv_append(
        _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(slot_mapping),
        k_new.shape[0], H_kv, D, P, num_pages, _ptr(err_flag), _stream(stream)))


def decode_workspace_size(batch: int, num_q_heads: int, num_kv_heads: int, head_dim: int) -> int:
    return int(lib().paged_attn_decode_workspace_size(batch, num_q_heads, num_kv_heads, head_dim))


# Decode workspaces kept by the binding for callers that pass none: one per
# (device, stream, head shape), zero-filled once and grown when a larger batch
# needs more.  The kernel leaves a workspace zero-filled after every call, so
# calls in one stream's order may share it; calls on different streams get
# different ones.
_WORKSPACES = {}


def shared_prefix_workspace_size(batch: int, num_q_heads: int, num_kv_heads: int,
                                 head_dim: int) -> int:
    return int(lib().paged_attn_decode_shared_prefix_workspace_size(batch, num_q_heads,
                                                                   num_kv_heads, head_dim))


def decode_workspace(device: torch.device, stream_handle: int, batch: int, num_q_heads: int,
                     num_kv_heads: int, head_dim: int, shared_prefix: bool = False) -> torch.Tensor:
    """The binding's cached decode workspace for this stream and shape: it
    allocates (and zero-fills) only when none is cached yet or the cached
    one is too small, so a CUDA-graph capture must be preceded by one call
    of the same shape on the capturing stream (or pass ``workspace``)."""
    size = shared_prefix_workspace_size if shared_prefix else decode_workspace_size
    need = max(size(batch, num_q_heads, num_kv_heads, head_dim), 256)
    key = (device.index if device.index is not None else torch.cuda.current_device(),
           int(stream_handle), num_q_heads, num_kv_heads, head_dim, shared_prefix)
    ws = _WORKSPACES.get(key)
    if ws is None or ws.numel() < need:
        ws = torch.zeros(need, dtype=torch.uint8, device=device)
        # the zero fill runs on torch's current stream: order the kernel's
        # stream after it
        cur = torch.cuda.current_stream(device)
        if int(stream_handle) != cur.cuda_stream:
            torch.cuda.ExternalStream(int(stream_handle), device=device).wait_stream(cur)
        _WORKSPACES[key] = ws
    return ws


def paged_attn_decode(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor,
                      v_cache: torch.Tensor, block_table: torch.Tensor, seq_lens: torch.Tensor,
                      max_seq_len: int, scale: float, window: int = 0,
                      workspace: Optional[torch.Tensor] = None,
                      err_flag: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """out/q [B, H_q, D]; block_table [B, max_blocks] int32; seq_lens [B] int32.
    Without ``workspace`` the binding's cached one for this stream is used
    (``decode_workspace``): it allocates only on the first call of a stream
    and shape, or when the batch outgrows it."""
    for n, t in (("out", out), ("q", q), ("k_cache", k_cache), ("v_cache", v_cache)):
        _bf16(t, n)
    if block_table.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise ValueError("block_table and seq_lens must be int32")
    B, H_q, D = q.shape
    num_pages, H_kv, P, _ = k_cache.shape
    if workspace is None:
        workspace = decode_workspace(q.device, _stream(stream), B, H_q, H_kv, D)
    _check("paged_attn_decode", lib().paged_attn_decode(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
        block_table.shape[1], _ptr(seq_lens), B, H_q, H_kv, D, P, num_pages, int(max_seq_len),
        float(scale), int(window), _ptr(workspace), workspace.numel(), _ptr(err_flag),
        _stream(stream)))
    return out


def paged_attn_decode_append(out: torch.Tensor, q: torch.Tensor, k_new: torch.Tensor,
                             v_new: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                             block_table: torch.Tensor, seq_lens: torch.Tensor,
                             max_seq_len: int, scale: float, window: int = 0,
                             workspace: Optional[torch.Tensor] = None,
                             err_flag: Optional[torch.Tensor] = None,
                             stream=None) -> torch.Tensor:
    """paged_attn_decode with each sequence's new K/V row ([B, H_kv, D]
    k_new/v_new) written to position seq_lens[b]-1 of its pages by the same
    launch.  Workspace handling as paged_attn_decode."""
    for n, t in (("out", out), ("q", q), ("k_new", k_new), ("v_new", v_new),
                 ("k_cache", k_cache), ("v_cache", v_cache)):
        _bf16(t, n)
    if block_table.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise ValueError("block_table and seq_lens must be int32")
    B, H_q, D = q.shape
    num_pages, H_kv, P, _ = k_cache.shape
    if tuple(k_new.shape) != (B, H_kv, D) or tuple(v_new.shape) != (B, H_kv, D):
        raise ValueError("k_new and v_new must be [batch, num_kv_heads, head_dim]")
    if workspace is None:
        workspace = decode_workspace(q.device, _stream(stream), B, H_q, H_kv, D)
    _check("paged_attn_decode_append", lib().paged_attn_decode_append(
        _ptr(out), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
        _ptr(block_table), block_table.shape[1], _ptr(seq_lens), B, H_q, H_kv, D, P, num_pages,
        int(max_seq_len), float(scale), int(window), _ptr(workspace), workspace.numel(),
        _ptr(err_flag), _stream(stream)))
    return out


def paged_attn_decode_shared_prefix(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor,
                                    v_cache: torch.Tensor, block_table: torch.Tensor,
                                    seq_lens: torch.Tensor, group_size: int,
                                    prefix_lens: torch.Tensor, max_seq_len: int, scale: float,
                                    workspace: Optional[torch.Tensor] = None,
                                    err_flag: Optional[torch.Tensor] = None,
                                    stream=None) -> torch.Tensor:
    """Decode for groups of ``group_size`` consecutive sequences that share
    their first ``prefix_lens[j]`` keys (pages aliased in their block
    tables): out/q [B, H_q, D]; prefix_lens [ceil(B / group_size)] int32.
    Same result as paged_attn_decode; the shared pages are read once per
    group.  Workspace handling as paged_attn_decode."""
    for n, t in (("out", out), ("q", q), ("k_cache", k_cache), ("v_cache", v_cache)):
        _bf16(t, n)
    for n, t in (("block_table", block_table), ("seq_lens", seq_lens),
                 ("prefix_lens", prefix_lens)):
        if t.dtype != torch.int32:
            raise ValueError(f"{n} must be int32")
    B, H_q, D = q.shape
    num_pages, H_kv, P, _ = k_cache.shape
    if workspace is None:
        workspace = decode_workspace(q.device, _stream(stream), B, H_q, H_kv, D,
                                     shared_prefix=True)
    _check("paged_attn_decode_shared_prefix", lib().paged_attn_decode_shared_prefix(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
        block_table.shape[1], _ptr(seq_lens), B, int(group_size), _ptr(prefix_lens), H_q, H_kv,
        D, P, num_pages, int(max_seq_len), float(scale), _ptr(workspace), workspace.numel(),
        _ptr(err_flag), _stream(stream)))
    return out


def paged_attn_varlen(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor,
                      v_cache: torch.Tensor, cu_seq_lens_q: torch.Tensor,
                      cu_seq_lens_k: torch.Tensor, block_table: torch.Tensor,
                      max_seqlen_q: int, max_seqlen_k: int, scale: float, causal: bool = True,
                      window: int = 0, err_flag: Optional[torch.Tensor] = None,
                      stream=None) -> torch.Tensor:
    """out/q [total_q, H_q, D]; cu_seq_lens_* [B+1] int32; block_table [B, max_blocks]."""
    for n, t in (("out", out), ("q", q), ("k_cache", k_cache), ("v_cache", v_cache)):
        _bf16(t, n)
    for n, t in (("cu_seq_lens_q", cu_seq_lens_q), ("cu_seq_lens_k", cu_seq_lens_k),
                 ("block_table", block_table)):
        if t.dtype != torch.int32:
            raise ValueError(f"{n} must be int32")
    total_q, H_q, D = q.shape
    num_pages, H_kv, P, _ = k_cache.shape
    _check("paged_attn_varlen", lib().paged_attn_varlen(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(cu_seq_lens_q),
        _ptr(cu_seq_lens_k), _ptr(block_table), block_table.shape[1],
        cu_seq_lens_q.shape[0] - 1, int(max_seqlen_q), int(max_seqlen_k), total_q, H_q, H_kv,
        D, P, num_pages, float(scale), 1 if causal else 0, int(window), _ptr(err_flag),
        _stream(stream)))
    return out


def paged_attn_mixed(dec_out: torch.Tensor, dec_q: torch.Tensor, dec_block_table: torch.Tensor,
                     dec_seq_lens: torch.Tensor, dec_max_seq_len: int, pre_out: torch.Tensor,
                     pre_q: torch.Tensor, cu_seq_lens_q: torch.Tensor,
                     cu_seq_lens_k: torch.Tensor, pre_block_table: torch.Tensor,
                     max_seqlen_q: int, max_seqlen_k: int, k_cache: torch.Tensor,
                     v_cache: torch.Tensor, scale: float, window: int = 0,
                     decode_ctas: int = 0, workspace: Optional[torch.Tensor] = None,
                     err_flag: Optional[torch.Tensor] = None, stream=None):
    """One continuous-batching step in one launch: decode rows (dec_q/dec_out
    [B, H_q, D]) and causal prefill chunks (pre_q/pre_out [total_q, H_q, D],
    cu_seq_lens_* [Bp+1]).  Workspace handling as paged_attn_decode."""
    for n, t in (("dec_out", dec_out), ("dec_q", dec_q), ("pre_out", pre_out),
                 ("pre_q", pre_q), ("k_cache", k_cache), ("v_cache", v_cache)):
        _bf16(t, n)
    for n, t in (("dec_block_table", dec_block_table), ("dec_seq_lens", dec_seq_lens),
                 ("cu_seq_lens_q", cu_seq_lens_q), ("cu_seq_lens_k", cu_seq_lens_k),
                 ("pre_block_table", pre_block_table)):
        if t.dtype != torch.int32:
            raise ValueError(f"{n} must be int32")
    B, H_q, D = dec_q.shape
    total_q = pre_q.shape[0]
    num_pages, H_kv, P, _ = k_cache.shape
    if workspace is None:
        workspace = decode_workspace(dec_q.device, _stream(stream), max(B, 1), H_q, H_kv, D)
    _check("paged_attn_mixed", lib().paged_attn_mixed(
        _ptr(dec_out), _ptr(dec_q), _ptr(dec_block_table), dec_block_table.shape[1],
        _ptr(dec_seq_lens), B, int(dec_max_seq_len), _ptr(pre_out), _ptr(pre_q),
        _ptr(cu_seq_lens_q), _ptr(cu_seq_lens_k), _ptr(pre_block_table),
        pre_block_table.shape[1], cu_seq_lens_q.shape[0] - 1, int(max_seqlen_q),
        int(max_seqlen_k), total_q, _ptr(k_cache), _ptr(v_cache), H_q, H_kv, D, P, num_pages,
        float(scale), int(window), int(decode_ctas), _ptr(workspace), workspace.numel(),
        _ptr(err_flag), _stream(stream)))


def paged_attn_mixed_append(dec_out: torch.Tensor, dec_q: torch.Tensor,
                            dec_block_table: torch.Tensor, dec_seq_lens: torch.Tensor,
                            dec_max_seq_len: int, pre_out: torch.Tensor, pre_q: torch.Tensor,
                            cu_seq_lens_q: torch.Tensor, cu_seq_lens_k: torch.Tensor,
                            pre_block_table: torch.Tensor, max_seqlen_q: int, max_seqlen_k: int,
                            k_new: torch.Tensor, v_new: torch.Tensor, slot_mapping: torch.Tensor,
                            k_cache: torch.Tensor, v_cache: torch.Tensor, scale: float,
                            window: int = 0, decode_ctas: int = 0,
                            workspace: Optional[torch.Tensor] = None,
                            err_flag: Optional[torch.Tensor] = None, stream=None):
    """paged_attn_mixed with the step's append (k_new/v_new [T, H_kv, D],
    slot_mapping [T] int64) in the same launch."""
    for n, t in (("dec_out", dec_out), ("dec_q", dec_q), ("pre_out", pre_out),
                 ("pre_q", pre_q), ("k_new", k_new), ("v_new", v_new), ("k_cache", k_cache),
                 ("v_cache", v_cache)):
        _bf16(t, n)
    for n, t in (("dec_block_table", dec_block_table), ("dec_seq_lens", dec_seq_lens),
                 ("cu_seq_lens_q", cu_seq_lens_q), ("cu_seq_lens_k", cu_seq_lens_k),
                 ("pre_block_table", pre_block_table)):
        if t.dtype != torch.int32:
            raise ValueError(f"{n} must be int32")
    if slot_mapping.dtype != torch.int64:
        raise ValueError("slot_mapping must be int64")
    B, H_q, D = dec_q.shape
    total_q = pre_q.shape[0]
    num_pages, H_kv, P, _ = k_cache.shape
    if workspace is None:
        workspace = decode_workspace(dec_q.device, _stream(stream), max(B, 1), H_q, H_kv, D)
    _check("paged_attn_mixed_append", lib().paged_attn_mixed_append(
        _ptr(dec_out), _ptr(dec_q), _ptr(dec_block_table), dec_block_table.shape[1],
        _ptr(dec_seq_lens), B, int(dec_max_seq_len), _ptr(pre_out), _ptr(pre_q),
        _ptr(cu_seq_lens_q), _ptr(cu_seq_lens_k), _ptr(pre_block_table),
        pre_block_table.shape[1], cu_seq_lens_q.shape[0] - 1, int(max_seqlen_q),
        int(max_seqlen_k), total_q, _ptr(k_new), _ptr(v_new), _ptr(slot_mapping),
        k_new.shape[0], _ptr(k_cache), _ptr(v_cache), H_q, H_kv, D, P, num_pages,
        float(scale), int(window), int(decode_ctas), _ptr(workspace), workspace.numel(),
        _ptr(err_flag), _stream(stream)))


def paged_attn_decode_static(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor,
                             v_cache: torch.Tensor, block_table: torch.Tensor,
                             seq_lens: torch.Tensor, max_seq_len: int, scale: float,
                             window: int = 0, err_flag: Optional[torch.Tensor] = None,
                             stream=None) -> torch.Tensor:
    """paged_attn_decode without a caller workspace: for callers that cannot
    allocate device memory (the library's own fixed 8 MiB scratch is used;
    calls that overlap on the GPU race on it)."""
    for n, t in (("out", out), ("q", q), ("k_cache", k_cache), ("v_cache", v_cache)):
        _bf16(t, n)
    if block_table.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise ValueError("block_table and seq_lens must be int32")
    B, H_q, D = q.shape
    num_pages, H_kv, P, _ = k_cache.shape
    _check("paged_attn_decode_static", lib().paged_attn_decode_static(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
        block_table.shape[1], _ptr(seq_lens), B, H_q, H_kv, D, P, num_pages, int(max_seq_len),
        float(scale), int(window), _ptr(err_flag), _stream(stream)))
    return out


def pkv_copy(dst: torch.Tensor, src: torch.Tensor, stream=None) -> torch.Tensor:
    """Copy src into dst (same byte size, both contiguous) with the SMs:
    device memory of the current device or pinned host memory on either
    side, 16-byte aligned, a multiple of 16 bytes."""
    if not (dst.is_contiguous() and src.is_contiguous()):
        raise ValueError("pkv_copy: dst and src must be contiguous")
    nbytes = dst.numel() * dst.element_size()
    if nbytes != src.numel() * src.element_size():
        raise ValueError("pkv_copy: dst and src differ in size")
    _check("pkv_copy", lib().pkv_copy(_ptr(dst), _ptr(src), nbytes, _stream(stream)))
    return dst


def rope_table(cos_sin: torch.Tensor, theta: float, stream=None) -> torch.Tensor:
    """Fill cos_sin [max_position, head_dim] float32 with the rotary table:
    column i < head_dim/2 is cos(p * theta^(-2i/head_dim)), column
    head_dim/2 + i the sine."""
    if cos_sin.dtype != torch.float32 or not cos_sin.is_contiguous() or cos_sin.dim() != 2:
        raise ValueError("cos_sin must be a contiguous [max_position, head_dim] float32 tensor")
    _check("pkv_rope_table", lib().pkv_rope_table(
        _ptr(cos_sin), cos_sin.shape[0], cos_sin.shape[1], float(theta), _stream(stream)))
    return cos_sin


def paged_kv_append_rope(q: Optional[torch.Tensor], k_new: torch.Tensor, v_new: torch.Tensor,
                         k_cache: torch.Tensor, v_cache: torch.Tensor,
                         slot_mapping: torch.Tensor, positions: torch.Tensor,
                         cos_sin: torch.Tensor, q_norm_weight: Optional[torch.Tensor] = None,
                         k_norm_weight: Optional[torch.Tensor] = None, eps: float = 1e-6,
                         err_flag: Optional[torch.Tensor] = None, stream=None) -> None:
    """q [T, H_q, D] (in place) or None; k_new/v_new [T, H_kv, D]; caches
    [num_pages, H_kv, P, D]; slots [T] int64; positions [T] int32; cos_sin
    [max_position, D] float32; norm weights [D] bf16 or None."""
    for n, t in (("k_new", k_new), ("v_new", v_new), ("k_cache", k_cache), ("v_cache", v_cache)):
        _bf16(t, n)
    for n, t in (("q", q), ("q_norm_weight", q_norm_weight), ("k_norm_weight", k_norm_weight)):
        if t is not None:
            _bf16(t, n)
    if slot_mapping.dtype != torch.int64 or positions.dtype != torch.int32:
        raise ValueError("slot_mapping must be int64 and positions int32")
    if cos_sin.dtype != torch.float32 or not cos_sin.is_contiguous():
        raise ValueError("cos_sin must be a contiguous float32 tensor")
    num_pages, H_kv, P, D = k_cache.shape
    H_q = q.shape[1] if q is not None else 0
    _check("paged_kv_append_rope", lib().paged_kv_append_rope(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(slot_mapping),
        _ptr(positions), _ptr(cos_sin), cos_sin.shape[0], _ptr(q_norm_weight),
        _ptr(k_norm_weight), float(eps), k_new.shape[0], H_q, H_kv, D, P, num_pages,
        _ptr(err_flag), _stream(stream)))
