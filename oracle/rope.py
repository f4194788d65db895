"""fp64 CPU oracle: the per-head QK RMSNorm and rotary embedding fused into
the KV append.

TEST INFRASTRUCTURE ONLY (see package docstring): no product code may
import it, and it imports nothing from the product.

Sources, by page and section:

* scripts/benchmarks commit log, Gemma-4 shared-KV commit: the store layer
  keeps its post-rotary k (and its v) before the paged update, i.e. the
  cache holds K after the rotary embedding and V as projected.
* same log, Llama-3.2 support commit ("Attention forward factory"): Qwen3
  runs a per-head RMSNorm on q and k, over head_dim of [B, S, H, D], before
  the rest of attention; Llama has no such norm.
* same log, Gemma-4 engine commit ("Dual attention regimes") and the
  README's Gemma-4 paragraph: the rotary (cos, sin) tables are precomputed
  per position and per regime, rope_theta = 1e6 for full attention.

Readings where the pages are silent:

* Rotary convention: rotate-half.  For i < D/2, dims i and i + D/2 form a
  pair rotated counter-clockwise by the angle pos * theta^(-2i/D), i.e.
  (x_i + j x_{i+D/2}) * exp(j * angle) read as a complex number.
* RMSNorm over head_dim: y = w * x / sqrt(mean(x^2) + eps), one weight
  vector of length head_dim shared by all heads of q (and another for k).
* Order: norm, then rotary.  Exact arithmetic (fp64) and one rounding to
  bfloat16 at the end, round-to-nearest-even.
* A token whose position lies outside [0, max_position) is skipped whole:
  q rows untouched, nothing appended.  A negative slot skips the append of
  that token only; its q rows are still transformed.
"""
from __future__ import annotations

import numpy as np

from .paged_attention import bf16_bits_to_f64


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float64 values to bfloat16 (round to nearest, ties to even)
    and return the uint16 bit patterns.  Finite inputs within bf16 range.

    bfloat16 keeps 8 significant bits and float32's exponent range, so the
    spacing next to |x| in [2^e, 2^(e+1)) is 2^(e-7), never below the
    subnormal spacing 2^-133.  Scaling by a power of two is exact, and
    np.rint rounds halves to even."""
    x = np.asarray(x, dtype=np.float64)
    if not np.all(np.isfinite(x)):
        raise ValueError("non-finite value")
    _, e = np.frexp(x)                     # |x| = m * 2^e, 0.5 <= m < 1
    q = np.maximum(e - 8, -133).astype(np.float64)
    y = np.ldexp(np.rint(np.ldexp(x, (-q).astype(np.int64))), q.astype(np.int64))
    if np.any(np.abs(y) > 3.3895313892515355e38):
        raise ValueError("outside the bfloat16 range")
    bits32 = y.astype(np.float32).view(np.uint32)  # y is exact in float32
    return (bits32 >> np.uint32(16)).astype(np.uint16)


def rms_norm_heads(x: np.ndarray, w, eps: float) -> np.ndarray:
    """Per-head RMSNorm over the last axis (head_dim): w * x / sqrt(mean(x^2)
    + eps).  w is a [D] float64 vector, or None for no norm (x returned)."""
    if w is None:
        return x
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * w


def rope_angles(pos: np.ndarray, D: int, theta: float) -> np.ndarray:
    """[T, D/2] angles pos_t * theta^(-2i/D)."""
    i = np.arange(D // 2, dtype=np.float64)
    inv_freq = theta ** (-2.0 * i / D)
    return np.asarray(pos, dtype=np.float64)[:, None] * inv_freq[None, :]


def rope_rotate(x: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """Rotate x [T, H, D] by the rotary embedding of positions pos [T]
    (rotate-half pairs (i, i + D/2))."""
    D = x.shape[-1]
    a = rope_angles(pos, D, theta)[:, None, :]        # [T, 1, D/2]
    c, s = np.cos(a), np.sin(a)
    lo, hi = x[..., : D // 2], x[..., D // 2:]
    return np.concatenate([lo * c - hi * s, hi * c + lo * s], axis=-1)


def norm_rope_rows(x_bits: np.ndarray, pos: np.ndarray, theta: float, w_bits, eps: float,
                   ) -> np.ndarray:
    """The fused row transform: bf16 rows x [T, H, D] -> RMSNorm (weight
    w_bits [D] bf16, or None) -> rotary at pos [T] -> bf16 bits."""
    x = bf16_bits_to_f64(x_bits)
    w = None if w_bits is None else bf16_bits_to_f64(w_bits)
    return f64_to_bf16_bits(rope_rotate(rms_norm_heads(x, w, eps), pos, theta))


def q_norm_rope(q_bits: np.ndarray, positions: np.ndarray, theta: float, q_w_bits, eps: float,
                max_position: int) -> np.ndarray:
    """q [T, H_q, D] bf16 bits after the fused transform; rows of tokens
    with a position outside [0, max_position) are returned unchanged."""
    pos = np.asarray(positions, dtype=np.int64)
    ok = (pos >= 0) & (pos < max_position)
    out = np.array(q_bits, dtype=np.uint16, copy=True)
    if np.any(ok):
        out[ok] = norm_rope_rows(q_bits[ok], pos[ok], theta, q_w_bits, eps)
    return out


def kv_append_rope(k_cache: np.ndarray, v_cache: np.ndarray, k_new: np.ndarray,
                   v_new: np.ndarray, slot_mapping: np.ndarray, positions: np.ndarray,
                   theta: float, k_w_bits, eps: float, max_position: int):
    """Append with the fused transform: row t of K is normalised and rotated
    at positions[t] before it is stored at slot_mapping[t]; V is stored as
    given.  Pools are uint16 bf16 bit patterns [num_pages, H_kv, P, D];
    returns copies (k', v') with every other byte unchanged."""
    num_pages, H_kv, P, D = k_cache.shape
    pos = np.asarray(positions, dtype=np.int64)
    slots = np.asarray(slot_mapping, dtype=np.int64)
    keep = (pos >= 0) & (pos < max_position) & (slots >= 0)
    live = slots[keep]
    if len(np.unique(live)) != len(live):
        raise ValueError("duplicate slot in one append")
    if np.any(live >= num_pages * P):
        raise ValueError("slot outside the pool")
    k_out = k_cache.copy()
    v_out = v_cache.copy()
    idx = np.nonzero(keep)[0]
    if len(idx) == 0:
        return k_out, v_out
    k_rot = norm_rope_rows(k_new[idx], pos[idx], theta, k_w_bits, eps)
    for n, t in enumerate(idx):
        page, row = int(slots[t]) // P, int(slots[t]) % P
        k_out[page, :, row, :] = k_rot[n]
        v_out[page, :, row, :] = v_new[t]
    return k_out, v_out
