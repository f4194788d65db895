"""fp64 CPU oracle: paged KV append and attention over a paged KV cache.

TEST INFRASTRUCTURE ONLY (see package docstring): no product code may
import it, and it imports nothing from the product.

Sources, by page and section:

* scripts/benchmarks commit log, "Why this works" (flex_attention + paged
  KV engine): the cache is one contiguous pool of fixed-size pages and a
  page table maps (sequence, logical block) -> physical page.  Token
  position p of a sequence lives in page table[p // page_size] at row
  p % page_size.
* same page, "Files" paragraph: new K/V rows are written in-kernel to their
  physical address (k_cache[addr] = k_val) before attention reads them.
* cb_sync_driver.py commit message (phase 2 fixes) and README "Integration
  notes": variable-length batches are described by cumulative sequence
  lengths cu_seq_lens_q / cu_seq_lens_k.
* scripts/benchmarks commit log, Gemma-4 sliding-window commit: the
  sliding mask is causal AND q_pos - kv_pos < window (strict less-than);
  full attention is plain causal.

Readings where the pages are silent:

* A decode step attends the new token: append first, then the query at
  position len-1 attends keys 0..len-1.
* A prefill chunk of q_len queries on a sequence of k_len keys is aligned
  bottom-right: query i sits at position k_len - q_len + i.
* GQA maps query head h to kv head h // (H_q / H_kv).
* A negative slot means "skip this row".  A query with no allowed key
  returns 0.

Layouts: pools [num_pages, H_kv, page_size, D]; q/out [tokens, H_q, D];
bf16 values are carried as uint16 bit patterns and widened exactly.
"""
from __future__ import annotations

import numpy as np


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns (uint16) to float64."""
    u32 = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


def kv_append(k_cache: np.ndarray, v_cache: np.ndarray, k_new: np.ndarray,
              v_new: np.ndarray, slot_mapping: np.ndarray):
    """Scatter new K/V rows into copies of the pools.

    Row t of k_new/v_new ([T, H_kv, D]) goes to slot slot_mapping[t], i.e.
    page slot // page_size, row slot % page_size, for every kv head.
    Negative slots are skipped.  Slots must be unique and inside the pool.
    Returns (k_cache', v_cache'); all other bytes are unchanged.
    """
    num_pages, H_kv, P, D = k_cache.shape
    k_out = k_cache.copy()
    v_out = v_cache.copy()
    slots = np.asarray(slot_mapping, dtype=np.int64)
    live = slots[slots >= 0]
    if len(np.unique(live)) != len(live):
        raise ValueError("duplicate slot in one append")
    if np.any(live >= num_pages * P):
        raise ValueError("slot outside the pool")
    for t, s in enumerate(slots):
        if s < 0:
            continue
        page, row = int(s) // P, int(s) % P
        k_out[page, :, row, :] = k_new[t]
        v_out[page, :, row, :] = v_new[t]
    return k_out, v_out


def gather_sequence(cache: np.ndarray, table_row: np.ndarray, length: int) -> np.ndarray:
    """Rebuild one sequence's [length, H_kv, D] rows in logical order."""
    P = cache.shape[2]
    out = np.empty((length,) + (cache.shape[1], cache.shape[3]), dtype=cache.dtype)
    for p in range(length):
        page = int(table_row[p // P])
        out[p] = cache[page, :, p % P, :]
    return out


def attend_rows(q: np.ndarray, K: np.ndarray, V: np.ndarray, q_pos: np.ndarray,
                scale: float, causal: bool = True, window: int = 0,
                return_lse: bool = False):
    """softmax(q K^T * scale + mask) V for the rows of one sequence, in fp64.

    q [n, H_q, D]; K, V [L, H_kv, D] in logical order; q_pos [n] absolute
    positions of the queries.  Key j is allowed for a query at position qp
    when (not causal or j <= qp) and (window <= 0 or qp - j < window).
    Returns out [n, H_q, D] (and the natural-log LSE [n, H_q] if asked).
    """
    n, H_q, D = q.shape
    L, H_kv, _ = K.shape
    G = H_q // H_kv
    out = np.zeros((n, H_q, D), dtype=np.float64)
    lse = np.full((n, H_q), -np.inf, dtype=np.float64)
    if n == 0 or L == 0:
        return (out, lse) if return_lse else out
    j = np.arange(L)[None, :]
    qp = np.asarray(q_pos, dtype=np.int64)[:, None]
    allowed = np.ones((n, L), dtype=bool)
    if causal:
        allowed &= j <= qp
        if window > 0:
            allowed &= (qp - j) < window
    has_key = allowed.any(axis=1)
    for g in range(H_kv):
        Kg = K[:, g, :]                              # [L, D]
        Vg = V[:, g, :]
        Qg = q[:, g * G:(g + 1) * G, :]              # [n, G, D]
        s = np.einsum("ngd,ld->ngl", Qg, Kg) * scale
        s = np.where(allowed[:, None, :], s, -np.inf)
        m = s.max(axis=2, keepdims=True)
        m = np.where(np.isfinite(m), m, 0.0)
        p = np.exp(s - m)                            # exp(-inf) = 0
        denom = p.sum(axis=2, keepdims=True)
        safe = np.where(denom > 0, denom, 1.0)
        out[:, g * G:(g + 1) * G, :] = np.einsum("ngl,ld->ngd", p, Vg) / safe
        with np.errstate(divide="ignore"):
            lse[:, g * G:(g + 1) * G] = (m + np.log(denom))[..., 0]
    out[~has_key] = 0.0
    lse[~has_key] = -np.inf
    return (out, lse) if return_lse else out


def paged_decode(q_bits: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                 block_table: np.ndarray, seq_lens: np.ndarray, scale: float,
                 window: int = 0) -> np.ndarray:
    """One query per sequence at position seq_lens[b]-1 over the paged cache.

    q_bits [B, H_q, D] bf16 bits; pools as stored after this step's append.
    Returns [B, H_q, D] float64.
    """
    B = q_bits.shape[0]
    out = np.zeros(q_bits.shape, dtype=np.float64)
    for b in range(B):
        L = int(seq_lens[b])
        if L <= 0:
            continue
        K = bf16_bits_to_f64(gather_sequence(k_cache, block_table[b], L))
        V = bf16_bits_to_f64(gather_sequence(v_cache, block_table[b], L))
        q = bf16_bits_to_f64(q_bits[b:b + 1])
        out[b] = attend_rows(q, K, V, np.array([L - 1]), scale, True, window)[0]
    return out


def paged_varlen(q_bits: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                 cu_seq_lens_q: np.ndarray, cu_seq_lens_k: np.ndarray,
                 block_table: np.ndarray, scale: float, causal: bool = True,
                 window: int = 0) -> np.ndarray:
    """Packed variable-length attention over the paged cache.

    Chunk b owns query rows cu_q[b]:cu_q[b+1] of q_bits [total_q, H_q, D]
    and keys 0..k_len-1 of its sequence (k_len = cu_k[b+1]-cu_k[b]), read
    through block_table[b].  Query i of the chunk is at position
    k_len - q_len + i.  Returns [total_q, H_q, D] float64.
    """
    out = np.zeros(q_bits.shape, dtype=np.float64)
    for b in range(len(cu_seq_lens_q) - 1):
        q0, q1 = int(cu_seq_lens_q[b]), int(cu_seq_lens_q[b + 1])
        k_len = int(cu_seq_lens_k[b + 1]) - int(cu_seq_lens_k[b])
        n = q1 - q0
        if n == 0:
            continue
        K = bf16_bits_to_f64(gather_sequence(k_cache, block_table[b], k_len))
        V = bf16_bits_to_f64(gather_sequence(v_cache, block_table[b], k_len))
        q = bf16_bits_to_f64(q_bits[q0:q1])
        pos = k_len - n + np.arange(n)
        out[q0:q1] = attend_rows(q, K, V, pos, scale, causal, window)
    return out
