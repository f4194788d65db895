"""Seeded synthetic inputs for the paged-KV attention path.

This module draws random numbers and builds index structures (page pools,
block tables, slot mappings, cumulative sequence lengths).  It contains none
of the attention arithmetic: both the CPU oracle (``oracle/``) and the CUDA
path (``paged_kv_attention_11_gb300``) consume what it produces, and neither
is imported here.

Workload shapes follow the benchmark scenarios of the pages this library is
built from (scripts/benchmarks commit log, "Why this works" section: a paged
KV cache read through a page table; README "Integration notes": cu_seq_lens
for varlen; Gemma-4 sliding window of 512 and shared-KV layers):

  tiny     4 decode sequences, cached {7,33,64,100}, H 4/2/64, page 16
  qwen3    64 decode sequences, cached ~U[256,2048], H 32/8/128, page 16,
           16384-page pool, K scaled per kv head by U(0.5,2)
  mixed    8 prefill chunks (len ~U[128,1024], prefix ~U[0,512]) +
           120 decode sequences (cached ~U[64,4096]), H 32/8/128, page 16
  sliding  H 8/1/256, window 512, page 64, 32 decode (cached ~U[1024,8192])
           + 4 prefill chunks of 2048 (prefix 0), two layers on one pool
  grpo     64 prompts x 4 generations, 256-token prefix pages shared by the
           4 generations, completion ~U[0,3840], H 32/8/128, page 16
  full_d512  full-attention layers with 512-wide heads: H 8/1/512, page 16,
           64 decode (cached ~U[1024,8192]) + 4 prefill chunks of 1024

Values are bf16 bit patterns (numpy uint16): fp32 draws rounded to nearest
even before either side sees them, so both sides start from identical bits.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional, Sequence

import numpy as np

BASE_SEED = 3407


# ---------------------------------------------------------------------------
# bf16 bit handling (input preparation only)
# ---------------------------------------------------------------------------
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round-to-nearest-even); uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def randn_bf16(rng: np.random.Generator, shape, scale=None) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if scale is not None:
        x = x * np.asarray(scale, dtype=np.float32)
    return f32_to_bf16_bits(x)


# ---------------------------------------------------------------------------
# Step structure
# ---------------------------------------------------------------------------
@dataclasses.dataclass
class Step:
    """One batch of the hot path: new K/V rows, decode rows, prefill chunks.

    Pool layout: k_cache/v_cache [num_pages, H_kv, P, D] (bf16 bits).
    Decode: sequence b has ``dec_cached[b]`` tokens cached before the step;
    its new token sits at position dec_cached[b]; attention length is
    dec_cached[b] + 1.
    Prefill: chunk c has ``pre_prefix[c]`` cached tokens and
    ``pre_qlen[c]`` new tokens; k_len = prefix + qlen.
    """
    name: str
    H_q: int
    H_kv: int
    D: int
    P: int
    num_pages: int
    window: int
    scale: float
    n_layers: int = 1                  # layers whose Q reads the same pool
    # decode part
    dec_cached: np.ndarray = None      # [Bd] int32
    dec_block_table: np.ndarray = None  # [Bd, maxblk] int32
    # prefill part
    pre_prefix: np.ndarray = None      # [Bp] int32
    pre_qlen: np.ndarray = None        # [Bp] int32
    pre_block_table: np.ndarray = None  # [Bp, maxblk] int32
    used_pages: np.ndarray = None      # pages referenced by any table
    k_head_scale: Optional[np.ndarray] = None  # [H_kv] fp32 or None
    layer_page_offset: int = 0         # for multi-layer pools (grpo)
    # decode sequences j*group_size .. j*group_size+group_size-1 share their
    # first prefix_lens[j] keys (the same physical pages in their tables)
    group_size: int = 1
    prefix_lens: Optional[np.ndarray] = None  # [ceil(Bd / group_size)] int32

    # ---- derived index arrays --------------------------------------------
    @property
    def Bd(self) -> int:
        return 0 if self.dec_cached is None else int(self.dec_cached.shape[0])

    @property
    def Bp(self) -> int:
        return 0 if self.pre_qlen is None else int(self.pre_qlen.shape[0])

    @property
    def dec_seq_lens(self) -> np.ndarray:
        return (self.dec_cached + 1).astype(np.int32)

    @property
    def cu_seq_lens_q(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.pre_qlen)]).astype(np.int32)

    @property
    def cu_seq_lens_k(self) -> np.ndarray:
        return np.concatenate(
            [[0], np.cumsum(self.pre_prefix + self.pre_qlen)]).astype(np.int32)

    @property
    def total_q(self) -> int:
        return 0 if self.pre_qlen is None else int(self.pre_qlen.sum())

    def _slot(self, table_row: np.ndarray, pos: np.ndarray) -> np.ndarray:
        pos = np.asarray(pos, dtype=np.int64)
        return table_row[pos // self.P].astype(np.int64) * self.P + pos % self.P

    @property
    def pre_slots(self) -> np.ndarray:
        """Slot of every new prefill token, in packed (cu_seq_lens_q) order."""
        out = []
        for c in range(self.Bp):
            pos = self.pre_prefix[c] + np.arange(self.pre_qlen[c])
            out.append(self._slot(self.pre_block_table[c], pos))
        return (np.concatenate(out) if out else np.zeros(0)).astype(np.int64)

    @property
    def dec_slots(self) -> np.ndarray:
        out = [self._slot(self.dec_block_table[b], [self.dec_cached[b]])
               for b in range(self.Bd)]
        return (np.concatenate(out) if out else np.zeros(0)).astype(np.int64)

    @property
    def all_positions(self) -> np.ndarray:
        """Position of every new token in its sequence, in append order
        (prefill tokens prefix + i, then each decode row's cached length)."""
        parts = [self.pre_prefix[c] + np.arange(self.pre_qlen[c]) for c in range(self.Bp)]
        if self.Bd:
            parts.append(np.asarray(self.dec_cached))
        return (np.concatenate(parts) if parts else np.zeros(0)).astype(np.int32)

    @property
    def n_new_tokens(self) -> int:
        return self.total_q + self.Bd

    @property
    def all_slots(self) -> np.ndarray:
        """Append order: prefill tokens first, then one row per decode seq."""
        return np.concatenate([self.pre_slots, self.dec_slots]).astype(np.int64)

    def max_seq_len_dec(self) -> int:
        return int(self.dec_seq_lens.max()) if self.Bd else 0

    def max_seqlen_q(self) -> int:
        return int(self.pre_qlen.max()) if self.Bp else 0

    def max_seqlen_k(self) -> int:
        return int((self.pre_prefix + self.pre_qlen).max()) if self.Bp else 0


@dataclasses.dataclass
class StepValues:
    """bf16 bit arrays for one step (host copies)."""
    k_cache: np.ndarray      # [num_pages, H_kv, P, D] uint16, pre-append
    v_cache: np.ndarray
    k_new: np.ndarray        # [n_new, H_kv, D] uint16 (append order)
    v_new: np.ndarray
    q_dec: List[np.ndarray]  # per layer [Bd, H_q, D]
    q_pre: List[np.ndarray]  # per layer [total_q, H_q, D]


class _PageAllocator:
    def __init__(self, rng: np.random.Generator, num_pages: int, first: int = 0,
                 count: Optional[int] = None):
        count = num_pages - first if count is None else count
        self.perm = first + rng.permutation(count).astype(np.int32)
        self.next = 0

    def take(self, n: int) -> np.ndarray:
        if self.next + n > self.perm.shape[0]:
            raise ValueError("page pool exhausted")
        out = self.perm[self.next:self.next + n]
        self.next += n
        return out


def _table(rows: Sequence[np.ndarray], maxblk: int) -> np.ndarray:
    t = np.full((len(rows), max(maxblk, 1)), -1, dtype=np.int32)
    for i, r in enumerate(rows):
        t[i, :len(r)] = r
    return t


def make_step(name: str, seed: int, *, H_q: int, H_kv: int, D: int, P: int,
              num_pages: int, dec_cached: Sequence[int] = (),
              pre_prefix: Sequence[int] = (), pre_qlen: Sequence[int] = (),
              window: int = 0, k_head_scale: Optional[np.ndarray] = None,
              n_layers: int = 1, maxblk: Optional[int] = None) -> Step:
    """Assign pages from a seeded permutation of the pool to each sequence."""
    rng = np.random.default_rng(seed)
    alloc = _PageAllocator(rng, num_pages)
    dec_cached = np.asarray(dec_cached, dtype=np.int32)
    pre_prefix = np.asarray(pre_prefix, dtype=np.int32)
    pre_qlen = np.asarray(pre_qlen, dtype=np.int32)
    need = [(-(-(int(c) + 1) // P)) for c in dec_cached]
    need_p = [(-(-(int(a) + int(b)) // P)) for a, b in zip(pre_prefix, pre_qlen)]
    mb = max(need + need_p + [1]) if maxblk is None else maxblk
    dec_rows = [alloc.take(n) for n in need]
    pre_rows = [alloc.take(n) for n in need_p]
    used = np.concatenate(dec_rows + pre_rows) if (dec_rows or pre_rows) \
        else np.zeros(0, np.int32)
    return Step(name=name, H_q=H_q, H_kv=H_kv, D=D, P=P, num_pages=num_pages,
                window=window, scale=float(1.0 / np.sqrt(D)), n_layers=n_layers,
                dec_cached=dec_cached if len(dec_cached) else None,
                dec_block_table=_table(dec_rows, mb) if len(dec_cached) else None,
                pre_prefix=pre_prefix if len(pre_qlen) else None,
                pre_qlen=pre_qlen if len(pre_qlen) else None,
                pre_block_table=_table(pre_rows, mb) if len(pre_qlen) else None,
                used_pages=np.sort(used), k_head_scale=k_head_scale)


def fill_values(step: Step, seed: int, fill_unused: bool = False) -> StepValues:
    """Draw Q, new K/V and the contents of every referenced page.

    Unreferenced pages stay zero unless ``fill_unused`` (the kernels never
    read them; the tiny workload fills all 32 pages).  Referenced pages are
    filled whole, including rows past a sequence's length, so that masking
    of those rows is exercised.
    """
    rng = np.random.default_rng(seed + 1_000_003)
    shape = (step.num_pages, step.H_kv, step.P, step.D)
    ks = None
    if step.k_head_scale is not None:
        ks = step.k_head_scale.astype(np.float32)[None, :, None, None]
    k_cache = np.zeros(shape, dtype=np.uint16)
    v_cache = np.zeros(shape, dtype=np.uint16)
    pages = np.arange(step.num_pages) if fill_unused else step.used_pages
    if len(pages):
        k_cache[pages] = randn_bf16(rng, (len(pages),) + shape[1:], ks)
        v_cache[pages] = randn_bf16(rng, (len(pages),) + shape[1:])
    n_new = step.n_new_tokens
    ksn = None if ks is None else ks[:, :, 0, :]
    k_new = randn_bf16(rng, (n_new, step.H_kv, step.D), ksn)
    v_new = randn_bf16(rng, (n_new, step.H_kv, step.D))
    q_dec = [randn_bf16(rng, (step.Bd, step.H_q, step.D))
             for _ in range(step.n_layers)]
    q_pre = [randn_bf16(rng, (step.total_q, step.H_q, step.D))
             for _ in range(step.n_layers)]
    return StepValues(k_cache, v_cache, k_new, v_new, q_dec, q_pre)


# ---------------------------------------------------------------------------
# Named workloads
# ---------------------------------------------------------------------------
def tiny(seed: int = BASE_SEED + 1) -> Step:
    return make_step("tiny", seed, H_q=4, H_kv=2, D=64, P=16, num_pages=32,
                     dec_cached=[7, 33, 64, 100])


def qwen3_decode(seed: int = BASE_SEED + 2, batch: int = 64,
                 num_pages: int = 16384) -> Step:
    rng = np.random.default_rng(seed)
    cached = rng.integers(256, 2048, size=batch, endpoint=True)
    khs = rng.uniform(0.5, 2.0, size=8).astype(np.float32)
    return make_step("qwen3_decode", seed, H_q=32, H_kv=8, D=128, P=16,
                     num_pages=num_pages, dec_cached=cached, k_head_scale=khs)


def mixed_step(seed: int = BASE_SEED + 3, H_q: int = 32, H_kv: int = 8,
               D: int = 128, n_chunks: int = 8, n_dec: int = 120,
               num_pages: int = 32768) -> Step:
    rng = np.random.default_rng(seed)
    qlen = rng.integers(128, 1024, size=n_chunks, endpoint=True)
    prefix = rng.integers(0, 512, size=n_chunks, endpoint=True)
    cached = rng.integers(64, 4096, size=n_dec, endpoint=True)
    return make_step("mixed_step", seed, H_q=H_q, H_kv=H_kv, D=D, P=16,
                     num_pages=num_pages, dec_cached=cached,
                     pre_prefix=prefix, pre_qlen=qlen)


def sliding(seed: int = BASE_SEED + 4, n_dec: int = 32, n_chunks: int = 4,
            chunk: int = 2048, prefix: int = 0, num_pages: int = 4096) -> Step:
    rng = np.random.default_rng(seed)
    cached = rng.integers(1024, 8192, size=n_dec, endpoint=True)
    return make_step("sliding", seed, H_q=8, H_kv=1, D=256, P=64,
                     num_pages=num_pages, dec_cached=cached,
                     pre_prefix=[prefix] * n_chunks, pre_qlen=[chunk] * n_chunks,
                     window=512, n_layers=2)


def full_d512(seed: int = BASE_SEED + 6, n_dec: int = 64, n_chunks: int = 4,
              chunk: int = 1024, num_pages: Optional[int] = None) -> Step:
    """The full-attention regime with 512-wide heads (the Gemma-4 engine
    commit's second attention regime: head_dim 512, rope_theta 1e6): 8 q
    heads on 1 kv head, page 16, decode rows cached ~U[1024,8192] plus
    prefill chunks of ``chunk`` tokens (prefix 0)."""
    rng = np.random.default_rng(seed)
    cached = rng.integers(1024, 8192, size=n_dec, endpoint=True)
    need = int(sum(-(-(int(c) + 1) // 16) for c in cached)) + n_chunks * (-(-chunk // 16))
    return make_step("full_d512", seed, H_q=8, H_kv=1, D=512, P=16,
                     num_pages=num_pages or need + 64, dec_cached=cached,
                     pre_prefix=[0] * n_chunks, pre_qlen=[chunk] * n_chunks)


def grpo_layer(seed: int = BASE_SEED + 5, n_prompts: int = 64, n_gen: int = 4,
               prefix: int = 256, max_completion: int = 3840,
               layers: int = 36, layer: int = 0) -> Step:
    """One layer's view of the rollout-scale decode step.

    All ``layers`` share one pool; layer ``layer`` owns the page range
    [layer*pages_per_layer, (layer+1)*pages_per_layer).  Each prompt's
    prefix pages are allocated once and referenced by all ``n_gen`` tables.
    """
    P = 16
    rng = np.random.default_rng(seed)
    comp = rng.integers(0, max_completion, size=n_prompts * n_gen, endpoint=True)
    pre_pages = -(-prefix // P)
    per_layer = n_prompts * pre_pages + int(sum(-(-(prefix + int(c) + 1) // P) - pre_pages
                                                for c in comp))
    num_pages = per_layer * layers
    lrng = np.random.default_rng(seed * 1000 + layer)
    alloc = _PageAllocator(lrng, num_pages, first=layer * per_layer, count=per_layer)
    rows = []
    for p in range(n_prompts):
        shared = alloc.take(pre_pages)
        for g in range(n_gen):
            c = int(comp[p * n_gen + g])
            own = alloc.take(-(-(prefix + c + 1) // P) - pre_pages)
            rows.append(np.concatenate([shared, own]))
    mb = max(len(r) for r in rows)
    cached = (prefix + comp).astype(np.int32)
    used = np.unique(np.concatenate(rows))
    return Step(name="grpo", H_q=32, H_kv=8, D=128, P=P, num_pages=num_pages,
                window=0, scale=float(1.0 / np.sqrt(128)), dec_cached=cached,
                dec_block_table=_table(rows, mb), used_pages=used,
                layer_page_offset=layer * per_layer, group_size=n_gen,
                prefix_lens=np.full(n_prompts, (prefix // P) * P, np.int32))


WORKLOADS = {
    "tiny": tiny,
    "qwen3_decode": qwen3_decode,
    "mixed_step": mixed_step,
    "sliding": sliding,
    "grpo": grpo_layer,
    "full_d512": full_d512,
}
