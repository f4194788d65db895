"""paged_attn_decode_static: decode for callers that cannot allocate device
memory (an engine that has handed all free HBM to its KV page pool, a plugin
host that passes a kernel only its inputs and outputs).  Its scratch is the
library's own fixed 8 MiB device array instead of a caller workspace.

Checked here through the C ABI on two calls in a row with different
batches, each with a sequence long enough to be split into chunks (so the
partial results really go through the fixed array):
  - against the fp64 oracle, at the attention tolerance;
  - against paged_attn_decode with a caller workspace, bit for bit (same
    kernel, same schedule, a merge order that does not depend on which CTA
    ran a chunk).
Also: a batch whose scratch would exceed the fixed array is rejected before
anything is enqueued.  This file is collected last so that a failure here
never hides the other tests.
"""
import ctypes

import numpy as np
import pytest

import oracle
import workloads as wl
from _util import assert_close_attn, bf16_dev_to_bits, bf16_dev_to_f64, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import torch  # noqa: F401
    from paged_kv_attention_11_gb300 import build
    build.build()
    import paged_kv_attention_11_gb300 as m
    return m.lib()


def _case(seed, B, long_len, H_q=32, H_kv=8, D=128, P=16):
    """B sequences of 1..3000 keys, sequence 0 of ``long_len`` keys."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(1, 3000, size=B).astype(np.int32)
    lens[0] = long_len
    need = [-(-int(L) // P) for L in lens]
    num_pages = sum(need) + 8
    perm = rng.permutation(num_pages).astype(np.int32)
    bt = np.full((B, max(need)), -1, np.int32)
    o = 0
    for b, n in enumerate(need):
        bt[b, :n] = perm[o:o + n]
        o += n
    kc = wl.randn_bf16(rng, (num_pages, H_kv, P, D))
    vc = wl.randn_bf16(rng, (num_pages, H_kv, P, D))
    q = wl.randn_bf16(rng, (B, H_q, D))
    return q, kc, vc, bt, lens


def _longest_segment_is_split(lens, H_q, H_kv, P, n_sms, D):
    """The decode kernel cuts a segment (a sequence and its HP kv heads: two
    at head_dim 128 with an even kv-head count and a GQA group of at most 4,
    else one) into chunks when it has more 16-key tiles than half of one
    CTA's share of the batch's head-tiles (16 keys of one kv head; one
    persistent CTA per SM) and more than 16, and the longest segment
    exceeds that cut by more than a merge's cost (480 KB of K+V, 64*D*HP
    bytes per tile of the segment)."""
    G = H_q // H_kv
    hp = 2 if (D == 128 and H_kv % 2 == 0 and G <= 4) else 1
    tiles = -(-lens.astype(np.int64) // 16)
    half_share = -(-int(tiles.sum()) * H_kv // (2 * n_sms))
    cut = max(16, half_share)
    return int(tiles.max()) > cut + (480 * 1024) // (64 * D * hp)


def _args(out, q, kc, vc, bt, lens, scale):
    B, H_q, D = q.shape
    num_pages, H_kv, P, _ = kc.shape
    return (ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(q.data_ptr()),
            ctypes.c_void_p(kc.data_ptr()), ctypes.c_void_p(vc.data_ptr()),
            ctypes.c_void_p(bt.data_ptr()), bt.shape[1], ctypes.c_void_p(lens.data_ptr()),
            B, H_q, H_kv, D, P, num_pages, int(lens.max().item()), ctypes.c_float(scale), 0)


def test_static_scratch_decode_matches_oracle_and_workspace_decode_twice(lib):
    import torch
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    n_sms = torch.cuda.get_device_properties(0).multi_processor_count
    for call, (seed, B, long_len) in enumerate([(101, 64, 20000), (202, 23, 9000)]):
        q, kc, vc, bt, lens = _case(seed, B, long_len)
        assert _longest_segment_is_split(lens, q.shape[1], kc.shape[1], kc.shape[2], n_sms,
                                         q.shape[2])
        qd, kd, vd = to_dev_bf16(q), to_dev_bf16(kc), to_dev_bf16(vc)
        btd, ld = to_dev(bt), to_dev(lens)
        scale = 1.0 / np.sqrt(q.shape[2])
        err = torch.zeros(1, dtype=torch.int32, device="cuda")

        out_static = torch.full_like(qd, float("nan"))
        st = lib.paged_attn_decode_static(*_args(out_static, qd, kd, vd, btd, ld, scale),
                                          ctypes.c_void_p(err.data_ptr()), stream)
        assert st == 0, f"call {call}: status {st}"

        ws_bytes = lib.paged_attn_decode_workspace_size(B, q.shape[1], kc.shape[1], q.shape[2])
        ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
        out_ws = torch.full_like(qd, float("nan"))
        st = lib.paged_attn_decode(*_args(out_ws, qd, kd, vd, btd, ld, scale),
                                   ctypes.c_void_p(ws.data_ptr()), ctypes.c_size_t(ws_bytes),
                                   ctypes.c_void_p(err.data_ptr()), stream)
        assert st == 0
        torch.cuda.synchronize()
        assert int(err.item()) == 0

        want = oracle.paged_decode(q, kc, vc, bt, lens, scale)
        assert_close_attn(bf16_dev_to_f64(out_static), want, f"static vs oracle, call {call}")
        assert np.array_equal(bf16_dev_to_bits(out_static), bf16_dev_to_bits(out_ws)), \
            f"static and workspace decode differ, call {call}"


def test_static_scratch_rejects_oversized_batch(lib):
    import torch
    B, H_q, H_kv, D = 4096, 32, 8, 256  # the largest decode batch; 135 MB of scratch
    need = lib.paged_attn_decode_workspace_size(B, H_q, H_kv, D)
    assert need > (8 << 20)
    dummy = torch.zeros(16, dtype=torch.int32, device="cuda")
    p = ctypes.c_void_p(dummy.data_ptr())
    st = lib.paged_attn_decode_static(p, p, p, p, p, 4, p, B, H_q, H_kv, D, 16, 64, 64,
                                      ctypes.c_float(0.1), 0, None, None)
    assert st == 2  # PKV_ERR_UNSUPPORTED, before anything is enqueued
    assert b"8388608" in lib.pkv_last_cuda_error()
