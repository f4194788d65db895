"""GPU parity of paged_attn_varlen (tcgen05 prefill) against the fp64 oracle,
through the C ABI: causal bottom-right chunks on cached prefixes, sliding
window, non-causal, GQA groups 1..8, head_dim 64/128/256, pages 16/64, and
the mixed / sliding workloads end to end (append -> varlen -> decode)."""
import numpy as np
import pytest

import oracle
import workloads as wl
from _util import assert_close_attn, bf16_dev_to_f64, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    import torch  # noqa: F401
    from paged_kv_attention_11_gb300 import build
    build.build()
    import paged_kv_attention_11_gb300 as m
    m.lib()
    return m


def _varlen(pkv, step, vals, layer=0, causal=True, window=None, dev=None):
    import torch
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    if dev is None:
        kc, vc = to_dev_bf16(vals.k_cache), to_dev_bf16(vals.v_cache)
        slots = step.all_slots
        pkv.paged_kv_append(to_dev_bf16(vals.k_new), to_dev_bf16(vals.v_new), kc, vc,
                            to_dev(slots), err_flag=err)
    else:
        kc, vc = dev
    w = step.window if window is None else window
    q = to_dev_bf16(vals.q_pre[layer])
    out = torch.full_like(q, float("nan"))
    pkv.paged_attn_varlen(out, q, kc, vc, to_dev(step.cu_seq_lens_q), to_dev(step.cu_seq_lens_k),
                          to_dev(step.pre_block_table), step.max_seqlen_q(), step.max_seqlen_k(),
                          step.scale, causal, w, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, f"device error flag {int(err.item())}"
    hk, hv = oracle.kv_append(vals.k_cache, vals.v_cache, vals.k_new, vals.v_new, step.all_slots)
    want = oracle.paged_varlen(vals.q_pre[layer], hk, hv, step.cu_seq_lens_q,
                               step.cu_seq_lens_k, step.pre_block_table, step.scale, causal, w)
    return bf16_dev_to_f64(out), want, (kc, vc)


def _prefill_step(seed, H_q, H_kv, D, P, prefix, qlen, window=0, num_pages=None):
    need = sum(-(-(a + b) // P) for a, b in zip(prefix, qlen))
    return wl.make_step("t", seed, H_q=H_q, H_kv=H_kv, D=D, P=P,
                        num_pages=num_pages or need + 8, pre_prefix=prefix, pre_qlen=qlen,
                        window=window)


def test_varlen_tiny_single_chunk(pkv):
    step = _prefill_step(1, 4, 2, 64, 16, [20], [40])
    vals = wl.fill_values(step, 1)
    got, want, _ = _varlen(pkv, step, vals)
    assert_close_attn(got, want, "tiny")


@pytest.mark.parametrize("D", [64, 128, 256, 512])
@pytest.mark.parametrize("H", [(8, 8), (8, 4), (8, 2), (8, 1), (32, 8)])
def test_varlen_shapes(pkv, D, H):
    P = 64 if D == 256 else 16
    prefix = [0, 37, 200, 5]
    qlen = [130, 1, 77, 300]
    step = _prefill_step(D + H[0] + H[1], H[0], H[1], D, P, prefix, qlen)
    vals = wl.fill_values(step, D)
    got, want, _ = _varlen(pkv, step, vals)
    assert_close_attn(got, want, f"D={D} H={H}")


@pytest.mark.parametrize("P", [16, 32, 64, 128, 256])
def test_varlen_page_sizes(pkv, P):
    step = _prefill_step(P, 8, 2, 128, P, [100, 0], [300, 129])
    vals = wl.fill_values(step, P)
    got, want, _ = _varlen(pkv, step, vals)
    assert_close_attn(got, want, f"P={P}")


@pytest.mark.parametrize("window", [1, 2, 64, 127, 128, 129, 512])
def test_varlen_sliding_window(pkv, window):
    step = _prefill_step(window, 8, 1, 256, 64, [0, 1024, 30], [700, 300, 513], window=window)
    vals = wl.fill_values(step, window)
    got, want, _ = _varlen(pkv, step, vals)
    assert_close_attn(got, want, f"window={window}")


def test_varlen_non_causal(pkv):
    step = _prefill_step(9, 8, 2, 128, 16, [0, 50], [200, 64])
    vals = wl.fill_values(step, 9)
    got, want, _ = _varlen(pkv, step, vals, causal=False)
    assert_close_attn(got, want, "non-causal")


def test_varlen_empty_chunks_and_single_rows(pkv):
    step = _prefill_step(10, 8, 2, 128, 16, [10, 0, 300, 0, 7], [0, 1, 0, 129, 1])
    vals = wl.fill_values(step, 10)
    got, want, _ = _varlen(pkv, step, vals)
    assert_close_attn(got, want, "empty")


def test_varlen_q1_equals_decode(pkv):
    """A chunk of one query is the decode step of the same sequence: both
    kernels match the oracle's varlen result and its decode result (the two
    oracle results are the same rows), and each other."""
    import torch
    prefix = [63, 500, 2000]
    step = _prefill_step(11, 32, 8, 128, 16, prefix, [1, 1, 1])
    vals = wl.fill_values(step, 11)
    got, want, (kc, vc) = _varlen(pkv, step, vals)
    assert_close_attn(got, want, "q1 varlen vs oracle")
    out = torch.empty_like(to_dev_bf16(vals.q_pre[0]))
    lens = (step.pre_prefix + step.pre_qlen).astype(np.int32)
    pkv.paged_attn_decode(out, to_dev_bf16(vals.q_pre[0]), kc, vc, to_dev(step.pre_block_table),
                          to_dev(lens), int(lens.max()), step.scale, 0)
    torch.cuda.synchronize()
    hk, hv = oracle.kv_append(vals.k_cache, vals.v_cache, vals.k_new, vals.v_new, step.all_slots)
    want_dec = oracle.paged_decode(vals.q_pre[0], hk, hv, step.pre_block_table, lens, step.scale)
    assert np.array_equal(want_dec, want), "oracle: decode and q_len=1 varlen rows differ"
    got_dec = bf16_dev_to_f64(out)
    assert_close_attn(got_dec, want_dec, "q1 decode vs oracle")
    assert_close_attn(got, got_dec, "q1 varlen vs decode")


def test_varlen_sharp_scores_rescale_path(pkv):
    """Scores growing along the sequence force the O rescale in TMEM."""
    step = _prefill_step(12, 8, 2, 128, 16, [0], [600])
    vals = wl.fill_values(step, 12)
    # K rows scaled by a ramp so later keys have larger logits
    K = oracle.bf16_bits_to_f64(vals.k_cache).astype(np.float32)
    ramp = np.linspace(0.2, 6.0, step.P, dtype=np.float32)[None, None, :, None]
    vals.k_cache = wl.f32_to_bf16_bits(K * ramp)
    kn = oracle.bf16_bits_to_f64(vals.k_new).astype(np.float32)
    vals.k_new = wl.f32_to_bf16_bits(kn * np.linspace(0.2, 8.0, kn.shape[0],
                                                      dtype=np.float32)[:, None, None])
    got, want, _ = _varlen(pkv, step, vals)
    assert_close_attn(got, want, "rescale")


def test_varlen_mixed_workload_end_to_end(pkv):
    """Continuous-batching mixed step: append all rows, varlen chunks, decode rows."""
    import torch
    step = wl.mixed_step()
    vals = wl.fill_values(step, 3)
    got, want, (kc, vc) = _varlen(pkv, step, vals)
    assert_close_attn(got, want, "mixed prefill")
    hk, hv = oracle.kv_append(vals.k_cache, vals.v_cache, vals.k_new, vals.v_new, step.all_slots)
    q = to_dev_bf16(vals.q_dec[0])
    out = torch.empty_like(q)
    pkv.paged_attn_decode(out, q, kc, vc, to_dev(step.dec_block_table), to_dev(step.dec_seq_lens),
                          step.max_seq_len_dec(), step.scale, 0)
    torch.cuda.synchronize()
    want_d = oracle.paged_decode(vals.q_dec[0], hk, hv, step.dec_block_table, step.dec_seq_lens,
                                 step.scale)
    assert_close_attn(bf16_dev_to_f64(out), want_d, "mixed decode")


def test_varlen_mixed_small_heads(pkv):
    """The mixed step at the tiny head shape (4 q heads, 2 kv heads, head_dim 64)."""
    step = wl.mixed_step(H_q=4, H_kv=2, D=64, n_dec=16, num_pages=8192)
    vals = wl.fill_values(step, 4)
    got, want, _ = _varlen(pkv, step, vals)
    assert_close_attn(got, want, "mixed 4/2/64")


def test_varlen_sliding_workload_two_layers(pkv):
    """Sliding-window workload: layer 0 appends and attends, layer 1 reads
    the same pool with its own queries (shared KV)."""
    step = wl.sliding()
    vals = wl.fill_values(step, 5)
    got, want, dev = _varlen(pkv, step, vals, layer=0)
    assert_close_attn(got, want, "sliding layer 0")
    got1, want1, _ = _varlen(pkv, step, vals, layer=1, dev=dev)
    assert_close_attn(got1, want1, "sliding layer 1")


def test_varlen_sliding_with_prefix(pkv):
    step = wl.sliding(prefix=1024, n_dec=4, n_chunks=2, chunk=1000)
    vals = wl.fill_values(step, 6)
    got, want, _ = _varlen(pkv, step, vals)
    assert_close_attn(got, want, "sliding + prefix")


def test_varlen_bad_page_flags_no_fault(pkv):
    import torch
    step = _prefill_step(13, 8, 2, 128, 16, [0, 0], [64, 64])
    vals = wl.fill_values(step, 13)
    kc, vc = to_dev_bf16(vals.k_cache), to_dev_bf16(vals.v_cache)
    bt = step.pre_block_table.copy()
    bt[1, 2] = 10 ** 6
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    q = to_dev_bf16(vals.q_pre[0])
    out = torch.empty_like(q)
    pkv.paged_attn_varlen(out, q, kc, vc, to_dev(step.cu_seq_lens_q), to_dev(step.cu_seq_lens_k),
                          to_dev(bt), step.max_seqlen_q(), step.max_seqlen_k(), step.scale, True,
                          0, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & 2
    want = oracle.paged_varlen(vals.q_pre[0], vals.k_cache, vals.v_cache, step.cu_seq_lens_q,
                               step.cu_seq_lens_k, step.pre_block_table, step.scale)
    assert_close_attn(bf16_dev_to_f64(out)[:64], want[:64], "untouched chunk")
    assert np.all(np.isfinite(bf16_dev_to_f64(out)))


def test_varlen_head_dim_512_workload(pkv):
    """The full-attention regime with 512-wide heads: 4 prefill chunks of
    1024 tokens, 8 q heads on 1 kv head, page 16 (each Q tile's O is
    computed in two 256-column halves)."""
    step = wl.full_d512(n_dec=4)
    vals = wl.fill_values(step, 512)
    got, want, _ = _varlen(pkv, step, vals)
    assert_close_attn(got, want, "head_dim 512 prefill")


@pytest.mark.parametrize("window,P", [(100, 16), (0, 64), (513, 32)])
def test_varlen_head_dim_512_window_pages(pkv, window, P):
    step = _prefill_step(5120 + window + P, 16, 2, 512, P, [0, 300, 17], [400, 129, 64],
                         window=window)
    vals = wl.fill_values(step, 77)
    got, want, _ = _varlen(pkv, step, vals)
    assert_close_attn(got, want, f"D=512 window={window} P={P}")
