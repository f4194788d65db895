"""GPU parity: paged_kv_append (bit-exact) and paged_attn_decode (bf16 vs the
fp64 oracle) through the C ABI, on the named workloads and edge cases."""
import numpy as np
import pytest

import oracle
import workloads as wl
from _util import (assert_close_attn, bf16_dev_to_bits, bf16_dev_to_f64, to_dev,
                   to_dev_bf16)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    import torch  # noqa: F401
    from paged_kv_attention_11_gb300 import build
    build.build()
    import paged_kv_attention_11_gb300 as m
    m.lib()
    return m


def _err(torch):
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def run_decode_step(pkv, step, vals, layer=0, do_append=True, dev=None):
    """Append this step's new rows, then decode; returns (gpu out, oracle out,
    device pools, host pools after append)."""
    import torch
    if dev is None:
        dev = dict(k=to_dev_bf16(vals.k_cache), v=to_dev_bf16(vals.v_cache))
    err = _err(torch)
    kc, vc = dev["k"], dev["v"]
    slots = step.all_slots
    if do_append and len(slots):
        pkv.paged_kv_append(to_dev_bf16(vals.k_new), to_dev_bf16(vals.v_new), kc, vc,
                            to_dev(slots), err_flag=err)
    hk, hv = oracle.kv_append(vals.k_cache, vals.v_cache, vals.k_new, vals.v_new, slots)
    q = to_dev_bf16(vals.q_dec[layer])
    out = torch.empty_like(q)
    pkv.paged_attn_decode(out, q, kc, vc, to_dev(step.dec_block_table),
                          to_dev(step.dec_seq_lens), step.max_seq_len_dec(), step.scale,
                          step.window, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    want = oracle.paged_decode(vals.q_dec[layer], hk, hv, step.dec_block_table,
                               step.dec_seq_lens, step.scale, step.window)
    return bf16_dev_to_f64(out), want, (kc, vc), (hk, hv)


@pytest.mark.parametrize("name", ["tiny", "qwen3_decode", "mixed_step", "sliding"])
def test_workload_append_and_decode(pkv, name):
    step = wl.WORKLOADS[name]()
    vals = wl.fill_values(step, 3407, fill_unused=(name == "tiny"))
    got, want, (kc, vc), (hk, hv) = run_decode_step(pkv, step, vals)
    assert np.array_equal(bf16_dev_to_bits(kc), hk), "K pool differs after append"
    assert np.array_equal(bf16_dev_to_bits(vc), hv), "V pool differs after append"
    assert_close_attn(got, want, name)
    if step.n_layers > 1:   # shared-KV layer: its own Q over the same pool, no append
        got2, want2, _, _ = run_decode_step(pkv, step, vals, layer=1, do_append=False,
                                            dev=dict(k=kc, v=vc))
        assert_close_attn(got2, want2, name + " layer 1")


def test_grpo_layer_prefix_sharing(pkv):
    """Rollout decode with prefix pages aliased by 4 generations (one layer)."""
    step = wl.grpo_layer(layers=1, n_prompts=16)
    vals = wl.fill_values(step, 11)
    got, want, _, _ = run_decode_step(pkv, step, vals)
    assert_close_attn(got, want, "grpo")


def _random_case(rng, B, H_q, H_kv, D, P, lens, num_pages=None, extra=4):
    need = [max(1, -(-L // P)) for L in lens]
    num_pages = num_pages or (sum(need) + extra)
    perm = rng.permutation(num_pages).astype(np.int32)
    bt = np.full((B, max(need)), -1, np.int32)
    o = 0
    for b, n in enumerate(need):
        bt[b, :n] = perm[o:o + n]
        o += n
    kc = wl.randn_bf16(rng, (num_pages, H_kv, P, D))
    vc = wl.randn_bf16(rng, (num_pages, H_kv, P, D))
    q = wl.randn_bf16(rng, (B, H_q, D))
    return q, kc, vc, bt, np.asarray(lens, np.int32)


def _decode(pkv, q, kc, vc, bt, lens, scale, window, max_len=None):
    import torch
    err = _err(torch)
    qd = to_dev_bf16(q)
    out = torch.empty_like(qd)
    pkv.paged_attn_decode(out, qd, to_dev_bf16(kc), to_dev_bf16(vc), to_dev(bt), to_dev(lens),
                          int(lens.max()) if max_len is None else max_len, scale, window,
                          err_flag=err)
    torch.cuda.synchronize()
    return out, int(err.item())


@pytest.mark.parametrize("D", [64, 128, 256, 512])
@pytest.mark.parametrize("H", [(8, 8), (8, 4), (8, 2), (8, 1), (16, 2)])
@pytest.mark.parametrize("P", [16, 64])
def test_decode_shapes(pkv, D, H, P):
    rng = np.random.default_rng(D * 100 + H[0] * 10 + H[1] + P)
    lens = [1, 15, 16, 17, 100, 333, 1000, 0, 64, 65]
    q, kc, vc, bt, L = _random_case(rng, len(lens), H[0], H[1], D, P, lens)
    out, err = _decode(pkv, q, kc, vc, bt, L, 1 / np.sqrt(D), 0)
    assert err == 0
    want = oracle.paged_decode(q, kc, vc, bt, L, 1 / np.sqrt(D))
    got = bf16_dev_to_f64(out)
    assert_close_attn(got, want, f"D={D} H={H} P={P}")
    assert np.all(got[lens.index(0)] == 0)


def test_decode_head_dim_256_large_call(pkv):
    """head_dim 256 above the small-call size (more than ~1 MB of K/V per
    SM): the launch with 4 consumer warps and 8 stages."""
    rng = np.random.default_rng(256)
    lens = list(rng.integers(1, 2048, size=24))
    lens[0] = 2048
    q, kc, vc, bt, L = _random_case(rng, len(lens), 8, 4, 256, 16, lens)
    out, err = _decode(pkv, q, kc, vc, bt, L, 1 / 16, 0)
    assert err == 0
    want = oracle.paged_decode(q, kc, vc, bt, L, 1 / 16)
    assert_close_attn(bf16_dev_to_f64(out), want, "d256 large")


@pytest.mark.parametrize("window", [1, 2, 16, 17, 100, 512])
def test_decode_window(pkv, window):
    rng = np.random.default_rng(window)
    lens = [1, 5, 16, 31, 64, 200, 777, 2048]
    q, kc, vc, bt, L = _random_case(rng, len(lens), 8, 2, 128, 16, lens)
    out, err = _decode(pkv, q, kc, vc, bt, L, 0.09, window)
    assert err == 0
    want = oracle.paged_decode(q, kc, vc, bt, L, 0.09, window)
    got = bf16_dev_to_f64(out)
    assert_close_attn(got, want, f"window={window}")
    if window == 1:  # only the query's own key: its V row, exactly
        for b, n in enumerate(lens):
            V = oracle.gather_sequence(vc, bt[b], n)[n - 1]
            for h in range(8):
                assert np.array_equal(got[b, h], oracle.bf16_bits_to_f64(V[h // 4]))


def test_decode_single_long_sequence_many_splits(pkv):
    rng = np.random.default_rng(5)
    q, kc, vc, bt, L = _random_case(rng, 1, 32, 8, 128, 16, [16000])
    out, err = _decode(pkv, q, kc, vc, bt, L, 1 / np.sqrt(128), 0)
    assert err == 0
    assert_close_attn(bf16_dev_to_f64(out), oracle.paged_decode(q, kc, vc, bt, L, 1 / np.sqrt(128)),
                      "long")


def test_decode_many_empty_and_tiny_sequences(pkv):
    rng = np.random.default_rng(6)
    lens = list(rng.integers(0, 4, size=300))
    lens[7] = 5000
    q, kc, vc, bt, L = _random_case(rng, len(lens), 4, 1, 64, 16, lens)
    out, err = _decode(pkv, q, kc, vc, bt, L, 0.125, 0)
    assert err == 0
    assert_close_attn(bf16_dev_to_f64(out), oracle.paged_decode(q, kc, vc, bt, L, 0.125),
                      "empty-mix")


def test_decode_sharp_and_large_scores(pkv):
    """Scores of order 1e2 must not overflow the exp2-domain softmax."""
    rng = np.random.default_rng(7)
    q, kc, vc, bt, L = _random_case(rng, 4, 8, 2, 128, 16, [50, 300, 1000, 17])
    q = wl.f32_to_bf16_bits(oracle.bf16_bits_to_f64(q).astype(np.float32) * 8)
    out, err = _decode(pkv, q, kc, vc, bt, L, 1.0, 0)
    assert err == 0
    assert_close_attn(bf16_dev_to_f64(out), oracle.paged_decode(q, kc, vc, bt, L, 1.0), "sharp")


def test_decode_is_deterministic(pkv):
    rng = np.random.default_rng(8)
    q, kc, vc, bt, L = _random_case(rng, 64, 32, 8, 128, 16, rng.integers(1, 3000, 64))
    a, _ = _decode(pkv, q, kc, vc, bt, L, 0.088, 0)
    b, _ = _decode(pkv, q, kc, vc, bt, L, 0.088, 0)
    assert np.array_equal(bf16_dev_to_bits(a), bf16_dev_to_bits(b))


def test_decode_bad_block_table_entry_flags_and_masks(pkv):
    rng = np.random.default_rng(9)
    lens = [40, 40, 40]
    q, kc, vc, bt, L = _random_case(rng, 3, 4, 2, 64, 16, lens)
    bad = bt.copy()
    bad[1, 1] = kc.shape[0] + 7      # keys 16..31 of sequence 1 point outside the pool
    bad[2, 0] = -3                   # keys 0..15 of sequence 2
    out, err = _decode(pkv, q, kc, vc, bad, L, 0.125, 0)
    assert err & 2                   # PKV_DEVERR_PAGE
    got = bf16_dev_to_f64(out)
    want0 = oracle.paged_decode(q[:1], kc, vc, bt[:1], L[:1], 0.125)
    assert_close_attn(got[:1], want0, "untouched row")
    # row 1 = attention over keys {0..15, 32..39} only
    K = oracle.bf16_bits_to_f64(oracle.gather_sequence(kc, bt[1], 40))
    V = oracle.bf16_bits_to_f64(oracle.gather_sequence(vc, bt[1], 40))
    keep = np.r_[0:16, 32:40]
    want1 = oracle.attend_rows(oracle.bf16_bits_to_f64(q[1:2]), K[keep], V[keep],
                               np.array([len(keep) - 1]), 0.125)
    assert_close_attn(got[1:2], want1, "masked page")


def test_decode_length_beyond_table_is_clamped_and_flagged(pkv):
    rng = np.random.default_rng(10)
    q, kc, vc, bt, L = _random_case(rng, 2, 4, 2, 64, 16, [32, 20])
    L2 = L.copy()
    L2[0] = 1000                     # table holds only 2 pages
    out, err = _decode(pkv, q, kc, vc, bt, L2, 0.125, 0, max_len=1000)
    assert err & 4                   # PKV_DEVERR_LEN
    want = oracle.paged_decode(q, kc, vc, bt, L, 0.125)
    assert_close_attn(bf16_dev_to_f64(out), want, "clamped")


def test_append_skip_and_out_of_pool_slots(pkv):
    import torch
    rng = np.random.default_rng(11)
    num_pages, H_kv, P, D = 6, 2, 16, 128
    kc = np.full((num_pages, H_kv, P, D), 0x7E57, np.uint16)
    vc = np.full_like(kc, 0x0BAD)
    T = 9
    k_new = wl.randn_bf16(rng, (T, H_kv, D))
    v_new = wl.randn_bf16(rng, (T, H_kv, D))
    slots = rng.permutation(num_pages * P)[:T].astype(np.int64)
    slots[2] = -1
    slots[5] = num_pages * P + 3     # outside the pool
    kd, vd = to_dev_bf16(kc), to_dev_bf16(vc)
    err = _err(torch)
    pkv.paged_kv_append(to_dev_bf16(k_new), to_dev_bf16(v_new), kd, vd, to_dev(slots),
                        err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & 1       # PKV_DEVERR_SLOT
    ok = slots.copy()
    ok[5] = -1
    hk, hv = oracle.kv_append(kc, vc, k_new, v_new, ok)
    assert np.array_equal(bf16_dev_to_bits(kd), hk)
    assert np.array_equal(bf16_dev_to_bits(vd), hv)


def test_append_large_prefill_sized(pkv):
    """A prefill-sized append (8 k rows of 2 KB) over a shuffled slot set."""
    import torch
    rng = np.random.default_rng(12)
    num_pages, H_kv, P, D = 1024, 8, 16, 128
    kc = wl.randn_bf16(rng, (num_pages, H_kv, P, D))
    vc = wl.randn_bf16(rng, (num_pages, H_kv, P, D))
    T = 8192
    slots = rng.permutation(num_pages * P)[:T].astype(np.int64)
    k_new = wl.randn_bf16(rng, (T, H_kv, D))
    v_new = wl.randn_bf16(rng, (T, H_kv, D))
    kd, vd = to_dev_bf16(kc), to_dev_bf16(vc)
    pkv.paged_kv_append(to_dev_bf16(k_new), to_dev_bf16(v_new), kd, vd, to_dev(slots))
    torch.cuda.synchronize()
    hk, hv = oracle.kv_append(kc, vc, k_new, v_new, slots)
    assert np.array_equal(bf16_dev_to_bits(kd), hk)
    assert np.array_equal(bf16_dev_to_bits(vd), hv)


@pytest.mark.parametrize("T,H_kv,D,P", [
    (1, 8, 128, 16),       # one token
    (3, 1, 512, 16),       # a 1 KB row: fewer vectors than lanes
    (40000, 8, 128, 16),   # more tokens than one wave of warps
    (5000, 1, 256, 64),
    (777, 2, 64, 32),
    (300, 24, 512, 16),    # 24 KB rows: many passes per warp
    (50, 64, 512, 16),     # 64 KB rows
])
def test_append_row_sizes_and_padding(pkv, T, H_kv, D, P):
    """Whole pools bit-exact against the oracle across token counts and row
    sizes (one or two vectors per lane per pass, many passes), with padding
    rows mixed in."""
    import torch
    rng = np.random.default_rng(T + H_kv + D)
    num_pages = -(-T // P) + 3
    kc = wl.randn_bf16(rng, (num_pages, H_kv, P, D))
    vc = wl.randn_bf16(rng, (num_pages, H_kv, P, D))
    slots = rng.permutation(num_pages * P)[:T].astype(np.int64)
    slots[::7] = -1
    k_new = wl.randn_bf16(rng, (T, H_kv, D))
    v_new = wl.randn_bf16(rng, (T, H_kv, D))
    kd, vd = to_dev_bf16(kc), to_dev_bf16(vc)
    err = _err(torch)
    pkv.paged_kv_append(to_dev_bf16(k_new), to_dev_bf16(v_new), kd, vd, to_dev(slots),
                        err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    hk, hv = oracle.kv_append(kc, vc, k_new, v_new, slots)
    assert np.array_equal(bf16_dev_to_bits(kd), hk)
    assert np.array_equal(bf16_dev_to_bits(vd), hv)


def test_decode_workspace_reuse_stays_clean(pkv):
    """One workspace across many calls of different shapes: the arrival
    counters must return to zero after every call."""
    import torch
    rng = np.random.default_rng(13)
    ws = torch.zeros(pkv.decode_workspace_size(300, 32, 8, 128) + 4096, dtype=torch.uint8,
                     device="cuda")
    for it in range(6):
        B = int(rng.integers(1, 300))
        lens = rng.integers(0, 4000, B)
        q, kc, vc, bt, L = _random_case(rng, B, 32, 8, 128, 16, lens)
        qd = to_dev_bf16(q)
        out = torch.empty_like(qd)
        err = _err(torch)
        pkv.paged_attn_decode(out, qd, to_dev_bf16(kc), to_dev_bf16(vc), to_dev(bt), to_dev(L),
                              int(L.max()), 0.088, 0, workspace=ws, err_flag=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert_close_attn(bf16_dev_to_f64(out), oracle.paged_decode(q, kc, vc, bt, L, 0.088),
                          f"reuse {it}")
    counters = ws[:300 * 8 * 4].view(torch.int32)
    assert int(counters.abs().sum().item()) == 0


def test_decode_head_dim_512_workload(pkv):
    """The full-attention regime with 512-wide heads (8 q heads on 1 kv
    head): 64 decode rows over contexts of 1k-8k tokens, append first."""
    step = wl.full_d512()
    vals = wl.fill_values(step, 512)
    got, want, (kc, vc), (hk, hv) = run_decode_step(pkv, step, vals)
    assert np.array_equal(bf16_dev_to_bits(kc), hk), "K pool differs after append"
    assert_close_attn(got, want, "head_dim 512")


@pytest.mark.parametrize("window", [1, 300])
def test_decode_head_dim_512_window_and_short(pkv, window):
    rng = np.random.default_rng(512 + window)
    lens = [1, 2, 16, 17, 700, 5000]
    q, kc, vc, bt, L = _random_case(rng, len(lens), 16, 2, 512, 16, lens)
    out, err = _decode(pkv, q, kc, vc, bt, L, 1 / np.sqrt(512), window)
    assert err == 0
    want = oracle.paged_decode(q, kc, vc, bt, L, 1 / np.sqrt(512), window)
    assert_close_attn(bf16_dev_to_f64(out), want, f"D=512 window={window}")
