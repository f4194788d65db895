"""Pins for the fp64 oracle, independent of the oracle's own code path.

The pages print no worked (Q, K, V) -> O example, so the oracle is pinned by
closed forms, invariants, a library-built dense reference and hand-derived
values.  Each test names the kind of mistake it is meant to catch.
"""
import math

import numpy as np
import pytest
from scipy.special import softmax as sp_softmax

import oracle
import workloads as wl

bf = wl.f32_to_bf16_bits
f64 = oracle.bf16_bits_to_f64


# ---------------------------------------------------------------------------
# helpers that build paged inputs from dense ones (index bookkeeping only)
# ---------------------------------------------------------------------------
def paginate(K_bits, V_bits, P, rng, num_pages=None, extra_pages=3):
    """Scatter a dense [L, H_kv, D] sequence into a shuffled page pool."""
    L, H_kv, D = K_bits.shape
    n = -(-L // P)
    num_pages = num_pages or (n + extra_pages)
    perm = rng.permutation(num_pages)[:n].astype(np.int32)
    kc = bf(rng.standard_normal((num_pages, H_kv, P, D)).astype(np.float32))
    vc = bf(rng.standard_normal((num_pages, H_kv, P, D)).astype(np.float32))
    for p in range(L):
        kc[perm[p // P], :, p % P] = K_bits[p]
        vc[perm[p // P], :, p % P] = V_bits[p]
    return kc, vc, perm


def rand_bits(rng, shape, s=1.0):
    return bf((rng.standard_normal(shape) * s).astype(np.float32))


# ---------------------------------------------------------------------------
# bf16 widening: fixed by the bfloat16 format (sign, 8-bit exponent, 7-bit
# mantissa), not by the oracle
# ---------------------------------------------------------------------------
def test_bf16_widening_known_patterns():
    bits = np.array([0x3F80, 0xC000, 0x3F81, 0x0001, 0x7F7F, 0x8000, 0x4049],
                    dtype=np.uint16)
    want = [1.0, -2.0, 1.0 + 2.0 ** -7, 2.0 ** -133,
            (2.0 - 2.0 ** -7) * 2.0 ** 127, -0.0, 3.140625]
    got = f64(bits)
    assert list(got) == want
    assert math.copysign(1.0, got[5]) == -1.0


def test_bf16_rounding_of_inputs_is_nearest_even():
    # 1 + 2^-8 is a tie between 1 and 1+2^-7: even mantissa (1.0) wins;
    # 1 + 3*2^-8 ties between 1+2^-7 and 1+2^-6: even (1+2^-6) wins.
    x = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, 1 + 2 ** -8 + 2 ** -20], np.float32)
    assert list(f64(bf(x))) == [1.0, 1 + 2 ** -6, 1 + 2 ** -7]


# ---------------------------------------------------------------------------
# hand-derived worked examples (closed forms)
# ---------------------------------------------------------------------------
def test_two_key_softmax_by_hand():
    # q=(2,0), keys (1,0),(0,1), scale 1/2 -> scores (1, 0);
    # p = (e/(e+1), 1/(e+1)); values (1,0),(0,3) -> o = (e/(e+1), 3/(e+1)).
    q = bf(np.array([[[2.0, 0.0]]], np.float32))
    K = bf(np.array([[[1.0, 0.0]], [[0.0, 1.0]]], np.float32))
    V = bf(np.array([[[1.0, 0.0]], [[0.0, 3.0]]], np.float32))
    out = oracle.attend_rows(f64(q), f64(K), f64(V), np.array([1]), 0.5)
    e = math.e
    np.testing.assert_allclose(out[0, 0], [e / (e + 1), 3 / (e + 1)], rtol=0, atol=1e-15)
    # the mask drops key 1 for a query at position 0 -> exactly V[0]
    out0 = oracle.attend_rows(f64(q), f64(K), f64(V), np.array([0]), 0.5)
    assert list(out0[0, 0]) == [1.0, 0.0]


def test_golden_fixture_three_keys():
    """tests/golden/three_key_window.txt: values derived by hand."""
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "three_key_window.txt")
    rows = {}
    for line in open(path):
        line = line.split("#", 1)[0].strip()
        if line:
            k, v = line.split("=", 1)
            rows[k.strip()] = v.strip()
    q = np.array(eval(rows["q"]), np.float32)[None, None, :]
    K = np.array(eval(rows["K"]), np.float32)[:, None, :]
    V = np.array(eval(rows["V"]), np.float32)[:, None, :]
    scale = float(rows["scale"])
    for key in ("full", "window2", "window1"):
        w = {"full": 0, "window2": 2, "window1": 1}[key]
        expect = np.array(eval(rows[key], {"e": math.e}), np.float64)
        got = oracle.attend_rows(f64(bf(q)), f64(bf(K)), f64(bf(V)), np.array([2]),
                                 scale, True, w)[0, 0]
        np.testing.assert_allclose(got, expect, rtol=0, atol=1e-14, err_msg=key)


# ---------------------------------------------------------------------------
# closed forms
# ---------------------------------------------------------------------------
def test_single_key_returns_its_value_exactly():
    rng = np.random.default_rng(1)
    q = rand_bits(rng, (1, 4, 32))
    K = rand_bits(rng, (1, 2, 32))
    V = rand_bits(rng, (1, 2, 32))
    out = oracle.attend_rows(f64(q), f64(K), f64(V), np.array([0]), 0.3)
    assert np.array_equal(out[0, :2], np.repeat(f64(V)[0, 0][None], 2, 0))
    assert np.array_equal(out[0, 2:], np.repeat(f64(V)[0, 1][None], 2, 0))


def test_window_one_returns_own_row_exactly():
    rng = np.random.default_rng(2)
    L = 40
    q = rand_bits(rng, (3, 2, 16))
    K = rand_bits(rng, (L, 1, 16))
    V = rand_bits(rng, (L, 1, 16))
    pos = np.array([0, 17, 39])
    out = oracle.attend_rows(f64(q), f64(K), f64(V), pos, 0.25, True, 1)
    for i, p in enumerate(pos):
        assert np.array_equal(out[i, 0], f64(V)[p, 0])
        assert np.array_equal(out[i, 1], f64(V)[p, 0])


def test_identical_keys_give_mean_of_allowed_values_bottom_right():
    """Pins bottom-right causal alignment and the strict window bound."""
    rng = np.random.default_rng(3)
    prefix, qlen, D = 11, 6, 8
    L = prefix + qlen
    k_row = rand_bits(rng, (1, 1, D))
    K = np.repeat(k_row, L, axis=0)
    V = rand_bits(rng, (L, 1, D))
    q = rand_bits(rng, (qlen, 1, D))
    kc, vc, perm = paginate(K, V, 4, rng)
    cu_q = np.array([0, qlen], np.int32)
    cu_k = np.array([0, L], np.int32)
    bt = perm[None, :]
    out = oracle.paged_varlen(q, kc, vc, cu_q, cu_k, bt, 0.5)
    Vf = f64(V)[:, 0]
    for i in range(qlen):
        np.testing.assert_allclose(out[i, 0], Vf[:prefix + i + 1].mean(0), atol=1e-13)
    for W in (1, 2, 5):
        out = oracle.paged_varlen(q, kc, vc, cu_q, cu_k, bt, 0.5, True, W)
        for i in range(qlen):
            qp = prefix + i
            lo = max(0, qp - W + 1)
            np.testing.assert_allclose(out[i, 0], Vf[lo:qp + 1].mean(0), atol=1e-13)


def test_zero_query_gives_mean():
    rng = np.random.default_rng(4)
    K = rand_bits(rng, (9, 1, 8))
    V = rand_bits(rng, (9, 1, 8))
    q = np.zeros((1, 1, 8), np.uint16)
    out = oracle.attend_rows(f64(q), f64(K), f64(V), np.array([8]), 1.0)
    np.testing.assert_allclose(out[0, 0], f64(V)[:, 0].mean(0), atol=1e-14)


def test_sharp_key_selects_its_row():
    D = 4
    q = bf(np.array([[[10.0, 0, 0, 0]]], np.float32))
    K = np.zeros((5, 1, D), np.float32)
    K[3, 0, 0] = 10.0                      # score 100*scale
    V = np.arange(20, dtype=np.float32).reshape(5, 1, D)
    out = oracle.attend_rows(f64(q), f64(bf(K)), f64(bf(V)), np.array([4]), 0.5)
    np.testing.assert_allclose(out[0, 0], V[3, 0], atol=1e-18)


def test_large_scores_stay_finite():
    """Catches a softmax without max subtraction (exp overflow)."""
    rng = np.random.default_rng(5)
    q = bf(np.full((1, 1, 16), 100.0, np.float32))
    K = bf((rng.uniform(50, 60, (7, 1, 16))).astype(np.float32))
    V = rand_bits(rng, (7, 1, 16))
    out = oracle.attend_rows(f64(q), f64(K), f64(V), np.array([6]), 1.0)
    assert np.all(np.isfinite(out))


def test_empty_sequence_and_no_key_rows_are_zero():
    rng = np.random.default_rng(6)
    q = rand_bits(rng, (2, 2, 8))
    kc = rand_bits(rng, (4, 1, 4, 8))
    vc = rand_bits(rng, (4, 1, 4, 8))
    bt = np.array([[0, 1], [2, 3]], np.int32)
    out = oracle.paged_decode(q, kc, vc, bt, np.array([0, 3]), 0.3)
    assert np.all(out[0] == 0)
    assert np.any(out[1] != 0)


# ---------------------------------------------------------------------------
# an independent dense reference built from library routines
# ---------------------------------------------------------------------------
def dense_reference(q, K, V, prefix, scale, window):
    """Contiguous K/V, mask from np.tril/np.triu, scipy softmax."""
    n, H_q, D = q.shape
    L, H_kv, _ = K.shape
    G = H_q // H_kv
    Kr = np.repeat(K, G, axis=1)            # [L, H_q, D]
    Vr = np.repeat(V, G, axis=1)
    allowed = np.tril(np.ones((n, L), bool), k=prefix)
    if window > 0:
        allowed &= np.triu(np.ones((n, L), bool), k=prefix - window + 1)
    out = np.zeros((n, H_q, D))
    for h in range(H_q):
        s = (q[:, h, :] @ Kr[:, h, :].T) * scale
        s = np.where(allowed, s, -np.inf)
        out[:, h, :] = sp_softmax(s, axis=1) @ Vr[:, h, :]
    return out


@pytest.mark.parametrize("P,window,H", [(4, 0, (4, 2)), (16, 0, (8, 1)),
                                        (4, 5, (4, 4)), (8, 3, (6, 2))])
def test_oracle_matches_library_dense_reference(P, window, H):
    rng = np.random.default_rng(7 + P + window)
    H_q, H_kv = H
    D, prefix, qlen = 16, 13, 9
    L = prefix + qlen
    K = rand_bits(rng, (L, H_kv, D))
    V = rand_bits(rng, (L, H_kv, D))
    q = rand_bits(rng, (qlen, H_q, D))
    kc, vc, perm = paginate(K, V, P, rng)
    got = oracle.paged_varlen(q, kc, vc, np.array([0, qlen]), np.array([0, L]),
                              perm[None], 0.37, True, window)
    want = dense_reference(f64(q), f64(K), f64(V), prefix, 0.37, window)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


def test_scalar_loop_reference_tiny():
    """A pure-Python loop with math.exp over 3 keys, 2 heads."""
    rng = np.random.default_rng(8)
    q = rand_bits(rng, (1, 2, 3))
    K = rand_bits(rng, (3, 1, 3))
    V = rand_bits(rng, (3, 1, 3))
    qf, Kf, Vf = f64(q), f64(K), f64(V)
    got = oracle.attend_rows(qf, Kf, Vf, np.array([2]), 0.7)
    for h in range(2):
        s = [sum(qf[0, h, d] * Kf[j, 0, d] for d in range(3)) * 0.7 for j in range(3)]
        w = [math.exp(x - max(s)) for x in s]
        z = sum(w)
        for d in range(3):
            ref = sum(w[j] * Vf[j, 0, d] for j in range(3)) / z
            assert abs(got[0, h, d] - ref) < 1e-14


# ---------------------------------------------------------------------------
# invariants
# ---------------------------------------------------------------------------
def _random_decode_case(rng, B=3, H_q=4, H_kv=2, D=16, P=8, lens=(5, 17, 30)):
    num_pages = 16
    kc = rand_bits(rng, (num_pages, H_kv, P, D))
    vc = rand_bits(rng, (num_pages, H_kv, P, D))
    perm = rng.permutation(num_pages).astype(np.int32)
    need = [-(-L // P) for L in lens]
    bt = np.full((B, max(need)), -1, np.int32)
    o = 0
    for b, n in enumerate(need):
        bt[b, :n] = perm[o:o + n]
        o += n
    q = rand_bits(rng, (B, H_q, D))
    return q, kc, vc, bt, np.array(lens, np.int32)


def test_convex_combination_bounds():
    rng = np.random.default_rng(9)
    q, kc, vc, bt, lens = _random_decode_case(rng)
    out = oracle.paged_decode(q, kc, vc, bt, lens, 0.25)
    for b in range(len(lens)):
        V = f64(oracle.gather_sequence(vc, bt[b], lens[b]))
        for h in range(q.shape[1]):
            g = h // 2
            assert np.all(out[b, h] <= V[:, g].max(0) + 1e-12)
            assert np.all(out[b, h] >= V[:, g].min(0) - 1e-12)


def test_page_permutation_invariance_bitwise():
    rng = np.random.default_rng(10)
    q, kc, vc, bt, lens = _random_decode_case(rng)
    out = oracle.paged_decode(q, kc, vc, bt, lens, 0.25, 7)
    sigma = rng.permutation(kc.shape[0])          # page p moves to sigma[p]
    kc2 = np.empty_like(kc)
    vc2 = np.empty_like(vc)
    kc2[sigma] = kc
    vc2[sigma] = vc
    bt2 = np.where(bt >= 0, sigma[np.maximum(bt, 0)], -1).astype(np.int32)
    out2 = oracle.paged_decode(q, kc2, vc2, bt2, lens, 0.25, 7)
    assert np.array_equal(out, out2)


def test_page_size_invariance_bitwise():
    rng = np.random.default_rng(11)
    L, H_kv, D = 45, 2, 8
    K = rand_bits(rng, (L, H_kv, D))
    V = rand_bits(rng, (L, H_kv, D))
    q = rand_bits(rng, (1, 4, D))
    outs = []
    for P in (4, 16, 64):
        kc, vc, perm = paginate(K, V, P, np.random.default_rng(P))
        outs.append(oracle.paged_decode(q, kc, vc, perm[None], np.array([L]), 0.3, 0))
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[1], outs[2])


def test_window_at_least_length_equals_no_window():
    rng = np.random.default_rng(12)
    q, kc, vc, bt, lens = _random_decode_case(rng)
    a = oracle.paged_decode(q, kc, vc, bt, lens, 0.25, 0)
    b = oracle.paged_decode(q, kc, vc, bt, lens, 0.25, int(lens.max()))
    c = oracle.paged_decode(q, kc, vc, bt, lens, 0.25, int(lens.max()) - 1)
    assert np.array_equal(a, b)
    assert not np.array_equal(a, c)


def test_decode_equals_last_row_of_varlen():
    rng = np.random.default_rng(13)
    q, kc, vc, bt, lens = _random_decode_case(rng)
    dec = oracle.paged_decode(q, kc, vc, bt, lens, 0.25, 6)
    cu_q = np.arange(len(lens) + 1, dtype=np.int32)
    cu_k = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    var = oracle.paged_varlen(q, kc, vc, cu_q, cu_k, bt, 0.25, True, 6)
    assert np.array_equal(dec, var)


def test_gqa_equals_mha_with_repeated_kv():
    """Pins the grouping h // (H_q/H_kv): kv head g serves q heads gG..gG+G-1."""
    rng = np.random.default_rng(14)
    H_q, H_kv, D, L = 8, 2, 16, 21
    K = rand_bits(rng, (L, H_kv, D))
    V = rand_bits(rng, (L, H_kv, D))
    q = rand_bits(rng, (3, H_q, D))
    pos = np.array([4, 12, 20])
    gqa = oracle.attend_rows(f64(q), f64(K), f64(V), pos, 0.25)
    Kr = np.repeat(K, H_q // H_kv, axis=1)
    Vr = np.repeat(V, H_q // H_kv, axis=1)
    mha = oracle.attend_rows(f64(q), f64(Kr), f64(Vr), pos, 0.25)
    np.testing.assert_allclose(gqa, mha, rtol=0, atol=1e-13)
    # an interleaved (h % H_kv) grouping would differ
    Ki = np.tile(K, (1, H_q // H_kv, 1))
    Vi = np.tile(V, (1, H_q // H_kv, 1))
    inter = oracle.attend_rows(f64(q), f64(Ki), f64(Vi), pos, 0.25)
    assert np.abs(inter - gqa).max() > 1e-3


def test_constant_score_shift_is_a_no_op():
    rng = np.random.default_rng(15)
    L, D = 12, 8
    K = rand_bits(rng, (L, 1, D))
    V = rand_bits(rng, (L, 1, D))
    q = rand_bits(rng, (2, 1, D))
    pos = np.array([5, 11])
    base = oracle.attend_rows(f64(q), f64(K), f64(V), pos, 0.5)
    # extra dim: q gets 3, every key gets 2 -> every score shifts by 3
    qx = np.concatenate([f64(q), np.full((2, 1, 1), 3.0)], axis=2)
    Kx = np.concatenate([f64(K), np.full((L, 1, 1), 2.0)], axis=2)
    Vx = np.concatenate([f64(V), np.zeros((L, 1, 1))], axis=2)
    shifted = oracle.attend_rows(qx, Kx, Vx, pos, 0.5)
    np.testing.assert_allclose(shifted[..., :D], base, rtol=0, atol=1e-13)


def test_lse_matches_log_sum_exp():
    rng = np.random.default_rng(16)
    K = rand_bits(rng, (6, 1, 4))
    V = rand_bits(rng, (6, 1, 4))
    q = rand_bits(rng, (1, 1, 4))
    _, lse = oracle.attend_rows(f64(q), f64(K), f64(V), np.array([5]), 0.5,
                                return_lse=True)
    s = (f64(K)[:, 0] @ f64(q)[0, 0]) * 0.5
    assert abs(lse[0, 0] - math.log(sum(math.exp(x) for x in s))) < 1e-13


def test_key_blocks_merged_by_lse_equal_whole_attention():
    # The split-KV decode and the shared-prefix (cascade) decode both rest on
    # this identity of softmax attention: attending over disjoint key blocks
    # and weighting each block's normalised output by exp(lse_i - lse), with
    # lse = log(sum_i exp(lse_i)), gives the attention over all keys.
    rng = np.random.default_rng(18)
    L, H_kv, G, D = 37, 2, 3, 8
    K, V = f64(rand_bits(rng, (L, H_kv, D))), f64(rand_bits(rng, (L, H_kv, D)))
    q = f64(rand_bits(rng, (1, H_kv * G, D)))
    whole = oracle.attend_rows(q, K, V, np.array([L - 1]), 0.35)
    parts = [oracle.attend_rows(q, K[a:b], V[a:b], np.array([L]), 0.35, causal=False,
                                return_lse=True) for a, b in ((0, 16), (16, 17), (17, L))]
    lses = np.stack([lse for _, lse in parts])            # [blocks, 1, H_q]
    total = np.log(np.exp(lses).sum(axis=0))
    merged = sum(np.exp(lse - total)[..., None] * o for o, lse in parts)
    np.testing.assert_allclose(merged, whole, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# append
# ---------------------------------------------------------------------------
def test_append_round_trip_and_untouched_bytes():
    rng = np.random.default_rng(17)
    num_pages, H_kv, P, D = 12, 2, 4, 8
    sentinel = np.uint16(0xABCD)
    kc = np.full((num_pages, H_kv, P, D), sentinel, np.uint16)
    vc = np.full_like(kc, 0x1234)
    L = 10
    table = rng.permutation(num_pages)[:3].astype(np.int32)
    K = rand_bits(rng, (L, H_kv, D))
    V = rand_bits(rng, (L, H_kv, D))
    slots = np.array([table[p // P] * P + p % P for p in range(L)], np.int64)
    slots_with_skip = np.concatenate([slots, [-1]])
    K2 = np.concatenate([K, rand_bits(rng, (1, H_kv, D))])
    V2 = np.concatenate([V, rand_bits(rng, (1, H_kv, D))])
    k2, v2 = oracle.kv_append(kc, vc, K2, V2, slots_with_skip)
    assert np.array_equal(oracle.gather_sequence(k2, table, L), K)
    assert np.array_equal(oracle.gather_sequence(v2, table, L), V)
    touched = np.zeros(kc.shape[:1] + kc.shape[2:3], bool)
    for s in slots:
        touched[s // P, s % P] = True
    mask = np.broadcast_to(touched[:, None, :, None], kc.shape)
    assert np.all(k2[~mask] == sentinel)
    assert np.all(v2[~mask] == 0x1234)
    assert np.array_equal(kc, np.full_like(kc, sentinel))   # inputs untouched


def test_append_rejects_duplicates_and_out_of_pool():
    kc = np.zeros((2, 1, 4, 8), np.uint16)
    rows = np.zeros((2, 1, 8), np.uint16)
    with pytest.raises(ValueError):
        oracle.kv_append(kc, kc, rows, rows, np.array([3, 3]))
    with pytest.raises(ValueError):
        oracle.kv_append(kc, kc, rows, rows, np.array([3, 8]))


def test_workload_slots_address_the_new_token_rows():
    """Decode slots land at position `cached` of each sequence's pages."""
    s = wl.tiny()
    for b in range(s.Bd):
        c = int(s.dec_cached[b])
        assert s.dec_slots[b] == s.dec_block_table[b, c // s.P] * s.P + c % s.P
    assert len(np.unique(s.all_slots)) == len(s.all_slots)
