"""Pins for the rope / QK-norm part of the fp64 oracle (oracle/rope.py).

The pages print no rotary or norm values, so these pin the oracle to
hand-derived numbers, closed forms, a library conversion (torch's float32
-> bfloat16 cast) and invariants of rotations.  Each test names the mistake
it is meant to catch.
"""
import math

import numpy as np
import pytest

import oracle
import workloads as wl

f64 = oracle.bf16_bits_to_f64
to_bf = oracle.f64_to_bf16_bits


# ------------------------------------------------------------ bf16 rounding
def test_every_finite_bf16_value_round_trips():
    # catches: a wrong spacing (off-by-one exponent) or sign handling
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore"):  # the NaN patterns
        x = f64(bits)
    fin = np.isfinite(x)
    got = to_bf(x[fin])
    want = bits[fin]
    # +0 and -0 both map to a zero; everything else must come back bitwise
    nz = x[fin] != 0
    assert np.array_equal(got[nz], want[nz])
    assert np.all(f64(got[~nz]) == 0)


def test_ties_go_to_even():
    # catches: round-half-up or truncation instead of ties-to-even
    cases = {
        1.0 + 2.0 ** -8: 0x3F80,            # tie between 1 and 1+2^-7: even is 1
        1.0 + 3 * 2.0 ** -8: 0x3F82,        # tie between 1+2^-7 (odd) and 1+2^-6
        -(1.0 + 2.0 ** -8): 0xBF80,
        1.0 + 2.0 ** -8 + 2.0 ** -30: 0x3F81,  # just above the tie
        1.0 + 2.0 ** -8 - 2.0 ** -30: 0x3F80,  # just below it
        2.0 ** -133: 0x0001,                # smallest subnormal
        2.0 ** -134: 0x0000,                # tie between 0 and 2^-133
        3 * 2.0 ** -134: 0x0002,            # tie between 2^-133 (odd) and 2^-132
        255.5: 0x4380,                      # spacing 1 in [128, 256): tie between
                                            # 255 (odd mantissa) and 256 -> 256
    }
    for x, b in cases.items():
        assert int(to_bf(np.array([x]))[0]) == b, (x, hex(b))


def test_agrees_with_torch_float32_cast():
    # catches: any rounding mistake on ordinary values (torch rounds float32
    # to bfloat16 to nearest, ties to even; float32 values are exact doubles)
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(11)
    x = (rng.standard_normal(200_000) * np.exp2(rng.integers(-30, 30, 200_000))).astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(to_bf(x.astype(np.float64)), want)


# ------------------------------------------------------------------ rotary
def test_hand_derived_rotations_d4():
    # D=4, theta=1e4: pair 0 = dims (0, 2) turns by pos, pair 1 = dims (1, 3)
    # by pos * 1e4^(-1/2) = pos / 100.  Catches: interleaved pairs (0,1),
    # a wrong frequency exponent, a clockwise rotation.
    p = 3.0
    e = np.eye(4)[:, None, :]                             # 4 rows, H=1
    got = oracle.rope_rotate(e, np.full(4, p), 1e4)[:, 0, :]
    c0, s0, c1, s1 = math.cos(3.0), math.sin(3.0), math.cos(0.03), math.sin(0.03)
    want = np.array([
        [c0, 0, s0, 0],     # e0 -> (cos, sin) in (dim0, dim2)
        [0, c1, 0, s1],     # e1 -> pair 1
        [-s0, 0, c0, 0],    # e2 -> (-sin, cos)
        [0, -s1, 0, c1],
    ])
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-15)


def test_frequency_ladder_d8():
    # theta=1e4, D=8: theta^(-2i/8) = 10^-i, so at pos 1 the angles are
    # 1, 0.1, 0.01, 0.001.  Catches: -i/D instead of -2i/D, or i+1.
    a = oracle.rope_angles(np.array([1.0]), 8, 1e4)[0]
    np.testing.assert_allclose(a, [1.0, 0.1, 0.01, 0.001], rtol=1e-15)


def test_rotation_is_complex_multiplication():
    # catches: a sign slip or a half swapped in the real form
    rng = np.random.default_rng(5)
    x = rng.standard_normal((7, 3, 64))
    pos = rng.integers(0, 40000, 7)
    got = oracle.rope_rotate(x, pos, 1e6)
    z = x[..., :32] + 1j * x[..., 32:]
    ang = pos[:, None].astype(float) * (1e6 ** (-np.arange(32) / 32.0))[None, :]
    w = z * np.exp(1j * ang)[:, None, :]
    np.testing.assert_allclose(got[..., :32], w.real, atol=1e-12)
    np.testing.assert_allclose(got[..., 32:], w.imag, atol=1e-12)


def test_position_zero_is_identity_and_inverse_undoes():
    rng = np.random.default_rng(6)
    x = rng.standard_normal((5, 2, 128))
    assert np.array_equal(oracle.rope_rotate(x, np.zeros(5), 1e6), x)
    pos = rng.integers(1, 9000, 5)
    back = oracle.rope_rotate(oracle.rope_rotate(x, pos, 1e6), -pos, 1e6)
    np.testing.assert_allclose(back, x, atol=1e-12)


def test_pair_norms_preserved():
    # catches: a scale error (e.g. cos applied twice)
    rng = np.random.default_rng(7)
    x = rng.standard_normal((9, 4, 256))
    y = oracle.rope_rotate(x, rng.integers(0, 5000, 9), 1e4)
    n = lambda v: v[..., :128] ** 2 + v[..., 128:] ** 2  # noqa: E731
    np.testing.assert_allclose(n(y), n(x), rtol=1e-12)


def test_scores_depend_on_relative_position_only():
    # the property rotary embeddings exist for: q(m).k(n) == q(m+s).k(n+s)
    rng = np.random.default_rng(8)
    q = rng.standard_normal((1, 1, 128))
    k = rng.standard_normal((1, 1, 128))
    for m, n, s in ((5, 2, 100), (0, 4000, 3), (8191, 17, 911)):
        d0 = np.sum(oracle.rope_rotate(q, [m], 1e6) * oracle.rope_rotate(k, [n], 1e6))
        d1 = np.sum(oracle.rope_rotate(q, [m + s], 1e6) * oracle.rope_rotate(k, [n + s], 1e6))
        assert abs(d0 - d1) < 1e-9


# ----------------------------------------------------------------- RMSNorm
def test_rmsnorm_hand_values():
    # [3, 4]: mean of squares 12.5 -> [3, 4] / sqrt(12.5)
    y = oracle.rms_norm_heads(np.array([[3.0, 4.0]]), np.ones(2), 0.0)
    np.testing.assert_allclose(y, [[0.848528137423857, 1.131370849898476]], rtol=1e-14)
    # eps enters under the root: [1, 1] with eps 1 -> 1/sqrt(2)
    y = oracle.rms_norm_heads(np.array([[1.0, 1.0]]), np.ones(2), 1.0)
    np.testing.assert_allclose(y, [[2 ** -0.5, 2 ** -0.5]], rtol=1e-15)
    # the zero row stays zero with eps > 0
    assert np.array_equal(oracle.rms_norm_heads(np.zeros((1, 8)), np.ones(8), 1e-6),
                          np.zeros((1, 8)))


def test_rmsnorm_invariants():
    # catches: mean over the wrong axis, sqrt dropped, weight misapplied
    rng = np.random.default_rng(9)
    x = rng.standard_normal((6, 4, 128))
    y = oracle.rms_norm_heads(x, np.ones(128), 0.0)
    np.testing.assert_allclose(np.mean(y * y, axis=-1), 1.0, rtol=1e-13)
    np.testing.assert_allclose(oracle.rms_norm_heads(3.7 * x, np.ones(128), 0.0), y, rtol=1e-13)
    w = rng.standard_normal(128)
    np.testing.assert_allclose(oracle.rms_norm_heads(x, w, 0.0), y * w, rtol=1e-13)
    assert oracle.rms_norm_heads(x, None, 1e-6) is x


# ------------------------------------------------------------------- fused
def test_fused_rows_without_norm_at_position_zero_are_unchanged():
    rng = np.random.default_rng(10)
    x = wl.randn_bf16(rng, (4, 2, 64))
    assert np.array_equal(oracle.norm_rope_rows(x, np.zeros(4), 1e6, None, 1e-6), x)


def test_append_rope_writes_only_live_slots():
    # catches: V transformed, K untransformed, a skipped token written, or
    # a byte outside the new rows touched
    rng = np.random.default_rng(12)
    num_pages, H, P, D = 6, 2, 16, 64
    sentinel = np.uint16(0x7FA1)
    kc = np.full((num_pages, H, P, D), sentinel, np.uint16)
    vc = np.full((num_pages, H, P, D), sentinel, np.uint16)
    T = 5
    k_new = wl.randn_bf16(rng, (T, H, D))
    v_new = wl.randn_bf16(rng, (T, H, D))
    slots = np.array([3, 40, -1, 95, 17], np.int64)
    pos = np.array([0, 7, 9, 4096, 12], np.int64)     # token 3: position out of range
    w = wl.randn_bf16(rng, (D,))
    k2, v2 = oracle.kv_append_rope(kc, vc, k_new, v_new, slots, pos, 1e6, w, 1e-6, 4096)
    rot = oracle.norm_rope_rows(k_new, pos, 1e6, w, 1e-6)
    written = {0: 3, 1: 40, 4: 17}
    touched = np.zeros((num_pages, P), bool)
    for t, s in written.items():
        pg, r = s // P, s % P
        touched[pg, r] = True
        assert np.array_equal(k2[pg, :, r], rot[t])
        assert np.array_equal(v2[pg, :, r], v_new[t])
    rows = lambda c: c.transpose(0, 2, 1, 3)  # noqa: E731  [page, row, head, dim]
    assert np.all(rows(k2)[~touched] == sentinel) and np.all(rows(v2)[~touched] == sentinel)
    # the slot of the out-of-range token stays untouched
    assert np.all(k2[95 // P, :, 95 % P] == sentinel)


def test_q_rows_of_invalid_positions_untouched():
    rng = np.random.default_rng(13)
    q = wl.randn_bf16(rng, (4, 8, 128))
    pos = np.array([-1, 5, 100, 100000], np.int64)
    out = oracle.q_norm_rope(q, pos, 1e6, None, 1e-6, 4096)
    assert np.array_equal(out[[0, 3]], q[[0, 3]])
    assert np.array_equal(out[[1, 2]], oracle.norm_rope_rows(q[[1, 2]], pos[[1, 2]], 1e6,
                                                             None, 1e-6))


def test_norm_precedes_rotation():
    # The order is only visible through a non-uniform weight (a rotation
    # keeps the mean square).  x = e0, w = [2, 1, 1, 1], eps 0, D 4:
    # norm first gives [4, 0, 0, 0] (rms of e0 is 1/2), then pair (0, 2)
    # turns by pos -> [4 cos p, 0, 4 sin p, 0]; rotating first would give
    # [4 cos p, 0, 2 sin p, 0].
    x = wl.f32_to_bf16_bits(np.array([[[1.0, 0.0, 0.0, 0.0]]], np.float32))
    w = wl.f32_to_bf16_bits(np.array([2.0, 1.0, 1.0, 1.0], np.float32))
    got = f64(oracle.norm_rope_rows(x, np.array([3]), 1e4, w, 0.0))[0, 0]
    want = np.array([4 * math.cos(3.0), 0.0, 4 * math.sin(3.0), 0.0])
    np.testing.assert_allclose(got, want, rtol=2.0 ** -8, atol=0)
