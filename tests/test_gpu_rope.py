"""GPU parity: pkv_rope_table and paged_kv_append_rope against the fp64 oracle
(oracle/rope.py), through the C ABI.

Tolerance, from the arithmetic: the kernel works in float32 from a float32
table and rounds once to bf16.  Its float32 result is within a few float32
ulps of the exact value: about 1e-6 of the magnitudes of the two inputs of
each rotary pair, far below a bf16 half-ulp (2^-9 relative).  So each output
is at most one bf16 ulp from the exact fp64 result, plus that 1e-6 floor
where the pair cancels.  It may differ from the oracle's correctly rounded
value only where the exact value lies within that error of a rounding
midpoint: at most 1 element in 1000.  V rows, and every byte the call does
not write, are bit-exact."""
import numpy as np
import pytest

import oracle
import workloads as wl
from _util import assert_close_attn, bf16_dev_to_bits, bf16_dev_to_f64, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu

f64 = oracle.bf16_bits_to_f64
MISMATCH_MAX = 1e-3


@pytest.fixture(scope="module")
def pkv():
    import torch  # noqa: F401
    from paged_kv_attention_11_gb300 import build
    build.build()
    import paged_kv_attention_11_gb300 as m
    m.lib()
    return m


def _table(pkv, max_pos, D, theta):
    import torch
    cs = torch.empty((max_pos, D), dtype=torch.float32, device="cuda")
    pkv.rope_table(cs, theta)
    return cs


def bf16_spacing(v: np.ndarray) -> np.ndarray:
    """Distance between adjacent bf16 values around |v| (2^(e-8) for |v| in
    [2^(e-1), 2^e)), floored at the subnormal spacing."""
    _, e = np.frexp(np.abs(v))
    return np.ldexp(1.0, np.maximum(e - 8, -133))


def check_rows(got_bits, x_bits, pos, theta, w_bits, eps, what):
    """got_bits [n, H, D] from the GPU vs the exact transform of x_bits."""
    x = f64(x_bits)
    w = None if w_bits is None else f64(w_bits)
    normed = oracle.rms_norm_heads(x, w, eps)
    exact = oracle.rope_rotate(normed, pos, theta)
    D = x.shape[-1]
    pair = np.abs(normed[..., : D // 2]) + np.abs(normed[..., D // 2:])
    floor = 1e-6 * np.concatenate([pair, pair], axis=-1)
    got = f64(got_bits)
    assert np.all(np.isfinite(got)), what
    gap = np.abs(got - exact)
    lim = bf16_spacing(np.maximum(np.abs(exact), np.abs(got))) + floor
    bad = gap > lim
    assert not bad.any(), (f"{what}: {int(bad.sum())} outputs beyond 1 bf16 ulp; worst gap "
                           f"{gap[bad].max():.3e} at {np.argwhere(bad)[0]}")
    want = oracle.f64_to_bf16_bits(exact)
    frac = float(np.mean(got_bits != want)) if got_bits.size else 0.0
    assert frac <= MISMATCH_MAX, f"{what}: {frac:.2e} of outputs differ from the oracle"


# ----------------------------------------------------------------- table
@pytest.mark.parametrize("D,theta", [(64, 1e4), (128, 1e6), (256, 1e4), (256, 1e6)])
def test_rope_table_is_the_rounded_exact_table(pkv, D, theta):
    max_pos = 9000
    got = _table(pkv, max_pos, D, theta).cpu().numpy().astype(np.float64)
    a = oracle.rope_angles(np.arange(max_pos), D, theta)
    exact = np.concatenate([np.cos(a), np.sin(a)], axis=1)
    half_ulp = 0.5 * np.spacing(np.abs(exact).astype(np.float32)).astype(np.float64)
    gap = np.abs(got - exact)
    assert np.all(gap <= half_ulp * (1 + 1e-6) + 1e-11), float((gap - half_ulp).max())


# ------------------------------------------------------ shapes and edges
CASES = [
    # D, H_q, H_kv, P, T, q_norm, k_norm, with_q, theta
    (64, 4, 2, 16, 37, True, True, True, 1e4),
    (128, 32, 8, 16, 1000, True, True, True, 1e6),
    (256, 8, 1, 64, 300, False, False, True, 1e4),
    (128, 32, 8, 16, 1, False, True, False, 1e6),
    (128, 16, 16, 16, 513, True, False, True, 1e6),
    (256, 8, 1, 64, 77, True, True, True, 1e6),
]


@pytest.mark.parametrize("D,H_q,H_kv,P,T,qn,kn,with_q,theta", CASES)
def test_append_rope_shapes(pkv, D, H_q, H_kv, P, T, qn, kn, with_q, theta):
    import torch
    rng = np.random.default_rng(D * 1000 + T)
    num_pages = -(-T // P) + 5
    max_pos = 8192
    eps = float(np.float32(1e-6))
    kc = wl.randn_bf16(rng, (num_pages, H_kv, P, D))  # unrelated contents: must survive
    vc = wl.randn_bf16(rng, (num_pages, H_kv, P, D))
    k_new = wl.randn_bf16(rng, (T, H_kv, D), 1.7)
    v_new = wl.randn_bf16(rng, (T, H_kv, D))
    q = wl.randn_bf16(rng, (T, H_q, D), 0.6)
    slots = rng.permutation(num_pages * P)[:T].astype(np.int64)
    pos = rng.integers(0, max_pos, T).astype(np.int32)
    pos[0] = 0
    if T > 3:
        slots[1] = -1                  # padding: no append, q still transformed
        pos[2] = max_pos               # out of the table: token skipped whole
        pos[-1] = max_pos - 1
    qw = wl.randn_bf16(rng, (D,)) if qn else None
    kw = wl.randn_bf16(rng, (D,)) if kn else None

    dkc, dvc, dq = to_dev_bf16(kc), to_dev_bf16(vc), to_dev_bf16(q)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    cs = _table(pkv, max_pos, D, theta)
    pkv.paged_kv_append_rope(dq if with_q else None, to_dev_bf16(k_new), to_dev_bf16(v_new),
                             dkc, dvc, to_dev(slots), to_dev(pos), cs,
                             None if qw is None else to_dev_bf16(qw),
                             None if kw is None else to_dev_bf16(kw), eps, err_flag=err)
    torch.cuda.synchronize()
    e = int(err.item())
    assert e == (pkv.DEVERR_POS if T > 3 else 0), e

    live = (pos >= 0) & (pos < max_pos)
    hk, hv = oracle.kv_append_rope(kc, vc, k_new, v_new, slots, pos, theta, kw, eps, max_pos)
    gk, gv = bf16_dev_to_bits(dkc), bf16_dev_to_bits(dvc)
    assert np.array_equal(gv, hv), "V pool differs"
    # K: every byte outside the appended rows exact, the rows within tolerance
    w = np.nonzero(live & (slots >= 0))[0]
    pg, rw = slots[w] // P, slots[w] % P
    mask = np.ones((num_pages, P), bool)
    mask[pg, rw] = False
    rows = lambda c: c.transpose(0, 2, 1, 3)  # noqa: E731
    assert np.array_equal(rows(gk)[mask], rows(hk)[mask]), "K pool bytes outside the new rows"
    check_rows(gk[pg, :, rw, :], k_new[w], pos[w], theta, kw, eps, "k rows")
    if with_q:
        gq = bf16_dev_to_bits(dq)
        assert np.array_equal(gq[~live], q[~live]), "q rows of skipped tokens changed"
        check_rows(gq[live], q[live], pos[live], theta, qw, eps, "q rows")


def test_append_rope_bad_slot_flags_and_skips(pkv):
    import torch
    rng = np.random.default_rng(4)
    D, H_q, H_kv, P, num_pages, T = 128, 8, 2, 16, 4, 6
    kc = wl.randn_bf16(rng, (num_pages, H_kv, P, D))
    vc = wl.randn_bf16(rng, (num_pages, H_kv, P, D))
    k_new = wl.randn_bf16(rng, (T, H_kv, D))
    v_new = wl.randn_bf16(rng, (T, H_kv, D))
    q = wl.randn_bf16(rng, (T, H_q, D))
    slots = np.array([0, 5, num_pages * P, 17, 40, 63], np.int64)   # token 2 outside the pool
    pos = np.arange(T, dtype=np.int32) * 100
    dkc, dvc, dq = to_dev_bf16(kc), to_dev_bf16(vc), to_dev_bf16(q)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    cs = _table(pkv, 1024, D, 1e6)
    pkv.paged_kv_append_rope(dq, to_dev_bf16(k_new), to_dev_bf16(v_new), dkc, dvc,
                             to_dev(slots), to_dev(pos), cs, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == pkv.DEVERR_SLOT
    keep = np.array([True, True, False, True, True, True])
    hk, hv = oracle.kv_append_rope(kc, vc, k_new[keep], v_new[keep], slots[keep], pos[keep],
                                   1e6, None, 1e-6, 1024)
    assert np.array_equal(bf16_dev_to_bits(dvc), hv)
    gk = bf16_dev_to_bits(dkc)
    s = slots[keep]
    check_rows(gk[s // P, :, s % P, :], k_new[keep], pos[keep], 1e6, None, 1e-6, "k rows")
    # q of the token with the bad slot is still transformed
    check_rows(bf16_dev_to_bits(dq), q, pos, 1e6, None, 1e-6, "q rows")


# ------------------------------------ full size: the mixed step, end to end
def test_mixed_step_with_fused_rope_end_to_end(pkv):
    """The mixed continuous-batching step (8 prefill chunks + 120 decode rows,
    H 32/8/128, page 16) with the input transform fused into the append:
    all 5645 new tokens' q and k normalised and rotated (theta 1e6), then
    varlen prefill and decode read the rotated q and the pool."""
    import torch
    step = wl.mixed_step()
    vals = wl.fill_values(step, 3407)
    rng = np.random.default_rng(99)
    theta, eps, max_pos = 1e6, float(np.float32(1e-6)), 8192
    qw = wl.f32_to_bf16_bits((1 + 0.1 * rng.standard_normal(step.D)).astype(np.float32))
    kw = wl.f32_to_bf16_bits((1 + 0.1 * rng.standard_normal(step.D)).astype(np.float32))
    q_all = np.concatenate([vals.q_pre[0], vals.q_dec[0]])
    pos = step.all_positions
    slots = step.all_slots

    kc, vc = to_dev_bf16(vals.k_cache), to_dev_bf16(vals.v_cache)
    dq = to_dev_bf16(q_all)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    cs = _table(pkv, max_pos, step.D, theta)
    pkv.paged_kv_append_rope(dq, to_dev_bf16(vals.k_new), to_dev_bf16(vals.v_new), kc, vc,
                             to_dev(slots), to_dev(pos), cs, to_dev_bf16(qw), to_dev_bf16(kw),
                             eps, err_flag=err)
    out_pre = torch.empty((step.total_q, step.H_q, step.D), dtype=torch.bfloat16, device="cuda")
    out_dec = torch.empty((step.Bd, step.H_q, step.D), dtype=torch.bfloat16, device="cuda")
    pkv.paged_attn_varlen(out_pre, dq[:step.total_q], kc, vc, to_dev(step.cu_seq_lens_q),
                          to_dev(step.cu_seq_lens_k), to_dev(step.pre_block_table),
                          step.max_seqlen_q(), step.max_seqlen_k(), step.scale, True,
                          step.window, err_flag=err)
    pkv.paged_attn_decode(out_dec, dq[step.total_q:], kc, vc, to_dev(step.dec_block_table),
                          to_dev(step.dec_seq_lens), step.max_seq_len_dec(), step.scale,
                          step.window, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0

    # the transform itself
    gq = bf16_dev_to_bits(dq)
    check_rows(gq, q_all, pos, theta, qw, eps, "q rows")
    hk, hv = oracle.kv_append_rope(vals.k_cache, vals.v_cache, vals.k_new, vals.v_new, slots,
                                   pos, theta, kw, eps, max_pos)
    P = step.P
    gk = kc.view(torch.int16)[torch.as_tensor(slots // P, device="cuda"), :,
                              torch.as_tensor(slots % P, device="cuda"), :]
    check_rows(gk.cpu().numpy().view(np.uint16), vals.k_new, pos, theta, kw, eps, "k rows")
    assert np.array_equal(bf16_dev_to_bits(vc), hv), "V pool differs"
    # attention end to end from the same host inputs: the oracle's own
    # transformed q (q_norm_rope) and pool (kv_append_rope) drive its
    # varlen and decode, and the GPU's outputs are compared with those
    hq = oracle.q_norm_rope(q_all, pos, theta, qw, eps, max_pos)
    want_pre = oracle.paged_varlen(hq[:step.total_q], hk, hv, step.cu_seq_lens_q,
                                   step.cu_seq_lens_k, step.pre_block_table, step.scale,
                                   True, step.window)
    assert_close_attn(bf16_dev_to_f64(out_pre), want_pre, "varlen after fused rope")
    want_dec = oracle.paged_decode(hq[step.total_q:], hk, hv, step.dec_block_table,
                                   step.dec_seq_lens, step.scale, step.window)
    assert_close_attn(bf16_dev_to_f64(out_dec), want_dec, "decode after fused rope")
