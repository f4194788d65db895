"""GPU parity of paged_attn_mixed (one persistent launch for a step's decode
rows and causal prefill chunks) against the fp64 oracle: the full mixed
continuous-batching workload (8 prefill chunks on cached prefixes + 120
decode rows, H 32/8/128, page 16) after this step's append, with the split
between decode-first and prefill-first CTAs chosen by the library and set
explicitly at both extremes; a sliding window; steps with only one half;
and two calls in a row on one workspace (the queue and counters reset)."""
import numpy as np
import pytest

import oracle
import workloads as wl
from _util import assert_close_attn, bf16_dev_to_bits, bf16_dev_to_f64, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    import torch  # noqa: F401
    from paged_kv_attention_11_gb300 import build
    build.build()
    import paged_kv_attention_11_gb300 as m
    m.lib()
    return m


@pytest.fixture(scope="module")
def mixed_case(pkv):
    """The mixed workload after its append: device pools, inputs, oracle outputs."""
    import torch
    step = wl.mixed_step()
    vals = wl.fill_values(step, 2024)
    kc, vc = to_dev_bf16(vals.k_cache), to_dev_bf16(vals.v_cache)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.paged_kv_append(to_dev_bf16(vals.k_new), to_dev_bf16(vals.v_new), kc, vc,
                        to_dev(step.all_slots), err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    hk, hv = oracle.kv_append(vals.k_cache, vals.v_cache, vals.k_new, vals.v_new, step.all_slots)
    return step, vals, kc, vc, hk, hv


def _run(pkv, step, vals, kc, vc, window=0, decode_ctas=0, dec=True, pre=True, ws=None):
    import torch
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    qd = to_dev_bf16(vals.q_dec[0]) if dec else torch.empty((0, step.H_q, step.D),
                                                            dtype=torch.bfloat16, device="cuda")
    qp = to_dev_bf16(vals.q_pre[0]) if pre else torch.empty((0, step.H_q, step.D),
                                                            dtype=torch.bfloat16, device="cuda")
    od = torch.full_like(qd, float("nan"))
    op = torch.full_like(qp, float("nan"))
    cu_q = step.cu_seq_lens_q if pre else np.zeros(1, np.int32)
    cu_k = step.cu_seq_lens_k if pre else np.zeros(1, np.int32)
    pbt = step.pre_block_table if pre else np.zeros((0, 1), np.int32)
    dbt = step.dec_block_table if dec else np.zeros((0, 1), np.int32)
    dl = step.dec_seq_lens if dec else np.zeros(0, np.int32)
    pkv.paged_attn_mixed(od, qd, to_dev(dbt), to_dev(dl), step.max_seq_len_dec() if dec else 0,
                         op, qp, to_dev(cu_q), to_dev(cu_k), to_dev(pbt),
                         step.max_seqlen_q() if pre else 0, step.max_seqlen_k() if pre else 0,
                         kc, vc, step.scale, window, decode_ctas, workspace=ws, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return od, op


def _want(step, vals, hk, hv, window=0):
    wd = oracle.paged_decode(vals.q_dec[0], hk, hv, step.dec_block_table, step.dec_seq_lens,
                             step.scale, window)
    wp = oracle.paged_varlen(vals.q_pre[0], hk, hv, step.cu_seq_lens_q, step.cu_seq_lens_k,
                             step.pre_block_table, step.scale, True, window)
    return wd, wp


@pytest.fixture(scope="module")
def want_full(mixed_case):
    step, vals, _, _, hk, hv = mixed_case
    return _want(step, vals, hk, hv)


@pytest.mark.parametrize("decode_ctas", [0, 1, 40, 100, 151])
def test_mixed_step_full_workload(pkv, mixed_case, want_full, decode_ctas):
    step, vals, kc, vc, _, _ = mixed_case
    od, op = _run(pkv, step, vals, kc, vc, decode_ctas=decode_ctas)
    wd, wp = want_full
    assert_close_attn(bf16_dev_to_f64(od), wd, f"mixed decode (split {decode_ctas})")
    assert_close_attn(bf16_dev_to_f64(op), wp, f"mixed prefill (split {decode_ctas})")


def test_mixed_step_sliding_window(pkv, mixed_case):
    step, vals, kc, vc, hk, hv = mixed_case
    od, op = _run(pkv, step, vals, kc, vc, window=300)
    wd, wp = _want(step, vals, hk, hv, window=300)
    assert_close_attn(bf16_dev_to_f64(od), wd, "mixed decode, window 300")
    assert_close_attn(bf16_dev_to_f64(op), wp, "mixed prefill, window 300")


def test_mixed_step_one_half_only(pkv, mixed_case, want_full):
    step, vals, kc, vc, _, _ = mixed_case
    wd, wp = want_full
    od, _ = _run(pkv, step, vals, kc, vc, pre=False)
    assert_close_attn(bf16_dev_to_f64(od), wd, "mixed, decode only")
    _, op = _run(pkv, step, vals, kc, vc, dec=False)
    assert_close_attn(bf16_dev_to_f64(op), wp, "mixed, prefill only")


def test_mixed_step_twice_on_one_workspace(pkv, mixed_case):
    """The workspace is left ready for the next call: a second call gives
    the same bits."""
    import torch
    step, vals, kc, vc, _, _ = mixed_case
    need = pkv.decode_workspace_size(step.Bd, step.H_q, step.H_kv, step.D)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    od1, op1 = _run(pkv, step, vals, kc, vc, ws=ws)
    od2, op2 = _run(pkv, step, vals, kc, vc, ws=ws)
    assert np.array_equal(bf16_dev_to_bits(od1), bf16_dev_to_bits(od2))
    assert np.array_equal(bf16_dev_to_bits(op1), bf16_dev_to_bits(op2))


@pytest.mark.parametrize("H_q,H_kv", [(8, 2), (8, 1), (12, 3), (4, 4)])
def test_mixed_step_small(pkv, H_q, H_kv):
    """A small mixed step (2 prefill chunks, 8 decode rows) with the split at
    3 decode-first CTAs: decode items of two kv heads (8/2, 4/4) and of one
    (a group of 8; an odd kv-head count)."""
    import torch
    step = wl.mixed_step(n_chunks=2, n_dec=8, H_q=H_q, H_kv=H_kv, num_pages=2048)
    vals = wl.fill_values(step, 11)
    kc, vc = to_dev_bf16(vals.k_cache), to_dev_bf16(vals.v_cache)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.paged_kv_append(to_dev_bf16(vals.k_new), to_dev_bf16(vals.v_new), kc, vc,
                        to_dev(step.all_slots), err_flag=err)
    hk, hv = oracle.kv_append(vals.k_cache, vals.v_cache, vals.k_new, vals.v_new, step.all_slots)
    od, op = _run(pkv, step, vals, kc, vc, decode_ctas=3)
    wd, wp = _want(step, vals, hk, hv)
    assert_close_attn(bf16_dev_to_f64(od), wd, "small mixed decode")
    assert_close_attn(bf16_dev_to_f64(op), wp, "small mixed prefill")


@pytest.mark.parametrize("H_q,H_kv", [(12, 4), (6, 2), (24, 8)])
def test_mixed_decode_only_group_of_three(pkv, H_q, H_kv):
    """Decode rows alone through the one-launch path with a GQA group of 3
    (query rows of two kv heads per item: 6); the longest rows (up to 4096
    keys against a share of ~20-40 tiles per CTA) are cut and merged."""
    import torch
    step = wl.mixed_step(n_chunks=2, n_dec=24, H_q=H_q, H_kv=H_kv, num_pages=8192)
    vals = wl.fill_values(step, 13)
    kc, vc = to_dev_bf16(vals.k_cache), to_dev_bf16(vals.v_cache)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.paged_kv_append(to_dev_bf16(vals.k_new), to_dev_bf16(vals.v_new), kc, vc,
                        to_dev(step.all_slots), err_flag=err)
    hk, hv = oracle.kv_append(vals.k_cache, vals.v_cache, vals.k_new, vals.v_new, step.all_slots)
    od, _ = _run(pkv, step, vals, kc, vc, pre=False)
    wd = oracle.paged_decode(vals.q_dec[0], hk, hv, step.dec_block_table, step.dec_seq_lens,
                             step.scale)
    assert_close_attn(bf16_dev_to_f64(od), wd, f"mixed decode-only {H_q}/{H_kv}")


def _run_fused(pkv, step, vals, kc, vc, slots, decode_ctas=0, dec=True, pre=True):
    """paged_attn_mixed_append from the pools before the step's append."""
    import torch
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    qd = to_dev_bf16(vals.q_dec[0]) if dec else torch.empty((0, step.H_q, step.D),
                                                            dtype=torch.bfloat16, device="cuda")
    qp = to_dev_bf16(vals.q_pre[0]) if pre else torch.empty((0, step.H_q, step.D),
                                                            dtype=torch.bfloat16, device="cuda")
    od = torch.full_like(qd, float("nan"))
    op = torch.full_like(qp, float("nan"))
    cu_q = step.cu_seq_lens_q if pre else np.zeros(1, np.int32)
    cu_k = step.cu_seq_lens_k if pre else np.zeros(1, np.int32)
    pbt = step.pre_block_table if pre else np.zeros((0, 1), np.int32)
    dbt = step.dec_block_table if dec else np.zeros((0, 1), np.int32)
    dl = step.dec_seq_lens if dec else np.zeros(0, np.int32)
    pkv.paged_attn_mixed_append(od, qd, to_dev(dbt), to_dev(dl),
                                step.max_seq_len_dec() if dec else 0, op, qp, to_dev(cu_q),
                                to_dev(cu_k), to_dev(pbt), step.max_seqlen_q() if pre else 0,
                                step.max_seqlen_k() if pre else 0, to_dev_bf16(vals.k_new),
                                to_dev_bf16(vals.v_new), to_dev(slots), kc, vc, step.scale,
                                0, decode_ctas, err_flag=err)
    torch.cuda.synchronize()
    return od, op, int(err.item())


@pytest.mark.parametrize("decode_ctas", [0, 1, 100])
def test_mixed_append_full_workload(pkv, decode_ctas):
    """The step's append fused into the one-launch mixed step: pools bit-exact
    with the oracle's append, outputs against the oracle, and bitwise equal
    to paged_kv_append followed by paged_attn_mixed."""
    step = wl.mixed_step()
    vals = wl.fill_values(step, 2025)
    kc, vc = to_dev_bf16(vals.k_cache), to_dev_bf16(vals.v_cache)
    od, op, err = _run_fused(pkv, step, vals, kc, vc, step.all_slots, decode_ctas)
    assert err == 0
    hk, hv = oracle.kv_append(vals.k_cache, vals.v_cache, vals.k_new, vals.v_new, step.all_slots)
    assert np.array_equal(bf16_dev_to_bits(kc), hk), "K pool"
    assert np.array_equal(bf16_dev_to_bits(vc), hv), "V pool"
    wd, wp = _want(step, vals, hk, hv)
    assert_close_attn(bf16_dev_to_f64(od), wd, f"fused decode (split {decode_ctas})")
    assert_close_attn(bf16_dev_to_f64(op), wp, f"fused prefill (split {decode_ctas})")
    # the two-call path on the same inputs
    import torch
    kc2, vc2 = to_dev_bf16(vals.k_cache), to_dev_bf16(vals.v_cache)
    pkv.paged_kv_append(to_dev_bf16(vals.k_new), to_dev_bf16(vals.v_new), kc2, vc2,
                        to_dev(step.all_slots))
    od2, op2 = _run(pkv, step, vals, kc2, vc2, decode_ctas=decode_ctas)
    torch.cuda.synchronize()
    assert np.array_equal(bf16_dev_to_bits(od), bf16_dev_to_bits(od2)), "decode vs two calls"
    assert np.array_equal(bf16_dev_to_bits(op), bf16_dev_to_bits(op2)), "prefill vs two calls"


@pytest.mark.parametrize("dec,pre", [(True, False), (False, True)])
def test_mixed_append_one_half(pkv, dec, pre):
    """Appending with only decode rows or only prefill chunks in the call
    (the other half's rows are appended too: every slot is written)."""
    step = wl.mixed_step(n_chunks=3, n_dec=16, H_q=8, H_kv=2, num_pages=4096)
    vals = wl.fill_values(step, 31)
    kc, vc = to_dev_bf16(vals.k_cache), to_dev_bf16(vals.v_cache)
    od, op, err = _run_fused(pkv, step, vals, kc, vc, step.all_slots, 0, dec, pre)
    assert err == 0
    hk, hv = oracle.kv_append(vals.k_cache, vals.v_cache, vals.k_new, vals.v_new, step.all_slots)
    assert np.array_equal(bf16_dev_to_bits(kc), hk) and np.array_equal(bf16_dev_to_bits(vc), hv)
    wd, wp = _want(step, vals, hk, hv)
    if dec:
        assert_close_attn(bf16_dev_to_f64(od), wd, "fused decode only")
    if pre:
        assert_close_attn(bf16_dev_to_f64(op), wp, "fused prefill only")


def test_mixed_append_skips_padding_and_flags_bad_slots(pkv):
    """Slot -1 rows are skipped; a slot past the pool is flagged and skipped;
    the rest are written (the attention then reads the pools as written)."""
    step = wl.mixed_step(n_chunks=2, n_dec=8, H_q=8, H_kv=2, num_pages=2048)
    vals = wl.fill_values(step, 37)
    slots = step.all_slots.copy()
    pad = [3, 10]
    slots[pad] = -1
    bad = 5
    slots[bad] = step.num_pages * step.P + 7
    kc, vc = to_dev_bf16(vals.k_cache), to_dev_bf16(vals.v_cache)
    _, _, err = _run_fused(pkv, step, vals, kc, vc, slots, 0)
    assert err & 1  # PKV_DEVERR_SLOT
    ok = slots.copy()
    ok[bad] = -1
    hk, hv = oracle.kv_append(vals.k_cache, vals.v_cache, vals.k_new, vals.v_new, ok)
    assert np.array_equal(bf16_dev_to_bits(kc), hk) and np.array_equal(bf16_dev_to_bits(vc), hv)
