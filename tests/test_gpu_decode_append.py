"""GPU parity of paged_attn_decode_append (the decode step with its append
in the same launch) against the fp64 oracle's append-then-decode, through
the C ABI: pools bit-exact, outputs within the attention tolerance, and
bitwise equal to the two-call path (paged_kv_append + paged_attn_decode)."""
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


def _case(rng, H_q, H_kv, D, P, lens, extra=4):
    """Random pools and block tables; lens include the new token."""
    need = [max(1, -(-L // P)) for L in lens]
    num_pages = sum(need) + extra
    perm = rng.permutation(num_pages).astype(np.int32)
    B = len(lens)
    bt = np.full((B, max(need)), -1, np.int32)
    o = 0
    for b, n in enumerate(need):
        bt[b, :n] = perm[o:o + n]
        o += n
    kc = wl.randn_bf16(rng, (num_pages, H_kv, P, D))
    vc = wl.randn_bf16(rng, (num_pages, H_kv, P, D))
    q = wl.randn_bf16(rng, (B, H_q, D))
    k_new = wl.randn_bf16(rng, (B, H_kv, D))
    v_new = wl.randn_bf16(rng, (B, H_kv, D))
    return q, kc, vc, bt, np.asarray(lens, np.int32), k_new, v_new


def _slots(bt, lens, P):
    """Slot of each sequence's newest token (-1: no token)."""
    return np.array([int(bt[b, (L - 1) // P]) * P + (L - 1) % P if L > 0 else -1
                     for b, L in enumerate(lens)], np.int64)


def _check(pkv, q, kc, vc, bt, lens, k_new, v_new, scale, window, label):
    import torch
    P = kc.shape[2]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    qd = to_dev_bf16(q)
    kd, vd = to_dev_bf16(kc), to_dev_bf16(vc)
    out = torch.full_like(qd, float("nan"))
    pkv.paged_attn_decode_append(out, qd, to_dev_bf16(k_new), to_dev_bf16(v_new), kd, vd,
                                 to_dev(bt), to_dev(lens), int(lens.max()), scale, window,
                                 err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, label
    slots = _slots(bt, lens, P)
    hk, hv = oracle.kv_append(kc, vc, k_new, v_new, slots)
    assert np.array_equal(bf16_dev_to_bits(kd), hk), f"{label}: K pool"
    assert np.array_equal(bf16_dev_to_bits(vd), hv), f"{label}: V pool"
    want = oracle.paged_decode(q, hk, hv, bt, lens, scale, window)
    assert_close_attn(bf16_dev_to_f64(out), want, label)
    # the two-call path on the same inputs gives the same bits
    kd2, vd2 = to_dev_bf16(kc), to_dev_bf16(vc)
    pkv.paged_kv_append(to_dev_bf16(k_new), to_dev_bf16(v_new), kd2, vd2, to_dev(slots),
                        err_flag=err)
    out2 = torch.full_like(qd, float("nan"))
    pkv.paged_attn_decode(out2, qd, kd2, vd2, to_dev(bt), to_dev(lens), int(lens.max()), scale,
                          window, err_flag=err)
    torch.cuda.synchronize()
    assert np.array_equal(bf16_dev_to_bits(out), bf16_dev_to_bits(out2)), f"{label}: two-call"


@pytest.mark.parametrize("D", [64, 128, 256, 512])
@pytest.mark.parametrize("H", [(8, 8), (32, 8), (8, 1)])
def test_decode_append_shapes(pkv, D, H):
    rng = np.random.default_rng(D * 7 + H[0] + H[1])
    lens = [1, 15, 16, 17, 100, 333, 1000, 0, 64, 65, 2049]
    case = _case(rng, H[0], H[1], D, 16, lens)
    _check(pkv, *case, 1 / np.sqrt(D), 0, f"D={D} H={H}")


@pytest.mark.parametrize("window,P", [(1, 16), (100, 16), (512, 64)])
def test_decode_append_window_pages(pkv, window, P):
    rng = np.random.default_rng(window + P)
    lens = [1, 5, 16, 31, 64, 200, 777, 3000]
    case = _case(rng, 8, 2, 128, P, lens)
    _check(pkv, *case, 0.09, window, f"window={window} P={P}")


def test_decode_append_long_sequence_cut_into_chunks(pkv):
    """One 16000-token sequence: cut into chunks; only the last chunk's CTA
    writes the new row, before it reads that tile."""
    rng = np.random.default_rng(17)
    case = _case(rng, 32, 8, 128, 16, [16000])
    _check(pkv, *case, 1 / np.sqrt(128), 0, "long")


def test_decode_append_qwen3_workload(pkv):
    """The headline step at full size: 64 sequences, cached U[256,2048]."""
    step = wl.qwen3_decode()
    vals = wl.fill_values(step, 3407)
    lens = step.dec_seq_lens
    k_new = vals.k_new.reshape(len(lens), step.H_kv, step.D)
    v_new = vals.v_new.reshape(len(lens), step.H_kv, step.D)
    assert np.array_equal(_slots(step.dec_block_table, lens, step.P), step.dec_slots)
    _check(pkv, vals.q_dec[0], vals.k_cache, vals.v_cache, step.dec_block_table, lens, k_new,
           v_new, step.scale, 0, "qwen3_decode")


def test_decode_append_bad_page_flags_and_skips(pkv):
    """A block-table entry past the pool at the new token's page: the row is
    not written, the device flag reports it, and nothing faults."""
    import torch
    rng = np.random.default_rng(23)
    q, kc, vc, bt, lens, k_new, v_new = _case(rng, 8, 2, 128, 16, [40, 70])
    bt[1, (int(lens[1]) - 1) // 16] = kc.shape[0] + 5
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kd, vd = to_dev_bf16(kc), to_dev_bf16(vc)
    out = torch.empty_like(to_dev_bf16(q))
    pkv.paged_attn_decode_append(out, to_dev_bf16(q), to_dev_bf16(k_new), to_dev_bf16(v_new),
                                 kd, vd, to_dev(bt), to_dev(lens), int(lens.max()), 0.1, 0,
                                 err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pkv.DEVERR_PAGE
    # sequence 0 is untouched by the bad entry: its row was appended
    slot0 = int(bt[0, (int(lens[0]) - 1) // 16]) * 16 + (int(lens[0]) - 1) % 16
    hk, _ = oracle.kv_append(kc, vc, k_new[:1], v_new[:1], np.array([slot0], np.int64))
    assert np.array_equal(bf16_dev_to_bits(kd), hk)
    assert np.all(np.isfinite(bf16_dev_to_f64(out)))
