"""GPU checks of pkv_copy (host transfers done by the SMs): every byte lands
where it belongs in each direction (pinned host -> device, device -> pinned
host, device -> device), at sizes from one 16-byte word to several MB and
at 16-byte offsets, the bytes around the target stay untouched, and a
decode step driven through it (inputs copied in, paged_attn_decode_append,
output copied out) matches the fp64 oracle and, bit for bit, the same step
on inputs placed with torch's copies."""
import numpy as np
import pytest

import oracle
import workloads as wl
from _util import assert_close_attn, bf16_dev_to_bits, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu

SIZES = [16, 4096, 4112, 818944, 16 * 1048583]


@pytest.fixture(scope="module")
def pkv():
    import torch  # noqa: F401
    from paged_kv_attention_11_gb300 import build
    build.build()
    import paged_kv_attention_11_gb300 as m
    m.lib()
    return m


def _bytes(n, seed):
    return np.random.default_rng(seed).integers(0, 256, size=n, dtype=np.uint8)


@pytest.mark.parametrize("direction", ["h2d", "d2h", "d2d"])
@pytest.mark.parametrize("n", SIZES)
def test_copy_moves_every_byte(pkv, direction, n):
    import torch
    data = _bytes(n, n % 1000 + len(direction))
    pad = 64  # sentinel bytes on both sides of the target range
    src_pinned = direction == "h2d"
    dst_pinned = direction == "d2h"
    src_buf = torch.empty(n + 2 * pad, dtype=torch.uint8)
    src_buf = src_buf.pin_memory() if src_pinned else src_buf.cuda()
    src_buf.copy_(torch.from_numpy(np.concatenate([_bytes(pad, 1), data, _bytes(pad, 2)])))
    dst_buf = torch.full((n + 2 * pad,), 0xA5, dtype=torch.uint8)
    dst_buf = dst_buf.pin_memory() if dst_pinned else dst_buf.cuda()
    torch.cuda.synchronize()
    # 16-byte offsets that differ on the two sides
    src = src_buf[pad:pad + n]
    dst = dst_buf[pad - 16:pad - 16 + n] if pad >= 16 else dst_buf[:n]
    pkv.pkv_copy(dst, src)
    torch.cuda.synchronize()
    got = dst_buf.cpu().numpy()
    assert np.array_equal(got[pad - 16:pad - 16 + n], data)
    assert np.all(got[:pad - 16] == 0xA5) and np.all(got[pad - 16 + n:] == 0xA5)


def test_copy_rejects_before_enqueueing(pkv):
    import torch
    lib = pkv.lib()
    dev = torch.zeros(64, dtype=torch.uint8, device="cuda")
    p = dev.data_ptr()
    # a size that is not a multiple of 16, a misaligned pointer, overlap
    assert lib.pkv_copy(p + 32, p, 8, None) == 1
    assert lib.pkv_copy(p + 32, p + 1, 16, None) == 1
    assert lib.pkv_copy(p + 16, p, 32, None) == 1
    assert lib.pkv_copy(None, p, 16, None) == 1
    assert lib.pkv_copy(p, p + 32, 0, None) == 0


def _decode_case(seed, B=48, H_q=32, H_kv=8, D=128, P=16):
    rng = np.random.default_rng(seed)
    lens = rng.integers(1, 1500, size=B).astype(np.int32)
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
    k_new = wl.randn_bf16(rng, (B, H_kv, D))
    v_new = wl.randn_bf16(rng, (B, H_kv, D))
    return q, kc, vc, bt, lens, k_new, v_new


def test_decode_step_through_host_copies(pkv):
    """Two steps in a row: each packs its inputs in one pinned buffer, copies
    them in with pkv_copy, runs paged_attn_decode_append and copies the
    output rows back with pkv_copy."""
    import torch
    for step, seed in enumerate((71, 72)):
        q, kc, vc, bt, lens, k_new, v_new = _decode_case(seed)
        P = kc.shape[2]
        scale = 1.0 / np.sqrt(q.shape[2])
        parts = [q.view(np.uint8), k_new.view(np.uint8), v_new.view(np.uint8),
                 bt.view(np.uint8), lens.view(np.uint8)]
        offs, off = [], 0
        for a in parts:
            offs.append(off)
            off += (a.nbytes + 255) // 256 * 256
        host = torch.zeros(off, dtype=torch.uint8).pin_memory()
        hn = host.numpy()
        for a, o in zip(parts, offs):
            hn[o:o + a.nbytes] = a.reshape(-1)
        dev = torch.empty(off, dtype=torch.uint8, device="cuda")

        def view(i, dtype, shape):
            import math
            n = math.prod(shape) * torch.empty((), dtype=dtype).element_size()
            return dev[offs[i]:offs[i] + n].view(dtype).view(shape)
        kd, vd = to_dev_bf16(kc), to_dev_bf16(vc)
        out = torch.full(q.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
        out_h = torch.zeros(q.shape, dtype=torch.bfloat16).pin_memory()
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        torch.cuda.synchronize()
        pkv.pkv_copy(dev, host)
        pkv.paged_attn_decode_append(
            out, view(0, torch.bfloat16, q.shape), view(1, torch.bfloat16, k_new.shape),
            view(2, torch.bfloat16, v_new.shape), kd, vd, view(3, torch.int32, bt.shape),
            view(4, torch.int32, lens.shape), int(lens.max()), scale, 0, err_flag=err)
        pkv.pkv_copy(out_h, out)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        got_bits = out_h.view(torch.int16).numpy().view(np.uint16)
        slots = np.array([int(bt[b, (L - 1) // P]) * P + (L - 1) % P for b, L in enumerate(lens)],
                         np.int64)
        hk, hv = oracle.kv_append(kc, vc, k_new, v_new, slots)
        want = oracle.paged_decode(q, hk, hv, bt, lens, scale)
        assert_close_attn(oracle.bf16_bits_to_f64(got_bits), want, f"step {step} vs oracle")
        # the same step with its inputs placed by torch's copies
        kd2, vd2 = to_dev_bf16(kc), to_dev_bf16(vc)
        out2 = torch.full_like(out, float("nan"))
        pkv.paged_attn_decode_append(out2, to_dev_bf16(q), to_dev_bf16(k_new), to_dev_bf16(v_new),
                                     kd2, vd2, to_dev(bt), to_dev(lens), int(lens.max()), scale,
                                     0, err_flag=err)
        torch.cuda.synchronize()
        assert np.array_equal(got_bits, bf16_dev_to_bits(out2)), f"step {step}: copy path"
        assert np.array_equal(bf16_dev_to_bits(kd), hk) and np.array_equal(bf16_dev_to_bits(vd), hv)
