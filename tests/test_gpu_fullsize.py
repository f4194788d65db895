"""GPU parity at full size for the GRPO rollout-scale decode step: 64 prompts x
4 generations (256 sequences), each prompt's 256-token prefix stored once and
its pages shared by the 4 generations' block tables, completions U[0,3840],
32/8 heads, head_dim 128, page 16, and the caches of 36 layers in one pool
(about 73 GB of K+V on the device).  The step runs through the C ABI as the
benchmark runs it (append every new row, then decode with a workspace) on the
last layer's page range; outputs are compared with the fp64 oracle on sampled
sequences, the appended pages bit-exactly.

Every page outside that layer's referenced pages holds NaN, so a read of a
wrong page shows up as a non-finite output anywhere in the batch."""
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


def test_grpo_rollout_full_size_sampled(pkv):
    import torch
    layers, layer = 36, 35
    step = wl.grpo_layer(layers=layers, layer=layer)
    H, P, D = step.H_kv, step.P, step.D
    B = step.Bd
    assert B == 256 and step.num_pages * H * P * D * 2 * 2 > 60e9

    shape = (step.num_pages, H, P, D)
    kc = torch.full(shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    vc = torch.full(shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    used = torch.as_tensor(step.used_pages, dtype=torch.int64, device="cuda")
    gen = torch.Generator(device="cuda").manual_seed(35)
    kc[used] = torch.randn((len(used), H, P, D), generator=gen, device="cuda").to(torch.bfloat16)
    vc[used] = torch.randn((len(used), H, P, D), generator=gen, device="cuda").to(torch.bfloat16)

    # sampled sequences: the longest, the shortest, all 4 generations of one
    # prompt (shared prefix pages) and a seeded random few
    rng = np.random.default_rng(3535)
    lens = step.dec_seq_lens
    pick = {int(np.argmax(lens)), int(np.argmin(lens)), 40, 41, 42, 43}
    pick.update(int(x) for x in rng.choice(B, size=8, replace=False))
    pick = np.array(sorted(pick))
    bt = step.dec_block_table
    pages_s = np.unique(np.concatenate([bt[b][: -(-int(lens[b]) // P)] for b in pick]))
    pages_s = pages_s[pages_s >= 0]
    remap = {int(p): i for i, p in enumerate(pages_s)}

    # host-generated contents for the sampled sequences' pages (the oracle's
    # inputs), written over the device fill
    hk = wl.randn_bf16(rng, (len(pages_s), H, P, D))
    hv = wl.randn_bf16(rng, (len(pages_s), H, P, D))
    idx = torch.as_tensor(pages_s, dtype=torch.int64, device="cuda")
    kc[idx] = to_dev_bf16(hk)
    vc[idx] = to_dev_bf16(hv)
    k_new = wl.randn_bf16(rng, (B, H, D))
    v_new = wl.randn_bf16(rng, (B, H, D))
    q = wl.randn_bf16(rng, (B, step.H_q, D))

    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    slots = step.dec_slots
    pkv.paged_kv_append(to_dev_bf16(k_new), to_dev_bf16(v_new), kc, vc, to_dev(slots),
                        err_flag=err)
    out = torch.empty((B, step.H_q, D), dtype=torch.bfloat16, device="cuda")
    pkv.paged_attn_decode(out, to_dev_bf16(q), kc, vc, to_dev(bt), to_dev(lens),
                          step.max_seq_len_dec(), step.scale, step.window, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got_all = bf16_dev_to_f64(out)
    assert np.all(np.isfinite(got_all)), "a sequence read a page outside its table"

    # oracle on the sampled sequences over a compact copy of their pages
    cbt = np.full((len(pick), bt.shape[1]), -1, np.int32)
    for i, b in enumerate(pick):
        n = -(-int(lens[b]) // P)
        cbt[i, :n] = [remap[int(p)] for p in bt[b][:n]]
    cslots = np.array([remap[int(slots[b] // P)] * P + int(slots[b] % P) for b in pick],
                      np.int64)
    ok, ov = oracle.kv_append(hk, hv, k_new[pick], v_new[pick], cslots)
    got_k = kc[idx].cpu().view(torch.int16).numpy().view(np.uint16)
    got_v = vc[idx].cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got_k, ok), "K pages differ after append"
    assert np.array_equal(got_v, ov), "V pages differ after append"
    want = oracle.paged_decode(q[pick], ok, ov, cbt, lens[pick], step.scale, step.window)
    assert_close_attn(got_all[pick], want, "grpo full size")

    # the same step through the shared-prefix (cascade) decode: each prompt's
    # 16 prefix pages read once per group of 4 generations
    out_c = torch.full((B, step.H_q, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    pkv.paged_attn_decode_shared_prefix(out_c, to_dev_bf16(q), kc, vc, to_dev(bt), to_dev(lens),
                                        step.group_size, to_dev(step.prefix_lens),
                                        step.max_seq_len_dec(), step.scale, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got_c = bf16_dev_to_f64(out_c)
    assert np.all(np.isfinite(got_c)), "a sequence read a page outside its table"
    assert_close_attn(got_c[pick], want, "grpo full size, cascade")
    del kc, vc
    torch.cuda.empty_cache()
