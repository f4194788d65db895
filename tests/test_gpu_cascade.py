"""GPU parity of paged_attn_decode_shared_prefix (cascade decode: a prefix
pass reads each group's shared pages once, the split-KV decode reads each
member's suffix and merges) against the fp64 oracle's plain decode -- the
cascade changes the order of the sums, not the result.

Covers the GRPO layer (16 prompts x 4 generations sharing a 256-token
prefix), members no longer than their prefix (decoded whole), groups with no
sharing, a prefix length that is not a whole number of pages (flagged,
treated as no sharing), a last group shorter than the others, groups of one,
and the row limits per head_dim (32 rows at 64, 16 at 128, 8 at 256)."""
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


def _cascade(pkv, q, kc, vc, bt, lens, group_size, prefix_lens, scale):
    import torch
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    qd = to_dev_bf16(q)
    out = torch.full_like(qd, float("nan"))
    pkv.paged_attn_decode_shared_prefix(out, qd, to_dev_bf16(kc), to_dev_bf16(vc), to_dev(bt),
                                        to_dev(lens), group_size, to_dev(prefix_lens),
                                        int(lens.max()), scale, err_flag=err)
    torch.cuda.synchronize()
    return bf16_dev_to_f64(out), int(err.item())


def _groups(rng, n_groups, group_size, prefix_pages, suffix_lens, H_q, H_kv, D, P):
    """Block tables where each group's members alias the group's prefix
    pages, then own pages for their suffixes."""
    B = n_groups * group_size
    lens = np.asarray(suffix_lens, np.int64)[:B] + np.repeat(np.asarray(prefix_pages) * P,
                                                             group_size)[:B]
    lens = lens.astype(np.int32)
    own = [max(0, -(-int(lens[b]) // P) - prefix_pages[b // group_size]) for b in range(B)]
    num_pages = int(sum(prefix_pages) + sum(own) + 4)
    perm = rng.permutation(num_pages).astype(np.int32)
    mb = max(prefix_pages[b // group_size] + own[b] for b in range(B))
    bt = np.full((B, max(mb, 1)), -1, np.int32)
    o = 0
    for j in range(n_groups):
        shared = perm[o:o + prefix_pages[j]]
        o += prefix_pages[j]
        for m in range(group_size):
            b = j * group_size + m
            bt[b, :prefix_pages[j]] = shared
            bt[b, prefix_pages[j]:prefix_pages[j] + own[b]] = perm[o:o + own[b]]
            o += own[b]
    kc = wl.randn_bf16(rng, (num_pages, H_kv, P, D))
    vc = wl.randn_bf16(rng, (num_pages, H_kv, P, D))
    q = wl.randn_bf16(rng, (B, H_q, D))
    return q, kc, vc, bt, lens


def test_cascade_grpo_layer(pkv):
    """16 prompts x 4 generations, 256-token prefix pages shared, after this
    step's append (the rollout decode step)."""
    import torch
    step = wl.grpo_layer(layers=1, n_prompts=16)
    vals = wl.fill_values(step, 21)
    kc, vc = to_dev_bf16(vals.k_cache), to_dev_bf16(vals.v_cache)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.paged_kv_append(to_dev_bf16(vals.k_new), to_dev_bf16(vals.v_new), kc, vc,
                        to_dev(step.all_slots), err_flag=err)
    hk, hv = oracle.kv_append(vals.k_cache, vals.v_cache, vals.k_new, vals.v_new, step.all_slots)
    q = to_dev_bf16(vals.q_dec[0])
    out = torch.empty_like(q)
    pkv.paged_attn_decode_shared_prefix(out, q, kc, vc, to_dev(step.dec_block_table),
                                        to_dev(step.dec_seq_lens), step.group_size,
                                        to_dev(step.prefix_lens), step.max_seq_len_dec(),
                                        step.scale, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    want = oracle.paged_decode(vals.q_dec[0], hk, hv, step.dec_block_table, step.dec_seq_lens,
                               step.scale)
    assert_close_attn(bf16_dev_to_f64(out), want, "cascade grpo")


@pytest.mark.parametrize("D,H,gs", [(128, (32, 8), 4), (128, (16, 2), 2), (64, (8, 2), 8),
                                    (256, (8, 1), 1), (128, (8, 8), 16)])
def test_cascade_shapes_and_edges(pkv, D, H, gs):
    rng = np.random.default_rng(D + 7 * gs)
    P = 16
    n_groups = 6
    # group 0: long prefix; group 1: members shorter than the prefix;
    # group 2: no sharing; group 3: one member exactly at the prefix length
    prefix_pages = [20, 8, 0, 4, 1, 3]
    B = n_groups * gs
    suffix = rng.integers(1, 700, size=B)
    suffix[gs:2 * gs] = -rng.integers(1, 100, size=gs)     # group 1: inside the prefix
    suffix[3 * gs] = 0                                       # length == prefix
    q, kc, vc, bt, lens = _groups(rng, n_groups, gs, prefix_pages, suffix, H[0], H[1], D, P)
    pl = np.array(prefix_pages, np.int32) * P
    got, err = _cascade(pkv, q, kc, vc, bt, lens, gs, pl, 1 / np.sqrt(D))
    assert err == 0
    want = oracle.paged_decode(q, kc, vc, bt, lens, 1 / np.sqrt(D))
    assert_close_attn(got, want, f"cascade D={D} H={H} group={gs}")


@pytest.mark.parametrize("D,H", [(128, (8, 2)), (256, (4, 2))])
def test_cascade_long_suffix_merges_with_prefix(pkv, D, H):
    """Suffixes long enough that the decode cuts them into chunks: the merge
    phase then weighs the prefix partial with the suffix chunks."""
    rng = np.random.default_rng(900 + D)
    P, gs = 16, 4
    prefix_pages = [16, 2, 0]
    suffix = np.array([6000, 5000, 40, 1, 3000, 7000, 2, 900, 4500, 10, 6500, 300])
    q, kc, vc, bt, lens = _groups(rng, 3, gs, prefix_pages, suffix, H[0], H[1], D, P)
    pl = np.array(prefix_pages, np.int32) * P
    got, err = _cascade(pkv, q, kc, vc, bt, lens, gs, pl, 1 / np.sqrt(D))
    assert err == 0
    want = oracle.paged_decode(q, kc, vc, bt, lens, 1 / np.sqrt(D))
    assert_close_attn(got, want, f"cascade long suffix D={D}")


def test_cascade_bad_prefix_and_short_last_group(pkv):
    rng = np.random.default_rng(99)
    P, D, gs = 16, 128, 4
    prefix_pages = [6, 6, 6]
    q, kc, vc, bt, lens = _groups(rng, 3, gs, prefix_pages, rng.integers(1, 300, size=12),
                                  32, 8, D, P)
    # drop the last member: the last group has 3 sequences
    q, bt, lens = q[:11], bt[:11], lens[:11]
    pl = np.array([96, 95, 96], np.int32)   # group 1: not a whole number of pages
    got, err = _cascade(pkv, q, kc, vc, bt, lens, gs, pl, 1 / np.sqrt(D))
    assert err == 4  # PKV_DEVERR_LEN: group 1 decoded without sharing
    want = oracle.paged_decode(q, kc, vc, bt, lens, 1 / np.sqrt(D))
    assert_close_attn(got, want, "cascade bad prefix")
