"""Host-side checks of the benchmark's accounting: the algorithmic bytes and
FLOPs it divides by are recounted here by brute force from the masks'
definitions (causal bottom-right, strict window), independently of the
closed forms in bench.py; and the reference arm runs on the host."""
import json
import os
import subprocess
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads as wl  # noqa: E402


def _pairs_brute(prefix, qlen, window):
    n = 0
    k_len = prefix + qlen
    for i in range(qlen):
        qpos = k_len - qlen + i
        for k in range(k_len):
            if k <= qpos and (window <= 0 or qpos - k < window):
                n += 1
    return n


def test_varlen_flops_counts_unmasked_pairs():
    for window in (0, 7, 64):
        step = wl.make_step("t", 5, H_q=8, H_kv=2, D=64, P=16, num_pages=64,
                            pre_prefix=[0, 37, 5], pre_qlen=[50, 1, 90], window=window)
        pairs = sum(_pairs_brute(int(p), int(q), window)
                    for p, q in zip(step.pre_prefix, step.pre_qlen))
        assert bench.varlen_flops(step) == 4.0 * step.D * step.H_q * pairs


def test_decode_bytes_counts_attended_kv_once():
    for window in (0, 100):
        step = wl.make_step("t", 6, H_q=8, H_kv=2, D=64, P=16, num_pages=256,
                            dec_cached=[7, 33, 300, 0], window=window)
        lens = step.dec_seq_lens
        kv = 0
        for L in lens:
            keys = [k for k in range(int(L)) if window <= 0 or (int(L) - 1) - k < window]
            kv += len(keys) * step.H_kv * step.D * 2 * 2
        qo = step.Bd * step.H_q * step.D * 2 * 2
        pages = sum(-(-min(int(L), window if window > 0 else int(L)) // step.P) for L in lens)
        assert bench.decode_bytes(step) == kv + qo + pages * 4 + step.Bd * 4


def test_append_bytes():
    step = wl.tiny()
    n = step.n_new_tokens
    # read new K and V, write them: 4 * H_kv * D bf16 values per row, plus the slot
    assert bench.append_bytes(step, n) == n * (4 * step.H_kv * step.D * 2 + 8)


def test_reference_arm_runs_on_host():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "0"], capture_output=True, text=True,
                         timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_append_rope_bytes_counts_every_tensor_once():
    # recount from the tensors the fused call touches, itemised
    step = wl.mixed_step()
    n = step.n_new_tokens
    bf16, f32 = 2, 4
    tensors = {
        "q read": n * step.H_q * step.D * bf16, "q write": n * step.H_q * step.D * bf16,
        "k_new": n * step.H_kv * step.D * bf16, "v_new": n * step.H_kv * step.D * bf16,
        "k pool rows": n * step.H_kv * step.D * bf16, "v pool rows": n * step.H_kv * step.D * bf16,
        "cos/sin rows": n * step.D * f32, "slots": n * 8, "positions": n * 4,
        "norm weights": 2 * step.D * bf16,
    }
    assert bench.append_rope_bytes(step, n) == sum(tensors.values())
    assert len(step.all_positions) == n


def test_multicore_oracle_baseline_runs():
    # spawned workers, two of them, one timed step
    out = bench.cpu_baseline_multicore(steps=1, max_workers=2)
    assert out["cores"] == 2 and out["kind"] == "oracle" and out["value"] > 0


def test_positions_agree_with_slots():
    # the position of each new token, looked up through its block table,
    # must land on the slot the append writes
    for step in (wl.mixed_step(), wl.tiny(), wl.sliding()):
        pos = step.all_positions.astype(np.int64)
        tables = ([step.pre_block_table[c] for c in range(step.Bp) for _ in range(int(step.pre_qlen[c]))]
                  + [step.dec_block_table[b] for b in range(step.Bd)])
        slots = np.array([int(t[p // step.P]) * step.P + p % step.P for t, p in zip(tables, pos)])
        assert np.array_equal(slots, step.all_slots)


def test_traffic_entries_name_existing_sources():
    # every captured-traffic entry hashes files that exist, and the value is
    # either the capture's byte count or None (sources changed since)
    for key, (nbytes, files, sha) in bench.TRAFFIC.items():
        for f in files:
            assert os.path.isfile(os.path.join(bench.ROOT, "paged_kv_attention_11_gb300", "csrc", f)), f
        assert len(sha) == 16 and nbytes > 0
        assert bench.traffic_bytes(key) in (nbytes, None)


def test_source_digest_ignores_comments_not_code():
    # a comment edit keeps a capture's traffic entry; a code edit (even one
    # inside a string literal, or a changed operator) retires it
    base = 'int f(int x) {  // twice x\n  /* doubled */ return 2 * x;\n}\nconst char* s = "a//b";\n'
    d = bench.source_digest([base])
    assert bench.source_digest([base.replace("twice x", "x times two")]) == d
    assert bench.source_digest([base.replace("/* doubled */", "/* a\nlonger\nnote */")]) == d
    assert bench.source_digest(["// header\n\n" + base + "\n\n"]) == d
    assert bench.source_digest([base.replace("2 * x", "3 * x")]) != d
    assert bench.source_digest([base.replace('"a//b"', '"a//c"')]) != d
    # file boundaries count: the same text split differently is another digest
    assert bench.source_digest([base, base]) != bench.source_digest([base + base])
