"""Benchmark of the paged-KV attention hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step of the default workload (Qwen3-4B-shaped decode step, one layer:
64 sequences with 256..2048 cached tokens, 32 query / 8 kv heads, head_dim
128, 16-token pages in a shuffled 16384-page pool) is:
    paged_kv_append (64 new K/V rows)  ->  paged_attn_decode (split + merge)
The headline value is achieved HBM GB/s: algorithmic bytes of the step
(every attended K/V byte once, q, out, the appended rows) divided by the
device time of the step.  L2 is flushed (a 512 MB read) before every step,
outside the timed events.  A second object reports the continuous-batching
mixed step (8 prefill chunks + 120 decode rows) in tokens/s.

--impl reference times the fp64 CPU oracle on a bounded sample of the same
workload and prints the same JSON line with "impl": "reference".
"""
from __future__ import annotations

import argparse
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = "paged decode-attn achieved HBM GB/s (% of 8 TB/s); mixed-step tokens/sec"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one launch,
# from an ncu capture on a GB300, with the SHA-256 prefix of the kernel's
# source files (concatenated, in the order listed, comments and blank lines
# removed: see source_digest) at capture time.  A value is reported only
# while the sources still have that hash; once the kernel's code changes the
# field is null until a new capture replaces the entry.  The summaries under
# profiles/ give the command and the other counters.
#   decode_qwen3: decode_split_kernel<128,4,12,0,2> on the qwen3_decode step
#   decode_d512:  decode_split_kernel<512,2,4,0,1> on the head_dim 512 step
#   varlen_mixed: varlen_fwd_kernel<128,2,128,1,3,2,128> on the mixed step
#   varlen_d512:  varlen_fwd_kernel<512,1,32,2,2,2,256> on the head_dim 512 step
#   mixed_single: mixed_step_kernel<12,2,0> on the mixed step
#   append_mixed: kv_append_kernel<2> on the mixed step (5645 rows)
#   append_rope_mixed: kv_append_rope_kernel<128> on the mixed step, both norms
_DEC_SRC = ("decode.cu", "decode_body.cuh", "tile16.cuh", "common.cuh")
_VAR_SRC = ("varlen.cu", "varlen_body.cuh", "tcgen05.cuh", "exp2_math.cuh", "common.cuh")
_MIX_SRC = ("mixed.cu", "decode_body.cuh", "varlen_body.cuh", "tile16.cuh", "tcgen05.cuh",
            "exp2_math.cuh", "common.cuh")
TRAFFIC = {
    "decode_qwen3": (320_193_536, _DEC_SRC, "3dd9f216abb9b4be"),
    "decode_d512": (573_851_648, _DEC_SRC, "3dd9f216abb9b4be"),
    "varlen_mixed": (91_294_464, _VAR_SRC, "abd6d5929394aa53"),
    "varlen_d512": (44_015_616, _VAR_SRC, "abd6d5929394aa53"),
    "mixed_single": (1_218_739_456, _MIX_SRC, "4227504b9f00f717"),
    "append_mixed": (23_259_648, ("append.cu", "common.cuh"), "afb5104dd69f82c8"),
    "append_rope_mixed": (83_629_312, ("rope_append.cu",), "4dad9297abe899eb"),
}


def traffic_bytes(key: str):
    """The captured traffic of TRAFFIC[key], or None when a kernel source
    file has changed since the capture."""
    nbytes, files, sha = TRAFFIC[key]
    texts = []
    try:
        for f in files:
            with open(os.path.join(ROOT, "paged_kv_attention_11_gb300", "csrc", f)) as fh:
                texts.append(fh.read())
    except OSError:
        return None
    return nbytes if source_digest(texts) == sha else None


_CODE_TOKENS = re.compile(r'"(?:\\.|[^"\\\n])*"|\'(?:\\.|[^\'\\\n])*\'|//[^\n]*|/\*.*?\*/',
                          re.DOTALL)


def source_digest(texts) -> str:
    """SHA-256 prefix (16 hex digits) of C/CUDA sources with their comments,
    trailing blanks and empty lines removed, so that an edit of a comment
    does not mark a capture as stale while any change of code does.  String
    and character literals are kept as written."""
    import hashlib
    m = hashlib.sha256()
    for text in texts:
        code = _CODE_TOKENS.sub(lambda t: t.group(0) if t.group(0)[0] in "\"'" else " ", text)
        lines = [ln.rstrip() for ln in code.splitlines()]
        m.update("\n".join(ln for ln in lines if ln).encode())
        m.update(b"\0")
    return m.hexdigest()[:16]


# ------------------------------------------------------------------ helpers
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(vals, device):
    """Each value's maximum over all ranks (the slowest replica sets the
    job's time); the values themselves at world size 1."""
    ws, _, _ = dist_env()
    if ws <= 1:
        return [float(v) for v in vals]
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in vals], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.cpu()]


def job_gb_s(ws: int, bytes_per_rank: int, step_ms: float) -> float:
    """Whole-job throughput: the bytes all ranks processed in one step over
    the (max-over-ranks) step time."""
    return ws * bytes_per_rank / (step_ms * 1e-3) / 1e9


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            hbm = d.get("hbm_gbs") or d.get("hbm_GBps") or d.get("hbm")
            tf = d.get("bf16_tflops") or d.get("bf16")
            tfs = d.get("bf16_tflops_sustained") or tf
            if hbm:
                return float(hbm), float(tf or FALLBACK_BF16_TFLOPS), float(
                    tfs or FALLBACK_BF16_TFLOPS), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during the timed region."""
    FIELDS = ("pci.bus_id,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id: str):
        self.bus = bus_id.lower()[-12:] if bus_id else ""
        self.rows = []
        self._stop = threading.Event()
        self._t = None

    def _run(self):
        while not self._stop.is_set():
            try:
                out = subprocess.run(["nvidia-smi", f"--query-gpu={self.FIELDS}",
                                      "--format=csv,noheader,nounits"], capture_output=True,
                                     text=True, timeout=5).stdout
                for line in out.strip().splitlines():
                    f = [x.strip() for x in line.split(",")]
                    if len(f) >= 9 and (not self.bus or f[0].lower().endswith(self.bus)):
                        self.rows.append(f)
                        break
            except Exception:
                pass
            self._stop.wait(0.2)

    def __enter__(self):
        self._t = threading.Thread(target=self._run, daemon=True)
        self._t.start()
        return self

    def __exit__(self, *a):
        self._stop.set()
        if self._t:
            self._t.join(timeout=10)

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4)
                          if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(self.rows)}


# -------------------------------------------------------------- byte models
def decode_bytes(step: wl.Step) -> int:
    """Algorithmic HBM bytes of one decode call: each attended K and V row
    once (window-limited), q in, out, block-table entries and lengths."""
    L = step.dec_seq_lens.astype(np.int64)
    if step.window > 0:
        L = np.minimum(L, step.window)
    kv = int(L.sum()) * step.H_kv * step.D * 2 * 2
    qo = step.Bd * step.H_q * step.D * 2 * 2
    bt = int(np.sum(-(-L // step.P))) * 4 + step.Bd * 4
    return kv + qo + bt


def append_bytes(step: wl.Step, n_rows: int) -> int:
    return n_rows * step.H_kv * step.D * 2 * 2 * 2 + n_rows * 8


def append_rope_bytes(step: wl.Step, n_rows: int) -> int:
    """Fused norm + rotary + append: q read and written in place, k and v
    read and written, one cos/sin table row (D float32) per token, slot and
    position per token, and the two [D] bf16 norm weights."""
    per_tok = (step.H_q * step.D * 2 * 2 + step.H_kv * step.D * 2 * 2 * 2 + step.D * 4 + 8 + 4)
    return n_rows * per_tok + 2 * step.D * 2


def varlen_flops(step: wl.Step) -> float:
    """4*D*H_q flops per unmasked (query, key) pair (QK^T and PV)."""
    pairs = 0
    for c in range(step.Bp):
        q, p = int(step.pre_qlen[c]), int(step.pre_prefix[c])
        pos = p + np.arange(q)
        n = pos + 1
        if step.window > 0:
            n = np.minimum(n, step.window)
        pairs += int(n.sum())
    return 4.0 * step.D * step.H_q * pairs


# --------------------------------------------------------- device workload
class DeviceStep:
    """A step's inputs resident on the GPU (values drawn on the device)."""

    def __init__(self, step: wl.Step, seed: int, device):
        import torch
        self.step = step
        g = torch.Generator(device=device)
        g.manual_seed(seed)
        shape = (step.num_pages, step.H_kv, step.P, step.D)
        bf = torch.bfloat16
        if step.num_pages * step.H_kv * step.P * step.D * 2 > (4 << 30):
            # a multi-layer pool: only this layer's referenced pages are drawn
            self.k_cache = torch.empty(shape, device=device, dtype=bf)
            self.v_cache = torch.empty(shape, device=device, dtype=bf)
            used = torch.from_numpy(step.used_pages.astype(np.int64)).to(device)
            for c in range(0, used.numel(), 8192):
                idx = used[c:c + 8192]
                sub = (idx.numel(),) + shape[1:]
                self.k_cache[idx] = torch.randn(sub, generator=g, device=device).to(bf)
                self.v_cache[idx] = torch.randn(sub, generator=g, device=device).to(bf)
        else:
            self.k_cache = torch.randn(shape, generator=g, device=device,
                                       dtype=torch.float32).to(bf)
            if step.k_head_scale is not None:
                s = torch.from_numpy(step.k_head_scale).to(device).view(1, -1, 1, 1)
                self.k_cache = (self.k_cache.float() * s).to(bf)
            self.v_cache = torch.randn(shape, generator=g, device=device,
                                       dtype=torch.float32).to(bf)
        n_new = step.n_new_tokens
        self.k_new = torch.randn((n_new, step.H_kv, step.D), generator=g, device=device).to(bf)
        self.v_new = torch.randn((n_new, step.H_kv, step.D), generator=g, device=device).to(bf)
        self.slots = torch.from_numpy(step.all_slots).to(device)
        self.q_dec = torch.randn((step.Bd, step.H_q, step.D), generator=g, device=device).to(bf) \
            if step.Bd else None
        self.out_dec = torch.empty_like(self.q_dec) if step.Bd else None
        self.q_pre = torch.randn((step.total_q, step.H_q, step.D), generator=g,
                                 device=device).to(bf) if step.Bp else None
        self.out_pre = torch.empty_like(self.q_pre) if step.Bp else None
        if step.Bd:
            self.dec_bt = torch.from_numpy(step.dec_block_table).to(device)
            self.dec_lens = torch.from_numpy(step.dec_seq_lens).to(device)
        if step.Bp:
            self.pre_bt = torch.from_numpy(step.pre_block_table).to(device)
            self.cu_q = torch.from_numpy(step.cu_seq_lens_q).to(device)
            self.cu_k = torch.from_numpy(step.cu_seq_lens_k).to(device)
        import paged_kv_attention_11_gb300 as pkv
        self.pkv = pkv
        need = pkv.decode_workspace_size(max(step.Bd, 1), step.H_q, step.H_kv, step.D)
        self.ws = torch.zeros(max(need, 256), dtype=torch.uint8, device=device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)

    def enable_rope(self, theta: float = 1e6, eps: float = 1e-6, max_position: int = 16384):
        """Set up the fused norm + rotary append: one contiguous q for all
        new tokens (prefill rows, then decode rows; the varlen and decode
        calls then read its two slices), positions, the cos/sin table and
        the two norm weights."""
        import torch
        s = self.step
        dev = self.k_cache.device
        parts = [t for t in (self.q_pre, self.q_dec) if t is not None]
        self.q_all = torch.cat(parts).contiguous()
        if s.Bp:
            self.q_pre = self.q_all[:s.total_q]
        if s.Bd:
            self.q_dec = self.q_all[s.total_q:]
        self.positions = torch.from_numpy(s.all_positions).to(dev)
        self.cos_sin = torch.empty((max_position, s.D), dtype=torch.float32, device=dev)
        self.pkv.rope_table(self.cos_sin, theta)
        g = torch.Generator(device=dev)
        g.manual_seed(77)
        self.q_w = (1 + 0.1 * torch.randn(s.D, generator=g, device=dev)).to(torch.bfloat16)
        self.k_w = (1 + 0.1 * torch.randn(s.D, generator=g, device=dev)).to(torch.bfloat16)
        self.rope_eps = eps

    def append_rope(self, stream):
        self.pkv.paged_kv_append_rope(self.q_all, self.k_new, self.v_new, self.k_cache,
                                      self.v_cache, self.slots, self.positions, self.cos_sin,
                                      self.q_w, self.k_w, self.rope_eps, err_flag=self.err,
                                      stream=stream)

    def append(self, stream):
        self.pkv.paged_kv_append(self.k_new, self.v_new, self.k_cache, self.v_cache, self.slots,
                                 err_flag=self.err, stream=stream)

    def varlen(self, stream):
        s = self.step
        self.pkv.paged_attn_varlen(self.out_pre, self.q_pre, self.k_cache, self.v_cache,
                                   self.cu_q, self.cu_k, self.pre_bt, s.max_seqlen_q(),
                                   s.max_seqlen_k(), s.scale, True, s.window,
                                   err_flag=self.err, stream=stream)

    def decode(self, stream):
        s = self.step
        self.pkv.paged_attn_decode(self.out_dec, self.q_dec, self.k_cache, self.v_cache,
                                   self.dec_bt, self.dec_lens, s.max_seq_len_dec(), s.scale,
                                   s.window, workspace=self.ws, err_flag=self.err,
                                   stream=stream)

    def decode_append(self, stream):
        """The decode step with its append fused (paged_attn_decode_append):
        decode-only steps, whose new rows are the decode rows in order."""
        s = self.step
        self.pkv.paged_attn_decode_append(self.out_dec, self.q_dec, self.k_new, self.v_new,
                                          self.k_cache, self.v_cache, self.dec_bt, self.dec_lens,
                                          s.max_seq_len_dec(), s.scale, s.window,
                                          workspace=self.ws, err_flag=self.err, stream=stream)

    def mixed(self, stream, decode_ctas=0):
        """Decode rows and prefill chunks in one paged_attn_mixed launch."""
        s = self.step
        self.pkv.paged_attn_mixed(self.out_dec, self.q_dec, self.dec_bt, self.dec_lens,
                                  s.max_seq_len_dec(), self.out_pre, self.q_pre, self.cu_q,
                                  self.cu_k, self.pre_bt, s.max_seqlen_q(), s.max_seqlen_k(),
                                  self.k_cache, self.v_cache, s.scale, s.window,
                                  decode_ctas=decode_ctas, workspace=self.ws, err_flag=self.err,
                                  stream=stream)

    def mixed_append(self, stream, decode_ctas=0):
        """The step's append, decode rows and prefill chunks in one
        paged_attn_mixed_append launch."""
        s = self.step
        self.pkv.paged_attn_mixed_append(
            self.out_dec, self.q_dec, self.dec_bt, self.dec_lens, s.max_seq_len_dec(),
            self.out_pre, self.q_pre, self.cu_q, self.cu_k, self.pre_bt, s.max_seqlen_q(),
            s.max_seqlen_k(), self.k_new, self.v_new, self.slots, self.k_cache, self.v_cache,
            s.scale, s.window, decode_ctas=decode_ctas, workspace=self.ws, err_flag=self.err,
            stream=stream)

    def decode_shared_prefix(self, stream):
        """The same decode through the shared-prefix (cascade) entry point."""
        import torch
        s = self.step
        if not hasattr(self, "ws_pfx"):
            need = self.pkv.shared_prefix_workspace_size(s.Bd, s.H_q, s.H_kv, s.D)
            self.ws_pfx = torch.zeros(need, dtype=torch.uint8, device=self.k_cache.device)
            self.prefix_lens = torch.from_numpy(s.prefix_lens).to(self.k_cache.device)
        self.pkv.paged_attn_decode_shared_prefix(
            self.out_dec, self.q_dec, self.k_cache, self.v_cache, self.dec_bt, self.dec_lens,
            s.group_size, self.prefix_lens, s.max_seq_len_dec(), s.scale,
            workspace=self.ws_pfx, err_flag=self.err, stream=stream)


def time_steps(fn_phases, steps, warmup, stream, flush, graphs=True, phase_events=True):
    """Run warmup + steps; returns per-step per-phase device ms (events).

    With ``graphs`` the whole step is captured once into one CUDA graph (the
    API calls are capture-safe: no allocation, no host sync), with timing
    events recorded as graph nodes, and replayed once per timed step, so the
    events time device work, not the host's graph launch.  With
    ``phase_events`` there is an event between consecutive phases (per-phase
    times; an event node between two kernels also stops the next kernel's
    prologue from overlapping the previous one through programmatic
    dependent launch); without, only around the step, and the single
    returned "phase" is the whole step as an engine would run it.  Without
    external-event capture support in torch, each phase gets its own graph
    and the events sit around the replays.  Every timed step starts after an
    L2 flush on the same stream.
    """
    import torch
    for _ in range(warmup):
        for f in fn_phases:
            f(stream)
    torch.cuda.synchronize()
    n = len(fn_phases)
    if graphs:
        try:
            gev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(n + 1)]
        except TypeError:
            gev = None
        if gev is not None:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                gev[0].record(stream)
                for i, f in enumerate(fn_phases):
                    f(stream)
                    if phase_events or i == n - 1:
                        gev[i + 1 if phase_events else 1].record(stream)
            if not phase_events:
                n = 1
            torch.cuda.synchronize()
            with torch.cuda.stream(stream):
                for _ in range(warmup):
                    g.replay()
            torch.cuda.synchronize()
            out = []
            for _ in range(steps):
                flush()
                with torch.cuda.stream(stream):
                    g.replay()
                torch.cuda.synchronize()
                out.append([gev[i].elapsed_time(gev[i + 1]) for i in range(n)])
            return out
        gs = []
        for f in fn_phases:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                f(stream)
            gs.append(g)
        torch.cuda.synchronize()

        def mk(g):
            return lambda s: g.replay()
        fn_phases = [mk(g) for g in gs]
        for _ in range(warmup):
            with torch.cuda.stream(stream):
                for f in fn_phases:
                    f(stream)
        torch.cuda.synchronize()
    recs = []
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
              for _ in range(steps)]
    with torch.cuda.stream(stream):
        for k in range(steps):
            flush()
            evs = events[k]
            evs[0].record(stream)
            for i, f in enumerate(fn_phases):
                f(stream)
                evs[i + 1].record(stream)
            recs.append(evs)
    torch.cuda.synchronize()
    return [[recs[k][i].elapsed_time(recs[k][i + 1]) for i in range(n)]
            for k in range(steps)]


# --------------------------------------------------------------- ours arm
def run_ours(args):
    import torch
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    from paged_kv_attention_11_gb300 import build
    build.build()

    hbm_peak, tf_peak, tf_sus, peak_src = peaks()
    stream = torch.cuda.Stream(device)
    # L2 flush between timed steps: READ 512 MB (4x L2) so that L2 holds
    # only clean lines of an unrelated buffer when a step starts (a write
    # flush would leave dirty lines whose write-back lands inside the step).
    flush_buf = torch.ones(512 << 20, dtype=torch.uint8, device=device)

    def flush():
        with torch.cuda.stream(stream):
            flush_buf.view(torch.int32).sum()

    def barrier():
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()

    sections = {"mixed": ("mixed_step", run_mixed), "sliding": ("sliding_step", run_sliding),
                "grpo": ("grpo_step", run_grpo), "d512": ("head_dim_512_step", run_full512)}
    if args.only in sections:
        # one section alone (profiling runs)
        key, fn = sections[args.only]
        res = fn(args, device, stream, flush, rank)
        if rank == 0:
            print(json.dumps({"metric": METRIC, key: res}), flush=True)
        return

    # ---- headline: Qwen3-shaped decode step -------------------------------
    step = wl.qwen3_decode()
    ds = DeviceStep(step, wl.BASE_SEED + 2 + 1000 * rank, device)
    torch.cuda.synchronize()
    bus = ""
    try:
        bus = torch.cuda.get_device_properties(device).pci_bus_id
    except Exception:
        pass
    barrier()
    torch.cuda.synchronize()
    assert step.Bp == 0 and step.n_new_tokens == step.Bd  # the fused path's precondition
    with ClockSampler(bus) as clocks:
        per_step = time_steps([ds.append, ds.decode], args.steps, args.warmup, stream, flush,
                              phase_events=False)
        per_fused = time_steps([ds.decode_append], args.steps, args.warmup, stream, flush,
                               phase_events=False)
    torch.cuda.synchronize()
    barrier()
    # per-kernel breakdown for the roofline: the same steps with an event
    # between the two kernels
    per = time_steps([ds.append, ds.decode], args.steps, args.warmup, stream, flush)
    torch.cuda.synchronize()
    assert int(ds.err.item()) == 0, f"device error flag {int(ds.err.item())}"
    two_ms = float(np.mean([sum(p) for p in per_step]))
    fused_ms = float(np.mean([sum(p) for p in per_fused]))
    dec_ms = float(np.mean([p[1] for p in per]))
    app_ms = float(np.mean([p[0] for p in per]))
    two_ms, fused_ms, dec_ms = max_over_ranks([two_ms, fused_ms, dec_ms], device)
    fused_best = fused_ms < two_ms
    step_ms = fused_ms if fused_best else two_ms
    dbytes = decode_bytes(step)
    abytes = append_bytes(step, step.n_new_tokens)
    value = job_gb_s(ws, dbytes + abytes, step_ms)
    dec_gbs = dbytes / (dec_ms * 1e-3) / 1e9

    # ---- end to end through the public API with host buffers ---------------
    e2e = None
    if not args.only:
        # copies on the copy engines (torch's copy_), then on the SMs
        # (pkv_copy); the line reports the SM path, the other beside it
        ce = run_e2e(ds, step, stream, flush, args, dbytes + abytes, fused=fused_best,
                     sm_copy=False)
        try:
            e2e = run_e2e(ds, step, stream, flush, args, dbytes + abytes, fused=fused_best)
            e2e["copy_engine"] = {"value": ce["value"], "ms_per_step": ce["ms_per_step"]}
        except Exception as ex:  # pkv_copy refused these buffers: keep the copy engines
            e2e = ce
            e2e["sm_copy"] = {"unavailable": f"{type(ex).__name__}: {ex}"[:200]}

    # ---- secondary: mixed continuous-batching step (tokens/s) -------------
    mixed = None if args.only == "decode" else run_mixed(args, device, stream, flush, rank)
    sliding = None if args.only else run_sliding(args, device, stream, flush, rank)
    grpo = None if args.only else run_grpo(args, device, stream, flush, rank)
    full512 = None if args.only else run_full512(args, device, stream, flush, rank)

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded, bf16 ~N(0,1), K scaled per kv head by U(0.5,2))",
        "config": {"workload": "qwen3_decode: one layer, batch 64, cached ~U[256,2048], "
                               "H_q 32 / H_kv 8, head_dim 128, page 16, 16384-page shuffled "
                               "pool; step = append 64 rows + decode"
                               + (" (one launch: paged_attn_decode_append)" if fused_best else
                                  " (paged_kv_append, then paged_attn_decode)"),
                   "l2": "flushed before every timed step (512 MB read, outside the timed events)",
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
        "pct_of_8TBs": round(100.0 * value / ws / NOMINAL_HBM_GBS, 2),
        "decode_only": {"gb_s": round(dec_gbs, 2), "us": round(dec_ms * 1e3, 2),
                        "pct_of_8TBs": round(100 * dec_gbs / NOMINAL_HBM_GBS, 2)},
        "append_us": round(app_ms * 1e3, 2),
        "two_launch_step": {"gb_s": round(job_gb_s(ws, dbytes + abytes, two_ms), 2),
                            "ms_per_step": round(two_ms, 5)},
        "fused_append_step": {"gb_s": round(job_gb_s(ws, dbytes + abytes, fused_ms), 2),
                              "ms_per_step": round(fused_ms, 5),
                              "frac_of_peak": round(job_gb_s(ws, dbytes + abytes, fused_ms) / ws
                                                    / hbm_peak, 4)},
        "step_us_with_event_between_kernels": round((app_ms + dec_ms) * 1e3, 2),
        "roofline": {"bound": "hbm", "kernel": "decode_split_kernel (split-KV with fused last-arriver merge)",
                     "achieved": round(dec_gbs, 2), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(dec_gbs / hbm_peak, 4), "peak_source": peak_src,
                     "algorithmic_bytes": dbytes, "traffic": traffic_bytes("decode_qwen3")},
        "e2e": e2e,
        # our kernels in the headline's timed region: one per step fused, else two
        "gpu_launches": (1 if fused_best else 2) * args.steps,
        "clocks": clocks.summary(),
        "mixed_step": mixed,
        "sliding_step": sliding,
        "grpo_step": grpo,
        "head_dim_512_step": full512,
    }
    if rank == 0:
        line["cpu_baseline"] = None if args.skip_cpu else cpu_baseline(step, ds, rank)
        if not args.skip_cpu:
            try:
                line["cpu_baseline_multicore"] = cpu_baseline_multicore()
            except Exception as e:  # reported, never fatal to the GPU line
                line["cpu_baseline_multicore"] = {"unavailable": f"{type(e).__name__}: {e}"}
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_e2e(ds: DeviceStep, step: wl.Step, stream, flush, args, nbytes, fused=True,
            sm_copy=True):
    """Same step through the public API, inputs from pinned host memory.

    The step's inputs (q, the new K/V rows, block table, lengths; the slot
    mapping too on the two-call path) sit in one pinned host buffer and go
    to the device in one copy, as an engine batches its step metadata; the
    output comes back in one copy.  ``fused``: paged_attn_decode_append
    (one launch), else paged_kv_append then paged_attn_decode.
    ``sm_copy``: both copies by the library's pkv_copy (the SMs), else by
    torch's copy_ (the copy engines)."""
    import torch
    parts = {"q": ds.q_dec, "k_new": ds.k_new, "v_new": ds.v_new, "bt": ds.dec_bt,
             "lens": ds.dec_lens}
    if not fused:
        parts["slots"] = ds.slots
    offs, off = {}, 0
    for k, t in parts.items():
        offs[k] = off
        off += (t.numel() * t.element_size() + 255) // 256 * 256
    host_buf = torch.empty(off, dtype=torch.uint8).pin_memory()
    dev_buf = torch.empty(off, dtype=torch.uint8, device=ds.q_dec.device)

    def view(buf, k):
        t = parts[k]
        n = t.numel() * t.element_size()
        return buf[offs[k]:offs[k] + n].view(t.dtype).view(t.shape)
    for k, t in parts.items():
        view(host_buf, k).copy_(t.cpu())
    dev = {k: view(dev_buf, k) for k in parts}
    out_h = torch.empty(ds.out_dec.shape, dtype=ds.out_dec.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in parts.values())
    d2h = out_h.numel() * out_h.element_size()
    pkv = ds.pkv

    def full(s):
        with torch.cuda.stream(s):
            if sm_copy:
                pkv.pkv_copy(dev_buf, host_buf, stream=s)
            else:
                dev_buf.copy_(host_buf, non_blocking=True)
            if fused:
                pkv.paged_attn_decode_append(ds.out_dec, dev["q"], dev["k_new"], dev["v_new"],
                                             ds.k_cache, ds.v_cache, dev["bt"], dev["lens"],
                                             step.max_seq_len_dec(), step.scale, step.window,
                                             workspace=ds.ws, err_flag=ds.err, stream=s)
            else:
                pkv.paged_kv_append(dev["k_new"], dev["v_new"], ds.k_cache, ds.v_cache,
                                    dev["slots"], err_flag=ds.err, stream=s)
                pkv.paged_attn_decode(ds.out_dec, dev["q"], ds.k_cache, ds.v_cache, dev["bt"],
                                      dev["lens"], step.max_seq_len_dec(), step.scale,
                                      step.window, workspace=ds.ws, err_flag=ds.err, stream=s)
            if sm_copy:
                pkv.pkv_copy(out_h, ds.out_dec, stream=s)
            else:
                out_h.copy_(ds.out_dec, non_blocking=True)

    per = time_steps([full], args.steps, args.warmup, stream, flush, graphs=False)
    ms = float(np.mean([p[0] for p in per]))
    return {"value": round(nbytes / (ms * 1e-3) / 1e9, 2), "unit": "GB/s",
            "ms_per_step": round(ms, 5), "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h),
            "path": (("one H2D copy, paged_attn_decode_append, one D2H copy" if fused else
                      "one H2D copy, paged_kv_append + paged_attn_decode, one D2H copy")
                     + (" (both copies by pkv_copy on the SMs)" if sm_copy else
                        " (both copies by the copy engines)"))}


def run_mixed(args, device, stream, flush, rank):
    """Continuous-batching mixed step: append all new rows, varlen prefill of
    8 chunks, decode of 120 sequences.  Tokens/s = new tokens / step time."""
    import torch
    try:
        step = wl.mixed_step()
        ds = DeviceStep(step, wl.BASE_SEED + 3 + 1000 * rank, device)
        per_step = time_steps([ds.append, ds.varlen, ds.decode], args.steps, args.warmup,
                              stream, flush, phase_events=False)
        per = time_steps([ds.append, ds.varlen, ds.decode], args.steps, args.warmup, stream,
                         flush)
        torch.cuda.synchronize()
        if int(ds.err.item()) != 0:
            return {"unavailable": f"device error flag {int(ds.err.item())}"}
    except Exception as e:  # varlen not available yet, etc.
        return {"unavailable": f"{type(e).__name__}: {e}"}
    ms = float(np.mean([sum(p) for p in per_step]))
    ph = np.mean(np.array(per), axis=0)
    tokens = step.n_new_tokens
    fl = varlen_flops(step)
    hbm_peak, tf_peak, _, src = peaks()
    # the same step with decode and prefill in one launch (paged_attn_mixed)
    try:
        fused_step = time_steps([ds.append, ds.mixed], args.steps, args.warmup, stream, flush,
                                phase_events=False)
        torch.cuda.synchronize()
        if int(ds.err.item()) != 0:
            raise RuntimeError(f"device error flag {int(ds.err.item())}")
        fms = float(np.mean([sum(p) for p in fused_step]))
        fused = {"value": round(tokens / (fms * 1e-3), 1), "unit": "tokens/s",
                 "ms_per_step": round(fms, 5),
                 "traffic": traffic_bytes("mixed_single"),
                 "note": "append, then paged_attn_mixed: decode rows and prefill chunks in one "
                         "persistent launch (split chosen by the library); traffic is the "
                         "mixed kernel's DRAM bytes per launch"}
    except Exception as e:
        fused = {"unavailable": f"{type(e).__name__}: {e}"}
    # ... and with the append in the same launch (paged_attn_mixed_append)
    try:
        app_step = time_steps([ds.mixed_append], args.steps, args.warmup, stream, flush,
                              phase_events=False)
        torch.cuda.synchronize()
        if int(ds.err.item()) != 0:
            raise RuntimeError(f"device error flag {int(ds.err.item())}")
        ams = float(np.mean([sum(p) for p in app_step]))
        fused_app = {"value": round(tokens / (ams * 1e-3), 1), "unit": "tokens/s",
                     "ms_per_step": round(ams, 5),
                     "note": "paged_attn_mixed_append: the step's append, decode rows and "
                             "prefill chunks in one launch (grid barrier after the append)"}
    except Exception as e:
        fused_app = {"unavailable": f"{type(e).__name__}: {e}"}
    # the same step with q/k RMSNorm and the rotary embedding fused into the
    # append (the attention layer's whole input transform)
    try:
        ds.enable_rope()
        rope_step = time_steps([ds.append_rope, ds.varlen, ds.decode], args.steps, args.warmup,
                               stream, flush, phase_events=False)
        rope_per = time_steps([ds.append_rope, ds.varlen, ds.decode], args.steps, args.warmup,
                              stream, flush)
        torch.cuda.synchronize()
        if int(ds.err.item()) != 0:
            raise RuntimeError(f"device error flag {int(ds.err.item())}")
        rms = float(np.mean([sum(p) for p in rope_step]))
        rph = np.mean(np.array(rope_per), axis=0)
        rb = append_rope_bytes(step, tokens)
        with_rope = {
            "value": round(tokens / (rms * 1e-3), 1), "unit": "tokens/s",
            "ms_per_step": round(rms, 5),
            "phase_us": {"append_rope": round(rph[0] * 1e3, 2), "varlen": round(rph[1] * 1e3, 2),
                         "decode": round(rph[2] * 1e3, 2)},
            "append_rope_roofline": {
                "bound": "hbm", "achieved": round(rb / (rph[0] * 1e-3) / 1e9, 2),
                "peak": hbm_peak, "unit": "GB/s",
                "frac": round(rb / (rph[0] * 1e-3) / 1e9 / hbm_peak, 4), "peak_source": src,
                "algorithmic_bytes": int(rb),
                "traffic": traffic_bytes("append_rope_mixed")},
            "note": "q and k RMSNorm + rotary (theta 1e6) over all new tokens fused into the "
                    "append; q transformed in place"}
    except Exception as e:
        with_rope = {"unavailable": f"{type(e).__name__}: {e}"}
    three = round(tokens / (ms * 1e-3), 1)
    # the fastest of the three paths is the step's value
    paths = [(three, round(ms, 5), "append + paged_attn_varlen + paged_attn_decode")]
    if fused.get("value") is not None:
        paths.append((fused["value"], fused["ms_per_step"],
                      "append + paged_attn_mixed (one launch for decode and prefill)"))
    if fused_app.get("value") is not None:
        paths.append((fused_app["value"], fused_app["ms_per_step"],
                      "paged_attn_mixed_append (append, decode and prefill in one launch)"))
    best = max(paths, key=lambda p: p[0])
    return {"metric": "mixed-step tokens/sec",
            "value": best[0],
            "path": best[2],
            "unit": "tokens/s",
            "ms_per_step": best[1],
            "tokens_per_step": int(tokens),
            "workload": "mixed_step: 8 prefill chunks (len ~U[128,1024] on prefix ~U[0,512]) + "
                        "120 decode rows (cached ~U[64,4096]); H 32/8/128, page 16",
            "three_launches": {"value": three, "unit": "tokens/s", "ms_per_step": round(ms, 5)},
            "phase_us": {"append": round(ph[0] * 1e3, 2), "varlen": round(ph[1] * 1e3, 2),
                         "decode": round(ph[2] * 1e3, 2)},
            "varlen_roofline": {"bound": "tensor", "achieved": round(fl / (ph[1] * 1e-3) / 1e12, 2),
                                "peak": tf_peak, "unit": "TFLOP/s",
                                "frac": round(fl / (ph[1] * 1e-3) / 1e12 / tf_peak, 4),
                                "peak_source": src, "algorithmic_flops": fl,
                                "traffic": traffic_bytes("varlen_mixed")},
            "decode_gb_s": round(decode_bytes(step) / (ph[2] * 1e-3) / 1e9, 2),
            "append_gb_s": round(append_bytes(step, tokens) / (ph[0] * 1e-3) / 1e9, 2),
            "append_bytes": int(append_bytes(step, tokens)),
            "append_roofline": {"bound": "hbm",
                                "achieved": round(append_bytes(step, tokens) / (ph[0] * 1e-3) / 1e9, 2),
                                "peak": hbm_peak, "unit": "GB/s",
                                "frac": round(append_bytes(step, tokens) / (ph[0] * 1e-3) / 1e9
                                              / hbm_peak, 4),
                                "peak_source": src, "algorithmic_bytes": int(append_bytes(step, tokens)),
                                "traffic": traffic_bytes("append_mixed"),
                                "note": "the phase between two graph events: the launch is inside"},
            "single_launch": fused,
            "single_launch_append": fused_app,
            "with_rope": with_rope}


def run_sliding(args, device, stream, flush, rank):
    """Sliding-window step (window 512, 8/1 heads, head_dim 256, page 64):
    layer 0 appends its rows, then prefill + decode; layer 1 reads the same
    pool with its own queries (shared KV), without an append."""
    try:
        step = wl.sliding()
        ds = DeviceStep(step, wl.BASE_SEED + 4 + 1000 * rank, device)
        l0 = time_steps([ds.append, ds.varlen, ds.decode], args.steps, args.warmup, stream,
                        flush)
        l1 = time_steps([ds.varlen, ds.decode], args.steps, args.warmup, stream, flush)
        import torch
        torch.cuda.synchronize()
        if int(ds.err.item()) != 0:
            return {"unavailable": f"device error flag {int(ds.err.item())}"}
    except Exception as e:
        return {"unavailable": f"{type(e).__name__}: {e}"}
    p0 = np.mean(np.array(l0), axis=0)
    p1 = np.mean(np.array(l1), axis=0)
    fl = varlen_flops(step)
    db = decode_bytes(step)
    return {"workload": "sliding: window 512, H 8/1/256, page 64; 32 decode rows (cached "
                        "~U[1024,8192]) + 4 prefill chunks of 2048; 2 layers on one pool",
            "layer0_us": {"append": round(p0[0] * 1e3, 2), "varlen": round(p0[1] * 1e3, 2),
                          "decode": round(p0[2] * 1e3, 2)},
            "layer1_us": {"varlen": round(p1[0] * 1e3, 2), "decode": round(p1[1] * 1e3, 2)},
            "varlen_tflops": round(fl / (p0[1] * 1e-3) / 1e12, 2),
            "decode_gb_s": round(db / (p0[2] * 1e-3) / 1e9, 2),
            "decode_bytes": int(db), "varlen_flops": fl,
            "note": "decode K/V (16.8 MB) fits in L2; L2 flushed before every timed step"}


def run_grpo(args, device, stream, flush, rank):
    """GRPO rollout decode step, one layer of 36 in one pool (the last layer's
    page range): append 256 rows, decode 256 sequences whose 256-token prefix
    pages are shared by 4 generations."""
    try:
        nl = max(1, int(getattr(args, "grpo_layers", 36)))
        step = wl.grpo_layer(layers=nl, layer=nl - 1)
        ds = DeviceStep(step, wl.BASE_SEED + 5 + 1000 * rank, device)
        per = time_steps([ds.append, ds.decode], args.steps, args.warmup, stream, flush,
                         phase_events=False)
        per_c = time_steps([ds.append, ds.decode_shared_prefix], args.steps, args.warmup, stream,
                           flush, phase_events=False)
        import torch
        torch.cuda.synchronize()
        if int(ds.err.item()) != 0:
            return {"unavailable": f"device error flag {int(ds.err.item())}"}
        del ds
        torch.cuda.empty_cache()
    except Exception as e:
        return {"unavailable": f"{type(e).__name__}: {e}"}
    ms = float(np.mean([sum(p) for p in per]))
    ms_c = float(np.mean([sum(p) for p in per_c]))
    logical = decode_bytes(step) + append_bytes(step, step.Bd)
    unique = grpo_unique_bytes(step) + append_bytes(step, step.Bd)
    return {"workload": "grpo: 64 prompts x 4 generations, prefix 256 shared, completion "
                        f"~U[0,3840], H 32/8/128, page 16, {nl} layers in one pool "
                        f"({step.num_pages} pages)",
            "layer_step_us": round(ms * 1e3, 2),
            "step_ms_36_layers": round(36 * ms, 3),
            "decode_tokens_per_s": round(step.Bd / (36 * ms * 1e-3), 1),
            "logical_gb_s": round(logical / (ms * 1e-3) / 1e9, 2),
            "logical_bytes_per_layer": int(logical),
            "shared_prefix": {
                "layer_step_us": round(ms_c * 1e3, 2),
                "step_ms_36_layers": round(36 * ms_c, 3),
                "decode_tokens_per_s": round(step.Bd / (36 * ms_c * 1e-3), 1),
                "unique_gb_s": round(unique / (ms_c * 1e-3) / 1e9, 2),
                "unique_bytes_per_layer": int(unique),
                "note": "append + paged_attn_decode_shared_prefix (prefix pass reads each "
                        "prompt's pages once, then the suffix decode with the merge); "
                        "unique bytes count each prompt's prefix once"},
            "note": "one layer timed (append + decode), scaled by 36; logical bytes count "
                    "each generation's shared prefix pages"}


def grpo_unique_bytes(step: wl.Step) -> int:
    """Algorithmic bytes of the cascade decode: each group's shared prefix
    K/V once per group, each member's suffix once, q, out, page ids."""
    L = step.dec_seq_lens.astype(np.int64)
    kvrow = step.H_kv * step.D * 2 * 2
    pl = np.repeat(step.prefix_lens.astype(np.int64), step.group_size)[:step.Bd]
    share = L > pl
    kv = int(np.sum(np.where(share, L - pl, L))) * kvrow
    kv += int(sum(int(step.prefix_lens[j]) for j in range(len(step.prefix_lens))
                  if np.any(share[j * step.group_size:(j + 1) * step.group_size]))) * kvrow
    qo = step.Bd * step.H_q * step.D * 2 * 2
    bt = int(np.sum(-(-L // step.P))) * 4 + step.Bd * 4
    return kv + qo + bt


def run_full512(args, device, stream, flush, rank):
    """Full attention with 512-wide heads (8 q heads on 1 kv head, page 16):
    append, varlen prefill of 4 chunks of 1024, decode of 64 rows over
    1k-8k tokens."""
    try:
        step = wl.full_d512()
        ds = DeviceStep(step, wl.BASE_SEED + 6 + 1000 * rank, device)
        per = time_steps([ds.append, ds.varlen, ds.decode], args.steps, args.warmup, stream,
                         flush)
        import torch
        torch.cuda.synchronize()
        if int(ds.err.item()) != 0:
            return {"unavailable": f"device error flag {int(ds.err.item())}"}
        del ds
        torch.cuda.empty_cache()
    except Exception as e:
        return {"unavailable": f"{type(e).__name__}: {e}"}
    ph = np.mean(np.array(per), axis=0)
    db = decode_bytes(step)
    fl = varlen_flops(step)
    hbm_peak, tf_peak, _, src = peaks()
    gbs = db / (ph[2] * 1e-3) / 1e9
    tfs = fl / (ph[1] * 1e-3) / 1e12
    return {"workload": "full_d512: H 8/1/512, page 16, 64 decode rows cached ~U[1024,8192] "
                        "+ 4 prefill chunks of 1024",
            "append_us": round(ph[0] * 1e3, 2), "varlen_us": round(ph[1] * 1e3, 2),
            "decode_us": round(ph[2] * 1e3, 2),
            "decode_roofline": {"bound": "hbm", "achieved": round(gbs, 2), "peak": hbm_peak,
                                "unit": "GB/s", "frac": round(gbs / hbm_peak, 4),
                                "peak_source": src, "algorithmic_bytes": int(db),
                                "traffic": traffic_bytes("decode_d512")},
            "varlen_roofline": {"bound": "tensor", "achieved": round(tfs, 2), "peak": tf_peak,
                                "unit": "TFLOP/s", "frac": round(tfs / tf_peak, 4),
                                "peak_source": src, "algorithmic_flops": fl,
                                "traffic": traffic_bytes("varlen_d512"),
                                "note": "algorithmic flops count QK^T once; the kernel "
                                        "computes it for each 256-column half of O"}}


# ---------------------------------------------------------- CPU baselines
def oracle_decode_sample(step: wl.Step, vals: wl.StepValues, seqs):
    """Time the oracle (append + decode) on the given sequences."""
    import oracle
    t0 = time.perf_counter()
    slots = step.dec_slots[seqs]
    hk, hv = oracle.kv_append(vals.k_cache, vals.v_cache, vals.k_new[seqs], vals.v_new[seqs],
                              slots)
    oracle.paged_decode(vals.q_dec[0][seqs], hk, hv, step.dec_block_table[seqs],
                        step.dec_seq_lens[seqs], step.scale, step.window)
    return time.perf_counter() - t0


def sample_bytes(step: wl.Step, seqs) -> int:
    L = step.dec_seq_lens[seqs].astype(np.int64)
    return int(L.sum()) * step.H_kv * step.D * 4 + len(seqs) * step.H_q * step.D * 4 + \
        len(seqs) * step.H_kv * step.D * 8


def host_values(step: wl.Step) -> wl.StepValues:
    return wl.fill_values(step, wl.BASE_SEED + 2)


def cpu_baseline(step: wl.Step, ds, rank, budget_s: float = 12.0):
    vals = host_values(step)
    seqs_all = np.arange(step.Bd)
    t = 0.0
    nbytes = 0
    k = 0
    while t < budget_s and k < 50:
        seqs = seqs_all[(k * 8) % step.Bd:(k * 8) % step.Bd + 8]
        t += oracle_decode_sample(step, vals, seqs)
        nbytes += sample_bytes(step, seqs)
        k += 1
    return {"value": round(nbytes / t / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{k} x (append + decode of 8 of the 64 sequences), {t:.1f} s of "
                      f"single-threaded numpy fp64 on host ({os.cpu_count()} cores present)"}


# workers of the multi-core oracle timing (spawned processes: each rebuilds
# the seeded host inputs of the headline workload once, then times the
# oracle on the sequences it is given)
_POOL_STATE = {}


def _pool_init():
    step = wl.qwen3_decode()
    _POOL_STATE["step"] = step
    _POOL_STATE["vals"] = host_values(step)


def _pool_task(seqs):
    return oracle_decode_sample(_POOL_STATE["step"], _POOL_STATE["vals"], np.asarray(seqs))


def cpu_baseline_multicore(steps: int = 3, max_workers: int = 8, timeout_s: float = 240.0):
    """The oracle sample of the headline workload over several host cores:
    the 64 sequences of one step split across a spawn process pool, timed by
    the wall clock after one untimed step (which also waits for every
    worker's inputs).  Each worker holds about 2 GB (the oracle copies both
    pools per call), hence the cap on workers."""
    import concurrent.futures as cf
    import multiprocessing as mp
    import bench as self_module  # the workers resolve the task functions by this name
    step = wl.qwen3_decode()
    n = max(1, min(os.cpu_count() or 1, max_workers, step.Bd))
    chunks = [c.tolist() for c in np.array_split(np.arange(step.Bd), n) if len(c)]
    task = self_module._pool_task
    ex = cf.ProcessPoolExecutor(max_workers=n, mp_context=mp.get_context("spawn"),
                                initializer=self_module._pool_init)
    try:
        for f in [ex.submit(task, c) for c in chunks]:
            f.result(timeout=timeout_s)
        t0 = time.perf_counter()
        for _ in range(steps):
            for f in [ex.submit(task, c) for c in chunks]:
                f.result(timeout=timeout_s)
        wall = time.perf_counter() - t0
    finally:
        ex.shutdown(wait=False, cancel_futures=True)
    nbytes = steps * sample_bytes(step, np.arange(step.Bd))
    return {"value": round(nbytes / wall / 1e9, 4), "unit": "GB/s", "cores": n,
            "kind": "oracle",
            "sample": f"{steps} x (append + decode of all 64 sequences, split over {n} "
                      f"processes), {wall:.1f} s wall ({os.cpu_count()} cores present)"}


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    step = wl.qwen3_decode()
    vals = host_values(step)
    for k in range(args.warmup):
        oracle_decode_sample(step, vals, np.arange(k % 8 * 8, k % 8 * 8 + 8))
    times, nbytes = [], 0
    for k in range(args.steps):
        seqs = np.arange((k * 8) % step.Bd, (k * 8) % step.Bd + 8)
        times.append(oracle_decode_sample(step, vals, seqs))
        nbytes += sample_bytes(step, seqs)
    t = sum(times)
    v = nbytes / t / 1e9
    line = {"metric": METRIC, "value": round(v, 4), "unit": "GB/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * t / args.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": "qwen3_decode (one step = append + decode of 8 of the 64 "
                                   "sequences, fp64 CPU oracle)"},
            "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": "8 sequences per step"},
            "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--skip-cpu", action="store_true",
                    help="omit the CPU oracle baseline (profiling runs)")
    ap.add_argument("--grpo-layers", type=int, default=36,
                    help="layers of the GRPO pool (the timed layer is the last; fewer layers "
                         "keep the same per-layer work in a smaller pool, for profilers)")
    ap.add_argument("--only", choices=["decode", "mixed", "sliding", "grpo", "d512"],
                    default=None,
                    help="run only one section: the headline decode step, the mixed step, "
                         "the sliding-window step, the GRPO step or the head_dim 512 step "
                         "(profiling runs)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
