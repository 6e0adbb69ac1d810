#!/usr/bin/env python3
"""Benchmark of the KDA layer's hot path on GB300: chunked prefill tokens/s and
decode-step HBM GB/s, each against the measured roofline, with the float64 CPU
oracle timed on the host cores beside it.

One step = one chunked prefill of the 4 x 8192-token, 32-head, d = 128 bf16
batch (gate products, chunk-local products, the fp32 state carry, outputs and a
state snapshot every 256 tokens into the block-indexed pool).  The decode step
(512 sequences x 32 heads, one token each, fp32 states updated in place) and the
snapshot gather/restore copies are timed in the same run and reported beside it.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

For N > 1 launch one process per GPU with torch.distributed.run; each rank runs
its own replica (the layer has no cross-device exchange), value = all ranks'
tokens / the slowest rank's time.  Rank 0 prints one JSON line.
"""
import argparse
import csv
import hashlib
import io
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "KDA prefill tokens/s (% bf16 TC peak) and decode-step HBM GB/s (% of 8 TB/s)"
PREFILL_CFG = "prefill_4x8k"
DECODE_CFG = "decode_512x32"

# Algorithmic traffic and work per token-head of the prefill (d_k = d_v = 128,
# chunk 64, snapshot every 256 tokens):
#   bytes: q, k, v bf16 (3 x 256) + alpha fp32 (512) + beta (4) + o bf16 (256)
#          + one 64 KiB fp32 snapshot per 256 tokens (256)            = 1796 B
#   flops: 6 d_k d_v (state products) + C (3 d_k + 2 d_v) (chunk-local) = 139264
PREFILL_BYTES_PER_TH = 3 * 256 + 512 + 4 + 256 + 256
PREFILL_FLOPS_PER_TH = 6 * 128 * 128 + 64 * (3 * 128 + 2 * 128)
CHUNK_RECORD_BYTES = 74240     # one (chunk, head) record between the two prefill stages


def decode_bytes(n, H, d):
    """State read + write (fp32) plus the token's q, k, v (bf16), alpha (fp32),
    beta (fp32) and o (bf16)."""
    return 2 * n * H * d * d * 4 + n * H * (3 * d * 2 + d * 4 + 4 + d * 2)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# ----------------------------------------------------------------------------- clocks

CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a timed region."""

    def __init__(self, device):
        self.proc = None
        self.path = None
        try:
            bus = torch.cuda.get_device_properties(device).pci_bus_id
        except Exception:
            bus = None
        self.sel = ["-i", bus] if bus else []

    def start(self):
        """Start sampling; the caller keeps the GPU busy from here on, so that
        every sample is taken under load."""
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", *self.sel, f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        with open(self.path) as f:
            rows = list(csv.reader(io.StringIO(f.read())))
        os.unlink(self.path)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1].strip().split()[0]))
                smax.append(float(r[2].strip().split()[0]))
            except ValueError:
                continue
            for name, val in zip(names, r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------- helpers

# The sources each prefill kernel is compiled from: its own file and the
# headers it includes.
KERNEL_SOURCES = {
    "chunk_local": ("csrc/chunk_local.cu", "csrc/chunk_common.cuh", "csrc/chunk_decay.cuh", "csrc/kda_common.cuh",
                    "csrc/tc05.cuh"),
    "chunk_recur": ("csrc/chunk_recur.cu", "csrc/chunk_common.cuh", "csrc/kda_common.cuh", "csrc/tc05.cuh"),
}


def _code_only(text: bytes) -> bytes:
    """C/C++ source without its comments and with whitespace collapsed: what a
    change must touch to change the compiled code.  (No source here has a
    comment marker inside a string literal.)"""
    t = re.sub(rb"/\*.*?\*/", b" ", text, flags=re.S)
    t = re.sub(rb"//[^\n]*", b" ", t)
    return b" ".join(t.split())


def kernel_fingerprint(kernel=None):
    """Hash of the code a kernel is built from (of every CUDA source when
    ``kernel`` is None), comments aside, to tie recorded ncu traffic to the code
    it measured."""
    h = hashlib.sha256()
    pkg = os.path.join(ROOT, "hybrid_linear_attention_kda_gb300")
    if kernel is None:
        files = tuple(sorted(os.path.join("csrc", fn) for fn in os.listdir(os.path.join(pkg, "csrc"))))
    else:
        files = KERNEL_SOURCES[kernel]
    for rel in files + ("../include/kda.h",):
        with open(os.path.normpath(os.path.join(pkg, rel)), "rb") as f:
            h.update(os.path.basename(rel).encode() + _code_only(f.read()))
    return h.hexdigest()[:16]


# DRAM bytes per launch of a prefill kernel on this workload from an ncu capture
# (dram__bytes_read.sum + dram__bytes_write.sum), keyed by (kernel, fingerprint
# of its sources); any other fingerprint reports null.  The capture ran 2 x 8192
# tokens x 32 heads (8192 items, 1,236.6 MB); chunk_local's traffic grows with
# the item count, so the 16,384-item workload here moves twice that.
RECORDED_TRAFFIC = {
    ("chunk_local", "63eca31be9c9665c"): 2 * (673_399_808 + 563_152_128),
}


def barrier(dist_on):
    if dist_on:
        torch.distributed.barrier()
    if torch.cuda.is_available():
        torch.cuda.synchronize()


def max_over_ranks(x, dist_on, dev):
    """The largest of every rank's x (all ranks receive it)."""
    if not dist_on:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(units_per_rank, local_ms, world, dist_on, dev):
    """Whole-job throughput of `world` independent replicas: all ranks' units
    over the slowest rank's time (units per second), and that time (ms)."""
    slowest = max_over_ranks(local_ms, dist_on, dev)
    return world * units_per_rank / (slowest / 1e3), slowest


# ----------------------------------------------------------------------------- CPU oracle

def oracle_prefill_sample(data, seconds_target=10.0):
    """Time the float64 oracle on a bounded sample of the prefill workload: the
    first n tokens of every sequence, all heads, n sized for about
    ``seconds_target`` of CPU time.  Returns (tokens/s, cores, sample text, secs)."""
    import oracle
    H = data["q"].shape[1]
    lens = data["seq_lens"]
    n_seq = len(lens)
    cu = [0]
    for L in lens:
        cu.append(cu[-1] + L)

    def run(n_tok):
        idx = torch.cat([torch.arange(cu[s], cu[s] + n_tok) for s in range(n_seq)])
        sub = {key: data[key][idx] for key in ("q", "k", "v", "alpha", "beta")}
        t0 = time.perf_counter()
        oracle.run(sub["q"], sub["k"], sub["v"], sub["alpha"], sub["beta"],
                   [i * n_tok for i in range(n_seq + 1)], want_final=True)
        return time.perf_counter() - t0

    cal = 64
    t_cal = max(run(cal), 1e-3)
    n_tok = int(min(min(lens), max(cal, cal * seconds_target / t_cal)))
    n_tok = max(64, (n_tok // 64) * 64)
    secs = run(n_tok)
    tokens = n_seq * n_tok
    sample = (f"first {n_tok} of {lens[0]} tokens of each of the {n_seq} sequences, all {H} heads "
              f"({tokens} tokens, {secs:.1f} s)")
    return tokens / secs, oracle.threads(), sample, secs


# ----------------------------------------------------------------------------- our arm

def make_pool_table(lens, starts, H, d, dev, extra_slots=0):
    """A pool with one slot per snapshot the batch writes (after ``extra_slots``
    leading slots) and the matching [n, stride] table."""
    n_ord = [(s0 + L) // 256 for s0, L in zip(starts, lens)]
    width = max(1, max(n_ord) if n_ord else 1)
    table = torch.full((len(lens), width), -1, dtype=torch.int32)
    slot = extra_slots
    n_snap = 0
    for i, (s0, m) in enumerate(zip(starts, n_ord)):
        first = s0 // 256
        if m > first:
            table[i, first:m] = torch.arange(slot, slot + m - first, dtype=torch.int32)
            slot += m - first
            n_snap += m - first
    pool = torch.zeros((max(1, slot), H, d, d), dtype=torch.float32, device=dev)
    return pool, table.to(dev), n_snap


def prefill_method_bytes(tokens, H, d, n_snap, n_final, n_init):
    """The method's own HBM traffic for a prefill (no intermediate of any design):
    per token-head q, k, v (bf16), alpha (fp32), beta, o (bf16); every fp32 state
    written (snapshots, final states) or read (initial states)."""
    th = tokens * H
    state = H * d * d * 4
    return th * (3 * d * 2 + d * 4 + 4 + d * 2) + (n_snap + n_final + n_init) * state


def time_prefill(kda, lib, pargs, stream, dev, steps, warm, dist_on, clocks_too=True):
    """CUDA-event time of ``steps`` plain kda_prefill_chunked calls after ``warm``
    untimed ones, with nvidia-smi clocks sampled over the timed region (the same
    step keeps the GPU busy from 0.6 s before to 0.4 s after it).  Returns
    (ms per step, clock record, kernels launched in the timed region)."""
    import ctypes
    pref = ctypes.byref(pargs)
    sh = stream.cuda_stream

    def once():
        st = lib.kda_prefill_chunked(pref, sh)
        if st != 0:
            raise RuntimeError(f"prefill failed: {kda.kda_status_string(st)}: {lib.kda_last_error()}")

    for _ in range(warm):
        once()
    torch.cuda.synchronize(dev)
    assert kda.kda_check_status(stream) == 0

    def soak(seconds):
        t_end = time.perf_counter() + seconds
        while time.perf_counter() < t_end:
            for _ in range(4):
                once()
            torch.cuda.synchronize(dev)

    clocks = ClockSampler(dev) if clocks_too else None
    if clocks:
        clocks.start()
        soak(0.6)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    barrier(dist_on)
    launches0 = kda.kda_launch_count()
    ev0.record(stream)
    for _ in range(steps):
        once()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(dist_on)
    launches = kda.kda_launch_count() - launches0
    clk = None
    if clocks:
        soak(0.4)
        clk = clocks.stop()
        clk["window"] = "0.6 s before to 0.4 s after the timed region, the same step running throughout"
    assert kda.kda_check_status(stream) == 0
    return ev0.elapsed_time(ev1) / steps, clk, launches


def stage_times(kda, pargs, stream, dev, steps):
    """Per-kernel CUDA-event times (ms per step) from a separate pass of the
    instrumented entry point, which records an event before each kernel."""
    n_marks = 12
    marks = [[torch.cuda.Event(enable_timing=True) for _ in range(n_marks)] for _ in range(steps)]
    for evs in marks:
        for e in evs:
            e.record(stream)
    torch.cuda.synchronize(dev)
    recorded = [kda.kda_prefill_chunked_events(pargs, marks[i], stream) for i in range(steps)]
    torch.cuda.synchronize(dev)
    stages = {}
    for rec in recorded:
        for (name, e_a), (_, e_b) in zip(rec[:-1], rec[1:]):
            stages[name] = stages.get(name, 0.0) + e_a.elapsed_time(e_b) / steps
    assert kda.kda_check_status(stream) == 0
    return stages


def roofline_of(stages, method_bytes, peaks, dominant_traffic=None):
    """The dominant kernel's roofline: the method's algorithmic bytes of one
    step (the per-token-head figure times the token-heads one launch covers)
    over that kernel's time, against the measured HBM copy bandwidth."""
    dom_name, dom_ms = max(stages.items(), key=lambda kv: kv[1])
    achieved = method_bytes / (dom_ms / 1e3) / 1e9
    return {"bound": "hbm", "kernel": dom_name, "achieved": achieved, "peak": peaks["hbm_gbs"],
            "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"], "traffic": dominant_traffic,
            "peak_source": peaks["source"] + " (MEASURED_PEAKS hbm_gbs)" if peaks["source"] == "measured"
            else peaks["source"], "algorithmic_bytes_per_launch": method_bytes, "ms_per_launch": dom_ms,
            "bytes_counted": "the method's bytes: q, k, v, alpha, beta, o per token-head and every fp32 "
                             "state snapshot / final state written; no intermediate of this design"}


def bench_extra_workload(name, kda, lib, dev, stream, peaks, steps, warm, dist_on):
    """Tokens/s and roofline fraction of the 2^20-token sequence or the mixed
    varlen batch, inputs drawn on the device (same recipe, float32 draws)."""
    from hybrid_linear_attention_kda_gb300 import inputs
    w = inputs.WORKLOADS[name]
    H, d = w["H"], w["d"]
    if name == "long_1m":
        data = inputs.gen_prefill_device([w["T"]], H, d, d, w["seed"], dev)
        starts, lens = [0], [w["T"]]
        init_slot = None
        pool, table, n_snap = make_pool_table(lens, starts, H, d, dev)
        n_init = 0
        desc = (f"long_1m: 1 sequence x {w['T']} tokens, H={H}, d_k=d_v={d}, bf16 q/k/v/o, fp32 gates/state, "
                "snapshot every 256 tokens (4096 per head), zero initial state")
    else:
        data = inputs.gen_varlen_resume_device(w["n_seqs"], H, d, d, w["max_len"], w["prefix_len"],
                                               w["n_resume"], w["seed"], dev)
        lens_full = data["lens"]
        starts = data["start_pos"].tolist()
        lens = [L - s0 for L, s0 in zip(lens_full, starts)]
        n_pref = w["prefix_len"] // 256
        pool, table, n_snap = make_pool_table(lens, starts, H, d, dev, extra_slots=n_pref)
        # the shared prefix's snapshots fill slots [0, n_pref) first (not timed)
        pr = data["prefix"]
        ptab = torch.arange(n_pref, dtype=torch.int32, device=dev)[None]
        kda.prefill(pr["q"], pr["k"], pr["v"], pr["alpha"], pr["beta"], pr["cu_seqlens_dev"],
                    total_tokens=w["prefix_len"], pool=pool, snap_table=ptab, want_final=False)
        init_slot = torch.tensor([(p // 256 - 1) if p > 0 else -1 for p in starts], dtype=torch.int32,
                                 device=dev)
        n_init = sum(1 for p in starts if p > 0)
        desc = (f"varlen_64: {w['n_seqs']} sequences, lengths uniform in [1, {w['max_len']}], "
                f"{w['n_resume']} resumed from a shared {w['prefix_len']}-token prefix's snapshots, H={H}, "
                f"d_k=d_v={d}, bf16 q/k/v/o, fp32 gates/state, snapshot every 256 tokens")
    total = int(data["cu_seqlens"][-1])
    n = len(lens)
    o = torch.empty((total, H, d), dtype=torch.bfloat16, device=dev)
    fin = torch.empty((n, H, d, d), dtype=torch.float32, device=dev)
    sp = torch.tensor(starts, dtype=torch.int32, device=dev)
    pargs = kda.make_prefill_args(data["q"], data["k"], data["v"], data["alpha"], data["beta"],
                                  data["cu_seqlens_dev"], total, o, start_pos=sp, init_slot=init_slot,
                                  pool=pool, snap_table=table, final_state=fin)
    need = kda.kda_prefill_workspace_size(pargs)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    pargs.workspace, pargs.workspace_bytes = ws.data_ptr(), need
    ms, clk, launches = time_prefill(kda, lib, pargs, stream, dev, steps, warm, dist_on)
    stages = stage_times(kda, pargs, stream, dev, min(steps, 3))
    mb = prefill_method_bytes(total, H, d, n_snap, n, n_init)
    out = {"workload": desc, "value": total / (ms / 1e3), "unit": "tokens/s", "ms_per_step": ms,
           "steps": steps, "tokens_per_step": total, "gpu_launches": launches,
           "roofline": roofline_of(stages, mb, peaks),
           "path": {"achieved_gbs": mb / (ms / 1e3) / 1e9, "frac_of_hbm": mb / (ms / 1e3) / 1e9 / peaks["hbm_gbs"],
                    "algorithmic_bytes_per_step": mb},
           "stage_ms": stages, "clocks": clk,
           "l2": f"inputs larger than L2: {mb / 1e9:.2f} GB of algorithmic traffic per step",
           "data": "synthetic, drawn on the device (seeded torch generator, float32 draws, same recipe)"}
    del data, o, fin, pool, ws
    torch.cuda.empty_cache()
    return out


def bench_ours(args, rank, world, dev, dist_on):
    import hybrid_linear_attention_kda_gb300 as kda
    from hybrid_linear_attention_kda_gb300 import inputs

    lib = kda.load()
    peaks = load_peaks()
    w = inputs.WORKLOADS[PREFILL_CFG]
    n, H, d, T = w["n_seqs"], w["H"], w["d"], w["T"]
    host = inputs.gen_prefill([T] * n, H, d, d, w["seed"] + 1000 * rank, pin=True)
    x = {key: host[key].to(dev) for key in ("q", "k", "v", "alpha", "beta", "cu_seqlens")}
    total = n * T
    n_ord = T // 256
    pool = torch.zeros((n * n_ord, H, d, d), dtype=torch.float32, device=dev)
    table = torch.arange(n * n_ord, dtype=torch.int32, device=dev).view(n, n_ord)
    o = torch.empty((total, H, d), dtype=torch.bfloat16, device=dev)
    fin = torch.empty((n, H, d, d), dtype=torch.float32, device=dev)
    pargs = kda.make_prefill_args(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["cu_seqlens"],
                                  total, o, pool=pool, snap_table=table, final_state=fin)
    need = kda.kda_prefill_workspace_size(pargs)
    ws = None
    if need:
        ws = torch.empty(need, dtype=torch.uint8, device=dev)
        pargs.workspace, pargs.workspace_bytes = ws.data_ptr(), need
    stream = torch.cuda.current_stream(dev)
    import ctypes
    pref = ctypes.byref(pargs)

    def prefill_once():
        st = lib.kda_prefill_chunked(pref, stream.cuda_stream)
        if st != 0:
            raise RuntimeError(f"prefill failed: {kda.kda_status_string(st)}: {lib.kda_last_error()}")

    warm = max(3, args.warmup)
    # ---- device-resident timed region: the plain entry point, K steps
    ms_per_step, clk, launches = time_prefill(kda, lib, pargs, stream, dev, args.steps, warm, dist_on)
    value, total_ms = replica_throughput(total * args.steps, ms_per_step * args.steps, world, dist_on, dev)
    ms_per_step = total_ms / args.steps
    # ---- per-kernel times from a separate pass of the instrumented entry point
    stages = stage_times(kda, pargs, stream, dev, args.steps)
    th = total * H
    method_bytes = th * PREFILL_BYTES_PER_TH                     # 1796 B per token-head
    path_bytes = method_bytes + n * H * d * d * 4                # + the final states
    alg_flops = th * PREFILL_FLOPS_PER_TH
    dom_name = max(stages.items(), key=lambda kv: kv[1])[0]
    traffic = RECORDED_TRAFFIC.get((dom_name, kernel_fingerprint(dom_name))) if dom_name in KERNEL_SOURCES else None
    roofline = roofline_of(stages, method_bytes, peaks, traffic)
    # the same bytes split by the kernel that must move them, and this design's
    # own intermediate (the per-(chunk, head) records) reported apart
    n_items = (T // 64) * n * H
    per_kernel = {}
    if "chunk_local" in stages:
        b = th * (3 * 256 + 512 + 4)
        per_kernel["chunk_local"] = {"method_bytes": b, "ms": stages["chunk_local"],
                                     "frac_of_hbm": b / (stages["chunk_local"] / 1e3) / 1e9 / peaks["hbm_gbs"],
                                     "counts": "q, k, v, alpha, beta"}
    if "chunk_recur" in stages:
        b = th * (256 + 256) + n * H * d * d * 4
        per_kernel["chunk_recur"] = {"method_bytes": b, "ms": stages["chunk_recur"],
                                     "frac_of_hbm": b / (stages["chunk_recur"] / 1e3) / 1e9 / peaks["hbm_gbs"],
                                     "counts": "o, snapshots, final states"}
    roofline["per_kernel"] = per_kernel
    roofline["design_overhead_bytes_per_step"] = {
        "value": 2 * n_items * CHUNK_RECORD_BYTES if "chunk_local" in stages else 0,
        "what": "per-(chunk, head) records written by the chunk-local stage and read back by the carry"}
    path = {"achieved_gbs": path_bytes / (ms_per_step / 1e3) / 1e9,
            "frac_of_hbm": path_bytes / (ms_per_step / 1e3) / 1e9 / peaks["hbm_gbs"],
            "algorithmic_bytes_per_step": path_bytes,
            "bytes_counted": "1796 B per token-head (q, k, v, alpha, beta, o, snapshot share) + final states"}
    tensor = {"achieved_tflops": alg_flops / (ms_per_step / 1e3) / 1e12,
              "peak_tflops": peaks["bf16_tflops"],
              "frac": alg_flops / (ms_per_step / 1e3) / 1e12 / peaks["bf16_tflops"],
              "algorithmic_flops_per_step": alg_flops}
    fp = kernel_fingerprint()

    # ---- end to end through the C ABI from pinned host buffers
    o_host = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
    fin_host = torch.empty(fin.shape, dtype=fin.dtype, pin_memory=True)
    h2d = sum(host[key].numel() * host[key].element_size()
              for key in ("q", "k", "v", "alpha", "beta", "cu_seqlens"))
    d2h = o_host.numel() * o_host.element_size() + fin_host.numel() * fin_host.element_size()

    def e2e_once():
        for key in ("q", "k", "v", "alpha", "beta", "cu_seqlens"):
            x[key].copy_(host[key], non_blocking=True)
        prefill_once()
        o_host.copy_(o, non_blocking=True)
        fin_host.copy_(fin, non_blocking=True)

    e2e_steps = max(3, min(args.steps, 10))
    for _ in range(2):
        e2e_once()
    barrier(dist_on)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_once()
    e1.record(stream)
    barrier(dist_on)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), dist_on, dev)
    e2e_serial = world * total * e2e_steps / (e2e_ms / 1e3)

    # the same, pipelined per sequence over three streams: the inputs of
    # sequence g+1 travel while sequence g is prefilled, and results travel
    # back while the next step's inputs come in (host->device runs at about
    # 210 GB/s and is the bound; the two directions overlap)
    s_in, s_comp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    cu_host = [torch.tensor([0, T], dtype=torch.int32).pin_memory() for _ in range(n)]
    cu_dev = [torch.empty(2, dtype=torch.int32, device=dev) for _ in range(n)]
    gargs = []
    for g in range(n):
        sl = slice(g * T, (g + 1) * T)
        ga = kda.make_prefill_args(x["q"][sl], x["k"][sl], x["v"][sl], x["alpha"][sl], x["beta"][sl], cu_dev[g],
                                   T, o[sl], pool=pool, snap_table=table[g:g + 1], final_state=fin[g:g + 1],
                                   workspace=ws)
        gargs.append(ga)
    ev_in = [torch.cuda.Event() for _ in range(n)]
    ev_comp = [torch.cuda.Event() for _ in range(n)]
    started = [False] * n

    def e2e_pipelined():
        for g in range(n):
            sl = slice(g * T, (g + 1) * T)
            if started[g]:
                s_in.wait_event(ev_comp[g])          # the previous step no longer reads these inputs
            with torch.cuda.stream(s_in):
                for key in ("q", "k", "v", "alpha", "beta"):
                    x[key][sl].copy_(host[key][sl], non_blocking=True)
                cu_dev[g].copy_(cu_host[g], non_blocking=True)
            ev_in[g].record(s_in)
            s_comp.wait_event(ev_in[g])
            st = lib.kda_prefill_chunked(ctypes.byref(gargs[g]), s_comp.cuda_stream)
            if st != 0:
                raise RuntimeError(f"prefill failed: {kda.kda_status_string(st)}")
            ev_comp[g].record(s_comp)
            started[g] = True
            s_out.wait_event(ev_comp[g])
            with torch.cuda.stream(s_out):
                o_host[sl].copy_(o[sl], non_blocking=True)
                fin_host[g:g + 1].copy_(fin[g:g + 1], non_blocking=True)

    for _ in range(2):
        e2e_pipelined()
    torch.cuda.synchronize(dev)
    barrier(dist_on)
    e0.record(s_in)
    for _ in range(e2e_steps):
        e2e_pipelined()
    s_in.wait_stream(s_comp)
    s_in.wait_stream(s_out)
    e1.record(s_in)
    torch.cuda.synchronize(dev)
    barrier(dist_on)
    e2e_pipe_ms = max_over_ranks(e0.elapsed_time(e1), dist_on, dev)
    assert kda.kda_check_status(stream) == 0
    e2e = {"value": world * total * e2e_steps / (e2e_pipe_ms / 1e3), "unit": "tokens/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "how": "per-sequence pipeline over three streams: host->device copy, prefill, device->host copy",
           "serial_value": e2e_serial,
           "h2d_gbs_floor_note": "host->device copies measured at about 210 GB/s bound this figure"}
    del x, o, pool, ws

    # ---- decode step, 512 x 32 heads, states updated in place
    dw = inputs.WORKLOADS[DECODE_CFG]
    dn, dH, dd = dw["n_seqs"], dw["H"], dw["d"]
    dpool = inputs.gen_states(dn, dH, dd, dd, dw["seed"], std=dw["state_std"]).to(dev)
    dslots = torch.arange(dn, dtype=torch.int32, device=dev)
    n_sets = 8                     # rotate inputs so they do not sit in L2 between steps
    dins = [{k_: t.to(dev) for k_, t in inputs.gen_decode(dn, dH, dd, dd, dw["seed"], s).items()}
            for s in range(n_sets)]
    do = torch.empty((dn, dH, dd), dtype=torch.bfloat16, device=dev)

    def decode_once(i):
        z = dins[i % n_sets]
        kda.kda_decode_step(z["q"], z["k"], z["v"], z["alpha"], z["beta"], dpool, dslots, do,
                            stream=stream)

    for i in range(warm):
        decode_once(i)
    barrier(dist_on)
    d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    d_launch0 = kda.kda_launch_count()
    d0.record(stream)
    for i in range(args.steps):
        decode_once(i)
    d1.record(stream)
    barrier(dist_on)
    d_launches = kda.kda_launch_count() - d_launch0
    dec_ms = max_over_ranks(d0.elapsed_time(d1), dist_on, dev) / args.steps
    dbytes = decode_bytes(dn, dH, dd)
    dec_gbs = dbytes / (dec_ms / 1e3) / 1e9
    assert kda.kda_check_status(stream) == 0

    # decode end to end: per step copy the token's inputs in and the outputs out
    dhost = [{k_: t.pin_memory() for k_, t in inputs.gen_decode(dn, dH, dd, dd, dw["seed"], s).items()}
             for s in range(2)]
    do_host = torch.empty(do.shape, dtype=do.dtype, pin_memory=True)
    d_h2d = sum(t.numel() * t.element_size() for t in dhost[0].values())
    d_d2h = do_host.numel() * do_host.element_size()
    z = dins[0]

    def decode_e2e(i):
        for k_, t in dhost[i % 2].items():
            z[k_].copy_(t, non_blocking=True)
        decode_once(0)
        do_host.copy_(do, non_blocking=True)

    for i in range(2):
        decode_e2e(i)
    barrier(dist_on)
    d0.record(stream)
    for i in range(args.steps):
        decode_e2e(i)
    d1.record(stream)
    barrier(dist_on)
    dec_e2e_ms = max_over_ranks(d0.elapsed_time(d1), dist_on, dev) / args.steps

    # ---- speculative decoding: 8 candidates per sequence verified, 5 accepted
    # (the pages' low-entropy average is 4.73 accepted tokens per step)
    sT, s_acc = 8, 5
    sins = [{k_: t.to(dev).reshape((dn, sT) + tuple(t.shape[1:]))
             for k_, t in inputs.gen_decode(dn * sT, dH, dd, dd, dw["seed"], 200 + s).items()} for s in range(2)]
    so = torch.empty((dn, sT, dH, dd), dtype=torch.bfloat16, device=dev)
    su = torch.empty((dn, sT, dH, dd), dtype=torch.float32, device=dev)
    sacc = torch.full((dn,), s_acc, dtype=torch.int32, device=dev)

    def spec_once(i, part):
        z = sins[i % 2]
        if part in ("verify", "both"):
            kda.kda_decode_verify(z["q"], z["k"], z["v"], z["alpha"], z["beta"], dpool, dslots, so, su,
                                  stream=stream)
        if part in ("commit", "both"):
            kda.kda_decode_commit(z["k"], z["alpha"], su, sacc, dpool, dslots, stream=stream)

    spec_ms = {}
    for part in ("verify", "commit", "both"):
        for i in range(warm):
            spec_once(i, part)
        barrier(dist_on)
        d0.record(stream)
        for i in range(args.steps):
            spec_once(i, part)
        d1.record(stream)
        barrier(dist_on)
        spec_ms[part] = max_over_ranks(d0.elapsed_time(d1), dist_on, dev) / args.steps
    assert kda.kda_check_status(stream) == 0
    st_bytes = dn * dH * dd * dd * 4
    tok_in = dn * sT * dH * (3 * dd * 2 + dd * 4 + 4)          # q, k, v bf16, alpha, beta
    ver_bytes = st_bytes + tok_in + dn * sT * dH * dd * (2 + 4)  # + o bf16, u fp32
    com_bytes = 2 * st_bytes + dn * s_acc * dH * dd * (2 + 4 + 4)  # + k, alpha, u of accepted tokens
    spec = {"workload": f"{dn} sequences x {dH} heads, d={dd}, {sT} candidate tokens verified and "
                        f"{s_acc} accepted per step",
            "value": dn * s_acc / (spec_ms["both"] / 1e3), "unit": "accepted tokens/s",
            "ms_per_step": spec_ms["both"], "verify_ms": spec_ms["verify"], "commit_ms": spec_ms["commit"],
            "verify_gbs": ver_bytes / (spec_ms["verify"] / 1e3) / 1e9,
            "commit_gbs": com_bytes / (spec_ms["commit"] / 1e3) / 1e9,
            "state_bytes_per_accepted_token": 3 * dd * dd * 4 / s_acc,
            "decode_state_bytes_per_token": 2 * dd * dd * 4}

    # ---- fused decode step: convolution, q/k norm, gates, update, gated RMSNorm
    fconv_w, fnorm_w = (t.to(dev) for t in inputs.gen_fused_params(dH, dd, dw["seed"]))
    fcpool = inputs.gen_conv_states(dn, dH, dd, dw["seed"]).to(dev)
    fins = [{k_: t.to(dev) for k_, t in inputs.gen_fused_step(dn, dH, dd, dw["seed"], 300 + s).items()}
            for s in range(4)]
    fy = torch.empty((dn, dH, dd), dtype=torch.bfloat16, device=dev)

    def fused_once(i):
        z = fins[i % 4]
        kda.decode_fused(z["xq"], z["xk"], z["xv"], z["a"], z["b"], z["g"], fconv_w, fnorm_w, dpool, fcpool,
                         dslots, fy, stream=stream)

    for i in range(warm):
        fused_once(i)
    barrier(dist_on)
    d0.record(stream)
    for i in range(args.steps):
        fused_once(i)
    d1.record(stream)
    barrier(dist_on)
    fused_ms = max_over_ranks(d0.elapsed_time(d1), dist_on, dev) / args.steps
    assert kda.kda_check_status(stream) == 0
    fbytes = (2 * dn * dH * dd * dd * 4                   # recurrent state read + write
              + 2 * dn * dH * 3 * 3 * dd * 2              # convolution state read + write
              + dn * dH * (5 * dd * 2 + 2)                # xq, xk, xv, a, g, b (bf16)
              + dn * dH * dd * 2                          # y (bf16)
              + dH * (3 * 4 * dd + dd) * 4)               # convolution taps and norm weight
    fused = {"workload": f"{dn} sequences x {dH} heads, d={dd}: causal convolution (width 4) with its state, "
                         "q/k L2 norm, gates, update, gated RMSNorm in one kernel",
             "value": fbytes / (fused_ms / 1e3) / 1e9, "unit": "GB/s", "ms_per_step": fused_ms,
             "frac_of_hbm": fbytes / (fused_ms / 1e3) / 1e9 / peaks["hbm_gbs"],
             "algorithmic_bytes_per_launch": fbytes}

    # ---- snapshot gather + restore of 128 states (64 KiB each)
    gsl = torch.arange(0, 2 * 128, 2, dtype=torch.int32, device=dev) % dn
    gbuf = torch.empty((128, dH, dd, dd), dtype=torch.float32, device=dev)
    rsl = torch.arange(1, 2 * 128, 2, dtype=torch.int32, device=dev) % dn
    for _ in range(2):
        kda.kda_snapshot_gather(dpool, gsl, gbuf, stream=stream)
        kda.kda_snapshot_restore(gbuf, dpool, rsl, stream=stream)
    barrier(dist_on)
    d0.record(stream)
    for _ in range(args.steps):
        kda.kda_snapshot_gather(dpool, gsl, gbuf, stream=stream)
        kda.kda_snapshot_restore(gbuf, dpool, rsl, stream=stream)
    d1.record(stream)
    barrier(dist_on)
    copy_ms = max_over_ranks(d0.elapsed_time(d1), dist_on, dev) / args.steps
    copy_bytes = 2 * 2 * gbuf.numel() * 4
    assert kda.kda_check_status(stream) == 0

    # ---- the long-context sequence and the mixed varlen batch, timed the same way
    extra = {}
    if not args.no_extra:
        del dpool, dins, sins, fins, fcpool, gbuf
        torch.cuda.empty_cache()
        for name in ("long_1m", "varlen_64"):
            extra[name] = bench_extra_workload(name, kda, lib, dev, stream, peaks, max(3, min(args.steps, 10)),
                                               warm, dist_on)

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": warm, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; q,k L2-normalised N(0,1), v N(0,1), alpha=exp(-softplus(N(0,1)+2)), beta=sigmoid(N(0,1)))",
        "config": prefill_config(world),
        "roofline": roofline,
        "path": path,
        "tensor": tensor,
        "stage_ms": stages,
        "e2e": e2e,
        "clocks": clk,
        "gpu_launches": launches,
        "decode": {"workload": f"{DECODE_CFG}: {dn} sequences x {dH} heads, d={dd}, one token each, "
                               "fp32 states N(0,0.05^2) updated in place in the pool",
                   "value": world * dec_gbs, "unit": "GB/s", "ms_per_step": dec_ms,
                   "frac_of_8tbs": dec_gbs / 8000.0,
                   "roofline": {"bound": "hbm", "achieved": dec_gbs, "peak": peaks["hbm_gbs"],
                                "unit": "GB/s", "frac": dec_gbs / peaks["hbm_gbs"],
                                "algorithmic_bytes_per_launch": dbytes},
                   "gpu_launches": d_launches,
                   "e2e": {"value": world * dbytes / (dec_e2e_ms / 1e3) / 1e9, "unit": "GB/s",
                           "ms_per_step": dec_e2e_ms, "h2d_bytes_per_step": d_h2d,
                           "d2h_bytes_per_step": d_d2h}},
        "fused_decode": fused,
        "speculative_decode": spec,
        "snapshot_copy": {"value": copy_bytes / (copy_ms / 1e3) / 1e9, "unit": "GB/s",
                          "ms_per_step": copy_ms, "states": 128},
        "kernel_fingerprint": fp,
    }
    line.update(extra)
    if rank == 0:
        line["prefix_cache"] = bench_prefix_cache()
    if world == 1 and rank == 0 and not args.no_cpu_baseline:
        tps, cores, sample, _ = oracle_prefill_sample(host, args.cpu_seconds)
        line["cpu_baseline"] = {"value": tps, "unit": "tokens/s", "cores": cores,
                                "kind": "oracle", "sample": sample}
    return line


def bench_prefix_cache(n_req=2000, seed=20266):
    """Host prefix-cache index on a synthetic serving stream: 16 system prompts of
    2K-8K tokens, each request one of them plus a 100-2000-token question, one
    step per 8 requests, second-hit admission, 32K-token interval retention."""
    import numpy as np
    from hybrid_linear_attention_kda_gb300.prefix_cache import PrefixCache
    rng = np.random.default_rng(seed)
    sys_prompts = [rng.integers(0, 163840, size=int(rng.integers(2048, 8192)), dtype=np.int32) for _ in range(16)]
    reqs = [np.concatenate([sys_prompts[int(rng.integers(0, 16))],
                            rng.integers(0, 163840, size=int(rng.integers(100, 2000)), dtype=np.int32)])
            for _ in range(n_req)]
    pc = PrefixCache(4096, retention_interval=32768, admit_on_second_hit=True)
    row = np.full(64, -1, dtype=np.int32)
    tokens = reused = 0
    t0 = time.perf_counter()
    ids = []
    for i, r in enumerate(reqs):
        p = pc.plan_request(r, snap_row=row)
        ids.append(p["request_id"])
        tokens += len(r)
        reused += p["start_pos"]
        if i % 8 == 7:
            pc.end_step(True)
            for rid in ids:
                pc.release(rid)
            ids = []
    dt = time.perf_counter() - t0
    st = pc.stats()
    return {"workload": f"{n_req} requests over 16 shared system prompts (2K-8K tokens) + 100-2000-token "
                        "questions, 8 per step, second-hit admission, 32K interval",
            "value": n_req / dt, "unit": "plans/s", "us_per_plan": dt / n_req * 1e6,
            "prompt_tokens_per_s": tokens / dt, "hit_rate": st["hits"] / max(1, st["requests"]),
            "prompt_tokens_reused": reused / max(1, tokens), "host": "1 thread"}


def prefill_config(world):
    """The prefill workload as both arms name it in their JSON lines."""
    from hybrid_linear_attention_kda_gb300 import inputs
    w = inputs.WORKLOADS[PREFILL_CFG]
    n, T, H, d = w["n_seqs"], w["T"], w["H"], w["d"]
    path_bytes = n * T * H * PREFILL_BYTES_PER_TH + n * H * d * d * 4
    return {"workload": f"{PREFILL_CFG}: {n} sequences x {T} tokens, H={H}, d_k=d_v={d}, "
                        "bf16 q/k/v/o, fp32 alpha/beta/state, chunk 64, snapshot every 256 "
                        "tokens into a block-indexed pool, zero initial state",
            "l2": f"inputs larger than L2: {path_bytes / 1e9:.2f} GB of algorithmic traffic per step",
            "parallelism": f"replicas x{world}"}


# ----------------------------------------------------------------------------- reference arm

def bench_reference(args, world=1):
    """The float64 oracle as it stands, on the host cores: each step a bounded
    sample of the prefill workload.  Under a launch of ``world`` ranks only rank
    0 runs it; its line names the same configuration as the GPU arm's."""
    from hybrid_linear_attention_kda_gb300 import inputs
    w = inputs.WORKLOADS[PREFILL_CFG]
    host = inputs.gen_prefill([w["T"]] * w["n_seqs"], w["H"], w["d"], w["d"], w["seed"])
    budget = max(2.0, 150.0 / (args.steps + max(3, args.warmup)))
    times, toks = [], 0
    warm = max(3, args.warmup)
    sample = None
    cores = None
    for i in range(warm + args.steps):
        tps, cores, sample, secs = oracle_prefill_sample(host, budget)
        if i >= warm:
            times.append(secs)
            toks += tps * secs
    value = toks / sum(times)
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": 1, "steps": args.steps, "warmup": warm,
            "ms_per_step": 1e3 * sum(times) / len(times), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": prefill_config(world),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def run_case(args):
    """One small case for profilers (ncu captures): ``--case prefill`` runs
    ``--reps`` chunked prefills of ``--seqs`` x ``--len`` tokens, ``--heads``
    heads, d = ``--dim``, after one warm-up; ``--case decode`` runs decode steps
    of ``--seqs`` x ``--heads`` states.  Prints the CUDA-event median (not a
    bench value when run under a profiler)."""
    import hybrid_linear_attention_kda_gb300 as kda
    from hybrid_linear_attention_kda_gb300 import inputs
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    kda.load()
    H, d = args.heads, args.dim
    dt = torch.bfloat16 if args.dtype == "bf16" else torch.float32
    times = []
    if args.case == "prefill":
        lens = [args.len] * args.seqs
        data = inputs.gen_prefill_device(lens, H, d, d, 20261, dev, dtype=dt, decay=args.decay)
        pool, table, _ = make_pool_table(lens, [0] * len(lens), H, d, dev)
        fin = torch.empty((len(lens), H, d, d), device=dev)
        o = torch.empty((sum(lens), H, d), dtype=dt, device=dev)
        pargs = kda.make_prefill_args(data["q"], data["k"], data["v"], data["alpha"], data["beta"],
                                      data["cu_seqlens_dev"], sum(lens), o, pool=pool, snap_table=table,
                                      final_state=fin)
        need = kda.kda_prefill_workspace_size(pargs)
        ws = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
        pargs.workspace, pargs.workspace_bytes = ws.data_ptr(), need
        fn = lambda: kda.kda_prefill_chunked(pargs)  # noqa: E731
        fn()
    else:
        pool = inputs.gen_states(args.seqs, H, d, d, 20263).to(dev)
        slots = torch.arange(args.seqs, dtype=torch.int32, device=dev)
        z = {k_: t.to(dev) for k_, t in inputs.gen_decode(args.seqs, H, d, d, 20263, 0, dtype=dt).items()}
        o = torch.empty((args.seqs, H, d), dtype=dt, device=dev)
        fn = lambda: kda.kda_decode_step(z["q"], z["k"], z["v"], z["alpha"], z["beta"], pool, slots, o)  # noqa: E731
        fn()
    torch.cuda.synchronize()
    for _ in range(args.reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b))
    assert kda.kda_check_status() == 0
    print(json.dumps({"case": args.case, "seqs": args.seqs, "len": args.len, "heads": H, "dim": d,
                      "dtype": args.dtype, "median_ms": statistics.median(times)}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the 2^20-token and mixed varlen prefill workloads")
    ap.add_argument("--case", choices=["prefill", "decode"], default=None,
                    help="run one small case for a profiler instead of the benchmark")
    ap.add_argument("--seqs", type=int, default=2)
    ap.add_argument("--len", type=int, default=8192)
    ap.add_argument("--heads", type=int, default=32)
    ap.add_argument("--dim", type=int, default=128)
    ap.add_argument("--dtype", choices=["bf16", "fp32"], default="bf16")
    ap.add_argument("--decay", choices=["config", "mild"], default="config")
    ap.add_argument("--reps", type=int, default=2)
    args = ap.parse_args()
    if args.case:
        run_case(args)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.gpus != world and world == 1 and args.gpus > 1:
        sys.exit("for --gpus > 1 launch one process per GPU with torch.distributed.run")

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(bench_reference(args, world)), flush=True)
        return

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist_on = world > 1
    if dist_on:
        torch.distributed.init_process_group("nccl", device_id=dev)
    line = bench_ours(args, rank, world, dev, dist_on)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist_on:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
