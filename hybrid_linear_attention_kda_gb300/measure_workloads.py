"""Time the five KDA workloads on cuda:0 through the C ABI, each beside the
float64 CPU oracle on a bounded sample of the same workload, and print one JSON
line per workload plus a markdown table.

    python -m hybrid_linear_attention_kda_gb300.measure_workloads [--reps 5] [--oracle-seconds 5]

GPU times are CUDA-event times on the launching stream after warm-up; every
workload's inputs except the tiny one are larger than L2.  The oracle is test
infrastructure and is only timed here, as a baseline.
"""
import argparse
import json
import statistics
import time

import torch

import hybrid_linear_attention_kda_gb300 as kda
from hybrid_linear_attention_kda_gb300 import inputs


def _time_gpu(fn, reps, warm=3):
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    times = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b))
    if kda.kda_check_status() != 0:
        raise RuntimeError("device status set")
    return statistics.median(times)


def _oracle_tokens_per_s(data, seconds):
    """Oracle on the first n tokens of every sequence (all heads), n sized for
    about `seconds`; returns (tokens/s, threads, description)."""
    import oracle
    lens = data["seq_lens"]
    cu = [0]
    for L in lens:
        cu.append(cu[-1] + L)

    def run(n_tok):
        ns = [min(n_tok, L) for L in lens]
        idx = torch.cat([torch.arange(cu[s], cu[s] + ns[s]) for s in range(len(lens))])
        sub = {k: data[k][idx] for k in ("q", "k", "v", "alpha", "beta")}
        cus = [0]
        for x in ns:
            cus.append(cus[-1] + x)
        t0 = time.perf_counter()
        oracle.run(sub["q"], sub["k"], sub["v"], sub["alpha"], sub["beta"], cus)
        return time.perf_counter() - t0, sum(ns)

    t_cal, _ = run(64)
    n_tok = int(max(64, min(max(lens), 64 * seconds / max(t_cal, 1e-3))))
    secs, toks = run(n_tok)
    return toks / secs, oracle.threads(), f"first {n_tok} tokens of each sequence ({toks} tokens, {secs:.1f} s)"


def _prefill_case(name, data, dev, reps, oracle_seconds, dtype_name, extra=None, start_pos=None):
    x = {k: data[k].to(dev) for k in ("q", "k", "v", "alpha", "beta", "cu_seqlens")}
    T, H, d = data["q"].shape
    lens = data["seq_lens"]
    starts = [0] * len(lens) if start_pos is None else [int(p) for p in start_pos]
    n_ord = [(s0 + L) // 256 for s0, L in zip(starts, lens)]
    table = torch.full((len(lens), max(1, max(n_ord))), -1, dtype=torch.int32)
    slot = 0
    for s, m in enumerate(n_ord):
        table[s, :m] = torch.arange(slot, slot + m, dtype=torch.int32)
        slot += m
    pool = torch.zeros((max(1, slot), H, d, d), device=dev)
    table = table.to(dev)
    o = torch.empty((T, H, d), dtype=data["v"].dtype, device=dev)
    fin = torch.empty((len(lens), H, d, d), device=dev)
    ws = {}

    sp = None if start_pos is None else torch.tensor(starts, dtype=torch.int32, device=dev)

    def call():
        out = kda.prefill(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["cu_seqlens"],
                          total_tokens=T, start_pos=sp, pool=pool, snap_table=table, o=o, final_state=fin,
                          workspace=ws.get("w"))
        return out

    ms = _time_gpu(call, reps)
    tps, cores, sample = _oracle_tokens_per_s(data, oracle_seconds)
    row = {"workload": name, "gpu_ms": ms, "gpu_tokens_per_s": T / (ms / 1e3), "dtype": dtype_name,
           "oracle_tokens_per_s": tps, "oracle_cores": cores, "oracle_sample": sample}
    if extra:
        row.update(extra)
    return row


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--reps", type=int, default=5)
    ap.add_argument("--oracle-seconds", type=float, default=5.0)
    ap.add_argument("--only", default=None, help="comma-separated workload names")
    args = ap.parse_args(argv)
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    W = inputs.WORKLOADS
    only = set(args.only.split(",")) if args.only else set(W)
    rows = []

    if "tiny_fp32" in only:
        w = W["tiny_fp32"]
        data = inputs.gen_prefill([w["T"]], w["H"], w["d"], w["d"], w["seed"], dtype=torch.float32)
        rows.append(_prefill_case("tiny_fp32", data, dev, args.reps, args.oracle_seconds, "fp32"))
    if "prefill_4x8k" in only:
        w = W["prefill_4x8k"]
        data = inputs.gen_prefill([w["T"]] * w["n_seqs"], w["H"], w["d"], w["d"], w["seed"])
        rows.append(_prefill_case("prefill_4x8k", data, dev, args.reps, args.oracle_seconds, "bf16"))
        del data
    if "long_1m" in only:
        w = W["long_1m"]
        data = inputs.gen_prefill([w["T"]], w["H"], w["d"], w["d"], w["seed"])
        rows.append(_prefill_case("long_1m", data, dev, max(1, args.reps // 2), args.oracle_seconds, "bf16"))
        del data
    if "varlen_64" in only:
        w = W["varlen_64"]
        data = inputs.gen_varlen_resume(w["n_seqs"], w["H"], w["d"], w["d"], w["max_len"], w["prefix_len"],
                                        w["n_resume"], w["seed"])
        data["seq_lens"] = [int(x) for x in (data["cu_seqlens"][1:] - data["cu_seqlens"][:-1])]
        # resumed sequences start at their positions inside the shared prefix; their
        # initial states are zero here (the same work as resuming from a snapshot)
        rows.append(_prefill_case("varlen_64", data, dev, args.reps, args.oracle_seconds, "bf16",
                                  {"note": "resume positions as in the workload; initial states zero"},
                                  start_pos=data["start_pos"]))
        del data
    if "decode_512x32" in only:
        w = W["decode_512x32"]
        n, H, d = w["n_seqs"], w["H"], w["d"]
        pool = inputs.gen_states(n, H, d, d, w["seed"], std=w["state_std"]).to(dev)
        slots = torch.arange(n, dtype=torch.int32, device=dev)
        zs = [{k: t.to(dev) for k, t in inputs.gen_decode(n, H, d, d, w["seed"], s).items()} for s in range(4)]
        o = torch.empty((n, H, d), dtype=torch.bfloat16, device=dev)
        it = [0]

        def step():
            z = zs[it[0] % 4]
            it[0] += 1
            kda.kda_decode_step(z["q"], z["k"], z["v"], z["alpha"], z["beta"], pool, slots, o)

        ms = _time_gpu(step, args.reps * 4)
        nbytes = 2 * n * H * d * d * 4 + n * H * (3 * d * 2 + d * 4 + 4 + d * 2)
        import oracle
        import numpy as np
        hz = inputs.gen_decode(n, H, d, d, w["seed"], 0)
        S0 = pool.double().cpu().numpy()
        t0 = time.perf_counter()
        oracle.run(hz["q"], hz["k"], hz["v"], hz["alpha"], hz["beta"], np.arange(n + 1), init_state=S0)
        osecs = time.perf_counter() - t0
        rows.append({"workload": "decode_512x32", "gpu_ms": ms, "gpu_gbs": nbytes / (ms / 1e3) / 1e9,
                     "gpu_states_per_s": n * H / (ms / 1e3), "dtype": "bf16",
                     "oracle_states_per_s": n * H / osecs, "oracle_cores": oracle.threads(),
                     "oracle_sample": f"one full step ({osecs:.1f} s)"})
    for r in rows:
        print(json.dumps(r))
    print("\n| Workload | GPU | Oracle (host) | Cores |\n|---|---|---|---|")
    for r in rows:
        if "gpu_gbs" in r:
            g = f"{r['gpu_ms']:.3f} ms/step, {r['gpu_gbs']:.0f} GB/s"
            c = f"{r['oracle_states_per_s']:.3g} states/s ({r['oracle_sample']})"
        else:
            g = f"{r['gpu_ms']:.3f} ms, {r['gpu_tokens_per_s'] / 1e6:.2f} M tok/s"
            c = f"{r['oracle_tokens_per_s']:.3g} tok/s ({r['oracle_sample']})"
        print(f"| {r['workload']} | {g} | {c} | {r['oracle_cores']} |")


if __name__ == "__main__":
    main()
