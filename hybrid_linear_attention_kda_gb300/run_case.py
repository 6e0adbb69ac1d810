"""Run one prefill or decode case of a chosen size through the C ABI, a few
times, on cuda:0 (a driver for profilers such as ncu and for quick checks).

    python -m hybrid_linear_attention_kda_gb300.run_case prefill --seqs 2 --len 8192 --heads 32 --reps 3
    python -m hybrid_linear_attention_kda_gb300.run_case decode --seqs 512 --heads 32 --reps 3

Prefill writes a snapshot every 256 tokens into a pool, like the benchmark.
"""
import argparse
import sys

import torch

import hybrid_linear_attention_kda_gb300 as kda
from hybrid_linear_attention_kda_gb300 import inputs


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("what", choices=["prefill", "decode"])
    ap.add_argument("--seqs", type=int, default=2)
    ap.add_argument("--len", type=int, default=8192)
    ap.add_argument("--heads", type=int, default=32)
    ap.add_argument("--d", type=int, default=128)
    ap.add_argument("--dtype", choices=["bf16", "fp32"], default="bf16")
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--seed", type=int, default=1)
    args = ap.parse_args(argv)
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    dt = inputs.torch_dtype(args.dtype)
    n, H, d = args.seqs, args.heads, args.d
    if args.what == "prefill":
        T = args.len
        host = inputs.gen_prefill([T] * n, H, d, d, args.seed, dtype=dt)
        x = {key: host[key].to(dev) for key in ("q", "k", "v", "alpha", "beta", "cu_seqlens")}
        n_ord = T // 256
        pool = torch.zeros((max(1, n * n_ord), H, d, d), device=dev)
        table = torch.arange(n * n_ord, dtype=torch.int32, device=dev).view(n, max(n_ord, 0))
        o = ws = None
        for _ in range(args.reps):
            o, fin = kda.prefill(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["cu_seqlens"],
                                 total_tokens=n * T, pool=pool,
                                 snap_table=table if n_ord else None, o=o)
    else:
        pool = inputs.gen_states(n, H, d, d, args.seed).to(dev)
        slots = torch.arange(n, dtype=torch.int32, device=dev)
        z = {key: t.to(dev) for key, t in inputs.gen_decode(n, H, d, d, args.seed, 0, dtype=dt).items()}
        o = torch.empty((n, H, d), dtype=dt, device=dev)
        for _ in range(args.reps):
            kda.kda_decode_step(z["q"], z["k"], z["v"], z["alpha"], z["beta"], pool, slots, o)
    torch.cuda.synchronize()
    bits = kda.kda_check_status()
    if bits:
        sys.exit(f"device status bits 0x{bits:x}")
    print(f"{args.what} ok: launches {kda.kda_launch_count()}")


if __name__ == "__main__":
    main()
