"""Shared helpers of the test suite: error measures and GPU plumbing.

The error measures follow the tolerances the layer is held to: per (sequence,
head), outputs by RMS(diff) / RMS(reference) and states by the same ratio for
bf16 inputs; relative Frobenius error for fp32 inputs.
"""
import numpy as np
import torch

BF16_OUT_TOL = 2e-2     # outputs, bf16 inputs: RMS(diff)/RMS(ref) per (seq, head)
BF16_STATE_TOL = 1e-2   # states, bf16 inputs
FP32_TOL = 1e-4         # relative Frobenius error per (seq, head), fp32 inputs


def rel_rms(got, ref):
    """RMS(got - ref) / RMS(ref) over all elements (inf if ref is all zero and got is not)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    num = np.sqrt(np.mean((got - ref) ** 2)) if ref.size else 0.0
    den = np.sqrt(np.mean(ref ** 2)) if ref.size else 0.0
    if den == 0.0:
        return 0.0 if num == 0.0 else float("inf")
    return float(num / den)


def worst_out_err(o_gpu, o_ref, cu_seqlens):
    """Worst per-(sequence, head) relative RMS error of packed outputs [T, H, d_v]."""
    o_gpu = np.asarray(o_gpu, dtype=np.float64)
    o_ref = np.asarray(o_ref, dtype=np.float64)
    worst = 0.0
    cu = [int(x) for x in cu_seqlens]
    for s in range(len(cu) - 1):
        a, b = cu[s], cu[s + 1]
        if a == b:
            continue
        for h in range(o_ref.shape[1]):
            worst = max(worst, rel_rms(o_gpu[a:b, h], o_ref[a:b, h]))
    return worst


def worst_state_err(s_gpu, s_ref):
    """Worst per-(entry, head) relative RMS error of states [n, H, d_k, d_v]."""
    s_gpu = np.asarray(s_gpu, dtype=np.float64)
    s_ref = np.asarray(s_ref, dtype=np.float64)
    worst = 0.0
    for i in range(s_ref.shape[0]):
        for h in range(s_ref.shape[1]):
            worst = max(worst, rel_rms(s_gpu[i, h], s_ref[i, h]))
    return worst


def to_dev(d, device, keys=("q", "k", "v", "alpha", "beta")):
    return {key: d[key].to(device) for key in keys}


def cpu64(t):
    return t.detach().to("cpu", torch.float64).numpy()
