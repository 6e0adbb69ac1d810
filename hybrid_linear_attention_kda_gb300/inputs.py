"""Seeded synthetic inputs for the KDA layer.

This module only draws random numbers; it holds none of the layer's arithmetic.
Both the GPU path and the float64 oracle read the exact bytes it produces.

Recipe (the value distributions of the layer's serving workloads):
  q, k ~ N(0, 1) per element, each [d_k] vector L2-normalised in float64, then
         rounded to the storage dtype (bf16 or fp32);
  v    ~ N(0, 1), rounded to the storage dtype;
  beta  = sigmoid(N(0, 1)) in fp32 (one per token and head);
  alpha = exp(-softplus(N(0, 1) + 2)) in fp32 per channel ("config" decay), or
          exp(-softplus(N(0, 1) - 5)) ("mild" decay: alpha near 1, so a state
          carried across many chunks still matters);
  decode states ~ N(0, 0.05^2) fp32.

Every sequence draws from its own stream, ``torch.Generator`` seeded with
``seed * 1000003 + seq``, in fixed blocks of 4096 tokens (q, k, v, alpha, beta in
that order per block), so any batch can be generated piecewise and a sequence's
values do not depend on the other sequences of its batch.  Large batches draw
their sequences on a thread pool (torch's CPU kernels release the GIL); each
sequence still draws from its own generator, so the bytes do not change.
"""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

BLOCK = 4096
_DECAY_SHIFT = {"config": 2.0, "mild": -5.0}


def _stream(seed: int, seq: int) -> torch.Generator:
    g = torch.Generator()
    g.manual_seed(int(seed) * 1000003 + int(seq))
    return g


def _for_each_sequence(fn, n_seqs, total_tokens):
    """fn(i) for every sequence i; on a thread pool when the batch is large (each
    call writes a disjoint slice of the packed outputs)."""
    workers = min(n_seqs, os.cpu_count() or 1, 32)
    if workers <= 1 or total_tokens < 4 * BLOCK:
        for i in range(n_seqs):
            fn(i)
        return
    with ThreadPoolExecutor(workers) as ex:
        for _ in ex.map(fn, range(n_seqs)):
            pass


def _unit_rows(x: torch.Tensor) -> torch.Tensor:
    return x / torch.linalg.vector_norm(x, dim=-1, keepdim=True)


def gen_sequence_block(g, n, H, d_k, d_v, decay):
    """One block of n tokens from generator g, all float64."""
    q = _unit_rows(torch.randn((n, H, d_k), generator=g, dtype=torch.float64))
    k = _unit_rows(torch.randn((n, H, d_k), generator=g, dtype=torch.float64))
    v = torch.randn((n, H, d_v), generator=g, dtype=torch.float64)
    shift = _DECAY_SHIFT[decay]
    alpha = torch.exp(-torch.nn.functional.softplus(
        torch.randn((n, H, d_k), generator=g, dtype=torch.float64) + shift))
    beta = torch.sigmoid(torch.randn((n, H), generator=g, dtype=torch.float64))
    return q, k, v, alpha, beta


def gen_prefill(seq_lens, H, d_k, d_v, seed, dtype=torch.bfloat16, decay="config",
                pin=False):
    """Packed prefill inputs on the host.

    Returns dict with q, k [T, H, d_k] and v [T, H, d_v] in ``dtype``, alpha
    [T, H, d_k] and beta [T, H] in fp32, cu_seqlens int32 [n+1] and seq_lens.
    ``seq_lens[i]`` tokens are drawn for sequence i from its own stream.
    """
    seq_lens = [int(x) for x in seq_lens]
    T = sum(seq_lens)
    kw = {"pin_memory": True} if pin else {}
    q = torch.empty((T, H, d_k), dtype=dtype, **kw)
    k = torch.empty((T, H, d_k), dtype=dtype, **kw)
    v = torch.empty((T, H, d_v), dtype=dtype, **kw)
    alpha = torch.empty((T, H, d_k), dtype=torch.float32, **kw)
    beta = torch.empty((T, H), dtype=torch.float32, **kw)
    offs = np.concatenate([[0], np.cumsum(seq_lens, dtype=np.int64)]) if seq_lens else [0]
    dst = {"q": q, "k": k, "v": v, "alpha": alpha, "beta": beta}
    _for_each_sequence(lambda s: _draw_into(_stream(seed, s), seq_lens[s], H, d_k, d_v, dtype, decay, dst,
                                            int(offs[s])), len(seq_lens), T)
    cu = torch.zeros(len(seq_lens) + 1, dtype=torch.int32)
    cu[1:] = torch.tensor(np.cumsum(seq_lens), dtype=torch.int32) if seq_lens else cu[1:]
    return {"q": q, "k": k, "v": v, "alpha": alpha, "beta": beta,
            "cu_seqlens": cu, "seq_lens": seq_lens}


def gen_decode(n_seqs, H, d_k, d_v, seed, step, dtype=torch.bfloat16, decay="config"):
    """Inputs of one batched decode step: one token per sequence.

    Sequence i of step ``step`` draws from stream (seed + 7919 * (step + 1), i).
    Returns q, k [n, H, d_k], v [n, H, d_v] in ``dtype``; alpha [n, H, d_k] and
    beta [n, H] fp32.
    """
    q = torch.empty((n_seqs, H, d_k), dtype=dtype)
    k = torch.empty((n_seqs, H, d_k), dtype=dtype)
    v = torch.empty((n_seqs, H, d_v), dtype=dtype)
    alpha = torch.empty((n_seqs, H, d_k), dtype=torch.float32)
    beta = torch.empty((n_seqs, H), dtype=torch.float32)
    # one generator per step; sequences take consecutive rows of its block
    g = _stream(seed + 7919 * (step + 1), 0)
    qb, kb, vb, ab, bb = gen_sequence_block(g, n_seqs, H, d_k, d_v, decay)
    q[:] = qb.to(dtype)
    k[:] = kb.to(dtype)
    v[:] = vb.to(dtype)
    alpha[:] = ab.to(torch.float32)
    beta[:] = bb.to(torch.float32)
    return {"q": q, "k": k, "v": v, "alpha": alpha, "beta": beta}


def gen_states(n, H, d_k, d_v, seed, std=0.05):
    """fp32 states [n, H, d_k, d_v] with N(0, std^2) entries."""
    g = _stream(seed, 999_999_937)
    return (torch.randn((n, H, d_k, d_v), generator=g, dtype=torch.float64) * std).to(
        torch.float32)


# The five workloads the layer is exercised on (sizes and seeds only).
WORKLOADS = {
    # tiny fp32 check: one sequence, resumed from its snapshot at t = 256
    "tiny_fp32": dict(n_seqs=1, H=2, T=512, d=64, dtype="fp32", seed=20260, resume_at=256),
    # prefill: 4 sequences x 8192 tokens, 32 heads, d = 128, bf16 q/k/v
    "prefill_4x8k": dict(n_seqs=4, H=32, T=8192, d=128, dtype="bf16", seed=20261),
    # long context: one sequence of 2^20 tokens, 8 heads, resumed at 2^19
    "long_1m": dict(n_seqs=1, H=8, T=1 << 20, d=128, dtype="bf16", seed=20262, resume_at=1 << 19),
    # decode: 512 sequences x 32 heads, 64 consecutive steps, states ~ N(0, 0.05^2)
    "decode_512x32": dict(n_seqs=512, H=32, d=128, dtype="bf16", seed=20263, steps=64, state_std=0.05),
    # mixed varlen: 64 sequences, lengths uniform in [1, 16384]; 32 of them resume
    # inside a shared 4096-token prefix at a multiple of 256
    "varlen_64": dict(n_seqs=64, H=32, d=128, dtype="bf16", seed=20264, max_len=16384,
                      prefix_len=4096, n_resume=32),
}

PREFIX_STREAM = 1_000_001
LAYOUT_STREAM = 1_000_000
TOKEN_TABLE_STREAM = 1_000_002


def gen_token_table(vocab, H, d_k, d_v, seed, dtype=torch.bfloat16, decay="mild"):
    """Layer inputs per token id, for serving-style runs driven by token ids.

    Row t holds the q, k, v, alpha, beta that token id t feeds the layer (drawn
    by the same recipe as above), a stand-in for the model's projections: equal
    prompt prefixes then give equal layer inputs, which is what prefix reuse
    relies on.  Returns dict of [vocab, H, .] tensors.
    """
    g = _stream(seed, TOKEN_TABLE_STREAM)
    qb, kb, vb, ab, bb = gen_sequence_block(g, vocab, H, d_k, d_v, decay)
    return {"q": qb.to(dtype), "k": kb.to(dtype), "v": vb.to(dtype),
            "alpha": ab.to(torch.float32), "beta": bb.to(torch.float32)}


FUSED_STREAM = 1_000_003


def gen_fused_params(H, d, seed):
    """Per-head parameters of the fused decode step: depthwise convolution taps
    conv_w [H, 3, 4, d] ~ N(0, 0.5^2) (q, k, v) and the RMSNorm weight
    norm_w [H, d] ~ 1 + N(0, 0.1^2), both fp32."""
    g = _stream(seed, FUSED_STREAM)
    conv_w = (0.5 * torch.randn((H, 3, 4, d), generator=g, dtype=torch.float64)).to(torch.float32)
    norm_w = (1.0 + 0.1 * torch.randn((H, d), generator=g, dtype=torch.float64)).to(torch.float32)
    return conv_w, norm_w


def gen_fused_step(n, H, d, seed, step):
    """Raw projections of one decode token per (sequence, head), bf16: xq, xk,
    xv, g ~ N(0, 1); a ~ N(2, 1) (decay logits, alpha = exp(-softplus(a)) as in
    the decay recipe above); b ~ N(0, 1) (beta logits, [n, H])."""
    g = _stream(seed + 7919 * (step + 1), FUSED_STREAM)
    out = {}
    for key in ("xq", "xk", "xv", "g"):
        out[key] = torch.randn((n, H, d), generator=g, dtype=torch.float64).to(torch.bfloat16)
    out["a"] = (torch.randn((n, H, d), generator=g, dtype=torch.float64) + 2.0).to(torch.bfloat16)
    out["b"] = torch.randn((n, H), generator=g, dtype=torch.float64).to(torch.bfloat16)
    return out


def gen_conv_states(n, H, d, seed):
    """Convolution states [n, H, 3, 3, d] bf16 ~ N(0, 1) (previous raw inputs)."""
    g = _stream(seed, FUSED_STREAM + 1)
    return torch.randn((n, H, 3, 3, d), generator=g, dtype=torch.float64).to(torch.bfloat16)


def embed(table, token_lists):
    """Packed inputs of several token-id lists: dict with q, k, v, alpha, beta
    ([sum of lengths, H, .]) and cu_seqlens."""
    lens = [len(t) for t in token_lists]
    ids = torch.tensor([x for t in token_lists for x in t], dtype=torch.long)
    out = {key: table[key].index_select(0, ids) for key in ("q", "k", "v", "alpha", "beta")}
    cu = torch.zeros(len(lens) + 1, dtype=torch.int32)
    if lens:
        cu[1:] = torch.tensor(np.cumsum(lens), dtype=torch.int32)
    out["cu_seqlens"] = cu
    return out


def torch_dtype(name):
    return {"bf16": torch.bfloat16, "fp32": torch.float32}[name]


def _draw_into(g, L, H, d_k, d_v, dtype, decay, dst, off):
    """Draw L tokens block by block from g into the packed tensors of dst at off."""
    for b in range(0, L, BLOCK):
        n = min(BLOCK, L - b)
        qb, kb, vb, ab, bb = gen_sequence_block(g, BLOCK, H, d_k, d_v, decay)
        sl = slice(off + b, off + b + n)
        dst["q"][sl] = qb[:n].to(dtype)
        dst["k"][sl] = kb[:n].to(dtype)
        dst["v"][sl] = vb[:n].to(dtype)
        dst["alpha"][sl] = ab[:n].to(torch.float32)
        dst["beta"][sl] = bb[:n].to(torch.float32)


def _empty(T, H, d_k, d_v, dtype, pin=False):
    kw = {"pin_memory": True} if pin else {}
    return {"q": torch.empty((T, H, d_k), dtype=dtype, **kw),
            "k": torch.empty((T, H, d_k), dtype=dtype, **kw),
            "v": torch.empty((T, H, d_v), dtype=dtype, **kw),
            "alpha": torch.empty((T, H, d_k), dtype=torch.float32, **kw),
            "beta": torch.empty((T, H), dtype=torch.float32, **kw)}


def gen_varlen_resume(n_seqs, H, d_k, d_v, max_len, prefix_len, n_resume, seed,
                      dtype=torch.bfloat16, decay="config", interval=256, pin=False):
    """A packed varlen batch in which some sequences resume inside a shared prefix.

    Lengths L_i are uniform in [1, max_len].  ``n_resume`` sequences chosen among
    those with L_i > interval share their first min(L_i, prefix_len) tokens with
    one common prefix (drawn from its own stream) and resume at p_i = interval * m,
    m uniform in [1, min(prefix_len, L_i - 1) // interval]; only their tokens
    [p_i, L_i) are packed.  The other sequences are packed whole from position 0.

    Returns dict: packed q, k, v, alpha, beta, cu_seqlens (int32), start_pos
    (int32), lens (full lengths), resumed (sorted indices), and ``prefix`` (the
    shared prefix's own tensors, [prefix_len, H, .]).
    """
    lens, resumed, start = varlen_layout(n_seqs, max_len, prefix_len, n_resume, seed, interval)

    prefix = _empty(prefix_len, H, d_k, d_v, dtype)
    _draw_into(_stream(seed, PREFIX_STREAM), prefix_len, H, d_k, d_v, dtype, decay, prefix, 0)

    packed_lens = [lens[i] - start[i] for i in range(n_seqs)]
    T = sum(packed_lens)
    out = _empty(T, H, d_k, d_v, dtype, pin)
    offs = np.concatenate([[0], np.cumsum(packed_lens, dtype=np.int64)])
    rs = set(resumed)

    def fill(i):
        L, p, off = lens[i], start[i], int(offs[i])
        if i in rs:
            own = _empty(L, H, d_k, d_v, dtype)
            _draw_into(_stream(seed, i), L, H, d_k, d_v, dtype, decay, own, 0)
            shared = min(L, prefix_len)
            for key in own:
                own[key][:shared] = prefix[key][:shared]
                out[key][off:off + L - p] = own[key][p:L]
        else:
            _draw_into(_stream(seed, i), L, H, d_k, d_v, dtype, decay, out, off)

    _for_each_sequence(fill, n_seqs, T)
    cu = torch.zeros(n_seqs + 1, dtype=torch.int32)
    cu[1:] = torch.tensor(np.cumsum(packed_lens), dtype=torch.int32)
    out.update({"cu_seqlens": cu, "start_pos": torch.tensor(start, dtype=torch.int32),
                "lens": lens, "resumed": resumed, "prefix": prefix})
    return out


# ----------------------------------------------------------------------------- device-side draws

def varlen_layout(n_seqs, max_len, prefix_len, n_resume, seed, interval=256):
    """The layout of the mixed varlen batch of ``gen_varlen_resume``: full lengths,
    the resumed sequences and their start positions (drawn on the host from the
    same stream, so both generators agree on it)."""
    g = _stream(seed, LAYOUT_STREAM)
    lens = torch.randint(1, max_len + 1, (n_seqs,), generator=g).tolist()
    eligible = [i for i in range(n_seqs) if lens[i] > interval]
    perm = torch.randperm(len(eligible), generator=g).tolist()
    resumed = sorted(eligible[j] for j in perm[:n_resume])
    start = [0] * n_seqs
    for i in resumed:
        m_max = min(prefix_len, lens[i] - 1) // interval
        start[i] = interval * int(torch.randint(1, m_max + 1, (1,), generator=g))
    return lens, resumed, start


def _device_block(g, n, H, d_k, d_v, decay, device, dtype):
    """n tokens of the recipe above drawn on ``device`` in float32."""
    q = torch.randn((n, H, d_k), generator=g, device=device)
    q = q / torch.linalg.vector_norm(q, dim=-1, keepdim=True)
    k = torch.randn((n, H, d_k), generator=g, device=device)
    k = k / torch.linalg.vector_norm(k, dim=-1, keepdim=True)
    v = torch.randn((n, H, d_v), generator=g, device=device)
    a = torch.randn((n, H, d_k), generator=g, device=device) + _DECAY_SHIFT[decay]
    alpha = torch.exp(-torch.nn.functional.softplus(a))
    beta = torch.sigmoid(torch.randn((n, H), generator=g, device=device))
    return q.to(dtype), k.to(dtype), v.to(dtype), alpha, beta


def gen_prefill_device(seq_lens, H, d_k, d_v, seed, device, dtype=torch.bfloat16, decay="config",
                       block=65536):
    """Packed prefill inputs drawn directly on ``device`` by the same recipe, in
    float32 with a seeded device generator: for timing runs at full size, where
    drawing gigabytes in float64 on the host would take minutes.  These are not
    the bytes ``gen_prefill`` produces.  Returns the same dict keys (tensors on
    ``device``; cu_seqlens on the host and on the device as ``cu_seqlens_dev``)."""
    seq_lens = [int(x) for x in seq_lens]
    T = sum(seq_lens)
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1000003 + 17)
    out = {"q": torch.empty((T, H, d_k), dtype=dtype, device=device),
           "k": torch.empty((T, H, d_k), dtype=dtype, device=device),
           "v": torch.empty((T, H, d_v), dtype=dtype, device=device),
           "alpha": torch.empty((T, H, d_k), dtype=torch.float32, device=device),
           "beta": torch.empty((T, H), dtype=torch.float32, device=device)}
    for b in range(0, T, block):
        n = min(block, T - b)
        for key, t in zip(("q", "k", "v", "alpha", "beta"), _device_block(g, n, H, d_k, d_v, decay, device, dtype)):
            out[key][b:b + n] = t
    cu = torch.zeros(len(seq_lens) + 1, dtype=torch.int32)
    cu[1:] = torch.tensor(np.cumsum(seq_lens), dtype=torch.int32) if seq_lens else cu[1:]
    out.update({"cu_seqlens": cu, "cu_seqlens_dev": cu.to(device), "seq_lens": seq_lens})
    return out


def gen_varlen_resume_device(n_seqs, H, d_k, d_v, max_len, prefix_len, n_resume, seed, device,
                             dtype=torch.bfloat16, decay="config", interval=256):
    """The mixed varlen batch of ``gen_varlen_resume`` (same layout), with its
    token values drawn on ``device`` as in ``gen_prefill_device``.  Resumed
    sequences share the prefix's values over their first min(L_i, prefix_len)
    tokens; only tokens [p_i, L_i) are packed.  Returns the packed tensors,
    cu_seqlens (host and ``cu_seqlens_dev``), start_pos (host), lens, resumed
    and ``prefix`` (its own tensors on ``device``)."""
    lens, resumed, start = varlen_layout(n_seqs, max_len, prefix_len, n_resume, seed, interval)
    prefix = gen_prefill_device([prefix_len], H, d_k, d_v, seed + 1, device, dtype, decay)
    packed = [lens[i] - start[i] for i in range(n_seqs)]
    body = gen_prefill_device(packed, H, d_k, d_v, seed + 2, device, dtype, decay)
    cu = body["cu_seqlens"].tolist()
    rs = set(resumed)
    for i in range(n_seqs):
        if i in rs:
            shared = min(lens[i], prefix_len) - start[i]      # packed tokens still inside the prefix
            if shared > 0:
                for key in ("q", "k", "v", "alpha", "beta"):
                    body[key][cu[i]:cu[i] + shared] = prefix[key][start[i]:start[i] + shared]
    body.update({"start_pos": torch.tensor(start, dtype=torch.int32), "lens": lens, "resumed": resumed,
                 "prefix": prefix})
    return body
