"""Python binding of libkda.so, the GB300 (sm_103a) KDA library.

Argument marshalling only: every step of the computation runs in the library's
CUDA kernels.  PyTorch supplies device memory and streams.  The functions carry
the names of the C entry points declared in ``include/kda.h``; see that header
for layouts, ownership and error behaviour.

KDA (Kimi Delta Attention) keeps one fp32 state S in R^{d_k x d_v} per head and
updates it in place for every token ("Kimi K3 Tech Intro", section 2.1):
    S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T ,
    o_t = scale * S_t^T q_t .
"""
import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "_lib", "libkda.so")

KDA_OK, KDA_ERR_INVALID_ARG, KDA_ERR_UNSUPPORTED, KDA_ERR_CUDA, KDA_ERR_DEVICE_STATUS, \
    KDA_ERR_TIMEOUT, KDA_ERR_NO_MEMORY = range(7)
KDA_BF16, KDA_FP32 = 0, 1
KDA_DEV_BAD_SLOT, KDA_DEV_BAD_START, KDA_DEV_BAD_SEQLENS, KDA_DEV_BAD_ORDINAL = 0x1, 0x2, 0x4, 0x8
KDA_DEV_WAIT_TIMEOUT, KDA_DEV_BAD_ACCEPT = 0x10, 0x20

CHUNK = 64
SNAP_INTERVAL = 256


class KdaError(RuntimeError):
    def __init__(self, status, message):
        super().__init__(f"{message} (status {status})")
        self.status = status


class PrefillArgs(ctypes.Structure):
    """Mirror of ``kda_prefill_args``."""
    _fields_ = [
        ("n_seqs", ctypes.c_int32), ("n_heads", ctypes.c_int32),
        ("d_k", ctypes.c_int32), ("d_v", ctypes.c_int32),
        ("chunk", ctypes.c_int32), ("snap_interval", ctypes.c_int32),
        ("dtype", ctypes.c_int32), ("scale", ctypes.c_float),
        ("total_tokens", ctypes.c_int64), ("n_slots", ctypes.c_int64),
        ("snap_table_stride", ctypes.c_int32), ("reserved0", ctypes.c_int32),
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("alpha", ctypes.c_void_p), ("beta", ctypes.c_void_p),
        ("cu_seqlens", ctypes.c_void_p), ("start_pos", ctypes.c_void_p),
        ("init_slot", ctypes.c_void_p), ("pool", ctypes.c_void_p),
        ("snap_table", ctypes.c_void_p), ("o", ctypes.c_void_p),
        ("final_state", ctypes.c_void_p), ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t),
    ]


class FusedDecodeArgs(ctypes.Structure):
    """Mirror of ``kda_fused_decode_args``."""
    _fields_ = [
        ("n_seqs", ctypes.c_int32), ("n_heads", ctypes.c_int32), ("d", ctypes.c_int32),
        ("conv_size", ctypes.c_int32), ("norm_eps", ctypes.c_float), ("reserved0", ctypes.c_int32),
        ("n_slots", ctypes.c_int64),
        ("xq", ctypes.c_void_p), ("xk", ctypes.c_void_p), ("xv", ctypes.c_void_p),
        ("a", ctypes.c_void_p), ("b", ctypes.c_void_p), ("g", ctypes.c_void_p),
        ("conv_w", ctypes.c_void_p), ("norm_w", ctypes.c_void_p), ("pool", ctypes.c_void_p),
        ("conv_state", ctypes.c_void_p), ("state_slot", ctypes.c_void_p), ("y", ctypes.c_void_p),
    ]


_lib = None


def lib_path() -> str:
    return LIB_PATH


def load():
    """Load libkda.so.  Raises when it has not been built: there is no fallback."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is missing; build it with "
            "`python -m hybrid_linear_attention_kda_gb300.build` (needs nvcc)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    lib.kda_abi_version.restype = i32
    lib.kda_launch_count.restype = ctypes.c_uint64
    lib.kda_status_string.restype = ctypes.c_char_p
    lib.kda_status_string.argtypes = [ctypes.c_int]
    lib.kda_last_error.restype = ctypes.c_char_p
    lib.kda_prefill_workspace_size.restype = sz
    lib.kda_prefill_workspace_size.argtypes = [ctypes.POINTER(PrefillArgs)]
    lib.kda_prefill_chunked.restype = ctypes.c_int
    lib.kda_prefill_chunked.argtypes = [ctypes.POINTER(PrefillArgs), vp]
    lib.kda_prefill_chunked_events.restype = ctypes.c_int
    lib.kda_prefill_chunked_events.argtypes = [ctypes.POINTER(PrefillArgs), vp, ctypes.POINTER(vp), i32,
                                               ctypes.POINTER(i32), ctypes.POINTER(ctypes.c_char_p)]
    lib.kda_decode_step.restype = ctypes.c_int
    lib.kda_decode_step.argtypes = [i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, i64, vp, vp, f32, vp]
    lib.kda_decode_fused.restype = ctypes.c_int
    lib.kda_decode_fused.argtypes = [ctypes.POINTER(FusedDecodeArgs), vp]
    lib.kda_decode_verify.restype = ctypes.c_int
    lib.kda_decode_verify.argtypes = [i32, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, i64, vp, vp, vp, f32, vp]
    lib.kda_decode_commit.restype = ctypes.c_int
    lib.kda_decode_commit.argtypes = [i32, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, i64, vp, vp]
    lib.kda_snapshot_gather.restype = ctypes.c_int
    lib.kda_snapshot_gather.argtypes = [vp, i64, vp, i32, i32, i32, i32, vp, vp]
    lib.kda_snapshot_restore.restype = ctypes.c_int
    lib.kda_snapshot_restore.argtypes = [vp, vp, i64, vp, i32, i32, i32, i32, vp]
    lib.kda_check_status.restype = ctypes.c_int
    lib.kda_check_status.argtypes = [vp, i32, ctypes.POINTER(ctypes.c_uint32)]
    from . import prefix_cache
    prefix_cache.declare(lib)
    _lib = lib
    return lib


def _check(status):
    if status != KDA_OK:
        lib = load()
        name = lib.kda_status_string(status).decode()
        raise KdaError(status, f"{name}: {lib.kda_last_error().decode()}")


def _dev(x, name, dtype=None, shape=None, device=None, min_numel=None):
    """Address of a device tensor, after the checks the C calls cannot make.

    They take bare pointers and trust the dtype, shape and dense row-major
    layout their header states.  A mismatch would make a kernel read or write
    outside the tensor, so it is refused here: the tensor must be on a CUDA
    device (``device``, when given), contiguous, of ``dtype`` (one dtype or a
    tuple) and of exactly ``shape``, or of at least ``min_numel`` elements."""
    import torch
    if not isinstance(x, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor (got {type(x).__name__})")
    if dtype is not None:
        allowed = dtype if isinstance(dtype, tuple) else (dtype,)
        if x.dtype not in allowed:
            raise TypeError(f"{name} must be {' or '.join(str(t) for t in allowed)} (got {x.dtype})")
    if shape is not None and tuple(x.shape) != tuple(int(e) for e in shape):
        raise ValueError(f"{name} must have shape {tuple(int(e) for e in shape)} (got {tuple(x.shape)})")
    if min_numel is not None and x.numel() < min_numel:
        raise ValueError(f"{name} must hold at least {min_numel} elements (got {x.numel()})")
    if not x.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if x.device.type != "cuda":
        raise ValueError(f"{name} must be on a CUDA device (got {x.device})")
    if device is not None and x.device != device:
        raise ValueError(f"{name} is on {x.device}, the other operands on {device}")
    return x.data_ptr()


def _opt_dev(x, name, **checks):
    return None if x is None else _dev(x, name, **checks)


def _dims(x, name, ndim):
    """Shape of a tensor that must have ``ndim`` dimensions."""
    if not hasattr(x, "shape") or len(x.shape) != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions (got {getattr(x, 'shape', None)})")
    return tuple(int(e) for e in x.shape)


def _stream_handle(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dtype_code(t):
    import torch
    if t.dtype == torch.bfloat16:
        return KDA_BF16
    if t.dtype == torch.float32:
        return KDA_FP32
    raise TypeError(f"q/k/v must be bf16 or fp32, got {t.dtype}")


def _torch():
    import torch
    return torch


def kda_status_string(status) -> str:
    return load().kda_status_string(int(status)).decode()


def kda_abi_version() -> int:
    return int(load().kda_abi_version())


def kda_launch_count() -> int:
    """Kernels launched by the library so far in this process."""
    return int(load().kda_launch_count())


def make_prefill_args(q, k, v, alpha, beta, cu_seqlens, total_tokens, o, *, start_pos=None,
                      init_slot=None, pool=None, snap_table=None, final_state=None,
                      workspace=None, scale=1.0, chunk=CHUNK, snap_interval=SNAP_INTERVAL):
    """Fill a ``PrefillArgs`` from device tensors.  ``total_tokens`` is the host
    copy of cu_seqlens[-1] (at most the rows of q); ``snap_table`` is
    [n_seqs, stride] int32.  Layouts are checked against the header's."""
    torch = _torch()
    T, H, d_k = _dims(q, "q", 3)
    d_v = _dims(v, "v", 3)[2]
    n = _dims(cu_seqlens, "cu_seqlens", 1)[0] - 1
    if not 0 <= int(total_tokens) <= T:
        raise ValueError(f"total_tokens {int(total_tokens)} outside [0, {T}] (the rows of q)")
    dev = q.device
    qk = (torch.bfloat16, torch.float32)
    a = PrefillArgs()
    a.q = _dev(q, "q", qk, (T, H, d_k))
    a.k = _dev(k, "k", q.dtype, (T, H, d_k), dev)
    a.v = _dev(v, "v", q.dtype, (T, H, d_v), dev)
    a.alpha = _dev(alpha, "alpha", torch.float32, (T, H, d_k), dev)
    a.beta = _dev(beta, "beta", torch.float32, (T, H), dev)
    a.cu_seqlens = _dev(cu_seqlens, "cu_seqlens", torch.int32, (n + 1,), dev)
    a.o = _dev(o, "o", v.dtype, (T, H, d_v), dev)
    a.start_pos = _opt_dev(start_pos, "start_pos", dtype=torch.int32, shape=(n,), device=dev)
    a.init_slot = _opt_dev(init_slot, "init_slot", dtype=torch.int32, shape=(n,), device=dev)
    n_slots = 0 if pool is None else _dims(pool, "pool", 4)[0]
    a.pool = _opt_dev(pool, "pool", dtype=torch.float32, shape=(n_slots, H, d_k, d_v), device=dev)
    stride = 0 if snap_table is None else _dims(snap_table, "snap_table", 2)[1]
    a.snap_table = _opt_dev(snap_table, "snap_table", dtype=torch.int32, shape=(n, stride), device=dev)
    a.final_state = _opt_dev(final_state, "final_state", dtype=torch.float32, shape=(n, H, d_k, d_v), device=dev)
    a.workspace = _opt_dev(workspace, "workspace", device=dev)
    a.n_seqs = n
    a.n_heads, a.d_k, a.d_v = H, d_k, d_v
    a.chunk, a.snap_interval = chunk, snap_interval
    a.dtype = _dtype_code(q)
    a.scale = float(scale)
    a.total_tokens = int(total_tokens)
    a.n_slots = n_slots
    a.snap_table_stride = stride
    a.reserved0 = 0
    a.workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return a


def kda_prefill_workspace_size(args: PrefillArgs) -> int:
    return int(load().kda_prefill_workspace_size(ctypes.byref(args)))


def kda_prefill_chunked(args: PrefillArgs, stream=None):
    """Launch the chunked prefill described by ``args`` on ``stream``."""
    _check(load().kda_prefill_chunked(ctypes.byref(args), _stream_handle(stream)))


def kda_prefill_chunked_events(args: PrefillArgs, events, stream=None):
    """``kda_prefill_chunked`` that also records ``events`` (``torch.cuda.Event``
    with timing, already recorded once so that they exist) before each of its
    kernels and after the last.  Returns [(kernel name, event), ...]; the last
    name is ``"end"``."""
    n = len(events)
    arr = (ctypes.c_void_p * n)(*[e.cuda_event for e in events])
    names = (ctypes.c_char_p * n)()
    nrec = ctypes.c_int32(0)
    _check(load().kda_prefill_chunked_events(ctypes.byref(args), _stream_handle(stream), arr, n,
                                             ctypes.byref(nrec), names))
    return [(names[i].decode(), events[i]) for i in range(nrec.value)]


def kda_decode_step(q, k, v, alpha, beta, pool, state_slot, o, scale=1.0, stream=None):
    """One decode step; the states in pool[state_slot[s]] are updated in place.
    q, k, alpha [n, H, d_k]; v, o [n, H, d_v]; beta [n, H]."""
    torch = _torch()
    n, H, d_k = _dims(q, "q", 3)
    d_v = _dims(v, "v", 3)[2]
    dev = q.device
    ptrs = (_dev(q, "q", (torch.bfloat16, torch.float32), (n, H, d_k)),
            _dev(k, "k", q.dtype, (n, H, d_k), dev), _dev(v, "v", q.dtype, (n, H, d_v), dev),
            _dev(alpha, "alpha", torch.float32, (n, H, d_k), dev), _dev(beta, "beta", torch.float32, (n, H), dev))
    n_slots = _dims(pool, "pool", 4)[0]
    pp = _dev(pool, "pool", torch.float32, (n_slots, H, d_k, d_v), dev)
    sp = _dev(state_slot, "state_slot", torch.int32, (n,), dev)
    op = _dev(o, "o", q.dtype, (n, H, d_v), dev)
    _check(load().kda_decode_step(n, H, d_k, d_v, _dtype_code(q), *ptrs, pp, n_slots, sp, op, float(scale),
                                  _stream_handle(stream)))


def kda_decode_fused(args: FusedDecodeArgs, stream=None):
    _check(load().kda_decode_fused(ctypes.byref(args), _stream_handle(stream)))


def decode_fused(xq, xk, xv, a, b, g, conv_w, norm_w, pool, conv_state, state_slot, y, norm_eps=1e-6,
                 stream=None):
    """One fused decode step (``kda_decode_fused``): convolution, q/k norm,
    gates, update and gated RMSNorm, with both states updated in place.
    xq, xk, xv, a, g, y bf16 [n, H, d]; b bf16 [n, H]; conv_w fp32 [H, 3, K, d];
    norm_w fp32 [H, d]; pool fp32 [S, H, d, d]; conv_state bf16 [S, H, 3, K-1, d]."""
    torch = _torch()
    n, H, d = _dims(xq, "xq", 3)
    K = _dims(conv_w, "conv_w", 4)[2]
    dev = xq.device
    bf, f32 = torch.bfloat16, torch.float32
    vec = [_dev(t, nm, bf, (n, H, d), dev) for t, nm in ((xq, "xq"), (xk, "xk"), (xv, "xv"), (a, "a"))]
    bp = _dev(b, "b", bf, (n, H), dev)
    gp = _dev(g, "g", bf, (n, H, d), dev)
    cw = _dev(conv_w, "conv_w", f32, (H, 3, K, d), dev)
    nw = _dev(norm_w, "norm_w", f32, (H, d), dev)
    n_slots = _dims(pool, "pool", 4)[0]
    pp = _dev(pool, "pool", f32, (n_slots, H, d, d), dev)
    cs = _dev(conv_state, "conv_state", bf, (n_slots, H, 3, max(K - 1, 0), d), dev)
    sp = _dev(state_slot, "state_slot", torch.int32, (n,), dev)
    yp = _dev(y, "y", bf, (n, H, d), dev)
    args = FusedDecodeArgs(n, H, d, K, float(norm_eps), 0, n_slots, *vec[:3], vec[3], bp, gp, cw, nw, pp, cs, sp,
                           yp)
    kda_decode_fused(args, stream)


def kda_decode_verify(q, k, v, alpha, beta, pool, state_slot, o, u, scale=1.0, stream=None):
    """Run T candidate tokens per sequence without touching the states:
    q, k, alpha [n, T, H, d_k]; v, o, u [n, T, H, d_v]; beta [n, T, H]."""
    torch = _torch()
    n, T, H, d_k = _dims(q, "q", 4)
    d_v = _dims(v, "v", 4)[3]
    dev = q.device
    ptrs = (_dev(q, "q", (torch.bfloat16, torch.float32), (n, T, H, d_k)),
            _dev(k, "k", q.dtype, (n, T, H, d_k), dev), _dev(v, "v", q.dtype, (n, T, H, d_v), dev),
            _dev(alpha, "alpha", torch.float32, (n, T, H, d_k), dev),
            _dev(beta, "beta", torch.float32, (n, T, H), dev))
    n_slots = _dims(pool, "pool", 4)[0]
    pp = _dev(pool, "pool", torch.float32, (n_slots, H, d_k, d_v), dev)
    sp = _dev(state_slot, "state_slot", torch.int32, (n,), dev)
    op = _dev(o, "o", q.dtype, (n, T, H, d_v), dev)
    up = _dev(u, "u", torch.float32, (n, T, H, d_v), dev)
    _check(load().kda_decode_verify(n, T, H, d_k, d_v, _dtype_code(q), *ptrs, pp, n_slots, sp, op, up,
                                    float(scale), _stream_handle(stream)))


def kda_decode_commit(k, alpha, u, n_accept, pool, state_slot, stream=None):
    """Apply the first n_accept[i] verified updates of sequence i to its state:
    k, alpha [n, T, H, d_k]; u fp32 [n, T, H, d_v] from kda_decode_verify."""
    torch = _torch()
    n, T, H, d_k = _dims(k, "k", 4)
    d_v = _dims(u, "u", 4)[3]
    dev = k.device
    kp = _dev(k, "k", (torch.bfloat16, torch.float32), (n, T, H, d_k))
    ap = _dev(alpha, "alpha", torch.float32, (n, T, H, d_k), dev)
    up = _dev(u, "u", torch.float32, (n, T, H, d_v), dev)
    np_ = _dev(n_accept, "n_accept", torch.int32, (n,), dev)
    n_slots = _dims(pool, "pool", 4)[0]
    pp = _dev(pool, "pool", torch.float32, (n_slots, H, d_k, d_v), dev)
    sp = _dev(state_slot, "state_slot", torch.int32, (n,), dev)
    _check(load().kda_decode_commit(n, T, H, d_k, d_v, _dtype_code(k), kp, ap, up, np_, pp, n_slots, sp,
                                    _stream_handle(stream)))


def _pool_and_slots(pool, slots):
    torch = _torch()
    n_slots, H, d_k, d_v = _dims(pool, "pool", 4)
    m = _dims(slots, "slots", 1)[0]
    pp = _dev(pool, "pool", torch.float32, (n_slots, H, d_k, d_v))
    sp = _dev(slots, "slots", torch.int32, (m,), pool.device)
    return pp, sp, (n_slots, m, H, d_k, d_v)


def kda_snapshot_gather(pool, slots, dst, stream=None):
    """dst[i] = pool[slots[i]] (zeros where slots[i] == -1); dst [m, H, d_k, d_v]."""
    pp, sp, (n_slots, m, H, d_k, d_v) = _pool_and_slots(pool, slots)
    dp = _dev(dst, "dst", _torch().float32, (m, H, d_k, d_v), pool.device)
    _check(load().kda_snapshot_gather(pp, n_slots, sp, m, H, d_k, d_v, dp, _stream_handle(stream)))


def kda_snapshot_restore(src, pool, slots, stream=None):
    """pool[slots[i]] = src[i] (entries with slots[i] == -1 are skipped)."""
    pp, sp, (n_slots, m, H, d_k, d_v) = _pool_and_slots(pool, slots)
    srp = _dev(src, "src", _torch().float32, (m, H, d_k, d_v), pool.device)
    _check(load().kda_snapshot_restore(srp, pp, n_slots, sp, m, H, d_k, d_v, _stream_handle(stream)))


def kda_check_status(stream=None, timeout_ms=0):
    """Drain ``stream`` and return the device status bits (0 when clean).  Raises
    on a CUDA error or a timeout."""
    bits = ctypes.c_uint32(0)
    st = load().kda_check_status(_stream_handle(stream), int(timeout_ms), ctypes.byref(bits))
    if st == KDA_ERR_DEVICE_STATUS:
        return int(bits.value)
    _check(st)
    return 0


def prefill(q, k, v, alpha, beta, cu_seqlens, total_tokens=None, *, start_pos=None,
            init_slot=None, pool=None, snap_table=None, want_final=True, scale=1.0,
            o=None, final_state=None, workspace=None, stream=None):
    """Allocate the outputs (and workspace) with torch, then call
    ``kda_prefill_chunked``.  Returns (o, final_state or None)."""
    import torch
    T, H, d_k = _dims(q, "q", 3)
    d_v = _dims(v, "v", 3)[2]
    n = _dims(cu_seqlens, "cu_seqlens", 1)[0] - 1
    if total_tokens is None:
        total_tokens = T
    if o is None:
        o = torch.empty((T, H, d_v), dtype=v.dtype, device=v.device)
    if final_state is None and want_final:
        final_state = torch.empty((n, H, d_k, d_v), dtype=torch.float32, device=v.device)
    args = make_prefill_args(q, k, v, alpha, beta, cu_seqlens, total_tokens, o,
                             start_pos=start_pos, init_slot=init_slot, pool=pool,
                             snap_table=snap_table, final_state=final_state, scale=scale)
    need = kda_prefill_workspace_size(args)
    if need:
        if workspace is None or workspace.numel() * workspace.element_size() < need:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
        args.workspace = _dev(workspace, "workspace", device=q.device)
        args.workspace_bytes = workspace.numel() * workspace.element_size()
    kda_prefill_chunked(args, stream)
    return o, final_state
