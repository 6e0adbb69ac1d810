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


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


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
    copy of cu_seqlens[-1]; ``snap_table`` is [n_seqs, stride] int32."""
    T, H, d_k = q.shape
    d_v = v.shape[2]
    a = PrefillArgs()
    a.n_seqs = cu_seqlens.shape[0] - 1
    a.n_heads, a.d_k, a.d_v = H, d_k, d_v
    a.chunk, a.snap_interval = chunk, snap_interval
    a.dtype = _dtype_code(q)
    a.scale = float(scale)
    a.total_tokens = int(total_tokens)
    a.n_slots = 0 if pool is None else pool.shape[0]
    a.snap_table_stride = 0 if snap_table is None else snap_table.shape[1]
    a.reserved0 = 0
    a.q, a.k, a.v, a.alpha, a.beta = (_ptr(x) for x in (q, k, v, alpha, beta))
    a.cu_seqlens = _ptr(cu_seqlens)
    a.start_pos = _ptr(start_pos)
    a.init_slot = _ptr(init_slot)
    a.pool = _ptr(pool)
    a.snap_table = _ptr(snap_table)
    a.o = _ptr(o)
    a.final_state = _ptr(final_state)
    a.workspace = _ptr(workspace)
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
    """One decode step; the states in pool[state_slot[s]] are updated in place."""
    n, H, d_k = q.shape
    d_v = v.shape[2]
    _check(load().kda_decode_step(n, H, d_k, d_v, _dtype_code(q), _ptr(q), _ptr(k), _ptr(v),
                                  _ptr(alpha), _ptr(beta), _ptr(pool), pool.shape[0],
                                  _ptr(state_slot), _ptr(o), float(scale), _stream_handle(stream)))


def kda_decode_fused(args: FusedDecodeArgs, stream=None):
    _check(load().kda_decode_fused(ctypes.byref(args), _stream_handle(stream)))


def decode_fused(xq, xk, xv, a, b, g, conv_w, norm_w, pool, conv_state, state_slot, y, norm_eps=1e-6,
                 stream=None):
    """One fused decode step (``kda_decode_fused``): convolution, q/k norm,
    gates, update and gated RMSNorm, with both states updated in place."""
    n, H, d = xq.shape
    args = FusedDecodeArgs(n, H, d, conv_w.shape[2], float(norm_eps), 0, pool.shape[0],
                           _ptr(xq), _ptr(xk), _ptr(xv), _ptr(a), _ptr(b), _ptr(g), _ptr(conv_w),
                           _ptr(norm_w), _ptr(pool), _ptr(conv_state), _ptr(state_slot), _ptr(y))
    kda_decode_fused(args, stream)


def kda_decode_verify(q, k, v, alpha, beta, pool, state_slot, o, u, scale=1.0, stream=None):
    """Run T candidate tokens per sequence without touching the states:
    q, k, alpha [n, T, H, d_k]; v, o, u [n, T, H, d_v]; beta [n, T, H]."""
    n, T, H, d_k = q.shape
    d_v = v.shape[3]
    _check(load().kda_decode_verify(n, T, H, d_k, d_v, _dtype_code(q), _ptr(q), _ptr(k), _ptr(v),
                                    _ptr(alpha), _ptr(beta), _ptr(pool), pool.shape[0], _ptr(state_slot),
                                    _ptr(o), _ptr(u), float(scale), _stream_handle(stream)))


def kda_decode_commit(k, alpha, u, n_accept, pool, state_slot, stream=None):
    """Apply the first n_accept[i] verified updates of sequence i to its state."""
    n, T, H, d_k = k.shape
    d_v = u.shape[3]
    _check(load().kda_decode_commit(n, T, H, d_k, d_v, _dtype_code(k), _ptr(k), _ptr(alpha), _ptr(u),
                                    _ptr(n_accept), _ptr(pool), pool.shape[0], _ptr(state_slot),
                                    _stream_handle(stream)))


def kda_snapshot_gather(pool, slots, dst, stream=None):
    """dst[i] = pool[slots[i]] (zeros where slots[i] == -1)."""
    _, H, d_k, d_v = pool.shape
    _check(load().kda_snapshot_gather(_ptr(pool), pool.shape[0], _ptr(slots), slots.shape[0],
                                      H, d_k, d_v, _ptr(dst), _stream_handle(stream)))


def kda_snapshot_restore(src, pool, slots, stream=None):
    """pool[slots[i]] = src[i] (entries with slots[i] == -1 are skipped)."""
    _, H, d_k, d_v = pool.shape
    _check(load().kda_snapshot_restore(_ptr(src), _ptr(pool), pool.shape[0], _ptr(slots),
                                       slots.shape[0], H, d_k, d_v, _stream_handle(stream)))


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
    T, H, d_k = q.shape
    d_v = v.shape[2]
    n = cu_seqlens.shape[0] - 1
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
        args.workspace = workspace.data_ptr()
        args.workspace_bytes = workspace.numel() * workspace.element_size()
    kda_prefill_chunked(args, stream)
    return o, final_state
