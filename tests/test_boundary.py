"""The C-ABI library on a host without a GPU: it builds, loads, exports every
function the public header declares, and rejects bad arguments on the host
before any launch (no call here reaches the CUDA driver)."""
import ctypes
import os
import re
import subprocess

import pytest
import torch

import hybrid_linear_attention_kda_gb300 as kda
from hybrid_linear_attention_kda_gb300 import build as kbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")


def _declared_functions():
    names = set()
    for fn in os.listdir(HEADER_DIR):
        if not fn.endswith(".h"):
            continue
        with open(os.path.join(HEADER_DIR, fn)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names.update(re.findall(r"^[A-Za-z_][\w\s\*]*?\b(kda_\w+)\s*\(", text, flags=re.M))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    kbuild.build()
    return kda.load()


def test_header_declares_the_boundary():
    names = _declared_functions()
    for required in ("kda_prefill_chunked", "kda_prefill_workspace_size", "kda_decode_step",
                     "kda_snapshot_gather", "kda_snapshot_restore", "kda_check_status",
                     "kda_status_string", "kda_pcache_create", "kda_pcache_plan_request",
                     "kda_pcache_end_step", "kda_pcache_release"):
        assert required in names


def test_every_declared_function_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", kda.lib_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT\s+(kda_\w+)", out))
    missing = [n for n in _declared_functions() if n not in exported]
    assert not missing, missing
    for n in _declared_functions():
        getattr(lib, n)        # resolvable through ctypes as well


def test_abi_version_and_status_strings(lib):
    assert kda.kda_abi_version() == 1
    assert kda.kda_status_string(kda.KDA_OK) == "KDA_OK"
    assert kda.kda_status_string(kda.KDA_ERR_TIMEOUT) == "KDA_ERR_TIMEOUT"
    assert kda.kda_status_string(kda.KDA_ERR_NO_MEMORY) == "KDA_ERR_NO_MEMORY"
    assert kda.kda_status_string(99) == "KDA_ERR_UNKNOWN"


def test_prefill_args_struct_matches_c_layout():
    # 8 int32 + float; int64 pair; 2 int32; 13 pointers; size_t (LP64)
    assert ctypes.sizeof(kda.PrefillArgs) == 4 * 8 + 8 * 2 + 4 * 2 + 8 * 13 + 8


def _args(**over):
    a = kda.PrefillArgs()
    a.n_seqs, a.n_heads, a.d_k, a.d_v = 1, 2, 128, 128
    a.chunk, a.snap_interval, a.dtype, a.scale = 64, 256, kda.KDA_BF16, 1.0
    a.total_tokens = 64
    for p in ("q", "k", "v", "alpha", "beta", "cu_seqlens", "o"):
        setattr(a, p, 0x10000)
    for key, val in over.items():
        setattr(a, key, val)
    return a


@pytest.mark.parametrize("over,status", [
    (dict(d_k=96, d_v=96), kda.KDA_ERR_UNSUPPORTED),
    (dict(d_k=128, d_v=64), kda.KDA_ERR_UNSUPPORTED),
    (dict(chunk=32), kda.KDA_ERR_UNSUPPORTED),
    (dict(snap_interval=128), kda.KDA_ERR_UNSUPPORTED),
    (dict(dtype=7), kda.KDA_ERR_UNSUPPORTED),
    (dict(n_heads=0), kda.KDA_ERR_INVALID_ARG),
    (dict(n_seqs=-1), kda.KDA_ERR_INVALID_ARG),
    (dict(total_tokens=-5), kda.KDA_ERR_INVALID_ARG),
    (dict(q=0), kda.KDA_ERR_INVALID_ARG),
    (dict(o=0x10008), kda.KDA_ERR_INVALID_ARG),             # not 16-byte aligned
    (dict(snap_table=0x20000, snap_table_stride=4), kda.KDA_ERR_INVALID_ARG),   # no pool
    (dict(init_slot=0x20000), kda.KDA_ERR_INVALID_ARG),     # no pool
    (dict(reserved0=1), kda.KDA_ERR_INVALID_ARG),
])
def test_prefill_rejects_bad_arguments_on_the_host(lib, over, status):
    a = _args(**over)
    assert lib.kda_prefill_chunked(ctypes.byref(a), None) == status
    assert lib.kda_last_error()                      # a message was recorded


def test_prefill_with_no_sequences_is_a_no_op(lib):
    a = _args(n_seqs=0, total_tokens=0)
    assert lib.kda_prefill_chunked(ctypes.byref(a), None) == kda.KDA_OK


@pytest.mark.parametrize("dims,status", [
    ((4, 2, 96, 96, kda.KDA_BF16), kda.KDA_ERR_UNSUPPORTED),
    ((4, 0, 128, 128, kda.KDA_BF16), kda.KDA_ERR_INVALID_ARG),
    ((4, 2, 128, 128, 5), kda.KDA_ERR_UNSUPPORTED),
    ((-1, 2, 128, 128, kda.KDA_BF16), kda.KDA_ERR_INVALID_ARG),
])
def test_decode_rejects_bad_arguments_on_the_host(lib, dims, status):
    n, H, dk, dv, dt = dims
    p = 0x10000
    assert lib.kda_decode_step(n, H, dk, dv, dt, p, p, p, p, p, p, 8, p, p, 1.0, None) == status


def test_decode_null_pointer_is_rejected(lib):
    p = 0x10000
    assert lib.kda_decode_step(4, 2, 128, 128, kda.KDA_BF16, p, None, p, p, p, p, 8, p, p,
                               1.0, None) == kda.KDA_ERR_INVALID_ARG


def test_copies_reject_bad_arguments_on_the_host(lib):
    p = 0x10000
    assert lib.kda_snapshot_gather(p, 4, p, -1, 2, 128, 128, p, None) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_snapshot_restore(p, p, 4, p, 3, 2, 64, 128, None) == kda.KDA_ERR_UNSUPPORTED
    assert lib.kda_snapshot_gather(p, 4, p, 0, 2, 128, 128, p, None) == kda.KDA_OK


def test_binding_raises_instead_of_falling_back(monkeypatch, tmp_path):
    monkeypatch.setattr(kda, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(kda, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        kda.load()


def test_workspace_size_of_an_empty_batch_is_zero(lib):
    assert kda.kda_prefill_workspace_size(_args(n_seqs=0, total_tokens=0)) == 0
    assert torch.tensor(0).numel() == 1


def test_workspace_size_is_zero_for_invalid_sizes(lib):
    """The header promises 0 when the sizes are invalid; no size wraps around."""
    assert kda.kda_prefill_workspace_size(_args()) > 0
    for over in (dict(n_heads=0), dict(n_heads=-3), dict(d_k=96, d_v=96), dict(d_k=128, d_v=64),
                 dict(dtype=7), dict(chunk=32), dict(snap_interval=128), dict(total_tokens=-64),
                 dict(total_tokens=1 << 31), dict(n_seqs=-1), dict(n_seqs=(1 << 20) + 1)):
        assert kda.kda_prefill_workspace_size(_args(**over)) == 0, over
    # every dtype and head size runs the chunked stages, so each needs a workspace:
    # the fp32 SIMT records (4 x 64 x d + 64 x 64 + d floats per (chunk, head))
    # are larger than the bf16 tensor-core records (74,240 bytes)
    bf = kda.kda_prefill_workspace_size(_args())
    f32 = kda.kda_prefill_workspace_size(_args(dtype=kda.KDA_FP32))
    d64 = kda.kda_prefill_workspace_size(_args(d_k=64, d_v=64))
    assert f32 > bf > 0 and d64 > 0


def test_fused_decode_args_struct_and_checks(lib):
    # 4 int32, float + int32, int64, 12 pointers (LP64)
    assert ctypes.sizeof(kda.FusedDecodeArgs) == 4 * 4 + 8 + 8 + 8 * 12
    a = kda.FusedDecodeArgs()
    a.n_seqs, a.n_heads, a.d, a.conv_size, a.n_slots = 1, 2, 96, 4, 1
    assert lib.kda_decode_fused(ctypes.byref(a), None) == kda.KDA_ERR_UNSUPPORTED
    a.d, a.conv_size = 128, 3
    assert lib.kda_decode_fused(ctypes.byref(a), None) == kda.KDA_ERR_UNSUPPORTED
    a.conv_size = 4
    assert lib.kda_decode_fused(ctypes.byref(a), None) == kda.KDA_ERR_INVALID_ARG     # NULL pointers
    a.reserved0 = 1
    assert lib.kda_decode_fused(ctypes.byref(a), None) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_decode_fused(None, None) == kda.KDA_ERR_INVALID_ARG


@pytest.mark.parametrize("T", [0, 17])
def test_verify_rejects_token_counts(lib, T):
    fake = 0x10000
    st = lib.kda_decode_verify(1, T, 2, 128, 128, kda.KDA_BF16, fake, fake, fake, fake, fake, fake, 1, fake,
                               fake, fake, 1.0, None)
    assert st == kda.KDA_ERR_UNSUPPORTED
