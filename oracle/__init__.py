"""Float64 CPU oracle of the KDA (Kimi Delta Attention) layer.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It shares no code with
the GPU library and never calls it; the GPU library never imports it.

Contents
--------
``run``            token-by-token float64 recurrence (C, OpenMP) over a packed
                   variable-length batch, with snapshots and resume
                   ("Kimi K3 Tech Intro", sections 2.1-2.3).
``chunked``        the chunked (block-matrix) form in float64 numpy, written from
                   the recurrence alone; used to check that blocking the
                   sequence into chunks of any size changes nothing
                   (the block-matrix form of the yunthe.com "Kimi K3 open-source
                   practice" page, FlashKDA paragraph).
``snapshot_positions`` / ``reusable_prefix``
                   which absolute positions carry snapshots, and how much of a
                   shared prefix a snapshot grid lets a request reuse
                   ("Kimi K3 Tech Intro", sections 2.1-2.2).
``PrefixCacheIndex`` / ``block_hashes``
                   the prefix-cache policy: chained 256-token hashes, interval
                   retention, second-hit admission, next-step reuse
                   ("Kimi K3 Tech Intro", sections 2.2-2.4 and 3).
``verify_steps`` / ``commit_steps``
                   a speculative decoding step: T candidate tokens run without
                   touching the state (outputs and update vectors), then the
                   accepted ones applied ("Kimi K3 Tech Intro", section 6).
``fused_step``     one fused decode step with the layer's prologue (causal
                   convolution with its state, q/k norm, gates) and epilogue
                   (gated RMSNorm) around the update ("Kimi K3 Tech Intro",
                   section 4.1).
``window_bound``   a rigorous upper bound on how much a state that is forgotten
                   at the start of a window can change the states inside it,
                   used to check long sequences on sampled windows.
"""
from .recurrent import run, threads, DT_BF16, DT_F32, DT_F64  # noqa: F401
from .chunked import chunked  # noqa: F401
from .positions import snapshot_positions, reusable_prefix  # noqa: F401
from .bounds import window_bound, state_norm_bound  # noqa: F401
from .prefix_cache import PrefixCacheIndex, block_hashes  # noqa: F401
from .speculative import verify_steps, commit_steps  # noqa: F401
from .fused_decode import fused_step  # noqa: F401
