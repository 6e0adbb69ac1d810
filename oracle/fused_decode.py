"""One fused KDA decode step: the layer's prologue and epilogue around the
recurrent update (test infrastructure).

"Kimi K3 Tech Intro", section 4.1: the decode kernel fuses the causal
convolution, the q/k norm, the gate computation, the recurrent update and the
gated RMSNorm, and updates the convolution state and the recurrent state in
place.  Section 2.1 names the two per-request states: the recurrent state S and
the convolution state C.

Readings (the page names the steps, not their exact forms):
* Causal convolution: depthwise per channel, width K = 4, over the raw q, k, v
  projections.  C holds the last K-1 raw inputs, oldest first.  The
  convolution output goes through SiLU:
      y_c = silu( sum_{tau<K} w[tau, c] * x_{t-K+1+tau}[c] )
  with tau = K-1 the current token.
* q/k norm: L2 normalisation, x * (sum x^2 + 1e-6)^(-1/2).
* Gates: alpha = exp(-softplus(a)) per channel, beta = sigmoid(b) per head.
* Recurrent update: the token recurrence of ``oracle.run`` with scale 1.
* Gated RMSNorm: y = gamma * o * (mean(o^2) + eps)^(-1/2) * sigmoid(g).
Everything is float64 numpy, step by step in the order above.
"""
import numpy as np

K_CONV = 4
QK_EPS = 1e-6


def _f64(x):
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float64)


def silu(x):
    return x / (1.0 + np.exp(-x))


def softplus(x):
    return np.logaddexp(0.0, x)


def sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def causal_conv(C, x, w):
    """C: [..., K-1, d] previous raw inputs (oldest first); x: [..., d] the
    current one; w: [K, d] taps (tau = K-1 multiplies x).  Returns
    (silu output [..., d], new C)."""
    window = np.concatenate([C, x[..., None, :]], axis=-2)        # [..., K, d]
    y = silu(np.sum(window * w, axis=-2))
    return y, window[..., 1:, :]


def l2norm(x):
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + QK_EPS)


def gated_rmsnorm(o, g, gamma, eps):
    return gamma * o / np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + eps) * sigmoid(g)


def fused_step(S, C, xq, xk, xv, a, b, g, conv_w, norm_w, eps=1e-6):
    """One decode step for n sequences x H heads.

    S: [n, H, d, d] recurrent states; C: [n, H, 3, K-1, d] raw q, k, v of the
    previous K-1 tokens; xq, xk, xv, a, g: [n, H, d]; b: [n, H];
    conv_w: [H, 3, K, d]; norm_w: [H, d].
    Returns (y [n, H, d], S', C')."""
    S, C = _f64(S).copy(), _f64(C).copy()
    xq, xk, xv, a, b, g = (_f64(t) for t in (xq, xk, xv, a, b, g))
    conv_w, norm_w = _f64(conv_w), _f64(norm_w)
    yq, Cq = causal_conv(C[:, :, 0], xq, conv_w[None, :, 0])
    yk, Ck = causal_conv(C[:, :, 1], xk, conv_w[None, :, 1])
    yv, Cv = causal_conv(C[:, :, 2], xv, conv_w[None, :, 2])
    q, k, v = l2norm(yq), l2norm(yk), yv
    alpha = np.exp(-softplus(a))
    beta = sigmoid(b)
    Sp = alpha[..., :, None] * S                                   # Diag(alpha) S
    u = beta[..., None] * (v - np.einsum("nhi,nhij->nhj", k, Sp))
    S = Sp + k[..., :, None] * u[..., None, :]
    o = np.einsum("nhi,nhij->nhj", q, S)
    y = gated_rmsnorm(o, g, norm_w[None], eps)
    return y, S, np.stack([Cq, Ck, Cv], axis=2)
