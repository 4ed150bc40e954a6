"""Random draws for the synthetic cache pairs (see the package docstring)."""
from __future__ import annotations

import numpy as np


def _rng(seed) -> np.random.Generator:
    return np.random.default_rng(seed)


def channel_scales(seed, L: int, H: int, d: int, sigma: float) -> np.ndarray:
    """Per-channel log-normal scales exp(N(0, sigma^2)), shape [L][H][1][d]."""
    r = _rng(seed)
    return np.exp(sigma * r.standard_normal((L, H, 1, d)))


def content(seed, L: int, H: int, T: int, d: int, sigma: float) -> np.ndarray:
    """Float64 content [L][H][T][d]: N(0,1) times per-channel log-normal scales."""
    r = _rng(seed)
    s = np.exp(sigma * r.standard_normal((L, H, 1, d)))
    return r.standard_normal((L, H, T, d)) * s


def hidden_selection(seed, L_src: int, L_tgt: int, k: int) -> np.ndarray:
    """Per target layer, k distinct source layers in ascending order: int32 [L_tgt][k]."""
    if not 1 <= k <= L_src:
        raise ValueError("need 1 <= k <= L_src")
    r = _rng(seed)
    out = np.empty((L_tgt, k), dtype=np.int32)
    for t in range(L_tgt):
        out[t] = np.sort(r.choice(L_src, size=k, replace=False))
    return out


def hidden_weights(seed, L_tgt: int, p: int, q: int, bias_std: float = 0.1):
    """Hidden affine maps: W [L_tgt][p][q] ~ N(0,1)/sqrt(p), b [L_tgt][q] ~ N(0, bias_std^2)."""
    r = _rng(seed)
    W = r.standard_normal((L_tgt, p, q)) / np.sqrt(p)
    b = bias_std * r.standard_normal((L_tgt, q))
    return W, b


def noise(seed, shape) -> np.ndarray:
    """Standard-normal noise draws; the consumer scales them."""
    return _rng(seed).standard_normal(shape)


def ragged_lengths(seed, n: int, lo: int, hi: int) -> np.ndarray:
    """n sequence lengths, uniform integers in [lo, hi]."""
    return _rng(seed).integers(lo, hi + 1, size=n).astype(np.int64)


def packed_positions(lengths) -> np.ndarray:
    """Positions for sequences packed on the token axis, restarting at 0 per sequence."""
    lengths = np.asarray(lengths, dtype=np.int64)
    if lengths.size == 0:
        return np.zeros(0, dtype=np.int32)
    return np.concatenate([np.arange(n, dtype=np.int32) for n in lengths])


# ---------------------------------------------------------------------------
# Device-side draws for workloads too large to generate on the host.  Same
# recipe, drawn with torch's seeded generator directly in device memory.
# ---------------------------------------------------------------------------

def torch_content(seed, L: int, H: int, T: int, d: int, sigma: float, dtype, device):
    """Content [L][H][T][d] in `dtype` on `device`, recipe as `content`."""
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    out = torch.empty((L, H, T, d), dtype=dtype, device=device)
    s = torch.exp(sigma * torch.randn((L, H, 1, d), generator=g, device=device, dtype=torch.float32))
    for l in range(L):  # one layer at a time bounds the fp32 temporary
        x = torch.randn((H, T, d), generator=g, device=device, dtype=torch.float32)
        out[l].copy_(x * s[l])
    return out


def torch_content_shared(seed, L: int, H: int, T: int, d: int, sigma: float, rho: float, dtype, device):
    """Content [L][H][T][d] whose layers share one component: for every layer,
    s_ch * (rho * z + sqrt(1 - rho^2) * e_l), z and e_l standard normal, z the
    same draw [H][T][d] for every layer.  Each channel is N(0, s_ch^2) as in
    `content`; two layers correlate by rho^2 channel by channel (the layers of
    one model's cache are correlated through its residual stream)."""
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    out = torch.empty((L, H, T, d), dtype=dtype, device=device)
    s = torch.exp(sigma * torch.randn((L, H, 1, d), generator=g, device=device, dtype=torch.float32))
    z = torch.randn((H, T, d), generator=g, device=device, dtype=torch.float32)
    a, b = float(rho), float(np.sqrt(1.0 - rho * rho))
    for l in range(L):
        x = torch.randn((H, T, d), generator=g, device=device, dtype=torch.float32)
        out[l].copy_((a * z + b * x) * s[l])
    return out


def torch_weights(seed, L_tgt: int, p: int, q: int, dtype, device, bias_std: float = 0.1,
                  out_major: bool = True):
    """Hidden weights on `device`.

    With out_major=True the weights come as [L_tgt][q][p] (row n holds the p input
    weights of output n), otherwise [L_tgt][p][q].  Bias is fp32 [L_tgt][q].
    """
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    shape = (L_tgt, q, p) if out_major else (L_tgt, p, q)
    W = torch.empty(shape, dtype=dtype, device=device)
    for t in range(L_tgt):
        w = torch.randn(shape[1:], generator=g, device=device, dtype=torch.float32)
        W[t].copy_(w / float(np.sqrt(p)))
    b = bias_std * torch.randn((L_tgt, q), generator=g, device=device, dtype=torch.float32)
    return W, b
