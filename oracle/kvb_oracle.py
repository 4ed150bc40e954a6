"""Float64 oracle: what closed-form cross-model KV-cache transfer computes.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Plain, slow and obvious:
NumPy float64, library primitives (matmul, `np.linalg.solve`, sort) as single
steps, no blocking or fusion.  Pages cited by title and section:

* [KVBridge] "KVBridge" README -- capability table under "What ships";
  "Loading" (centered Chan/Welford statistics, ridge and intercept formula,
  planner sizes); "Real-model T2 evidence" (stride-sampled observations, mapper
  size); "Fitting from out-of-core shards" (FitConfig: top_k, ridge_alpha,
  float32 accumulation).
* [Velox] "Cross-Model KV Transfer -- Reuse One Model's Prefill in Another" --
  "The mapping" (K and V formulas, top-k selection, ridge on centered data,
  content space); "Configuration" (k=8, lambda=0.01, stride 4, 500 x 1024
  calibration); "Metal kernel" (single-rotation recode); "The honesty crux"
  item 7 (refused configurations).
* [Ember] "Before Mapping KV Caches, Make Them Measurable" -- "what became
  first-class" (cache order [layer][kv_head][position][dimension]).
* [React] "KV-Cache zwischen Qwen3-Modellen uebertragen statt neu zu prefillen"
  -- "Eine lineare Bruecke reicht" (fit_ridge / map_cache sketch, 500 x 1024
  calibration downsampled to ~128K observations per target head).

Conventions (readings where the pages leave a step open):

* cache tensors are [L][H][T][d] (Ember, "what became first-class");
* RoPE is rotate-half: pair (i, i + d/2), frequency w_i = theta^(-2i/d)
  (Velox "Metal kernel" prints a garbled exponent; rotate-half because the
  interleaved "traditional" form is refused, Velox "honesty crux" item 7);
* keys are RoPE-stripped with the source theta before mapping, the bias is
  added before the target RoPE, values carry no RoPE (Velox "The mapping");
* the features of target layer t are the selected source layers in ascending
  index, then kv head, then dim: column (j*H + h)*d + e (cross-head features,
  KVBridge "What ships"; the order itself is not printed);
* W is [p][q] with p = k*H*d inputs and q = H*d outputs; per-head maps with
  shared cross-head features are column blocks of this one ridge;
* lambda is absolute, added to the un-normalised centered Gram;
* stride keeps the tokens whose position is a multiple of the stride;
* K and V have separate selections; R^2 per head is pooled over the head's d
  columns (1 - sum SSE / sum SST), then averaged over heads; ties in R^2 go to
  the lower source index; the k selected layers are returned ascending.

Parity pins (tests/test_oracle_pins.py): rope, recode, ridge, centered_stats,
chan_merge, single_source_r2, select_top_k, map_apply, fit_mapper, the size
formulas and the attention-output cosine are all pinned.  `synthesize_pair`
builds test inputs and is checked only through the recovery pins.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Sequence

import numpy as np

__all__ = [
    "inv_freq", "rope", "strip", "recode", "features", "all_layer_features",
    "Stats", "centered_stats", "chan_merge", "stats_from_batches",
    "ridge_from_stats", "fit_ridge", "single_source_r2", "select_top_k",
    "map_apply", "fit_mapper", "FitResult", "retain_stride",
    "synthesize_pair", "head_pooled_r2", "mapper_param_count",
    "fit_stats_bytes", "stride_observations", "attention_output",
    "attention_cosine",
]


# ---------------------------------------------------------------------------
# RoPE: strip (inverse rotation) and apply (forward rotation)
# Velox "The mapping": K_hat = (strip_rope(K_s) . W_K + b_K) . target_rope.
# KVBridge "What ships": exact inverse/forward RoPE.
# ---------------------------------------------------------------------------

def inv_freq(theta: float, d: int) -> np.ndarray:
    """w_i = theta^(-2i/d) for pair index i < d/2, float64."""
    if d % 2:
        raise ValueError("head_dim must be even")
    i = np.arange(d // 2, dtype=np.float64)
    return np.power(np.float64(theta), -2.0 * i / d)


def rope(x: np.ndarray, pos: np.ndarray, theta: float, sign: int = +1) -> np.ndarray:
    """Rotate pairs (i, i+d/2) of x[..., T, d] by sign * pos[T] * w_i (float64).

    sign=+1 applies RoPE (as a model stores its keys), sign=-1 strips it.
    """
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    half = d // 2
    ang = np.asarray(pos, dtype=np.float64)[:, None] * inv_freq(theta, d)[None, :]
    c = np.cos(ang)
    s = np.sin(ang) * float(sign)
    x1 = x[..., :half]
    x2 = x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def strip(x, pos, theta):
    """Inverse RoPE: keys back to position-free content space."""
    return rope(x, pos, theta, -1)


def recode(x: np.ndarray, pos: np.ndarray, theta_s: float, theta_t: float) -> np.ndarray:
    """One rotation by pos * (w_t - w_s) per pair (Velox "Metal kernel").

    Valid only when no map sits between strip and apply; kept as a closed form
    that strip-then-apply must equal.
    """
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    half = d // 2
    dw = inv_freq(theta_t, d) - inv_freq(theta_s, d)
    ang = np.asarray(pos, dtype=np.float64)[:, None] * dw[None, :]
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


# ---------------------------------------------------------------------------
# Features: top-k cross-layer, cross-head concatenation
# KVBridge "What ships" (top-k cross-layer features, cross-head features);
# React "Eine lineare Bruecke reicht" (x concatenates the selected layers).
# ---------------------------------------------------------------------------

def features(cache: np.ndarray, sel_row: Sequence[int], pos=None, theta=None) -> np.ndarray:
    """X [T, k*H*d]: column (j*H + h)*d + e = cache[sel_row[j]][h][:, e].

    If theta is given the selected layers are RoPE-stripped with it first
    (keys); values pass theta=None.
    """
    cache = np.asarray(cache, dtype=np.float64)
    _, H, T, d = cache.shape
    blocks = []
    for l in sel_row:
        c = cache[int(l)]
        if theta is not None:
            c = strip(c, pos, theta)
        blocks.append(np.transpose(c, (1, 0, 2)).reshape(T, H * d))
    return np.concatenate(blocks, axis=1)


def all_layer_features(cache, pos=None, theta=None) -> np.ndarray:
    """Features over every layer of a cache, [T, L*H*d] (selection = all layers)."""
    return features(cache, range(np.asarray(cache).shape[0]), pos, theta)


def retain_stride(pos: np.ndarray, stride: int) -> np.ndarray:
    """Boolean mask of tokens kept by the deterministic stride (pos % stride == 0).

    Velox "Configuration" (stride 4); KVBridge "Modest-host fitting"
    (deterministic token stride).
    """
    return (np.asarray(pos) % int(stride)) == 0


# ---------------------------------------------------------------------------
# Centered sufficient statistics with Chan merges
# KVBridge "Loading": only centered sufficient statistics are retained;
# batchwise Chan/Welford updates accumulate the centered covariance directly.
# ---------------------------------------------------------------------------

@dataclass
class Stats:
    n: int
    xbar: np.ndarray      # [p]
    ybar: np.ndarray      # [q]
    M: np.ndarray         # [p][p]  sum (x - xbar)(x - xbar)^T
    C: np.ndarray         # [p][q]  sum (x - xbar)(y - ybar)^T
    syy: np.ndarray       # [q]     sum (y - ybar)^2


def centered_stats(X: np.ndarray, Y: np.ndarray) -> Stats:
    """Two-pass centered statistics of one batch of observations (rows)."""
    X = np.asarray(X, dtype=np.float64)
    Y = np.asarray(Y, dtype=np.float64)
    n = X.shape[0]
    xbar = X.mean(axis=0)
    ybar = Y.mean(axis=0)
    Xc = X - xbar
    Yc = Y - ybar
    return Stats(n, xbar, ybar, Xc.T @ Xc, Xc.T @ Yc, (Yc * Yc).sum(axis=0))


def chan_merge(a: Stats, b: Stats) -> Stats:
    """Merge two centered summaries (Chan, Golub & LeVeque pairwise update)."""
    if a.n == 0:
        return b
    if b.n == 0:
        return a
    n = a.n + b.n
    dx = b.xbar - a.xbar
    dy = b.ybar - a.ybar
    f = a.n * b.n / n
    return Stats(
        n,
        a.xbar + dx * (b.n / n),
        a.ybar + dy * (b.n / n),
        a.M + b.M + f * np.outer(dx, dx),
        a.C + b.C + f * np.outer(dx, dy),
        a.syy + b.syy + f * dy * dy,
    )


def stats_from_batches(batches) -> Stats:
    """Fold (X_b, Y_b) batches in order with Chan merges."""
    acc = None
    for X, Y in batches:
        s = centered_stats(X, Y)
        acc = s if acc is None else chan_merge(acc, s)
    return acc


# ---------------------------------------------------------------------------
# Ridge on centered data, intercept unpenalised
# KVBridge "Loading": W = (X^T X + lambda I)^-1 X^T Y, b = Ybar - Xbar W.
# React "Eine lineare Bruecke reicht": fit_ridge centers x and y, solves, and
# forms b from the means.  Velox "The mapping": lambda = 0.01.
# ---------------------------------------------------------------------------

def ridge_from_stats(st: Stats, lam: float):
    """W [p][q] = solve(M + lam I, C); b [q] = ybar - xbar W."""
    p = st.M.shape[0]
    W = np.linalg.solve(st.M + lam * np.eye(p), st.C)
    b = st.ybar - st.xbar @ W
    return W, b


def fit_ridge(X: np.ndarray, Y: np.ndarray, lam: float = 0.01):
    """Ridge with intercept on raw observations (rows of X, Y)."""
    return ridge_from_stats(centered_stats(X, Y), lam)


# ---------------------------------------------------------------------------
# Single-source R^2 and top-k selection
# KVBridge "What ships": head-averaged single-source R^2, then top-k.
# Velox "The mapping" item 1: each target layer is fit from its k best
# predicting source layers.
# ---------------------------------------------------------------------------

def head_pooled_r2(Y_true: np.ndarray, Y_pred: np.ndarray, H: int, d: int,
                   ybar: np.ndarray | None = None) -> float:
    """Mean over heads of 1 - sum SSE / sum SST over each head's d columns.

    SST is taken about ybar (the column means of Y_true unless given).
    """
    Y_true = np.asarray(Y_true, dtype=np.float64)
    Y_pred = np.asarray(Y_pred, dtype=np.float64)
    if ybar is None:
        ybar = Y_true.mean(axis=0)
    sse = ((Y_true - Y_pred) ** 2).sum(axis=0)
    sst = ((Y_true - ybar) ** 2).sum(axis=0)
    r = [1.0 - sse[h * d:(h + 1) * d].sum() / sst[h * d:(h + 1) * d].sum() for h in range(H)]
    return float(np.mean(r))


def single_source_r2(Xs: Sequence[np.ndarray], Yt: Sequence[np.ndarray], lam: float,
                     H: int, d: int) -> np.ndarray:
    """R2[t][s]: in-sample head-averaged R^2 of a ridge fit of target t from source s.

    Xs[s] is [N, H*d] (source layer s over the retained observations), Yt[t]
    is [N, H*d].  Every pair is fitted explicitly and its residual formed
    directly (no closed-form shortcut).
    """
    L_s, L_t = len(Xs), len(Yt)
    out = np.empty((L_t, L_s), dtype=np.float64)
    for t in range(L_t):
        for s in range(L_s):
            W, b = fit_ridge(Xs[s], Yt[t], lam)
            pred = np.asarray(Xs[s], dtype=np.float64) @ W + b
            out[t, s] = head_pooled_r2(Yt[t], pred, H, d)
    return out


def select_top_k(r2: np.ndarray, k: int):
    """Per target row: the k source layers with largest R^2, ties to the lower index.

    Returns (sel int32 [L_t][k] ascending, margin float64 [L_t]) where margin is
    the gap between the k-th and (k+1)-th ranked R^2 (inf when k == L_s).
    """
    r2 = np.asarray(r2, dtype=np.float64)
    L_t, L_s = r2.shape
    sel = np.empty((L_t, k), dtype=np.int32)
    margin = np.full(L_t, np.inf)
    for t in range(L_t):
        order = sorted(range(L_s), key=lambda s: (-r2[t, s], s))
        sel[t] = np.sort(order[:k])
        if k < L_s:
            margin[t] = r2[t, order[k - 1]] - r2[t, order[k]]
    return sel, margin


# ---------------------------------------------------------------------------
# Apply: Velox "The mapping" and React map_cache
#   K_hat = rope_t(strip_s(K_s)[sel] W_K + b_K),  V_hat = V_s[sel] W_V + b_V
# ---------------------------------------------------------------------------

def map_apply(src_k, src_v, pos, sel_k, sel_v, W_k, b_k, W_v, b_v, theta_s, theta_t, H, d):
    """Target caches [L_t][H][T][d] (float64) from source caches [L_s][H][T][d]."""
    src_k = np.asarray(src_k, dtype=np.float64)
    src_v = np.asarray(src_v, dtype=np.float64)
    T = src_k.shape[2]
    L_t = len(sel_k)
    out_k = np.empty((L_t, H, T, d))
    out_v = np.empty((L_t, H, T, d))
    for t in range(L_t):
        Xk = features(src_k, sel_k[t], pos, theta_s)
        Yk = Xk @ np.asarray(W_k[t], dtype=np.float64) + np.asarray(b_k[t], dtype=np.float64)
        out_k[t] = rope(np.transpose(Yk.reshape(T, H, d), (1, 0, 2)), pos, theta_t, +1)
        Xv = features(src_v, sel_v[t])
        Yv = Xv @ np.asarray(W_v[t], dtype=np.float64) + np.asarray(b_v[t], dtype=np.float64)
        out_v[t] = np.transpose(Yv.reshape(T, H, d), (1, 0, 2))
    return out_k, out_v


# ---------------------------------------------------------------------------
# Whole fit, in the pages' order (KVBridge "System design" flowchart and
# "Loading"): strip source RoPE -> stride -> centered statistics -> single
# source R^2 -> top-k -> ridge per target layer.
# ---------------------------------------------------------------------------

@dataclass
class FitResult:
    sel_k: np.ndarray
    sel_v: np.ndarray
    W_k: np.ndarray      # [L_t][p][q]
    b_k: np.ndarray      # [L_t][q]
    W_v: np.ndarray
    b_v: np.ndarray
    r2_k: np.ndarray     # [L_t][L_s]
    r2_v: np.ndarray
    margin_k: np.ndarray
    margin_v: np.ndarray
    n_obs: int


def _layer_block(F: np.ndarray, l: int, width: int) -> np.ndarray:
    return F[:, l * width:(l + 1) * width]


def fit_mapper(calib, theta_s: float, theta_t: float, k: int, lam: float = 0.01,
               stride: int = 4) -> FitResult:
    """Fit K and V maps from calibration sequences.

    calib: iterable of (src_k, src_v, tgt_k, tgt_v, pos) with caches
    [L][H][T][d] (keys as stored, i.e. with RoPE) and pos [T].
    """
    XK, XV, YK, YV = [], [], [], []
    H = d = None
    for src_k, src_v, tgt_k, tgt_v, pos in calib:
        pos = np.asarray(pos)
        keep = retain_stride(pos, stride)
        _, H, _, d = np.asarray(src_k).shape
        XK.append(all_layer_features(src_k, pos, theta_s)[keep])
        XV.append(all_layer_features(src_v)[keep])
        YK.append(all_layer_features(tgt_k, pos, theta_t)[keep])
        YV.append(all_layer_features(tgt_v)[keep])
    XK, XV, YK, YV = (np.concatenate(a, axis=0) for a in (XK, XV, YK, YV))
    q = H * d
    L_s = XK.shape[1] // q
    L_t = YK.shape[1] // q

    out = {}
    for name, X, Y in (("k", XK, YK), ("v", XV, YV)):
        Xs = [_layer_block(X, s, q) for s in range(L_s)]
        Yt = [_layer_block(Y, t, q) for t in range(L_t)]
        r2 = single_source_r2(Xs, Yt, lam, H, d)
        sel, margin = select_top_k(r2, k)
        W = np.empty((L_t, k * q, q))
        b = np.empty((L_t, q))
        for t in range(L_t):
            Xt = np.concatenate([Xs[s] for s in sel[t]], axis=1)
            W[t], b[t] = fit_ridge(Xt, Yt[t], lam)
        out[name] = (sel, W, b, r2, margin)
    return FitResult(out["k"][0], out["v"][0], out["k"][1], out["k"][2], out["v"][1],
                     out["v"][2], out["k"][3], out["v"][3], out["k"][4], out["v"][4],
                     XK.shape[0])


# ---------------------------------------------------------------------------
# Test-input composition (not part of the method; builds synthetic pairs)
# ---------------------------------------------------------------------------

def synthesize_pair(content_k, content_v, pos, theta_s, theta_t, sel_k, sel_v,
                    W_k, b_k, W_v, b_v, noise_k=None, noise_v=None, noise_scale=0.0):
    """Stored caches of a synthetic pair with a hidden cross-layer affine map.

    Source keys are stored with source RoPE applied to their content; the target
    content is features(content) W + b + noise_scale * noise, and target keys
    are stored with target RoPE.  noise_scale may be a scalar or an array
    broadcastable to [L_t][q].
    """
    content_k = np.asarray(content_k, dtype=np.float64)
    content_v = np.asarray(content_v, dtype=np.float64)
    _, H, T, d = content_k.shape
    L_t = len(sel_k)
    ns = np.broadcast_to(np.asarray(noise_scale, dtype=np.float64), (L_t, H * d))
    src_k = rope(content_k, pos, theta_s, +1)
    src_v = content_v.copy()
    tgt_k = np.empty((L_t, H, T, d))
    tgt_v = np.empty((L_t, H, T, d))
    for t in range(L_t):
        yk = features(content_k, sel_k[t]) @ W_k[t] + b_k[t]
        yv = features(content_v, sel_v[t]) @ W_v[t] + b_v[t]
        if noise_k is not None:
            yk = yk + ns[t] * noise_k[t]
        if noise_v is not None:
            yv = yv + ns[t] * noise_v[t]
        tgt_k[t] = rope(np.transpose(yk.reshape(T, H, d), (1, 0, 2)), pos, theta_t, +1)
        tgt_v[t] = np.transpose(yv.reshape(T, H, d), (1, 0, 2))
    return src_k, src_v, tgt_k, tgt_v


# ---------------------------------------------------------------------------
# Size formulas (KVBridge "Loading" planner figures; "Real-model T2 evidence";
# React "Eine lineare Bruecke reicht" observation count)
# ---------------------------------------------------------------------------

def mapper_param_count(L_t: int, k: int, H: int, d: int) -> int:
    """Parameters of a K+V mapper: per target layer W_K, W_V [k*H*d][H*d] and b_K, b_V [H*d]."""
    p, q = k * H * d, H * d
    return L_t * 2 * (p * q + q)


def fit_stats_bytes(k: int, H: int, d: int, layers_per_block: int = 1, itemsize: int = 4) -> int:
    """Bytes of the centered Gram (K and V) and cross statistics (K and V) of one block."""
    p, q = k * H * d, H * d
    return layers_per_block * itemsize * (2 * p * p + 2 * p * q)


def stride_observations(n_sequences: int, seq_len: int, stride: int) -> int:
    """Observations kept from n_sequences x seq_len tokens with positions 0..seq_len-1."""
    return n_sequences * int(np.sum(retain_stride(np.arange(seq_len), stride)))


# ---------------------------------------------------------------------------
# Attention-output cosine (quality diagnostic)
# KVBridge "Real-model T2 evidence": the gate is on the mean and the minimum
# of the attention-output cosine; KVBridge "Scope and limitations" and Velox
# "The honesty crux" item 6: this cosine, not the calibration R^2, tracks
# downstream retention; Velox "What is not implemented" lists it as the
# screen to run on a pair before deploying it.
# ---------------------------------------------------------------------------

def attention_output(q, q_pos, k, v, kv_pos) -> np.ndarray:
    """o[l][hq][i] = sum over visible j of softmax_j(q_i . k_j / sqrt(d)) v_j.

    q is [L][Hq][Tq][d] (post-RoPE target queries), k and v are [L][H][T][d]
    (post-RoPE keys, as caches store them).  Query head hq reads KV head
    hq // (Hq / H) (grouped-query attention).  Key j is visible to query i
    iff kv_pos[j] <= q_pos[i] (causal by position within one sequence).  A
    query with no visible key gets the zero vector.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    L, Hq, Tq, d = q.shape
    H = k.shape[1]
    if Hq % H:
        raise ValueError("query heads must be a multiple of the KV heads")
    g = Hq // H
    visible = np.asarray(kv_pos)[None, :] <= np.asarray(q_pos)[:, None]   # [Tq][T]
    out = np.zeros((L, Hq, Tq, d))
    for l in range(L):
        for hq in range(Hq):
            kh = hq // g
            scores = q[l, hq] @ k[l, kh].T / np.sqrt(d)
            for i in range(Tq):
                if not visible[i].any():
                    continue
                s = scores[i][visible[i]]
                w = np.exp(s - s.max())
                out[l, hq, i] = (w / w.sum()) @ v[l, kh][visible[i]]
    return out


def attention_cosine(q, q_pos, k_a, v_a, k_b, v_b, kv_pos) -> np.ndarray:
    """cos(o_a, o_b) per [L][Hq][Tq] row, o_x = attention_output with cache x.

    Cache a is the one under test (the mapped cache), cache b the reference
    (the target's own prefill).  The cosine is 0 where either output is zero.
    """
    oa = attention_output(q, q_pos, k_a, v_a, kv_pos)
    ob = attention_output(q, q_pos, k_b, v_b, kv_pos)
    dot = (oa * ob).sum(axis=-1)
    den = np.sqrt((oa * oa).sum(axis=-1)) * np.sqrt((ob * ob).sum(axis=-1))
    return np.where(den > 0, dot / np.where(den > 0, den, 1.0), 0.0)
