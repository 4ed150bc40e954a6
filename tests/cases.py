"""Shared helpers of the GPU parity tests: seeded inputs, oracle calls on
(possibly sampled) slices, error measures.  Tests only."""
from __future__ import annotations

import numpy as np

import oracle as O
import synth

# Tolerances stated for this path: relative Frobenius error of mapped caches.
TOL_F32 = 1e-4
TOL_BF16 = 1e-2
TOL_W = 1e-3
# Attention-output cosine: absolute error per row.  fp32 dot products of
# length d <= 128 and softmax sums over a few thousand keys carry relative
# errors near 1e-6 (plus the fast exponential's ~2^-21); a cosine moves by at
# most the relative error of its two outputs, so 1e-4 leaves a wide margin.
TOL_COS = 1e-4


def rel_fro(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def to_host64(t) -> np.ndarray:
    import torch
    return t.detach().to(device="cpu", dtype=torch.float64).numpy()


class ApplyCase:
    """Inputs of one kvb_map_apply call, on the device, plus their exact host values."""

    def __init__(self, L_s, L_t, H, d, k, T, theta_s, theta_t, dtype, seed, positions=None, sigma=1.0,
                 device="cuda", host=True):
        import torch
        self.L_s, self.L_t, self.H, self.d, self.k, self.T = L_s, L_t, H, d, k, T
        self.theta_s, self.theta_t = theta_s, theta_t
        self.dtype = dtype
        p, q = k * H * d, H * d
        self.sel_k = synth.hidden_selection(seed + 1, L_s, L_t, k)
        self.sel_v = synth.hidden_selection(seed + 2, L_s, L_t, k)
        if positions is None:
            positions = np.arange(T, dtype=np.int32)
        self.positions_host = np.asarray(positions, dtype=np.int32)
        self.positions = torch.from_numpy(self.positions_host).to(device)
        if host:
            ck = synth.content(seed + 3, L_s, H, T, d, sigma)
            cv = synth.content(seed + 4, L_s, H, T, d, sigma)
            Wk, bk = synth.hidden_weights(seed + 5, L_t, p, q)
            Wv, bv = synth.hidden_weights(seed + 6, L_t, p, q)
            self.src_k = torch.from_numpy(ck).to(device=device, dtype=dtype)
            self.src_v = torch.from_numpy(cv).to(device=device, dtype=dtype)
            # device weights are output-major [L_t][q][p]
            self.W_k = torch.from_numpy(np.ascontiguousarray(np.transpose(Wk, (0, 2, 1)))).to(device=device, dtype=dtype)
            self.W_v = torch.from_numpy(np.ascontiguousarray(np.transpose(Wv, (0, 2, 1)))).to(device=device, dtype=dtype)
            self.b_k = torch.from_numpy(bk).to(device=device, dtype=torch.float32)
            self.b_v = torch.from_numpy(bv).to(device=device, dtype=torch.float32)
        else:
            self.src_k = synth.torch_content(seed + 3, L_s, H, T, d, sigma, dtype, device)
            self.src_v = synth.torch_content(seed + 4, L_s, H, T, d, sigma, dtype, device)
            self.W_k, self.b_k = synth.torch_weights(seed + 5, L_t, p, q, dtype, device)
            self.W_v, self.b_v = synth.torch_weights(seed + 6, L_t, p, q, dtype, device)
        self.out_k = torch.empty((L_t, H, T, d), dtype=dtype, device=device)
        self.out_v = torch.empty((L_t, H, T, d), dtype=dtype, device=device)

    def run(self, kvb, ctx):
        kvb.kvb_map_apply(ctx, self.src_k, self.src_v, self.positions, self.sel_k, self.sel_v, self.W_k,
                          self.W_v, self.b_k, self.b_v, self.out_k, self.out_v)

    def oracle(self, layers=None, tokens=None):
        """Oracle caches for target `layers` (default all) at `tokens` (default all)."""
        if layers is None:
            layers = np.arange(self.L_t)
        if tokens is None:
            tokens = np.arange(self.T)
        tokens = np.asarray(tokens)
        import torch
        idx = torch.from_numpy(tokens).to(self.src_k.device)
        sk = to_host64(self.src_k.index_select(2, idx))
        sv = to_host64(self.src_v.index_select(2, idx))
        li = torch.from_numpy(np.asarray(layers)).to(self.src_k.device)
        Wk = np.transpose(to_host64(self.W_k.index_select(0, li)), (0, 2, 1))
        Wv = np.transpose(to_host64(self.W_v.index_select(0, li)), (0, 2, 1))
        bk = to_host64(self.b_k.index_select(0, li))
        bv = to_host64(self.b_v.index_select(0, li))
        return O.map_apply(sk, sv, self.positions_host[tokens], self.sel_k[layers], self.sel_v[layers], Wk, bk,
                           Wv, bv, self.theta_s, self.theta_t, self.H, self.d)

    def gpu(self, layers=None, tokens=None):
        import torch
        ok, ov = self.out_k, self.out_v
        if layers is not None:
            li = torch.from_numpy(np.asarray(layers)).to(ok.device)
            ok, ov = ok.index_select(0, li), ov.index_select(0, li)
        if tokens is not None:
            ti = torch.from_numpy(np.asarray(tokens)).to(ok.device)
            ok, ov = ok.index_select(2, ti), ov.index_select(2, ti)
        return to_host64(ok), to_host64(ov)


def spec(L, H, d, theta):
    return {"n_layers": L, "n_kv_heads": H, "head_dim": d, "rope_theta": theta}


def make_pair(seed, L_s, L_t, H, d, k, T, n_seq, theta_s, theta_t, noise=1e-3, sigma=0.5, positions=None):
    """Synthetic calibration pair with a hidden cross-layer affine map (composed by the oracle).

    Returns dict(calib=[(src_k, src_v, tgt_k, tgt_v, pos)] * n_seq, holdout=(...), sel_k, sel_v, ...),
    float64 host arrays.  `positions` (list per sequence) defaults to 0..T-1.
    """
    p, q = k * H * d, H * d
    sel_k = synth.hidden_selection(seed + 1, L_s, L_t, k)
    sel_v = synth.hidden_selection(seed + 2, L_s, L_t, k)
    Wk, bk = synth.hidden_weights(seed + 3, L_t, p, q)
    Wv, bv = synth.hidden_weights(seed + 4, L_t, p, q)
    seqs = []
    for i in range(n_seq + 1):
        pos = np.arange(T) if positions is None else np.asarray(positions[i])
        Ti = len(pos)
        ck = synth.content(seed + 100 + i, L_s, H, Ti, d, sigma)
        cv = synth.content(seed + 200 + i, L_s, H, Ti, d, sigma)
        nk = synth.noise(seed + 300 + i, (L_t, Ti, q))
        nv = synth.noise(seed + 400 + i, (L_t, Ti, q))
        seqs.append(O.synthesize_pair(ck, cv, pos, theta_s, theta_t, sel_k, sel_v, Wk, bk, Wv, bv, nk, nv,
                                      noise) + (pos,))
    return dict(calib=seqs[:n_seq], holdout=seqs[n_seq], sel_k=sel_k, sel_v=sel_v, theta_s=theta_s,
                theta_t=theta_t, L_s=L_s, L_t=L_t, H=H, d=d, k=k)


def round_pair(pair, dtype):
    """Round every cache of a pair to `dtype` (torch dtype); returns host float64 copies of the rounded values."""
    import torch

    def r(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dtype).to(torch.float64).numpy()

    out = dict(pair)
    out["calib"] = [tuple(r(x) for x in s[:4]) + (s[4],) for s in pair["calib"]]
    h = pair["holdout"]
    out["holdout"] = tuple(r(x) for x in h[:4]) + (h[4],)
    return out


def oracle_full_stats(pair, stride=4):
    """Oracle centered statistics over ALL source features / target columns, K and V."""
    XK, XV, YK, YV = [], [], [], []
    for src_k, src_v, tgt_k, tgt_v, pos in pair["calib"]:
        keep = O.retain_stride(pos, stride)
        XK.append(O.all_layer_features(src_k, pos, pair["theta_s"])[keep])
        XV.append(O.all_layer_features(src_v)[keep])
        YK.append(O.all_layer_features(tgt_k, pos, pair["theta_t"])[keep])
        YV.append(O.all_layer_features(tgt_v)[keep])
    cat = lambda a: np.concatenate(a, axis=0)
    return O.centered_stats(cat(XK), cat(YK)), O.centered_stats(cat(XV), cat(YV))
