"""Pins for the float64 oracle, against what the pages and the mathematics fix.

No test here re-types an oracle formula: each one checks the oracle against an
independent route (a hand-computed value, a different formulation, a library
special case, brute force, a printed figure of the pages or an identity).
"""
import itertools
import math
import os

import numpy as np
import pytest

import oracle as O
import synth


def _golden(golden_dir):
    vals = {}
    with open(os.path.join(golden_dir, "page_figures.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, v = (s.strip() for s in line.split("="))
                vals[k] = float(v)
    return vals


# --------------------------------------------------------------------------
# RoPE
# --------------------------------------------------------------------------

def test_rope_hand_values():
    # d = 2: one pair, frequency theta^0 = 1, so position 1 rotates by 1 rad.
    y = O.rope(np.array([[[1.0, 0.0]]]), np.array([1]), 1e4, +1)
    assert np.allclose(y[0, 0], [math.cos(1.0), math.sin(1.0)], atol=1e-15)
    # d = 4, theta = 1e4: pair 1 is (index 1, index 3) with frequency 1e4^(-1/2) = 0.01;
    # position 100 rotates it by exactly 1 rad, pair 0 by 100 rad.
    x = np.zeros((1, 1, 4))
    x[0, 0, 1] = 1.0
    y = O.rope(x, np.array([100]), 1e4, +1)
    assert np.allclose(y[0, 0], [0.0, math.cos(1.0), 0.0, math.sin(1.0)], atol=1e-14)
    x = np.zeros((1, 1, 4))
    x[0, 0, 0] = 1.0
    y = O.rope(x, np.array([100]), 1e4, +1)
    assert np.allclose(y[0, 0], [math.cos(100.0), 0.0, math.sin(100.0), 0.0], atol=1e-13)


def test_rope_bias_is_rotated_after_being_added():
    # W = 0, b = (1, 0): the mapped key at position 1 is the rotated bias (cos 1, sin 1).
    src = np.zeros((1, 1, 2, 2))
    pos = np.array([0, 1])
    out_k, out_v = O.map_apply(src, src, pos, [[0]], [[0]], np.zeros((1, 2, 2)),
                               np.array([[1.0, 0.0]]), np.zeros((1, 2, 2)),
                               np.array([[1.0, 0.0]]), 1e4, 5e4, 1, 2)
    assert np.allclose(out_k[0, 0, 0], [1.0, 0.0])
    assert np.allclose(out_k[0, 0, 1], [math.cos(1.0), math.sin(1.0)])
    assert np.allclose(out_v[0, 0, 1], [1.0, 0.0])   # values carry no RoPE


def test_rope_complex_multiplication_form():
    rng = np.random.default_rng(0)
    d, T, theta = 16, 37, 5e5
    x = rng.standard_normal((3, T, d))
    pos = rng.integers(0, 40000, size=T)
    y = O.rope(x, pos, theta, +1)
    z = x[..., : d // 2] + 1j * x[..., d // 2:]
    i = np.arange(d // 2)
    rot = np.exp(1j * np.outer(pos, np.exp(-(2.0 * i / d) * np.log(theta))))
    zz = z * rot
    assert np.allclose(y, np.concatenate([zz.real, zz.imag], axis=-1), atol=1e-12)


def test_rope_roundtrip_norm_and_position_zero():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((2, 3, 50, 128))
    pos = rng.integers(0, 32768, size=50)
    for theta in (1e4, 5e5, 1e6):
        a = O.rope(O.strip(x, pos, theta), pos, theta, +1)
        b = O.strip(O.rope(x, pos, theta, +1), pos, theta)
        assert np.max(np.abs(a - x)) < 1e-13 and np.max(np.abs(b - x)) < 1e-13
        y = O.rope(x, pos, theta, +1)
        assert np.allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-14)
    z = O.rope(x, np.zeros(50, dtype=int), 1e6, +1)
    assert np.array_equal(z, x)


def test_rope_relative_position_property():
    # <rope(q, m), rope(k, n)> depends on m - n only (the defining RoPE property).
    rng = np.random.default_rng(2)
    q = rng.standard_normal((1, 1, 64))
    k = rng.standard_normal((1, 1, 64))
    for m, n, s in ((5, 3, 100), (0, 17, 31000), (1234, 1000, 7)):
        a = np.sum(O.rope(q, [m], 1e6) * O.rope(k, [n], 1e6))
        b = np.sum(O.rope(q, [m + s], 1e6) * O.rope(k, [n + s], 1e6))
        assert abs(a - b) < 1e-10


def test_recode_equals_strip_then_apply():
    # Velox "Metal kernel": strip with theta_s then apply theta_t is one rotation by
    # pos * (w_t - w_s) per pair.
    rng = np.random.default_rng(3)
    x = rng.standard_normal((4, 64, 128))
    pos = np.arange(64) * 511
    two = O.rope(O.strip(x, pos, 1e4), pos, 1e6, +1)
    assert np.max(np.abs(two - O.recode(x, pos, 1e4, 1e6))) < 1e-11


# --------------------------------------------------------------------------
# Features
# --------------------------------------------------------------------------

def test_feature_column_order_layer_then_head_then_dim():
    L, H, T, d = 5, 3, 4, 6
    idx = np.zeros((L, H, T, d))
    for l, h, t, e in itertools.product(range(L), range(H), range(T), range(d)):
        idx[l, h, t, e] = 1000 * l + 100 * h + 10 * t + e
    sel = [1, 4]
    X = O.features(idx, sel)
    assert X.shape == (T, len(sel) * H * d)
    for j, l in enumerate(sel):
        for h in range(H):
            for e in range(d):
                assert np.all(X[:, (j * H + h) * d + e] == 1000 * l + 100 * h + 10 * np.arange(T) + e)


# --------------------------------------------------------------------------
# Ridge
# --------------------------------------------------------------------------

def _gauss_jordan_solve(A, B):
    """Plain Gauss-Jordan elimination with partial pivoting on [A | B]."""
    A = np.array(A, dtype=np.float64)
    B = np.array(B, dtype=np.float64)
    n = A.shape[0]
    Aug = np.concatenate([A, B], axis=1)
    for c in range(n):
        r = c + int(np.argmax(np.abs(Aug[c:, c])))
        Aug[[c, r]] = Aug[[r, c]]
        Aug[c] /= Aug[c, c]
        for rr in range(n):
            if rr != c:
                Aug[rr] -= Aug[rr, c] * Aug[c]
    return Aug[:, n:]


def test_ridge_equals_bruteforce_normal_equations():
    rng = np.random.default_rng(4)
    X = rng.standard_normal((40, 6)) * np.array([1, 3, 0.2, 5, 1, 1]) + 7.0
    Y = rng.standard_normal((40, 3)) - 2.0
    lam = 0.37
    W, b = O.fit_ridge(X, Y, lam)
    xm = X.sum(0) / 40
    ym = Y.sum(0) / 40
    Xc = X - xm
    Yc = Y - ym
    A = np.zeros((6, 6))
    for i in range(6):
        for j in range(6):
            A[i, j] = sum(Xc[n, i] * Xc[n, j] for n in range(40)) + (lam if i == j else 0.0)
    Bm = np.array([[sum(Xc[n, i] * Yc[n, j] for n in range(40)) for j in range(3)] for i in range(6)])
    Wg = _gauss_jordan_solve(A, Bm)
    assert np.allclose(W, Wg, atol=1e-12)
    assert np.allclose(b, ym - xm @ Wg, atol=1e-12)


def test_ridge_matches_sklearn():
    sk = pytest.importorskip("sklearn.linear_model")
    rng = np.random.default_rng(5)
    X = rng.standard_normal((200, 12)) * rng.uniform(0.1, 4, 12) + rng.standard_normal(12)
    Y = X @ rng.standard_normal((12, 5)) + rng.standard_normal((200, 5))
    for lam in (0.01, 3.0):
        W, b = O.fit_ridge(X, Y, lam)
        m = sk.Ridge(alpha=lam, fit_intercept=True, solver="cholesky").fit(X, Y)
        assert np.allclose(W, m.coef_.T, atol=1e-10)
        assert np.allclose(b, m.intercept_, atol=1e-10)


def test_ridge_limits_and_shift_invariance():
    rng = np.random.default_rng(6)
    X = rng.standard_normal((100, 8))
    Y = X @ rng.standard_normal((8, 4)) + 0.1 * rng.standard_normal((100, 4)) + 3.0
    # lambda -> 0: ordinary least squares with an intercept column.
    W0, b0 = O.fit_ridge(X, Y, 1e-12)
    coef, *_ = np.linalg.lstsq(np.concatenate([X, np.ones((100, 1))], axis=1), Y, rcond=None)
    assert np.allclose(W0, coef[:8], atol=1e-9) and np.allclose(b0, coef[8], atol=1e-9)
    # lambda -> infinity: W -> 0, b -> mean of Y.
    Wi, bi = O.fit_ridge(X, Y, 1e12)
    assert np.max(np.abs(Wi)) < 1e-8 and np.allclose(bi, Y.mean(0), atol=1e-8)
    # the intercept is unpenalised: shifting X leaves W unchanged.
    W1, _ = O.fit_ridge(X, Y, 0.5)
    W2, _ = O.fit_ridge(X + 100.0, Y, 0.5)
    assert np.allclose(W1, W2, atol=1e-9)


def test_ridge_scalar_textbook_form():
    rng = np.random.default_rng(7)
    x = rng.standard_normal((50, 1))
    y = 2.5 * x + 1.0 + 0.3 * rng.standard_normal((50, 1))
    lam = 4.0
    W, b = O.fit_ridge(x, y, lam)
    xc = x[:, 0] - x[:, 0].mean()
    yc = y[:, 0] - y[:, 0].mean()
    assert abs(W[0, 0] - float(xc @ yc) / (float(xc @ xc) + lam)) < 1e-12


def test_ridge_per_head_equals_joint_columns():
    rng = np.random.default_rng(8)
    X = rng.standard_normal((300, 24))
    Y = rng.standard_normal((300, 12))
    W, b = O.fit_ridge(X, Y, 0.01)
    for h in range(3):
        Wh, bh = O.fit_ridge(X, Y[:, 4 * h:4 * h + 4], 0.01)
        assert np.allclose(Wh, W[:, 4 * h:4 * h + 4], atol=1e-12)
        assert np.allclose(bh, b[4 * h:4 * h + 4], atol=1e-12)


def test_ridge_recovers_exact_linear_relation():
    # Velox "The honesty crux" item 1: the fit recovers a known linear relation.
    rng = np.random.default_rng(9)
    X = rng.standard_normal((500, 10))
    Wt = rng.standard_normal((10, 3))
    bt = rng.standard_normal(3)
    W, b = O.fit_ridge(X, X @ Wt + bt, 1e-10)
    assert np.allclose(W, Wt, atol=1e-9) and np.allclose(b, bt, atol=1e-9)


# --------------------------------------------------------------------------
# Statistics
# --------------------------------------------------------------------------

def test_two_pass_stats_match_numpy_covariance():
    rng = np.random.default_rng(10)
    X = rng.standard_normal((77, 5)) * 3 + 1e3
    Y = rng.standard_normal((77, 2)) - 5
    st = O.centered_stats(X, Y)
    full = np.cov(np.concatenate([X, Y], axis=1).T, bias=True) * 77
    assert np.allclose(st.M, full[:5, :5], rtol=1e-10, atol=1e-8)
    assert np.allclose(st.C, full[:5, 5:], rtol=1e-10, atol=1e-8)
    assert np.allclose(st.syy, np.diag(full[5:, 5:]), rtol=1e-10)
    assert np.allclose(st.xbar, np.average(X, axis=0)) and st.n == 77


@pytest.mark.parametrize("parts", [[1] * 12, [5, 7], [1, 11], [3, 3, 3, 3], [11, 1]])
def test_chan_merge_equals_two_pass(parts):
    rng = np.random.default_rng(11)
    X = rng.standard_normal((12, 4)) * 10 + 1e4
    Y = rng.standard_normal((12, 3)) + 50
    cuts = np.cumsum([0] + parts)
    merged = O.stats_from_batches((X[a:b], Y[a:b]) for a, b in zip(cuts[:-1], cuts[1:]))
    ref = O.centered_stats(X, Y)
    assert merged.n == ref.n
    for f in ("xbar", "ybar", "M", "C", "syy"):
        assert np.allclose(getattr(merged, f), getattr(ref, f), rtol=1e-12, atol=1e-9), f


def test_gram_symmetric_psd():
    rng = np.random.default_rng(12)
    st = O.centered_stats(rng.standard_normal((30, 10)), rng.standard_normal((30, 2)))
    assert np.array_equal(st.M, st.M.T)
    assert np.min(np.linalg.eigvalsh(st.M)) > -1e-10


# --------------------------------------------------------------------------
# R^2 and selection
# --------------------------------------------------------------------------

def test_head_pooled_r2_matches_sklearn_variance_weighted():
    skm = pytest.importorskip("sklearn.metrics")
    rng = np.random.default_rng(13)
    H, d = 3, 4
    Yt = rng.standard_normal((60, H * d)) * rng.uniform(0.5, 3, H * d)
    Yp = Yt + 0.5 * rng.standard_normal((60, H * d))
    ref = np.mean([skm.r2_score(Yt[:, h * d:(h + 1) * d], Yp[:, h * d:(h + 1) * d],
                                multioutput="variance_weighted") for h in range(H)])
    assert abs(O.head_pooled_r2(Yt, Yp, H, d) - ref) < 1e-12


def test_single_source_r2_closed_form_sse():
    # SSE = S_yy - diag(C^T W) - lam diag(W^T W) for the ridge solution W.
    rng = np.random.default_rng(14)
    H, d, lam = 2, 3, 0.7
    Xs = [rng.standard_normal((40, H * d)) for _ in range(3)]
    Yt = [Xs[1] @ rng.standard_normal((H * d, H * d)) + rng.standard_normal((40, H * d))]
    r2 = O.single_source_r2(Xs, Yt, lam, H, d)
    for s in range(3):
        st = O.centered_stats(Xs[s], Yt[0])
        W, _ = O.ridge_from_stats(st, lam)
        sse = st.syy - np.einsum("ij,ij->j", st.C, W) - lam * np.einsum("ij,ij->j", W, W)
        r = np.mean([1 - sse[h * d:(h + 1) * d].sum() / st.syy[h * d:(h + 1) * d].sum() for h in range(H)])
        assert abs(r - r2[0, s]) < 1e-12
    assert np.argmax(r2[0]) == 1


def test_single_source_r2_of_a_copied_layer_is_one():
    rng = np.random.default_rng(15)
    Xs = [rng.standard_normal((200, 8)) for _ in range(4)]
    r2 = O.single_source_r2(Xs, [Xs[2].copy()], 0.01, 2, 4)
    assert 1.0 - r2[0, 2] < 1e-6 and np.all(r2[0, [0, 1, 3]] < 0.2)


def test_select_top_k_ordering_ties_and_margin():
    r2 = np.array([[0.1, 0.9, 0.5, 0.9, 0.2],
                   [0.3, 0.3, 0.3, 0.3, 0.3]])
    sel, margin = O.select_top_k(r2, 2)
    assert sel.tolist() == [[1, 3], [0, 1]]
    assert abs(margin[0] - 0.4) < 1e-15 and margin[1] == 0.0
    sel3, _ = O.select_top_k(r2, 3)
    assert sel3.tolist() == [[1, 2, 3], [0, 1, 2]]
    full, m = O.select_top_k(r2, 5)
    assert full.tolist() == [[0, 1, 2, 3, 4]] * 2 and np.all(np.isinf(m))


# --------------------------------------------------------------------------
# Apply and the whole fit
# --------------------------------------------------------------------------

def test_apply_with_identity_map_is_the_single_rotation_recode():
    rng = np.random.default_rng(16)
    L, H, T, d = 3, 2, 33, 8
    k_s = rng.standard_normal((L, H, T, d))
    v_s = rng.standard_normal((L, H, T, d))
    pos = rng.integers(0, 30000, size=T)
    eye = np.stack([np.eye(H * d)] * L)
    zero = np.zeros((L, H * d))
    sel = [[l] for l in range(L)]
    out_k, out_v = O.map_apply(k_s, v_s, pos, sel, sel, eye, zero, eye, zero, 1e4, 5e5, H, d)
    assert np.max(np.abs(out_k - O.recode(k_s, pos, 1e4, 5e5))) < 1e-11
    assert np.array_equal(out_v, v_s)


def _tiny_pair(seed, L_s=4, L_t=6, H=2, d=16, k=2, T=256, n_seq=4, noise=1e-3,
               theta_s=1e4, theta_t=5e4, sigma=0.5):
    sel_k = synth.hidden_selection(seed + 1, L_s, L_t, k)
    sel_v = synth.hidden_selection(seed + 2, L_s, L_t, k)
    Wk, bk = synth.hidden_weights(seed + 3, L_t, k * H * d, H * d)
    Wv, bv = synth.hidden_weights(seed + 4, L_t, k * H * d, H * d)
    pos = np.arange(T)
    seqs = []
    for i in range(n_seq + 1):
        ck = synth.content(seed + 100 + i, L_s, H, T, d, sigma)
        cv = synth.content(seed + 200 + i, L_s, H, T, d, sigma)
        nk = synth.noise(seed + 300 + i, (L_t, T, H * d))
        nv = synth.noise(seed + 400 + i, (L_t, T, H * d))
        seqs.append(O.synthesize_pair(ck, cv, pos, theta_s, theta_t, sel_k, sel_v, Wk, bk,
                                      Wv, bv, nk, nv, noise) + (pos,))
    return dict(calib=seqs[:n_seq], holdout=seqs[n_seq], sel_k=sel_k, sel_v=sel_v,
                theta_s=theta_s, theta_t=theta_t, H=H, d=d, k=k)


def _holdout_r2(fit, pair):
    src_k, src_v, tgt_k, tgt_v, pos = pair["holdout"]
    H, d = pair["H"], pair["d"]
    out_k, out_v = O.map_apply(src_k, src_v, pos, fit.sel_k, fit.sel_v, fit.W_k, fit.b_k,
                               fit.W_v, fit.b_v, pair["theta_s"], pair["theta_t"], H, d)
    r = []
    for t in range(out_k.shape[0]):
        for a, b in ((tgt_k[t], out_k[t]), (tgt_v[t], out_v[t])):
            A = np.transpose(a, (1, 0, 2)).reshape(-1, H * d)
            B = np.transpose(b, (1, 0, 2)).reshape(-1, H * d)
            r.append(O.head_pooled_r2(A, B, H, d))
    return np.array(r)


def test_noise_free_synthetic_target_is_reproduced_by_apply():
    pair = _tiny_pair(20, noise=0.0, n_seq=1)
    src_k, src_v, tgt_k, tgt_v, pos = pair["holdout"]
    Wk, bk = synth.hidden_weights(23, 6, 64, 32)
    Wv, bv = synth.hidden_weights(24, 6, 64, 32)
    out_k, out_v = O.map_apply(src_k, src_v, pos, pair["sel_k"], pair["sel_v"], Wk, bk, Wv, bv,
                               1e4, 5e4, 2, 16)
    assert np.max(np.abs(out_k - tgt_k)) < 1e-11 and np.max(np.abs(out_v - tgt_v)) < 1e-11


@pytest.mark.parametrize("seed", [0, 1000])
def test_fit_recovers_hidden_layers_on_the_tiny_pair(seed, golden_dir):
    # KVBridge "Thirty-second proof": every true source layer recovered, holdout R^2 high.
    pair = _tiny_pair(seed)
    fit = O.fit_mapper(pair["calib"], pair["theta_s"], pair["theta_t"], pair["k"], 0.01, 4)
    assert fit.n_obs == 4 * 64
    assert np.array_equal(fit.sel_k, pair["sel_k"]) and np.array_equal(fit.sel_v, pair["sel_v"])
    assert np.min(fit.margin_k) > 1e-3 and np.min(fit.margin_v) > 1e-3
    r2 = _holdout_r2(fit, pair)
    assert np.min(r2) > 0.9999
    # noise 1e-3 against unit-scale signal: the pages' demo level is reached too.
    assert np.median(r2) > _golden(golden_dir)["demo_holdout_r2_min"]


@pytest.mark.parametrize("geom", [(3, 2, 2, 4, 64), (5, 4, 2, 8, 128), (8, 6, 4, 16, 256)])
def test_fit_recovers_on_the_kvbridge_local_geometries(geom):
    # KVBridge "Local evidence": micro / small / medium cache geometries.
    L_s, L_t, H, d, T = geom
    pair = _tiny_pair(50 + L_s, L_s=L_s, L_t=L_t, H=H, d=d, k=2, T=T, n_seq=8)
    fit = O.fit_mapper(pair["calib"], pair["theta_s"], pair["theta_t"], 2, 0.01, 4)
    assert np.array_equal(fit.sel_k, pair["sel_k"]) and np.array_equal(fit.sel_v, pair["sel_v"])
    assert np.min(_holdout_r2(fit, pair)) > 0.9999


def test_top_k_single_source_choice_is_the_best_subset_by_brute_force():
    pair = _tiny_pair(77)
    fit = O.fit_mapper(pair["calib"], pair["theta_s"], pair["theta_t"], 2, 0.01, 4)
    src_k, src_v, tgt_k, tgt_v, pos = pair["holdout"]
    H, d = 2, 16
    # refit every 2-subset explicitly, score on the held-out sequence
    calib = pair["calib"]
    keep = [O.retain_stride(c[4], 4) for c in calib]
    Xall = np.concatenate([O.all_layer_features(c[0], c[4], 1e4)[m] for c, m in zip(calib, keep)])
    Yall = np.concatenate([O.all_layer_features(c[2], c[4], 5e4)[m] for c, m in zip(calib, keep)])
    Xh = O.all_layer_features(src_k, pos, 1e4)
    Yh = O.all_layer_features(tgt_k, pos, 5e4)
    q = H * d
    for t in range(6):
        best, best_r2 = None, -np.inf
        for sub in itertools.combinations(range(4), 2):
            cols = np.concatenate([np.arange(s * q, (s + 1) * q) for s in sub])
            W, b = O.fit_ridge(Xall[:, cols], Yall[:, t * q:(t + 1) * q], 0.01)
            r = O.head_pooled_r2(Yh[:, t * q:(t + 1) * q], Xh[:, cols] @ W + b, H, d)
            if r > best_r2:
                best, best_r2 = sub, r
        assert list(best) == fit.sel_k[t].tolist()


def test_stride_keeps_multiples_of_the_stride():
    pos = np.concatenate([np.arange(10), np.arange(7)])
    assert np.flatnonzero(O.retain_stride(pos, 4)).tolist() == [0, 4, 8, 10, 14]


# --------------------------------------------------------------------------
# Sizes printed on the pages
# --------------------------------------------------------------------------

def test_sizes_match_the_pages(golden_dir):
    g = _golden(golden_dir)
    # 14B -> 32B: 64 target layers, 8 KV heads, head_dim 128, k = 8
    n = O.mapper_param_count(64, 8, 8, 128)
    assert n == int(g["mapper_params_qwen3_14b_32b_k8"])
    assert round(n * 4 / 2**30, 4) == g["mapper_gib_fp32_qwen3_14b_32b_k8"]
    assert round(O.fit_stats_bytes(8, 8, 128) / 2**30, 2) == g["fit_stats_gib_one_layer_block"]
    # Qwen3 0.6B -> 1.7B T2 run: 28 target layers, 8 x 128, k = 1
    assert O.mapper_param_count(28, 1, 8, 128) == int(g["mapper_params_t2_qwen3_0p6b_1p7b"])
    assert O.stride_observations(16, 512, int(g["calib_stride"])) == int(g["t2_observations"])
    obs = O.stride_observations(int(g["calib_sequences"]), int(g["calib_seq_len"]), int(g["calib_stride"]))
    assert abs(obs - g["calib_observations_approx"]) / g["calib_observations_approx"] < 0.01
    # the oracle's fit produces W of exactly the counted shape
    pair = _tiny_pair(5, n_seq=1)
    fit = O.fit_mapper(pair["calib"], 1e4, 5e4, 2, 0.01, 4)
    assert fit.W_k.size + fit.W_v.size + fit.b_k.size + fit.b_v.size == O.mapper_param_count(6, 2, 2, 16)


# --------------------------------------------------------------------------
# Attention-output cosine
# --------------------------------------------------------------------------

def _attn_inputs(seed, L=2, H=2, g=3, T=37, d=16):
    q = synth.content(seed, L, H * g, T, d, 0.5)
    k = synth.content(seed + 1, L, H, T, d, 0.5)
    v = synth.content(seed + 2, L, H, T, d, 0.5)
    return q, k, v


def test_attention_output_matches_torch_sdpa_causal_gqa():
    # library route: scaled_dot_product_attention (default scale 1/sqrt(d),
    # is_causal) with each KV head repeated for its group of query heads
    torch = pytest.importorskip("torch")
    q, k, v = _attn_inputs(70)
    g = q.shape[1] // k.shape[1]
    pos = np.arange(q.shape[2])
    o = O.attention_output(q, pos, k, v, pos)
    kt = torch.from_numpy(k).repeat_interleave(g, dim=1)
    vt = torch.from_numpy(v).repeat_interleave(g, dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(torch.from_numpy(q), kt, vt, is_causal=True)
    assert np.abs(o - ref.numpy()).max() < 1e-12


def test_attention_output_subset_queries_equal_rows_of_the_full_result():
    q, k, v = _attn_inputs(71)
    pos = np.arange(q.shape[2]) + 100
    full = O.attention_output(q, pos, k, v, pos)
    rows = np.array([0, 5, 36])
    part = O.attention_output(q[:, :, rows], pos[rows], k, v, pos)
    assert np.abs(part - full[:, :, rows]).max() < 1e-13


def test_attention_output_first_position_sees_only_the_first_key():
    q, k, v = _attn_inputs(72)
    g = q.shape[1] // k.shape[1]
    pos = np.arange(q.shape[2])
    o = O.attention_output(q[:, :, :1], pos[:1], k, v, pos)
    for hq in range(q.shape[1]):
        assert np.array_equal(o[:, hq, 0], v[:, hq // g, 0])


def test_attention_output_query_with_no_visible_key_is_zero():
    q, k, v = _attn_inputs(73)
    o = O.attention_output(q[:, :, :2], np.array([-1, 0]), k, v, np.arange(q.shape[2]))
    assert np.all(o[:, :, 0] == 0) and np.all(o[:, :, 1] != 0)


def test_attention_cosine_invariants():
    q, k, v = _attn_inputs(74)
    pos = np.arange(q.shape[2])
    one = O.attention_cosine(q, pos, k, v, k, v, pos)
    assert np.abs(one - 1).max() < 1e-12
    # scaling the values scales every output: +1 for c > 0, -1 for c < 0
    assert np.abs(O.attention_cosine(q, pos, k, v, k, 2.5 * v, pos) - 1).max() < 1e-12
    assert np.abs(O.attention_cosine(q, pos, k, v, k, -0.5 * v, pos) + 1).max() < 1e-12
    # one vector added to every key of a head shifts each query's scores by a
    # constant: softmax, hence the output, is unchanged
    u = synth.content(75, k.shape[0], k.shape[1], 1, k.shape[3], 0.0)
    assert np.abs(O.attention_cosine(q, pos, k, v, k + u, v, pos) - 1).max() < 1e-10
    # a perturbed cache gives a cosine strictly inside (-1, 1), equal to the
    # library cosine of the two outputs
    torch = pytest.importorskip("torch")
    k2 = k + 0.5 * synth.noise(76, k.shape)
    v2 = v + 0.5 * synth.noise(77, v.shape)
    c = O.attention_cosine(q, pos, k2, v2, k, v, pos)
    oa = torch.from_numpy(O.attention_output(q, pos, k2, v2, pos))
    ob = torch.from_numpy(O.attention_output(q, pos, k, v, pos))
    assert np.abs(c - torch.nn.functional.cosine_similarity(oa, ob, dim=-1).numpy()).max() < 1e-12
    assert c.max() < 1 and c.min() > -1 and c.mean() > 0.5
