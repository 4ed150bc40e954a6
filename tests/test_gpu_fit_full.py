"""Full-size parity of the calibration fit against the float64 oracle.

Qwen3-14B -> 32B shapes: 40 -> 64 layers, 8 KV heads, head_dim 128, k = 8;
256 sequences x 1024 tokens streamed in 32 batches of 8192, stride 4, so
65,536 observations; lambda = 0.01 ("Cross-Model KV Transfer", "Configuration";
KVBridge README, "Loading").  The ridge systems have 8192 unknowns and 1024
right-hand sides, 128 of them (K and V of every target layer).

The source layers share one component (any two layers correlate by 0.8,
channel by channel, as the layers of one model's cache do through its
residual stream): each 8192-unknown system then has a condition number of
about 150 after Jacobi scaling instead of about 4 for independent layers.
Targets are fixed mixtures of 8 hidden source layers plus noise (values also
get a bias), built with plain torch arithmetic on the device.

Checked against the oracle: sampled (layer, head) slabs of the statistics,
the single-source R^2 of the two pairs at the selection boundary of one
target, and W and b of four target layers (K and V) -- with the solver's
default workspace and with a cap that splits the systems over several
batches.  The selection must recover the hidden layers with a margin.
"""
import numpy as np
import pytest

import oracle as O
import synth
from cases import TOL_W, rel_fro, spec, to_host64

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

L_S, L_T, H, D, K = 40, 64, 8, 128, 8
TB, N_BATCH, SEQ, STRIDE, LAM, THETA = 8192, 32, 1024, 4, 0.01, 1e6
RHO = 0.8 ** 0.5                      # layers correlate by RHO^2 = 0.8
W_TARGETS = (0, 21, 42, 63)            # target layers whose W and b are compared
T_STAR = 21                            # target whose boundary R^2 are compared
SRC_SLABS = ((0, 0), (17, 3), (39, 7))
TGT_SLABS = ((0, 0), (31, 5), (63, 7))
WS_CAP_MB = 12 * 1024                  # several solver batches: 3 for selection, 4 for the ridge


@pytest.fixture(scope="module")
def calib():
    from cross_model_kv_gb300 import build
    build.build()
    import cross_model_kv_gb300 as kvb
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = "cuda"
    sel = {0: synth.hidden_selection(501, L_S, L_T, K), 1: synth.hidden_selection(502, L_S, L_T, K)}
    coef = torch.linspace(1.0, 0.6, K).tolist()
    g = torch.Generator(device=dev)
    g.manual_seed(503)
    b_true_v = 0.1 * torch.randn((L_T, H, 1, D), generator=g, device=dev)
    pos = torch.arange(SEQ, dtype=torch.int32, device=dev).repeat(TB // SEQ)
    keep = torch.arange(0, TB, STRIDE, device=dev)  # pos % 4 == 0
    ctx = kvb.kvb_ctx_create(spec(L_S, H, D, THETA), spec(L_T, H, D, THETA), K, SEQ)
    st = kvb.kvb_stats_create(ctx, kvb.KVB_BF16, TB)
    tgt_layers = sorted({t for t, _ in TGT_SLABS} | set(W_TARGETS) | {T_STAR})
    host_src = {0: [], 1: []}
    host_tgt = {0: [], 1: []}
    li = torch.tensor(tgt_layers, device=dev)
    for b in range(N_BATCH):
        src = {0: synth.torch_content_shared(600 + b, L_S, H, TB, D, 1.0, RHO, torch.bfloat16, dev),
               1: synth.torch_content_shared(700 + b, L_S, H, TB, D, 1.0, RHO, torch.bfloat16, dev)}
        tgt = {kv: torch.empty((L_T, H, TB, D), dtype=torch.bfloat16, device=dev) for kv in (0, 1)}
        for kv in (0, 1):
            for t in range(L_T):
                acc = 0.1 * torch.randn((H, TB, D), generator=g, device=dev)
                for j in range(K):
                    acc += coef[j] * src[kv][int(sel[kv][t][j])].float()
                if kv == 1:
                    acc += b_true_v[t]
                tgt[kv][t].copy_(acc)
        kvb.kvb_stats_accumulate(ctx, st, src[0], src[1], tgt[0], tgt[1], pos, STRIDE)
        for kv in (0, 1):
            host_src[kv].append(src[kv].index_select(2, keep).cpu())
            host_tgt[kv].append(tgt[kv].index_select(0, li).index_select(2, keep).cpu())
        del src, tgt
    kvb.kvb_ctx_check(ctx)
    src_all = {kv: torch.cat(host_src[kv], dim=2) for kv in (0, 1)}   # [L_s][H][N][d] bf16, host
    tgt_all = {kv: torch.cat(host_tgt[kv], dim=2) for kv in (0, 1)}   # [len(tgt_layers)][H][N][d]
    del host_src, host_tgt
    pos_kept = np.tile(np.arange(0, SEQ, STRIDE), N_BATCH * (TB // SEQ))
    return dict(kvb=kvb, ctx=ctx, st=st, sel=sel, src=src_all, tgt=tgt_all, tgt_index={t: i for i, t in
                enumerate(tgt_layers)}, pos=pos_kept)


def _host64(x):
    return x.to(torch.float64).numpy()


def _features(c, kv, layers):
    """Oracle features [N][len(layers)*H*d] of source layers (keys RoPE-stripped)."""
    cache = _host64(c["src"][kv][list(layers)])
    return O.features(cache, range(len(layers)), c["pos"] if kv == 0 else None, THETA if kv == 0 else None)


def _target(c, kv, t):
    y = _host64(c["tgt"][kv][c["tgt_index"][t]])[None]
    return O.features(y, [0], c["pos"] if kv == 0 else None, THETA if kv == 0 else None)


def _slabs(arr, slabs, kv, c):
    cols = []
    for l, h in slabs:
        x = _host64(arr[l, h])
        cols.append(O.strip(x, c["pos"], THETA) if kv == 0 else x)
    return np.concatenate(cols, axis=1)


def _select(c, r2, cap_mb, monkeypatch):
    kvb = c["kvb"]
    if cap_mb:
        monkeypatch.setenv("KVB_FIT_WORKSPACE_MB", str(cap_mb))
    kvb.kvb_profile_enable(c["ctx"], True)
    sk, sv = kvb.kvb_layer_select(c["ctx"], c["st"], LAM, r2)
    kvb.kvb_profile_enable(c["ctx"], False)
    batches = kvb.kvb_profile_read(c["ctx"])["r2_solve_batch"][0]
    monkeypatch.delenv("KVB_FIT_WORKSPACE_MB", raising=False)
    return sk, sv, batches


def test_statistics_selection_and_boundary_r2(calib, monkeypatch):
    c, kvb = calib, calib["kvb"]
    assert kvb.kvb_stats_count(c["st"]) == N_BATCH * TB // STRIDE
    q, Fs, Ft = H * D, L_S * H * D, L_T * H * D
    f_src = np.concatenate([np.arange((l * H + h) * D, (l * H + h + 1) * D) for l, h in SRC_SLABS])
    f_tgt = np.concatenate([np.arange((l * H + h) * D, (l * H + h + 1) * D) for l, h in TGT_SLABS])
    tgt_slabs_local = [(c["tgt_index"][l], h) for l, h in TGT_SLABS]
    for kv in (0, 1):
        ref = O.centered_stats(_slabs(c["src"][kv], SRC_SLABS, kv, c), _slabs(c["tgt"][kv], tgt_slabs_local, kv, c))
        f = lambda *s: torch.empty(s, dtype=torch.float32, device="cuda")
        mx, my, gram, cross, syy = f(Fs), f(Ft), f(Fs, Fs), f(Fs, Ft), f(Ft)
        n = kvb.kvb_stats_export(c["st"], kv, mx, my, gram, cross, syy)
        assert n == ref.n
        gram, cross = to_host64(gram[f_src][:, f_src]), to_host64(cross[f_src][:, f_tgt])
        scale_m = np.sqrt(np.outer(np.diag(ref.M), np.diag(ref.M)))
        assert np.max(np.abs(gram - ref.M) / scale_m) < 1e-4
        scale_c = np.sqrt(np.outer(np.diag(ref.M), ref.syy))
        assert np.max(np.abs(cross - ref.C) / scale_c) < 1e-4
        assert rel_fro(to_host64(syy)[f_tgt], ref.syy) < 1e-4
        assert np.max(np.abs(to_host64(mx)[f_src] - ref.xbar)) < 1e-4
        assert np.max(np.abs(to_host64(my)[f_tgt] - ref.ybar)) < 1e-4
        del gram, cross

    torch.cuda.empty_cache()
    r2 = torch.empty((2, L_T, L_S), dtype=torch.float32, device="cuda")
    r2_cap = torch.empty_like(r2)
    sk, sv, n_default = _select(c, r2, 0, monkeypatch)
    sk_c, sv_c, n_capped = _select(c, r2_cap, WS_CAP_MB, monkeypatch)
    assert n_default == 1 and n_capped >= 3, (n_default, n_capped)
    for got_k, got_v in ((sk, sv), (sk_c, sv_c)):
        assert np.array_equal(got_k, c["sel"][0]) and np.array_equal(got_v, c["sel"][1])
    r2h, r2c = to_host64(r2), to_host64(r2_cap)
    assert np.max(np.abs(r2h - r2c)) <= 1e-5
    # selection margin: k-th minus (k+1)-th ranked R^2, every target, K and V
    ranked = -np.sort(-r2h, axis=2)
    margin = ranked[:, :, K - 1] - ranked[:, :, K]
    print(f"\nselection margin at 14B->32B shapes: min K {margin[0].min():.4g}, min V {margin[1].min():.4g}")
    assert margin.min() > 1e-3  # ten times the R^2 agreement checked below

    # boundary pairs of one target against the oracle's explicit single-source fits
    for kv in (0, 1):
        order = sorted(range(L_S), key=lambda s: (-r2h[kv, T_STAR, s], s))
        pair = (order[K - 1], order[K])  # lowest selected, best unselected
        Xs = [_features(c, kv, [s]) for s in pair]
        ref = O.single_source_r2(Xs, [_target(c, kv, T_STAR)], LAM, H, D)[0]
        got = r2h[kv, T_STAR, list(pair)]
        assert np.max(np.abs(got - ref)) < 1e-4, (kv, got, ref)
        assert ref[0] > ref[1]


@pytest.fixture(scope="module")
def oracle_fits(calib):
    """The oracle's ridge W, b (and the first 4096 feature rows) of every compared system."""
    c = calib
    out = {}
    for kv in (0, 1):
        for t in W_TARGETS:
            X = _features(c, kv, c["sel"][kv][t])
            W_o, b_o = O.fit_ridge(X, _target(c, kv, t), LAM)
            out[kv, t] = (W_o, b_o, X[:4096].copy())
            del X
    return out


@pytest.mark.parametrize("cap_mb", [0, WS_CAP_MB], ids=["default_workspace", "capped_workspace"])
def test_ridge_w_and_b_match_the_oracle(calib, oracle_fits, cap_mb, monkeypatch):
    c, kvb = calib, calib["kvb"]
    q, p = H * D, K * H * D
    torch.cuda.empty_cache()
    Wk = torch.empty((L_T, q, p), dtype=torch.float32, device="cuda")
    Wv = torch.empty_like(Wk)
    bk = torch.empty((L_T, q), dtype=torch.float32, device="cuda")
    bv = torch.empty_like(bk)
    if cap_mb:
        monkeypatch.setenv("KVB_FIT_WORKSPACE_MB", str(cap_mb))
    kvb.kvb_profile_enable(c["ctx"], True)
    kvb.kvb_ridge_solve(c["ctx"], c["st"], c["sel"][0], c["sel"][1], LAM, Wk, Wv, bk, bv)
    kvb.kvb_profile_enable(c["ctx"], False)
    batches = kvb.kvb_profile_read(c["ctx"])["ridge_solve_batch"][0]
    assert batches == (4 if cap_mb else 1), batches
    li = torch.tensor(W_TARGETS, device="cuda")
    gW = {0: to_host64(Wk.index_select(0, li)), 1: to_host64(Wv.index_select(0, li))}
    gb = {0: to_host64(bk.index_select(0, li)), 1: to_host64(bv.index_select(0, li))}
    del Wk, Wv
    errs = []
    for kv in (0, 1):
        for i, t in enumerate(W_TARGETS):
            W_o, b_o, X = oracle_fits[kv, t]
            W_g, b_g = gW[kv][i].T, gb[kv][i]
            ew = rel_fro(W_g, W_o)
            # the mapped output on the first 4096 observations: W and b together
            ey = rel_fro(X @ W_g + b_g, X @ W_o + b_o)
            eb = rel_fro(b_g, b_o)
            errs.append((kv, t, ew, ey, eb))
            assert ew <= TOL_W and ey <= TOL_W, (kv, t, ew, ey)
            if kv == 1:  # values carry a bias of N(0, 0.1^2), so b is far from zero
                assert eb <= TOL_W, (t, eb)
    print("\nW / output / b relative errors (kv, t, W, XW+b, b):", [tuple(round(x, 7) if isinstance(x, float)
                                                                             else x for x in e) for e in errs])
