"""W against the float64 oracle when the ridge systems are ill-conditioned.

Source layers that share one component correlate channel by channel (rho^2 =
0.99 here, as strongly correlated neighbouring layers of one model's cache
might); the 2048-unknown systems of k = 8 selected layers (2 KV heads,
head_dim 128) then have condition numbers of about 800-950 after Jacobi
scaling, against ~150 in the full-size fit test.  W's distance from the
oracle grows about in proportion to the condition number, and it comes from
the float32 accumulation of the statistics ("KVBridge" README, "Loading":
centered statistics accumulated in float32), not from the solver: the same
statistics solved in float64 on the host are as far from the oracle.
16,384 observations (8 batches of 8192 tokens, stride 4), lambda 0.01
("Cross-Model KV Transfer", "Configuration").
"""
import numpy as np
import pytest

import oracle as O
import synth
from cases import TOL_W, rel_fro, spec, to_host64

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

L_S, L_T, H, D, K = 10, 2, 2, 128, 8
TB, N_BATCH, SEQ, STRIDE, LAM, THETA = 8192, 8, 1024, 4, 0.01, 1e6
RHO2 = 0.99


@pytest.fixture(scope="module")
def fit():
    from cross_model_kv_gb300 import build
    build.build()
    import cross_model_kv_gb300 as kvb
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = "cuda"
    q, p = H * D, K * H * D
    sel = {0: synth.hidden_selection(511, L_S, L_T, K), 1: synth.hidden_selection(512, L_S, L_T, K)}
    coef = torch.linspace(1.0, 0.6, K).tolist()
    g = torch.Generator(device=dev)
    g.manual_seed(513)
    keep = torch.arange(0, TB, STRIDE, device=dev)
    pos = torch.arange(SEQ, dtype=torch.int32, device=dev).repeat(TB // SEQ)
    ctx = kvb.kvb_ctx_create(spec(L_S, H, D, THETA), spec(L_T, H, D, THETA), K, SEQ)
    st = kvb.kvb_stats_create(ctx, kvb.KVB_BF16, TB)
    host_src, host_tgt = {0: [], 1: []}, {0: [], 1: []}
    for b in range(N_BATCH):
        src = {kv: synth.torch_content_shared(610 + 100 * kv + b, L_S, H, TB, D, 1.0, RHO2 ** 0.5, torch.bfloat16,
                                              dev) for kv in (0, 1)}
        tgt = {kv: torch.empty((L_T, H, TB, D), dtype=torch.bfloat16, device=dev) for kv in (0, 1)}
        for kv in (0, 1):
            for t in range(L_T):
                acc = 0.1 * torch.randn((H, TB, D), generator=g, device=dev)
                for j in range(K):
                    acc += coef[j] * src[kv][int(sel[kv][t][j])].float()
                tgt[kv][t].copy_(acc)
        kvb.kvb_stats_accumulate(ctx, st, src[0], src[1], tgt[0], tgt[1], pos, STRIDE)
        for kv in (0, 1):
            host_src[kv].append(src[kv].index_select(2, keep).cpu())
            host_tgt[kv].append(tgt[kv].index_select(2, keep).cpu())
    kvb.kvb_ctx_check(ctx)
    Wk = torch.empty((L_T, q, p), dtype=torch.float32, device=dev)
    Wv = torch.empty_like(Wk)
    bk = torch.empty((L_T, q), dtype=torch.float32, device=dev)
    bv = torch.empty_like(bk)
    kvb.kvb_ridge_solve(ctx, st, sel[0], sel[1], LAM, Wk, Wv, bk, bv)
    W = {0: to_host64(Wk), 1: to_host64(Wv)}
    Fs, Ft = L_S * q, L_T * q
    exported = {}
    for kv in (0, 1):
        f = lambda *sh: torch.empty(sh, dtype=torch.float32, device=dev)
        mx, my, gram, cross, syy = f(Fs), f(Ft), f(Fs, Fs), f(Fs, Ft), f(Ft)
        kvb.kvb_stats_export(st, kv, mx, my, gram, cross, syy)
        exported[kv] = (to_host64(gram), to_host64(cross))
    kvb.kvb_stats_destroy(st)
    kvb.kvb_ctx_destroy(ctx)
    pos_kept = np.tile(np.arange(0, SEQ, STRIDE), N_BATCH * (TB // SEQ))
    out = {}
    for kv in (0, 1):
        src_h = torch.cat(host_src[kv], dim=2).to(torch.float64).numpy()
        tgt_h = torch.cat(host_tgt[kv], dim=2).to(torch.float64).numpy()
        strip = (pos_kept, THETA) if kv == 0 else (None, None)
        gram, cross = exported[kv]
        for t in range(L_T):
            stats = O.centered_stats(O.features(src_h, sel[kv][t], *strip), O.features(tgt_h, [t], *strip))
            W_o = O.ridge_from_stats(stats, LAM)[0]
            A = stats.M + LAM * np.eye(p)
            dsc = 1.0 / np.sqrt(np.diag(A))
            ev = np.linalg.eigvalsh(A * np.outer(dsc, dsc))
            # the GPU's own float32 statistics of this system (lower half kept), solved in float64
            fi = np.concatenate([np.arange(int(s) * q, (int(s) + 1) * q) for s in sel[kv][t]])
            G = np.tril(gram[np.ix_(fi, fi)])
            G = G + np.tril(G, -1).T
            W_s = np.linalg.solve(G + LAM * np.eye(p), cross[fi][:, t * q:(t + 1) * q])
            out[kv, t] = dict(cond=ev[-1] / ev[0], w=rel_fro(W[kv][t].T, W_o), stats=rel_fro(W_s, W_o))
    return out


def test_w_within_the_bound_at_condition_numbers_near_a_thousand(fit):
    for (kv, t), r in fit.items():
        assert r["cond"] > 500, (kv, t, r)  # as ill-conditioned as intended
        assert r["w"] <= TOL_W, (kv, t, r)
    print("\n(kv, t): condition number, W error, W error of the same statistics solved in float64:",
          {k: (round(r["cond"]), f"{r['w']:.2e}", f"{r['stats']:.2e}") for k, r in fit.items()})


def test_w_error_comes_from_the_statistics_not_the_solver(fit):
    # the float64 solve of the GPU's float32 statistics is as far from the oracle
    # as the GPU's own W (within a factor 1.5), so the solver adds little
    for (kv, t), r in fit.items():
        assert r["w"] <= 1.5 * r["stats"], (kv, t, r)
