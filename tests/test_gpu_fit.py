"""GPU parity of the fit path (statistics, selection, ridge) against the float64 oracle."""
import numpy as np
import pytest

import oracle as O
from cases import TOL_F32, TOL_W, make_pair, oracle_full_stats, rel_fro, round_pair, spec, to_host64

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvb():
    from cross_model_kv_gb300 import build
    build.build()
    import cross_model_kv_gb300 as m
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return m


def _dev(a, dtype):
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda", dtype)


def _accumulate(kvb, ctx, st, seqs, dtype, stride=4):
    for src_k, src_v, tgt_k, tgt_v, pos in seqs:
        kvb.kvb_stats_accumulate(ctx, st, _dev(src_k, dtype), _dev(src_v, dtype), _dev(tgt_k, dtype),
                                 _dev(tgt_v, dtype), _dev(pos.astype(np.int32), torch.int32), stride)


def _export(kvb, st, kv, Fs, Ft):
    f = lambda *s: torch.empty(s, dtype=torch.float32, device="cuda")
    mx, my, g, c, y = f(Fs), f(Ft), f(Fs, Fs), f(Fs, Ft), f(Ft)
    n = kvb.kvb_stats_export(st, kv, mx, my, g, c, y)
    return n, to_host64(mx), to_host64(my), to_host64(g), to_host64(c), to_host64(y)


def _ctx(kvb, pair, max_pos):
    return kvb.kvb_ctx_create(spec(pair["L_s"], pair["H"], pair["d"], pair["theta_s"]),
                              spec(pair["L_t"], pair["H"], pair["d"], pair["theta_t"]), pair["k"], max_pos)


def _check_stats(kvb, st, pair, tol):
    q = pair["H"] * pair["d"]
    Fs, Ft = pair["L_s"] * q, pair["L_t"] * q
    ref = oracle_full_stats(pair)
    for kv in (0, 1):
        n, mx, my, g, c, y = _export(kvb, st, kv, Fs, Ft)
        o = ref[kv]
        assert n == o.n
        assert rel_fro(mx, o.xbar) < tol and rel_fro(my, o.ybar) < tol
        assert rel_fro(g, o.M) < tol, rel_fro(g, o.M)
        assert rel_fro(c, o.C) < tol, rel_fro(c, o.C)
        assert rel_fro(y, o.syy) < tol


def _run_fit(kvb, ctx, st, pair, w_dtype):
    L_t, k, q = pair["L_t"], pair["k"], pair["H"] * pair["d"]
    r2 = torch.empty((2, L_t, pair["L_s"]), dtype=torch.float32, device="cuda")
    sel_k, sel_v = kvb.kvb_layer_select(ctx, st, 0.01, r2)
    Wk = torch.empty((L_t, q, k * q), dtype=w_dtype, device="cuda")
    Wv = torch.empty_like(Wk)
    bk = torch.empty((L_t, q), dtype=torch.float32, device="cuda")
    bv = torch.empty_like(bk)
    kvb.kvb_ridge_solve(ctx, st, sel_k, sel_v, 0.01, Wk, Wv, bk, bv)
    return sel_k, sel_v, to_host64(r2), Wk, Wv, bk, bv


def _check_fit(kvb, ctx, st, pair, w_dtype, w_tol):
    fit = O.fit_mapper(pair["calib"], pair["theta_s"], pair["theta_t"], pair["k"], 0.01, 4)
    sel_k, sel_v, r2, Wk, Wv, bk, bv = _run_fit(kvb, ctx, st, pair, w_dtype)
    assert np.array_equal(sel_k, fit.sel_k) and np.array_equal(sel_v, fit.sel_v)
    assert np.array_equal(fit.sel_k, pair["sel_k"]) and np.array_equal(fit.sel_v, pair["sel_v"])
    assert np.max(np.abs(r2[0] - fit.r2_k)) < 1e-4 and np.max(np.abs(r2[1] - fit.r2_v)) < 1e-4
    gWk = np.transpose(to_host64(Wk), (0, 2, 1))
    gWv = np.transpose(to_host64(Wv), (0, 2, 1))
    ek, ev = rel_fro(gWk, fit.W_k), rel_fro(gWv, fit.W_v)
    assert ek <= w_tol and ev <= w_tol, (ek, ev)
    assert rel_fro(to_host64(bk), fit.b_k) <= w_tol and rel_fro(to_host64(bv), fit.b_v) <= w_tol
    return fit, (sel_k, sel_v, Wk, Wv, bk, bv)


def test_tiny_pair_fp32_fit_matches_oracle_and_recovers(kvb):
    # tiny pair: 4 -> 6 layers, 2 KV heads, head_dim 16, k = 2, theta 1e4 -> 5e4,
    # 4 calibration sequences x 256 tokens, stride 4, noise 1e-3
    pair = make_pair(0, 4, 6, 2, 16, 2, 256, 4, 1e4, 5e4)
    ctx = _ctx(kvb, pair, 256)
    st = kvb.kvb_stats_create(ctx, kvb.KVB_F32, 256)
    _accumulate(kvb, ctx, st, pair["calib"], torch.float32)
    assert kvb.kvb_stats_count(st) == 256
    _check_stats(kvb, st, pair, 1e-5)
    fit, (sel_k, sel_v, Wk, Wv, bk, bv) = _check_fit(kvb, ctx, st, pair, torch.float32, 1e-4)
    # apply the GPU-fitted mapper on the held-out sequence
    src_k, src_v, tgt_k, tgt_v, pos = pair["holdout"]
    out_k = torch.empty((6, 2, 256, 16), dtype=torch.float32, device="cuda")
    out_v = torch.empty_like(out_k)
    kvb.kvb_map_apply(ctx, _dev(src_k, torch.float32), _dev(src_v, torch.float32),
                      _dev(pos.astype(np.int32), torch.int32), sel_k, sel_v, Wk, Wv, bk, bv, out_k, out_v)
    ok, ov = O.map_apply(src_k, src_v, pos, fit.sel_k, fit.sel_v, fit.W_k, fit.b_k, fit.W_v, fit.b_v, 1e4, 5e4, 2, 16)
    assert rel_fro(to_host64(out_k), ok) < TOL_F32 and rel_fro(to_host64(out_v), ov) < TOL_F32
    for t in range(6):
        for a, b in ((tgt_k[t], to_host64(out_k)[t]), (tgt_v[t], to_host64(out_v)[t])):
            A = np.transpose(a, (1, 0, 2)).reshape(256, 32)
            B = np.transpose(b, (1, 0, 2)).reshape(256, 32)
            assert O.head_pooled_r2(A, B, 2, 16) > 0.9999


def test_fp32_fit_system_size_not_a_multiple_of_the_panels(kvb):
    # head_dim 24, 4 KV heads, k = 5: ridge systems of 480 unknowns (7.5 panels of 64,
    # a partial last 128-wide super-panel) whose large trailing updates run on the
    # tensor cores; 8 sequences x 512 tokens, stride 4 -> 1024 observations
    pair = make_pair(5, 5, 2, 4, 24, 5, 512, 8, 1e4, 1e6)
    ctx = _ctx(kvb, pair, 512)
    st = kvb.kvb_stats_create(ctx, kvb.KVB_F32, 512)
    _accumulate(kvb, ctx, st, pair["calib"], torch.float32)
    assert kvb.kvb_stats_count(st) == 1024
    _check_fit(kvb, ctx, st, pair, torch.float32, 1e-4)


def test_fp32_fit_ragged_tensor_core_updates(kvb):
    # head_dim 64, 5 KV heads, k = 3: ridge systems of 960 unknowns whose trailing
    # updates (704 and 448 rows and columns) and right-hand-side updates (320 columns)
    # run on the tensor cores with partial 128 x 256 tiles in both directions
    pair = make_pair(6, 4, 3, 5, 64, 3, 512, 8, 1e4, 1e6)
    ctx = _ctx(kvb, pair, 512)
    st = kvb.kvb_stats_create(ctx, kvb.KVB_F32, 512)
    _accumulate(kvb, ctx, st, pair["calib"], torch.float32)
    assert kvb.kvb_stats_count(st) == 1024
    _check_fit(kvb, ctx, st, pair, torch.float32, 1e-4)


def test_chan_merge_over_ragged_batches_and_offsets(kvb):
    # unequal batch lengths, positions not starting at 0: merges must equal two-pass statistics
    rng = np.random.default_rng(3)
    positions = [np.arange(o, o + n) for o, n in ((0, 64), (5, 200), (17, 33), (100, 128), (0, 10))]
    pair = make_pair(7, 3, 2, 2, 16, 2, None, 4, 1e4, 1e6, positions=positions)
    ctx = _ctx(kvb, pair, 512)
    st = kvb.kvb_stats_create(ctx, kvb.KVB_F32, 256)
    _accumulate(kvb, ctx, st, pair["calib"], torch.float32)
    _check_stats(kvb, st, pair, 1e-5)


def test_checkpoint_export_import_resume(kvb):
    pair = make_pair(9, 3, 2, 2, 16, 2, 128, 4, 1e4, 1e6)
    q = 32
    Fs, Ft = 3 * q, 2 * q
    ctx = _ctx(kvb, pair, 128)
    a = kvb.kvb_stats_create(ctx, kvb.KVB_F32, 128)
    _accumulate(kvb, ctx, a, pair["calib"][:2], torch.float32)
    b = kvb.kvb_stats_create(ctx, kvb.KVB_F32, 128)
    f = lambda *s: torch.empty(s, dtype=torch.float32, device="cuda")
    for kv in (0, 1):
        bufs = (f(Fs), f(Ft), f(Fs, Fs), f(Fs, Ft), f(Ft))
        n = kvb.kvb_stats_export(a, kv, *bufs)
        kvb.kvb_stats_import(b, kv, n, *bufs)
    _accumulate(kvb, ctx, b, pair["calib"][2:], torch.float32)
    _check_stats(kvb, b, pair, 1e-5)


def test_bf16_fit_matches_oracle(kvb):
    # bf16 caches, head_dim 128: 4 -> 3 layers, 2 KV heads, k = 2, 8 sequences x 1024 tokens;
    # 1024 source features x 768 target columns tile by 128 x 256: tensor-core statistics
    pair = round_pair(make_pair(11, 4, 3, 2, 128, 2, 1024, 8, 1e4, 1e6, noise=1e-2, sigma=1.0), torch.bfloat16)
    ctx = _ctx(kvb, pair, 1024)
    st = kvb.kvb_stats_create(ctx, kvb.KVB_BF16, 1024)
    kvb.kvb_profile_enable(ctx, True)
    _accumulate(kvb, ctx, st, pair["calib"], torch.bfloat16)
    assert kvb.kvb_profile_read(ctx)["stats_gemm_tcgen05"][0] == 8
    assert kvb.kvb_stats_count(st) == 2048
    _check_stats(kvb, st, pair, 1e-4)
    _check_fit(kvb, ctx, st, pair, torch.float32, TOL_W)


def test_statistics_on_cta_pairs_and_single_ctas_agree(kvb, monkeypatch):
    # sizes that are multiples of 256 run on CTA pairs (256 x 256 tiles) unless
    # KVB_STATS_PAIR=0 when the statistics are created; both merge the same sums
    pair = round_pair(make_pair(12, 4, 3, 2, 128, 2, 1024, 6, 1e4, 1e6, noise=1e-2, sigma=1.0), torch.bfloat16)
    ctx = _ctx(kvb, pair, 1024)
    st_pair = kvb.kvb_stats_create(ctx, kvb.KVB_BF16, 1024)
    monkeypatch.setenv("KVB_STATS_PAIR", "0")
    st_one = kvb.kvb_stats_create(ctx, kvb.KVB_BF16, 1024)
    monkeypatch.delenv("KVB_STATS_PAIR")
    for st in (st_pair, st_one):
        _accumulate(kvb, ctx, st, pair["calib"], torch.bfloat16)
        _check_stats(kvb, st, pair, 1e-4)
    q = pair["H"] * pair["d"]
    for kv in (0, 1):
        a = _export(kvb, st_pair, kv, pair["L_s"] * q, pair["L_t"] * q)
        b = _export(kvb, st_one, kv, pair["L_s"] * q, pair["L_t"] * q)
        assert a[0] == b[0]
        for x, y in zip(a[1:], b[1:]):
            assert rel_fro(x, y) <= 1e-6


def test_fp32_statistics_on_tensor_cores_match_cuda_cores(kvb, monkeypatch):
    # fp32 caches whose shapes tile (1024 source x 768 target features): the statistics
    # run on the tensor cores with three bf16 parts per operand (six products), and on
    # the CUDA cores with KVB_STATS_TC_F32=0; both are fp32-accurate
    pair = make_pair(14, 4, 3, 2, 128, 2, 512, 8, 1e4, 1e6, noise=1e-2, sigma=1.0)
    ctx = _ctx(kvb, pair, 512)
    kvb.kvb_profile_enable(ctx, True)
    st_tc = kvb.kvb_stats_create(ctx, kvb.KVB_F32, 512)
    _accumulate(kvb, ctx, st_tc, pair["calib"], torch.float32)
    assert "stats_gemm_tcgen05" in kvb.kvb_profile_read(ctx)
    monkeypatch.setenv("KVB_STATS_TC_F32", "0")
    st_cc = kvb.kvb_stats_create(ctx, kvb.KVB_F32, 512)
    monkeypatch.delenv("KVB_STATS_TC_F32")
    _accumulate(kvb, ctx, st_cc, pair["calib"], torch.float32)
    assert "stats_gemm_simt" in kvb.kvb_profile_read(ctx)
    _check_stats(kvb, st_tc, pair, 1e-5)
    q = pair["H"] * pair["d"]
    for kv in (0, 1):
        a = _export(kvb, st_tc, kv, pair["L_s"] * q, pair["L_t"] * q)
        b = _export(kvb, st_cc, kv, pair["L_s"] * q, pair["L_t"] * q)
        # both sum ~1024 fp32 products per entry and batch in different orders: each is
        # within ~sqrt(1024) * 2^-24 ~ 2e-6 of the exact sums, as the oracle checks bound
        for x, y in zip(a[1:], b[1:]):
            assert rel_fro(x, y) <= 1e-5
    _check_fit(kvb, ctx, st_tc, pair, torch.float32, 1e-4)


def test_persistent_and_per_tile_solver_updates_agree(kvb, monkeypatch):
    # 1024-wide systems with 768 right-hand sides: the tensor-core updates run on the
    # persistent kernel by default and on the per-tile kernel with KVB_SOLVE_PERSIST=0
    pair = round_pair(make_pair(13, 4, 3, 2, 128, 2, 1024, 6, 1e4, 1e6, noise=1e-2, sigma=1.0), torch.bfloat16)
    ctx = _ctx(kvb, pair, 1024)
    st = kvb.kvb_stats_create(ctx, kvb.KVB_BF16, 1024)
    _accumulate(kvb, ctx, st, pair["calib"], torch.bfloat16)
    a = _run_fit(kvb, ctx, st, pair, torch.float32)
    monkeypatch.setenv("KVB_SOLVE_PERSIST", "0")
    b = _run_fit(kvb, ctx, st, pair, torch.float32)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    assert np.abs(a[2] - b[2]).max() <= 1e-5
    for x, y in zip(a[3:], b[3:]):
        assert rel_fro(to_host64(x), to_host64(y)) <= 1e-5
    _check_fit(kvb, ctx, st, pair, torch.float32, TOL_W)


@pytest.mark.parametrize("d,H", [(32, 8), (64, 4), (16, 16), (128, 2)])
def test_bf16_tensor_core_statistics_head_dims_packed_short_sequences(kvb, d, H):
    # H*d = 256, so the statistics run on the tensor cores; the single-pass gather
    # uses the four-matrix kernel for head_dim 128 (kept rows unevenly spaced at every
    # sequence boundary: one copy per row), its streaming kernel for 64 and the
    # register kernel for 16 / 32.
    # Each batch packs 200 sequences of 1-3 tokens (positions restart at 0), so
    # more rows are kept than T / stride and a CTA walks more than one chunk.
    rng = np.random.default_rng(d)
    positions = [np.concatenate([np.arange(n) for n in rng.integers(1, 4, size=200)]) for _ in range(5)]
    pair = round_pair(make_pair(40 + d, 3, 2, H, d, 2, None, 4, 1e4, 1e6, noise=1e-2, sigma=1.0,
                                positions=positions), torch.bfloat16)
    ctx = _ctx(kvb, pair, 8)
    st = kvb.kvb_stats_create(ctx, kvb.KVB_BF16, 1024)
    kvb.kvb_profile_enable(ctx, True)
    _accumulate(kvb, ctx, st, pair["calib"], torch.bfloat16)
    assert "stats_gemm_tcgen05" in kvb.kvb_profile_read(ctx)
    assert kvb.kvb_stats_count(st) == 800
    _check_stats(kvb, st, pair, 1e-4)


@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 128), (torch.float32, 16)])
def test_target_layer_blocks_reproduce_the_full_fit(kvb, dtype, d):
    # statistics of a target-layer block hold only that block's target columns;
    # one calibration pass per block gives the selections, R^2 and maps of the
    # object that holds every target layer, and of the float64 oracle
    # 8 sequences x 512 tokens, stride 4: 1024 observations for 2 x 2 x d features
    pair = make_pair(31, 4, 5, 2, d, 2, 512, 8, 1e4, 1e6, noise=1e-2, sigma=1.0)
    if dtype == torch.bfloat16:
        pair = round_pair(pair, torch.bfloat16)
    code = kvb.KVB_BF16 if dtype == torch.bfloat16 else kvb.KVB_F32
    ctx = _ctx(kvb, pair, 512)
    L_t, L_s, k, q = 5, 4, 2, 2 * d
    full = kvb.kvb_stats_create(ctx, code, 512)
    _accumulate(kvb, ctx, full, pair["calib"], dtype)
    sel_k, sel_v, r2, Wk, Wv, bk, bv = _run_fit(kvb, ctx, full, pair, torch.float32)
    _, _, _, cross_full, _ = _export(kvb, full, 0, L_s * q, L_t * q)[1:]

    bsk = np.zeros((L_t, k), dtype=np.int32)
    bsv = np.zeros((L_t, k), dtype=np.int32)
    br2 = torch.zeros((2, L_t, L_s), dtype=torch.float32, device="cuda")
    bWk, bWv = torch.zeros_like(Wk), torch.zeros_like(Wv)
    bbk, bbv = torch.zeros_like(bk), torch.zeros_like(bv)
    for t0, t1 in ((0, 2), (2, 5)):
        st = kvb.kvb_stats_create_block(ctx, code, 512, t0, t1)
        _accumulate(kvb, ctx, st, pair["calib"], dtype)
        n, _, _, _, cross_blk, _ = _export(kvb, st, 0, L_s * q, (t1 - t0) * q)
        assert np.abs(cross_blk - cross_full[:, t0 * q:t1 * q]).max() <= 1e-5 * np.abs(cross_full).max()
        kvb.kvb_layer_select(ctx, st, 0.01, br2, sel_k=bsk, sel_v=bsv)
        kvb.kvb_ridge_solve(ctx, st, bsk, bsv, 0.01, bWk, bWv, bbk, bbv)
        kvb.kvb_stats_destroy(st)
    assert np.array_equal(bsk, sel_k) and np.array_equal(bsv, sel_v)
    assert np.abs(to_host64(br2) - r2).max() <= 1e-5
    for a, b in ((bWk, Wk), (bWv, Wv), (bbk, bk), (bbv, bv)):
        assert rel_fro(to_host64(a), to_host64(b)) <= 1e-5
    # the blocked fit against the float64 oracle (KVBridge "Loading": blocking changes
    # how many passes the fit takes, not what it computes)
    fit = O.fit_mapper(pair["calib"], pair["theta_s"], pair["theta_t"], k, 0.01, 4)
    assert np.array_equal(bsk, fit.sel_k) and np.array_equal(bsv, fit.sel_v)
    assert np.array_equal(fit.sel_k, pair["sel_k"]) and np.array_equal(fit.sel_v, pair["sel_v"])
    br2h = to_host64(br2)
    assert np.max(np.abs(br2h[0] - fit.r2_k)) < 1e-4 and np.max(np.abs(br2h[1] - fit.r2_v)) < 1e-4
    w_tol = TOL_W if dtype == torch.bfloat16 else 1e-4
    for gw, ow in ((bWk, fit.W_k), (bWv, fit.W_v)):
        e = rel_fro(np.transpose(to_host64(gw), (0, 2, 1)), ow)
        assert e <= w_tol, e
    for gb, ob in ((bbk, fit.b_k), (bbv, fit.b_v)):
        assert rel_fro(to_host64(gb), ob) <= w_tol


def test_target_block_range_is_validated(kvb):
    pair = make_pair(32, 3, 4, 2, 16, 2, 64, 1, 1e4, 1e6)
    ctx = _ctx(kvb, pair, 64)
    for t0, t1 in ((-1, 2), (2, 2), (3, 2), (0, 5)):
        with pytest.raises(kvb.KvbError):
            kvb.kvb_stats_create_block(ctx, kvb.KVB_F32, 64, t0, t1)


def test_bad_calibration_position_is_reported(kvb):
    pair = make_pair(13, 3, 2, 2, 16, 2, 64, 1, 1e4, 1e6)
    ctx = _ctx(kvb, pair, 32)  # positions reach 63 >= max_pos
    st = kvb.kvb_stats_create(ctx, kvb.KVB_F32, 64)
    _accumulate(kvb, ctx, st, pair["calib"], torch.float32)
    with pytest.raises(kvb.KvbError):
        kvb.kvb_ctx_check(ctx)


def test_bf16_fit_cuda_core_statistics_path(kvb):
    # head_dim 64 and 3 target layers: 384 target columns do not tile by 256, so the
    # statistics run on the CUDA-core kernel (float32 centered operands)
    pair = round_pair(make_pair(12, 3, 3, 2, 64, 2, 512, 8, 1e4, 1e6, noise=1e-2, sigma=1.0), torch.bfloat16)
    ctx = _ctx(kvb, pair, 512)
    st = kvb.kvb_stats_create(ctx, kvb.KVB_BF16, 512)
    _accumulate(kvb, ctx, st, pair["calib"], torch.bfloat16)
    _check_stats(kvb, st, pair, 1e-5)
    _check_fit(kvb, ctx, st, pair, torch.bfloat16, 5e-3)


def test_no_observations_and_zero_lambda_is_a_numeric_error(kvb):
    # Nothing accumulated and lambda = 0: every system is zero, not positive definite.
    pair = make_pair(21, 3, 2, 2, 16, 2, 64, 1, 1e4, 1e6)
    ctx = _ctx(kvb, pair, 64)
    st = kvb.kvb_stats_create(ctx, kvb.KVB_F32, 64)
    with pytest.raises(kvb.KvbError) as e:
        kvb.kvb_layer_select(ctx, st, 0.0)
    assert e.value.status == 5
    Wk = torch.empty((2, 32, 64), dtype=torch.float32, device="cuda")
    bk = torch.empty((2, 32), dtype=torch.float32, device="cuda")
    sel = np.array([[0, 1], [1, 2]], dtype=np.int32)
    with pytest.raises(kvb.KvbError) as e:
        kvb.kvb_ridge_solve(ctx, st, sel, sel, 0.0, Wk, Wk.clone(), bk, bk.clone())
    assert e.value.status == 5


@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 128), (torch.float32, 16)])
def test_non_finite_calibration_value_is_a_numeric_error(kvb, dtype, d):
    # One NaN in one source value reaches the statistics of its feature; the
    # factorisations meet a pivot that is not a positive number and the fit calls
    # return KVB_ERR_NUMERIC instead of a selection or W built on it.
    pair = make_pair(22, 3, 2, 2, d, 2, 256, 4, 1e4, 1e6, noise=1e-2, sigma=1.0)
    if dtype == torch.bfloat16:
        pair = round_pair(pair, torch.bfloat16)
    src_k, src_v, tgt_k, tgt_v, pos = pair["calib"][1]
    src_v = src_v.copy()
    src_v[1, 0, 40, 3] = np.nan
    pair["calib"][1] = (src_k, src_v, tgt_k, tgt_v, pos)
    ctx = _ctx(kvb, pair, 256)
    st = kvb.kvb_stats_create(ctx, kvb.KVB_BF16 if dtype == torch.bfloat16 else kvb.KVB_F32, 256)
    _accumulate(kvb, ctx, st, pair["calib"], dtype)
    with pytest.raises(kvb.KvbError) as e:
        kvb.kvb_layer_select(ctx, st, 0.01)
    assert e.value.status == 5
    q = pair["H"] * d
    Wk = torch.empty((2, q, 2 * q), dtype=torch.float32, device="cuda")
    bk = torch.empty((2, q), dtype=torch.float32, device="cuda")
    sel = np.array([[0, 1], [1, 2]], dtype=np.int32)  # both systems of V read source layer 1
    with pytest.raises(kvb.KvbError) as e:
        kvb.kvb_ridge_solve(ctx, st, sel, sel, 0.01, Wk, Wk.clone(), bk, bk.clone())
    assert e.value.status == 5
    kvb.kvb_ctx_check(ctx)  # the context itself stays usable


def test_top_k_equal_to_all_source_layers(kvb):
    # k = L_src: every source layer is selected; the fit uses all of them.
    pair = make_pair(22, 3, 2, 2, 16, 3, 256, 4, 1e4, 5e4)
    ctx = _ctx(kvb, pair, 256)
    st = kvb.kvb_stats_create(ctx, kvb.KVB_F32, 256)
    _accumulate(kvb, ctx, st, pair["calib"], torch.float32)
    sel_k, sel_v, r2, Wk, Wv, bk, bv = _run_fit(kvb, ctx, st, pair, torch.float32)
    assert sel_k.tolist() == [[0, 1, 2]] * 2 and sel_v.tolist() == [[0, 1, 2]] * 2
    fit = O.fit_mapper(pair["calib"], 1e4, 5e4, 3, 0.01, 4)
    assert rel_fro(np.transpose(to_host64(Wk), (0, 2, 1)), fit.W_k) < 1e-4


@pytest.mark.parametrize("stride", [1, 3, 7])
def test_other_strides(kvb, stride):
    pair = make_pair(23, 3, 2, 2, 16, 2, 100, 3, 1e4, 1e6)
    ctx = _ctx(kvb, pair, 128)
    st = kvb.kvb_stats_create(ctx, kvb.KVB_F32, 128)
    _accumulate(kvb, ctx, st, pair["calib"], torch.float32, stride=stride)
    ref = oracle_full_stats(pair, stride)
    for kv in (0, 1):
        n, mx, my, g, c, y = _export(kvb, st, kv, 96, 64)
        assert n == ref[kv].n and rel_fro(g, ref[kv].M) < 1e-5 and rel_fro(c, ref[kv].C) < 1e-5


def test_reset_then_accumulate_again(kvb):
    pair = round_pair(make_pair(24, 2, 2, 2, 128, 1, 512, 2, 1e4, 1e6, sigma=1.0), torch.bfloat16)
    ctx = _ctx(kvb, pair, 512)
    st = kvb.kvb_stats_create(ctx, kvb.KVB_BF16, 512)
    _accumulate(kvb, ctx, st, pair["calib"][::-1], torch.bfloat16)  # other order first
    kvb.kvb_stats_reset(st)
    assert kvb.kvb_stats_count(st) == 0
    _accumulate(kvb, ctx, st, pair["calib"], torch.bfloat16)
    _check_stats(kvb, st, pair, 1e-4)


def test_four_matrix_gather_matches_oracle_and_per_matrix_path(kvb, monkeypatch):
    # bf16 caches, head_dim 128, 8 -> 8 layers x 8 KV heads (8192 source and target features):
    # the four matrices of a batch go through one gather launch (2048 items, ~13 per SM, so
    # CTAs cross chunk and matrix boundaries), S_yy is updated in the merge.  Two batches:
    # 4096 tokens (1024 kept rows, 8 chunks), then 3000 tokens at positions 7..3006 (750 kept
    # rows, a ragged last chunk).  Checked against the oracle and against one launch per
    # matrix (KVB_GATHER_ALL=0, which also keeps the separate S_yy pass and rounds the
    # stripped keys once more): both within 1e-6 of each other.
    import synth
    L, H, d = 8, 8, 128
    Fs = Ft = L * H * d
    batches = []
    for b, (T, p0) in enumerate(((4096, 0), (3000, 7))):
        caches = [synth.torch_content(900 + 10 * b + i, L, H, T, d, 1.0, torch.bfloat16, "cuda") for i in range(4)]
        batches.append((caches, torch.arange(p0, p0 + T, dtype=torch.int32, device="cuda")))
    ctx = kvb.kvb_ctx_create(spec(L, H, d, 1e4), spec(L, H, d, 1e6), 2, 4096)
    kvb.kvb_profile_enable(ctx, True)
    st_all = kvb.kvb_stats_create(ctx, kvb.KVB_BF16, 4096)
    monkeypatch.setenv("KVB_GATHER_ALL", "0")
    st_one = kvb.kvb_stats_create(ctx, kvb.KVB_BF16, 4096)
    monkeypatch.delenv("KVB_GATHER_ALL")
    for st in (st_all, st_one):
        for caches, pos in batches:
            kvb.kvb_stats_accumulate(ctx, st, *caches, pos, 4)
    kvb.kvb_ctx_check(ctx)
    kvb.kvb_profile_read(ctx)
    # oracle: two-pass centered statistics over the kept rows of both batches
    X, Y = {0: [], 1: []}, {0: [], 1: []}
    for caches, pos in batches:
        ph = pos.cpu().numpy()
        keep = O.retain_stride(ph, 4)
        sk, sv, tk, tv = (to_host64(c) for c in caches)
        X[0].append(O.all_layer_features(sk, ph, 1e4)[keep])
        X[1].append(O.all_layer_features(sv)[keep])
        Y[0].append(O.all_layer_features(tk, ph, 1e6)[keep])
        Y[1].append(O.all_layer_features(tv)[keep])
    for kv in (0, 1):
        ref = O.centered_stats(np.concatenate(X[kv]), np.concatenate(Y[kv]))
        a = _export(kvb, st_all, kv, Fs, Ft)
        b = _export(kvb, st_one, kv, Fs, Ft)
        assert a[0] == b[0] == ref.n == 1024 + 750
        # independent sources and targets: the cross statistics are sqrt(n)-sized noise, so
        # their errors are also taken against the Cauchy-Schwarz scale sqrt(M_ii S_yy_j)
        for got, want in zip(a[1:], (ref.xbar, ref.ybar, ref.M, ref.C, ref.syy)):
            assert rel_fro(got, want) < 1e-4, rel_fro(got, want)
        # per entry: fp32 accumulation in the tensor cores over ~110 K steps per batch
        dm = np.sqrt(np.diag(ref.M))
        assert np.max(np.abs(a[3] - ref.M) / np.outer(dm, dm)) < 5e-5
        assert np.max(np.abs(a[4] - ref.C) / np.outer(dm, np.sqrt(ref.syy))) < 5e-5
        for x, y in zip(a[1:], b[1:]):
            assert rel_fro(x, y) <= 1e-6, rel_fro(x, y)
