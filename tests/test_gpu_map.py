"""GPU parity of kvb_map_apply against the float64 oracle, through the C ABI.

Small cases compare every element; the full-size pair shapes compare sampled
target layers x sampled tokens (rows and layers are independent, so the
oracle on a slice is exact for that slice)."""
import os
import numpy as np
import pytest

from cases import TOL_BF16, TOL_F32, ApplyCase, rel_fro, spec

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


def _ctx(kvb, c, max_pos):
    return kvb.kvb_ctx_create(spec(c.L_s, c.H, c.d, c.theta_s), spec(c.L_t, c.H, c.d, c.theta_t), c.k, max_pos)


def _check_all(kvb, c, max_pos, tol, layers=None, tokens=None):
    ctx = _ctx(kvb, c, max_pos)
    kvb.kvb_profile_enable(ctx, True)
    c.run(kvb, ctx)
    kvb.kvb_ctx_check(ctx)
    ran = kvb.kvb_profile_read(ctx)
    tensor_core = c.d == 128 and (c.H * c.d) % 256 == 0
    tc_name = "map_gemm_tcgen05" if c.dtype == torch.bfloat16 else "map_gemm_tcgen05_split3"
    assert (tc_name in ran) == tensor_core and ("map_simt" in ran) != tensor_core, ran
    ok, ov = c.oracle(layers, tokens)
    gk, gv = c.gpu(layers, tokens)
    ek, ev = rel_fro(gk, ok), rel_fro(gv, ov)
    assert ek <= tol and ev <= tol, (ek, ev)
    return ek, ev


def test_tiny_pair_fp32(kvb):
    # tiny synthetic pair: 4 -> 6 layers, 2 KV heads, head_dim 16, k = 2, theta 1e4 -> 5e4
    c = ApplyCase(4, 6, 2, 16, 2, 256, 1e4, 5e4, torch.float32, seed=11, sigma=0.5)
    ek, ev = _check_all(kvb, c, 256, TOL_F32)
    assert ek < 1e-5 and ev < 1e-5


def test_tiny_pair_fp32_ragged_positions(kvb):
    from synth import packed_positions, ragged_lengths
    pos = packed_positions(ragged_lengths(3, 5, 1, 120))
    c = ApplyCase(4, 6, 2, 16, 2, len(pos), 1e4, 5e4, torch.float32, seed=12, positions=pos, sigma=0.5)
    _check_all(kvb, c, 128, TOL_F32)


def test_bf16_tensor_core_ragged_tail(kvb):
    # 2 heads x 128 = one 256-wide N tile, T = 300 (two full M tiles and a ragged one)
    c = ApplyCase(3, 2, 2, 128, 2, 300, 1e6, 1e6, torch.bfloat16, seed=21)
    _check_all(kvb, c, 512, TOL_BF16)


def test_bf16_tensor_core_several_n_tiles_random_positions(kvb):
    rng = np.random.default_rng(5)
    pos = rng.integers(0, 32768, size=1000).astype(np.int32)
    c = ApplyCase(5, 3, 8, 128, 3, 1000, 1e4, 5e5, torch.bfloat16, seed=22, positions=pos)
    _check_all(kvb, c, 32768, TOL_BF16)


def test_bf16_tensor_core_single_token(kvb):
    c = ApplyCase(2, 2, 2, 128, 1, 1, 1e4, 1e6, torch.bfloat16, seed=23, positions=[7])
    _check_all(kvb, c, 8, TOL_BF16)


@pytest.mark.parametrize("pair", ["1", "0"])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_tensor_core_largest_top_k(kvb, monkeypatch, pair, dtype):
    # top_k = 16, the most a context takes: the producer steps through 16 selected
    # source layers x 2 heads x 2 K blocks per head (and past the last selection
    # entry after the final block), on the CTA-pair and the single-CTA kernels
    monkeypatch.setenv("KVB_MAP_PAIR", pair)
    dt, tol = (torch.bfloat16, TOL_BF16) if dtype == "bf16" else (torch.float32, TOL_F32)
    c = ApplyCase(17, 3, 2, 128, 16, 300, 1e4, 1e6, dt, seed=26)
    _check_all(kvb, c, 512, tol)


def test_bf16_cuda_core_path_head_dim_64(kvb):
    c = ApplyCase(3, 2, 4, 64, 2, 200, 1e4, 1e6, torch.bfloat16, seed=24)
    _check_all(kvb, c, 256, TOL_BF16)


def test_fp32_tensor_core_split_head_dim_128(kvb):
    # fp32 caches on the tensor cores (bf16 hi/lo operand pairs, three passes)
    c = ApplyCase(3, 2, 2, 128, 2, 130, 1e6, 5e5, torch.float32, seed=25, positions=np.arange(130) * 200)
    _check_all(kvb, c, 32768, TOL_F32)


def test_fp32_tensor_core_split_ragged_tail_two_n_tiles(kvb):
    # 4 KV heads (two 256-wide output tiles), T = 1001 (ragged last token block), random positions
    pos = np.random.default_rng(5).integers(0, 30000, size=1001).astype(np.int32)
    c = ApplyCase(5, 3, 4, 128, 3, 1001, 1e4, 1e6, torch.float32, seed=34, positions=pos)
    ek, ev = _check_all(kvb, c, 30000, TOL_F32)
    assert ek < 2e-5 and ev < 2e-5, (ek, ev)  # the split keeps ~16 bits per operand


def test_fp32_cuda_core_path_head_dim_128_one_head(kvb):
    # one KV head (H*d = 128, not a multiple of the 256-wide output tile): CUDA cores
    c = ApplyCase(3, 2, 1, 128, 2, 70, 1e6, 5e5, torch.float32, seed=35, positions=np.arange(70) * 100)
    _check_all(kvb, c, 8192, TOL_F32)


def test_fp32_bad_position_is_reported_and_row_zeroed(kvb):
    pos = np.arange(200, dtype=np.int32)
    pos[33] = -4
    c = ApplyCase(2, 2, 2, 128, 1, 200, 1e4, 1e6, torch.float32, seed=36, positions=pos)
    ctx = _ctx(kvb, c, 256)
    c.run(kvb, ctx)
    with pytest.raises(kvb.KvbError) as e:
        kvb.kvb_ctx_check(ctx)
    assert e.value.status == 1
    assert torch.count_nonzero(c.out_k[:, :, 33]).item() == 0
    assert torch.count_nonzero(c.out_v[:, :, 33]).item() == 0
    assert torch.count_nonzero(c.out_k[:, :, 32]).item() > 0
    kvb.kvb_ctx_check(ctx)


def test_fused_and_separate_strip_give_identical_bits(kvb, monkeypatch):
    # the strip runs inside the map kernel by default (epilogue warps, during the
    # value tiles); KVB_MAP_FUSED_STRIP=0 runs the separate strip pass instead
    pos = np.random.default_rng(6).integers(0, 30000, size=1500).astype(np.int32)
    c = ApplyCase(6, 4, 4, 128, 3, 1500, 1e4, 1e6, torch.bfloat16, seed=38, positions=pos)
    ctx = _ctx(kvb, c, 30000)
    kvb.kvb_profile_enable(ctx, True)
    c.run(kvb, ctx)
    kvb.kvb_ctx_check(ctx)
    assert "rope_strip_bf16" not in kvb.kvb_profile_read(ctx)
    fused = (c.out_k.clone(), c.out_v.clone())
    monkeypatch.setenv("KVB_MAP_FUSED_STRIP", "0")
    c.out_k.zero_()
    c.out_v.zero_()
    c.run(kvb, ctx)
    kvb.kvb_ctx_check(ctx)
    assert "rope_strip_bf16" in kvb.kvb_profile_read(ctx)
    assert torch.equal(fused[0], c.out_k) and torch.equal(fused[1], c.out_v)
    ok, ov = c.oracle([0, 3], None)
    gk, gv = c.gpu([0, 3], None)
    assert rel_fro(gk, ok) <= TOL_BF16 and rel_fro(gv, ov) <= TOL_BF16


@pytest.mark.parametrize("shape", ["ragged_two_n_tiles", "ragged_two_n_tiles_fp32", "qwen3_0p6b_to_1p7b_T4096"])
def test_pair_kernel_schedules_and_single_cta_kernel(kvb, monkeypatch, shape):
    # maps run on CTA pairs with tiles claimed from a counter (bf16, and fp32 caches as
    # bf16 hi/lo parts); the same pair kernel with the fixed tile-per-pair assignment
    # (KVB_MAP_PAIR_STATIC=1) computes every tile identically, and the single-CTA
    # kernel (KVB_MAP_PAIR=0) is checked on its own
    tol = TOL_BF16
    if shape == "ragged_two_n_tiles":
        c = ApplyCase(5, 4, 4, 128, 2, 1500, 1e4, 1e6, torch.bfloat16, seed=39)
        layers, tokens, max_pos = None, None, 1500
    elif shape == "ragged_two_n_tiles_fp32":
        c = ApplyCase(5, 4, 4, 128, 2, 700, 1e4, 1e6, torch.float32, seed=41)
        layers, tokens, max_pos, tol = None, None, 700, TOL_F32
    else:
        c = ApplyCase(28, 28, 8, 128, 4, 4096, 1e6, 1e6, torch.bfloat16, seed=40, host=False)
        layers, tokens, max_pos = [0, 27], _sampled_tokens(4096, 256, 5), 4096
    ctx = _ctx(kvb, c, max_pos)
    ok, ov = c.oracle(layers, tokens)
    outs = {}
    for name, env in [("dynamic", {}), ("static", {"KVB_MAP_PAIR_STATIC": "1"}), ("single", {"KVB_MAP_PAIR": "0"})]:
        for k in ("KVB_MAP_PAIR_STATIC", "KVB_MAP_PAIR"):
            monkeypatch.delenv(k, raising=False)
        for k, v in env.items():
            monkeypatch.setenv(k, v)
        c.out_k.zero_()
        c.out_v.zero_()
        c.run(kvb, ctx)
        kvb.kvb_ctx_check(ctx)
        outs[name] = (c.out_k.clone(), c.out_v.clone())
        gk, gv = c.gpu(layers, tokens)
        assert rel_fro(gk, ok) <= tol and rel_fro(gv, ov) <= tol, name
    assert torch.equal(outs["dynamic"][0], outs["static"][0]) and torch.equal(outs["dynamic"][1], outs["static"][1])
    del c, outs
    torch.cuda.empty_cache()


def test_empty_input_is_a_no_op(kvb):
    c = ApplyCase(2, 2, 2, 128, 1, 0, 1e4, 1e4, torch.bfloat16, seed=26)
    ctx = _ctx(kvb, c, 8)
    c.run(kvb, ctx)
    kvb.kvb_ctx_check(ctx)


def test_deterministic_bits(kvb):
    c = ApplyCase(4, 2, 8, 128, 2, 777, 1e6, 1e6, torch.bfloat16, seed=27)
    ctx = _ctx(kvb, c, 1024)
    c.run(kvb, ctx)
    a = (c.out_k.clone(), c.out_v.clone())
    c.out_k.zero_()
    c.out_v.zero_()
    c.run(kvb, ctx)
    assert torch.equal(a[0], c.out_k) and torch.equal(a[1], c.out_v)


def test_bad_position_is_reported_and_row_zeroed(kvb):
    pos = np.arange(256, dtype=np.int32)
    pos[17] = 5000  # beyond max_pos = 256
    c = ApplyCase(2, 2, 2, 128, 1, 256, 1e4, 1e6, torch.bfloat16, seed=28, positions=pos)
    ctx = _ctx(kvb, c, 256)
    c.run(kvb, ctx)
    with pytest.raises(kvb.KvbError) as e:
        kvb.kvb_ctx_check(ctx)
    assert e.value.status == 1
    assert torch.count_nonzero(c.out_k[:, :, 17]).item() == 0
    kvb.kvb_ctx_check(ctx)  # cleared once reported


def test_invalid_selection_rejected_before_launch(kvb):
    c = ApplyCase(3, 2, 2, 128, 2, 64, 1e4, 1e4, torch.bfloat16, seed=29)
    ctx = _ctx(kvb, c, 64)
    bad = c.sel_k.copy()
    bad[0] = [1, 1]
    with pytest.raises(kvb.KvbError):
        kvb.kvb_map_apply(ctx, c.src_k, c.src_v, c.positions, bad, c.sel_v, c.W_k, c.W_v, c.b_k, c.b_v,
                          c.out_k, c.out_v)
    bad[0] = [0, 3]
    with pytest.raises(kvb.KvbError):
        kvb.kvb_map_apply(ctx, c.src_k, c.src_v, c.positions, bad, c.sel_v, c.W_k, c.W_v, c.b_k, c.b_v,
                          c.out_k, c.out_v)


def _sampled_tokens(T, n, seed):
    rng = np.random.default_rng(seed)
    idx = np.unique(np.concatenate([rng.choice(T, size=n, replace=False), [0, T - 1]]))
    return idx


def test_qwen3_0p6b_to_1p7b_shape_T4096(kvb):
    # 28 -> 28 layers, 8 KV heads, head_dim 128, theta 1e6 both, k = 4, T = 4096
    c = ApplyCase(28, 28, 8, 128, 4, 4096, 1e6, 1e6, torch.bfloat16, seed=31, host=False)
    _check_all(kvb, c, 4096, TOL_BF16, layers=[0, 13, 27], tokens=_sampled_tokens(4096, 512, 1))
    del c
    torch.cuda.empty_cache()


def test_qwen3_14b_to_32b_shape_T32768(kvb):
    # 40 -> 64 layers, 8 KV heads, head_dim 128, theta 1e6, k = 8, T = 32768
    c = ApplyCase(40, 64, 8, 128, 8, 32768, 1e6, 1e6, torch.bfloat16, seed=32, host=False)
    _check_all(kvb, c, 32768, TOL_BF16, layers=[0, 31, 63], tokens=_sampled_tokens(32768, 384, 2))
    del c
    torch.cuda.empty_cache()


def test_qwen3_14b_to_32b_shape_fp32_T4096(kvb):
    # fp32 caches and maps at the 14B -> 32B shape on the split tensor-core path
    c = ApplyCase(40, 64, 8, 128, 8, 4096, 1e6, 1e6, torch.float32, seed=37, host=False)
    _check_all(kvb, c, 4096, TOL_F32, layers=[0, 40, 63], tokens=_sampled_tokens(4096, 256, 4))
    del c
    torch.cuda.empty_cache()


def test_llama_8b_to_70b_shape_ragged_batch(kvb):
    # 32 -> 80 layers, 8 KV heads, head_dim 128, theta 5e5, k = 8; 16 sequences with
    # lengths uniform in [2048, 32768] packed on the token axis, positions restart.
    from synth import packed_positions, ragged_lengths
    lens = ragged_lengths(7, 16, 2048, 32768)
    pos = packed_positions(lens)
    c = ApplyCase(32, 80, 8, 128, 8, len(pos), 5e5, 5e5, torch.bfloat16, seed=33, positions=pos, host=False)
    starts = np.concatenate([[0], np.cumsum(lens)[:-1]])
    tok = np.unique(np.concatenate([_sampled_tokens(len(pos), 256, 3), starts, starts + lens - 1]))
    _check_all(kvb, c, 32768, TOL_BF16, layers=[0, 79], tokens=tok)
    del c
    torch.cuda.empty_cache()
