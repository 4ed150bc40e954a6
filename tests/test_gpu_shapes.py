"""Other pair shapes through kvb_map_apply: the big->small direction and odd
token counts, sampled against the float64 oracle."""
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


def _run(kvb, c, max_pos, layers, tokens):
    ctx = kvb.kvb_ctx_create(spec(c.L_s, c.H, c.d, c.theta_s), spec(c.L_t, c.H, c.d, c.theta_t), c.k, max_pos)
    c.run(kvb, ctx)
    kvb.kvb_ctx_check(ctx)
    ok, ov = c.oracle(layers, tokens)
    gk, gv = c.gpu(layers, tokens)
    assert rel_fro(gk, ok) <= TOL_BF16 and rel_fro(gv, ov) <= TOL_BF16


def test_big_to_small_qwen3_32b_to_14b_shape(kvb):
    # 64 -> 40 layers (the reverse direction of the 14B -> 32B pair), k = 8, T = 3000
    c = ApplyCase(64, 40, 8, 128, 8, 3000, 1e6, 1e6, torch.bfloat16, seed=61, host=False)
    tok = np.unique(np.concatenate([np.random.default_rng(1).choice(3000, 256, replace=False), [0, 2999]]))
    _run(kvb, c, 3000, [0, 21, 39], tok)


def test_different_thetas_and_odd_token_count(kvb):
    # 12 -> 20 layers, 4 KV heads (two 256-wide output tiles), k = 5, theta 1e4 -> 5e5, T = 1001
    rng = np.random.default_rng(2)
    pos = rng.integers(0, 20000, size=1001).astype(np.int32)
    c = ApplyCase(12, 20, 4, 128, 5, 1001, 1e4, 5e5, torch.bfloat16, seed=62, positions=pos)
    _run(kvb, c, 20000, None, None)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_largest_supported_geometry(kvb, dtype):
    # 255 source layers, 128 target layers, k = 16 (the limits of the selection
    # table), 2 KV heads x 128: every K block of a 4096-wide feature row comes
    # from a different (layer, head) slab
    pos = np.random.default_rng(3).integers(0, 4096, size=300).astype(np.int32)
    c = ApplyCase(255, 128, 2, 128, 16, 300, 1e4, 1e6, dtype, seed=63, positions=pos)
    tol = TOL_BF16 if dtype == torch.bfloat16 else TOL_F32
    ctx = kvb.kvb_ctx_create(spec(c.L_s, c.H, c.d, c.theta_s), spec(c.L_t, c.H, c.d, c.theta_t), c.k, 4096)
    c.run(kvb, ctx)
    kvb.kvb_ctx_check(ctx)
    ok, ov = c.oracle([0, 64, 127], None)
    gk, gv = c.gpu([0, 64, 127], None)
    assert rel_fro(gk, ok) <= tol and rel_fro(gv, ov) <= tol
