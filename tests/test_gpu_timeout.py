"""Failure detection on the GPU without a fault: a bounded wait that runs out.

With KVB_WAIT_TIMEOUT_MS=0 every mbarrier wait of the tensor-core map kernel
gives up as soon as it would have to wait; the kernel records KVB_ERR_TIMEOUT,
stops its other roles, drains its own copies and MMAs, frees TMEM and returns.
The host reads the status, and the device keeps working: a second context
with the default limit maps the same inputs correctly."""
import numpy as np
import pytest

from cases import TOL_BF16, ApplyCase, rel_fro, spec

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

KVB_ERR_TIMEOUT = 7


@pytest.fixture(scope="module")
def kvb():
    from cross_model_kv_gb300 import build
    build.build()
    import cross_model_kv_gb300 as m
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return m


def test_wait_limit_runs_out_status_reported_and_device_usable(kvb, monkeypatch):
    # 8 -> 8 layers, 8 KV heads, k = 4, T = 8192: a map of a few milliseconds, so the
    # epilogue warps wait on the first accumulator long enough to give up
    c = ApplyCase(8, 8, 8, 128, 4, 8192, 1e6, 1e6, torch.bfloat16, seed=71, host=False)
    mk = lambda: kvb.kvb_ctx_create(spec(c.L_s, c.H, c.d, c.theta_s), spec(c.L_t, c.H, c.d, c.theta_t), c.k, 8192)
    monkeypatch.setenv("KVB_WAIT_TIMEOUT_MS", "0")
    ctx0 = mk()
    c.run(kvb, ctx0)
    with pytest.raises(kvb.KvbError) as e:
        kvb.kvb_ctx_check(ctx0)
    assert e.value.status == KVB_ERR_TIMEOUT
    kvb.kvb_ctx_check(ctx0)  # reported once, then cleared
    monkeypatch.delenv("KVB_WAIT_TIMEOUT_MS")
    ctx1 = mk()
    c.out_k.zero_()
    c.out_v.zero_()
    c.run(kvb, ctx1)
    kvb.kvb_ctx_check(ctx1)
    tok = np.unique(np.concatenate([np.random.default_rng(0).choice(8192, 128, replace=False), [0, 8191]]))
    ok, ov = c.oracle([0, 7], tok)
    gk, gv = c.gpu([0, 7], tok)
    assert rel_fro(gk, ok) <= TOL_BF16 and rel_fro(gv, ov) <= TOL_BF16
