"""kvb_map_apply_noalloc: the mapper apply for callers that may not allocate
device memory (code living inside another framework's memory pool, or a
runtime that owns the whole device budget).  It keeps its scratch in a fixed
array of the library; its results must match kvb_map_apply's.

This file is collected last on purpose, so a run that stops at the first
failure has already run every other test."""
import numpy as np
import pytest

from cases import TOL_BF16, ApplyCase, rel_fro, spec, to_host64

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def kvb():
    from cross_model_kv_gb300 import build
    build.build()
    import cross_model_kv_gb300 as m
    return m


def _noalloc(kvb, c, max_pos, out_k, out_v):
    kvb.kvb_map_apply_noalloc(spec(c.L_s, c.H, c.d, c.theta_s), spec(c.L_t, c.H, c.d, c.theta_t), c.k, max_pos,
                              c.src_k, c.src_v, c.positions, c.sel_k, c.sel_v, c.W_k, c.W_v, c.b_k, c.b_v,
                              out_k, out_v)


@pytest.mark.gpu
def test_noalloc_matches_the_context_entry_point_on_two_calls_in_a_row(kvb):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    rng = np.random.default_rng(41)
    pos_b = rng.integers(0, 600, size=500).astype(np.int32)
    cases = [ApplyCase(6, 4, 8, 128, 3, 500, 1e4, 1e6, torch.bfloat16, seed=40),
             ApplyCase(6, 4, 8, 128, 3, 500, 1e4, 1e6, torch.bfloat16, seed=80, positions=pos_b)]
    for c in cases:  # two different inputs, one call each, back to back
        ctx = kvb.kvb_ctx_create(spec(c.L_s, c.H, c.d, c.theta_s), spec(c.L_t, c.H, c.d, c.theta_t), c.k, 600)
        c.run(kvb, ctx)
        kvb.kvb_ctx_check(ctx)
        ref_k, ref_v = to_host64(c.out_k), to_host64(c.out_v)
        out_k = torch.full_like(c.out_k, float("nan"))
        out_v = torch.full_like(c.out_v, float("nan"))
        _noalloc(kvb, c, 600, out_k, out_v)
        torch.cuda.synchronize()
        ek, ev = rel_fro(to_host64(out_k), ref_k), rel_fro(to_host64(out_v), ref_v)
        assert ek <= TOL_BF16 and ev <= TOL_BF16, (ek, ev)
        kvb.kvb_ctx_destroy(ctx)


def test_noalloc_rejects_sizes_beyond_its_scratch(kvb):
    # 40 source layers x 8 heads x 128 dims x 2 bytes = 80 KiB per token: 1000 tokens exceed 64 MiB.
    # Rejected on the host, before any device work.
    import ctypes
    from cross_model_kv_gb300 import _binding as b
    lib = b.load_library()
    s = b.kvb_model_spec(40, 8, 128, 1e6, 0, 0)
    t = b.kvb_model_spec(64, 8, 128, 1e6, 0, 0)
    sel = np.zeros((64, 8), dtype=np.int32)
    st = lib.kvb_map_apply_noalloc(ctypes.byref(s), ctypes.byref(t), 8, 1000, None, None, None, 1000,
                                   sel.ctypes.data_as(b._I32P), sel.ctypes.data_as(b._I32P), None, None, None,
                                   None, None, None, None)
    assert st == b.KVB_ERR_INVALID_ARG and b"64 MiB" in lib.kvb_last_error()
