"""kvb_map_apply_noalloc: the mapper apply for callers that may not allocate
device memory at all -- code running inside another framework's memory pool
(which owns every byte of the device), or a runtime that hands the library a
fixed budget up front.  Such callers cannot create a context, so this entry
point keeps its scratch in a fixed array inside the library instead.

Its results must be the same bits as kvb_map_apply's (both run the same strip
and map kernels; the separate strip pass and the one fused into the map kernel
are bit-identical), agree with the float64 oracle, leave the device's free
memory unchanged, and report a bad position through the status it returns.

This file is collected last on purpose, so a run that stops at the first
failure has already run every other test."""
import numpy as np
import pytest

from cases import TOL_BF16, ApplyCase, rel_fro, spec

torch = pytest.importorskip("torch")

MAX_POS = 600


@pytest.fixture(scope="module")
def kvb():
    from cross_model_kv_gb300 import build
    build.build()
    import cross_model_kv_gb300 as m
    return m


def _noalloc(kvb, c, out_k, out_v, positions=None):
    kvb.kvb_map_apply_noalloc(spec(c.L_s, c.H, c.d, c.theta_s), spec(c.L_t, c.H, c.d, c.theta_t), c.k, MAX_POS,
                              c.src_k, c.src_v, c.positions if positions is None else positions, c.sel_k, c.sel_v,
                              c.W_k, c.W_v, c.b_k, c.b_v, out_k, out_v)


def _cases():
    rng = np.random.default_rng(41)
    pos_b = rng.integers(0, MAX_POS, size=500).astype(np.int32)
    return [ApplyCase(6, 4, 8, 128, 3, 500, 1e4, 1e6, torch.bfloat16, seed=40),
            ApplyCase(6, 4, 8, 128, 3, 500, 1e4, 1e6, torch.bfloat16, seed=80, positions=pos_b)]


@pytest.mark.gpu
def test_noalloc_matches_the_context_entry_point_on_two_calls_in_a_row(kvb):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cases = _cases()
    refs = []
    for c in cases:
        ctx = kvb.kvb_ctx_create(spec(c.L_s, c.H, c.d, c.theta_s), spec(c.L_t, c.H, c.d, c.theta_t), c.k, MAX_POS)
        c.run(kvb, ctx)
        kvb.kvb_ctx_check(ctx)
        refs.append((c.out_k.clone(), c.out_v.clone()))
        kvb.kvb_ctx_destroy(ctx)
    outs = [(torch.full_like(c.out_k, float("nan")), torch.full_like(c.out_v, float("nan"))) for c in cases]
    # first call on this device: sets up the scratch address (and loads the kernels' modules)
    _noalloc(kvb, cases[0], *outs[0])
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    for c, (ok, ov) in zip(cases, outs):  # two different inputs, back to back
        ok.fill_(float("nan"))
        ov.fill_(float("nan"))
        _noalloc(kvb, c, ok, ov)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free_before
    rng = np.random.default_rng(7)
    for c, (ok, ov), (rk, rv) in zip(cases, outs, refs):
        assert torch.equal(ok, rk) and torch.equal(ov, rv)
        layers = np.array([0, c.L_t - 1])
        tokens = np.sort(rng.choice(c.T, size=96, replace=False))
        ek_o, ev_o = c.oracle(layers, tokens)
        c.out_k, c.out_v = ok, ov
        gk, gv = c.gpu(layers, tokens)
        ek, ev = rel_fro(gk, ek_o), rel_fro(gv, ev_o)
        assert ek <= TOL_BF16 and ev <= TOL_BF16, (ek, ev)


@pytest.mark.gpu
def test_noalloc_reports_a_position_beyond_max_pos(kvb):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    c = _cases()[0]
    bad = c.positions.clone()
    bad[123] = MAX_POS  # one position outside [0, max_pos): its rows become zeros, the call reports it
    ok, ov = torch.empty_like(c.out_k), torch.empty_like(c.out_v)
    with pytest.raises(kvb.KvbError) as e:
        _noalloc(kvb, c, ok, ov, positions=bad)
    assert e.value.status == 1
    assert torch.count_nonzero(ok[:, :, 123]) == 0
    # the error word is cleared by the next call, which maps correctly again
    _noalloc(kvb, c, ok, ov)
    torch.cuda.synchronize()
    rk, rv = c.oracle(np.array([1]), np.arange(0, c.T, 7))
    c.out_k, c.out_v = ok, ov
    gk, gv = c.gpu(np.array([1]), np.arange(0, c.T, 7))
    assert rel_fro(gk, rk) <= TOL_BF16 and rel_fro(gv, rv) <= TOL_BF16


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
