"""The C ABI: the library builds, loads, exports every declared symbol and
rejects bad arguments on the host before touching a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "kvb.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kvb_[a-z_0-9]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    from cross_model_kv_gb300 import build
    build.build()
    import cross_model_kv_gb300 as kvb
    return kvb.load_library()


def test_header_declares_the_boundary_calls():
    names = _declared_functions()
    for call in ("kvb_stats_accumulate", "kvb_layer_select", "kvb_ridge_solve", "kvb_map_apply"):
        assert call in names


def test_library_exports_every_declared_symbol(lib):
    import cross_model_kv_gb300 as kvb
    for name in _declared_functions():
        assert hasattr(lib, name), name
        assert name in kvb.SIGNATURES, name


def _spec(L, H=8, d=128, theta=1e6, **kw):
    from cross_model_kv_gb300 import kvb_model_spec
    return kvb_model_spec(L, H, d, theta, kw.get("interleaved", 0), kw.get("scaling", 0))


def _create(lib, src, tgt, k=2, max_pos=64):
    h = ctypes.c_void_p()
    st = lib.kvb_ctx_create(ctypes.byref(src), ctypes.byref(tgt), k, max_pos, 0, ctypes.byref(h))
    return st, h


def test_refusals_are_host_side_statuses(lib):
    # "Cross-Model KV Transfer", "The honesty crux" item 7: mismatched KV shapes,
    # rope_scaling and interleaved RoPE are refused, not approximated.
    st, h = _create(lib, _spec(4, H=8), _spec(6, H=4))
    assert st == 2 and not h.value and b"KV heads" in lib.kvb_last_error()
    st, _ = _create(lib, _spec(4, d=128), _spec(6, d=64))
    assert st == 2
    st, _ = _create(lib, _spec(4, scaling=1), _spec(6))
    assert st == 3 and b"rope_scaling" in lib.kvb_last_error()
    st, _ = _create(lib, _spec(4), _spec(6, interleaved=1))
    assert st == 3
    st, _ = _create(lib, _spec(4, d=17), _spec(6, d=17))
    assert st == 3
    st, _ = _create(lib, _spec(4), _spec(6), k=5)
    assert st == 1
    st, _ = _create(lib, _spec(4), _spec(6), k=0)
    assert st == 1
    st, _ = _create(lib, _spec(4), _spec(6), max_pos=0)
    assert st == 1
    # the largest geometry the tables hold: 255 source layers, 128 target layers, k = 16
    st, _ = _create(lib, _spec(256), _spec(6))
    assert st == 3 and b"255" in lib.kvb_last_error()
    st, _ = _create(lib, _spec(40), _spec(129))
    assert st == 3 and b"128" in lib.kvb_last_error()
    st, _ = _create(lib, _spec(40), _spec(64), k=17)
    assert st == 3 and b"16" in lib.kvb_last_error()


def test_null_arguments_are_rejected(lib):
    assert lib.kvb_ctx_destroy(None) == 0
    assert lib.kvb_map_apply(None, 1, None, None, None, 1, None, None, None, None, None, None, None, None,
                             None) == 1
    assert lib.kvb_ctx_reserve(None, 10) == 1
    assert lib.kvb_stats_destroy(None) == 0
    assert lib.kvb_last_error() is not None
    assert lib.kvb_version() >= 1


def test_python_binding_fails_loudly_without_the_library(tmp_path):
    from cross_model_kv_gb300 import _binding
    with pytest.raises(RuntimeError, match="not built"):
        _load_missing(tmp_path)


def _load_missing(tmp_path):
    from cross_model_kv_gb300 import _binding
    saved = _binding._lib
    _binding._lib = None
    try:
        _binding.load_library(str(tmp_path / "missing.so"))
    finally:
        _binding._lib = saved


def test_binding_rejects_wrong_selection_shape_before_the_library():
    import numpy as np
    from cross_model_kv_gb300 import _binding
    with pytest.raises(ValueError, match="selection"):
        _binding._host_sel(np.zeros((3, 2), dtype=np.int32), 4, 2)
