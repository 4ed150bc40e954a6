"""ctypes binding of libkvb (include/kvb.h): argument marshalling only.

Torch supplies device memory (data_ptr) and the stream
(torch.cuda.current_stream().cuda_stream); every step of the computation runs
in the library's kernels.  If libkvb.so is missing, every call raises: there is
no fallback.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
# KVB_LIBRARY=checked loads the checked build (index checks on the hot kernels'
# CUDA-core global accesses; build.build(checked=True) makes it)
LIB_PATH = os.path.join(_HERE, "_lib", "libkvb_checked.so" if os.environ.get("KVB_LIBRARY") == "checked"
                        else "libkvb.so")

KVB_OK = 0
KVB_ERR_INVALID_ARG = 1
KVB_ERR_SHAPE_MISMATCH = 2
KVB_ERR_UNSUPPORTED = 3
KVB_ERR_CUDA = 4
KVB_ERR_NUMERIC = 5
KVB_ERR_OOM = 6
KVB_ERR_TIMEOUT = 7
STATUS_NAMES = {0: "KVB_OK", 1: "KVB_ERR_INVALID_ARG", 2: "KVB_ERR_SHAPE_MISMATCH", 3: "KVB_ERR_UNSUPPORTED",
                4: "KVB_ERR_CUDA", 5: "KVB_ERR_NUMERIC", 6: "KVB_ERR_OOM", 7: "KVB_ERR_TIMEOUT"}

KVB_F32 = 0
KVB_BF16 = 1

# Every function include/kvb.h declares, with (restype, argtypes).
_P = ctypes.c_void_p
_I32P = ctypes.POINTER(ctypes.c_int32)
_I64P = ctypes.POINTER(ctypes.c_int64)


class kvb_model_spec(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("rope_theta", ctypes.c_double), ("rope_interleaved", ctypes.c_int32),
                ("rope_scaling", ctypes.c_int32)]


_SPEC_P = ctypes.POINTER(kvb_model_spec)


class kvb_kernel_time(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 32), ("launches", ctypes.c_int64), ("total_ms", ctypes.c_double)]

SIGNATURES = {
    "kvb_last_error": (ctypes.c_char_p, []),
    "kvb_version": (ctypes.c_int32, []),
    "kvb_ctx_create": (ctypes.c_int, [_SPEC_P, _SPEC_P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                      ctypes.POINTER(_P)]),
    "kvb_ctx_destroy": (ctypes.c_int, [_P]),
    "kvb_ctx_reserve": (ctypes.c_int, [_P, ctypes.c_int64]),
    "kvb_ctx_check": (ctypes.c_int, [_P, _P]),
    "kvb_profile_enable": (ctypes.c_int, [_P, ctypes.c_int32]),
    "kvb_profile_read": (ctypes.c_int, [_P, ctypes.POINTER(kvb_kernel_time), ctypes.c_int32, _I32P]),
    "kvb_map_apply": (ctypes.c_int, [_P, ctypes.c_int, _P, _P, _P, ctypes.c_int64, _I32P, _I32P, _P, _P, _P, _P,
                                     _P, _P, _P]),
    "kvb_map_apply_noalloc": (ctypes.c_int, [_SPEC_P, _SPEC_P, ctypes.c_int32, ctypes.c_int32, _P, _P, _P,
                                             ctypes.c_int64, _I32P, _I32P, _P, _P, _P, _P, _P, _P, _P]),
    "kvb_stats_create": (ctypes.c_int, [_P, ctypes.c_int, ctypes.c_int64, ctypes.POINTER(_P)]),
    "kvb_stats_create_block": (ctypes.c_int, [_P, ctypes.c_int, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                              ctypes.POINTER(_P)]),
    "kvb_stats_destroy": (ctypes.c_int, [_P]),
    "kvb_stats_reset": (ctypes.c_int, [_P, _P]),
    "kvb_stats_accumulate": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, ctypes.c_int64, ctypes.c_int32, _P]),
    "kvb_stats_count": (ctypes.c_int, [_P, _I64P, _P]),
    "kvb_stats_export": (ctypes.c_int, [_P, ctypes.c_int32, _I64P, _P, _P, _P, _P, _P, _P]),
    "kvb_stats_import": (ctypes.c_int, [_P, ctypes.c_int32, ctypes.c_int64, _P, _P, _P, _P, _P, _P]),
    "kvb_layer_select": (ctypes.c_int, [_P, _P, ctypes.c_double, _I32P, _I32P, _P, _P]),
    "kvb_ridge_solve": (ctypes.c_int, [_P, _P, _I32P, _I32P, ctypes.c_double, ctypes.c_int, _P, _P, _P, _P, _P]),
    "kvb_attention_cosine": (ctypes.c_int, [_P, ctypes.c_int, _P, ctypes.c_int32, _P, ctypes.c_int64, _P, _P, _P,
                                            _P, _P, ctypes.c_int64, _P, _P]),
}

_lib = None


class KvbError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libkvb.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        how = "build(checked=True)" if path.endswith("_checked.so") else "build()"
        raise RuntimeError(f"{os.path.basename(path)} is not built ({path}); run cross_model_kv_gb300.build.{how}")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def _check(status: int):
    if status != KVB_OK:
        msg = load_library().kvb_last_error()
        raise KvbError(status, msg.decode() if msg else "")


def _spec(s) -> kvb_model_spec:
    if isinstance(s, kvb_model_spec):
        return s
    return kvb_model_spec(int(s["n_layers"]), int(s["n_kv_heads"]), int(s["head_dim"]), float(s["rope_theta"]),
                          int(s.get("rope_interleaved", 0)), int(s.get("rope_scaling", 0)))


def _stream(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _dev(t):
    """Device pointer of a CUDA tensor (must be contiguous)."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _host_sel(sel, L_t: int, k: int) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(sel.cpu() if hasattr(sel, "cpu") else sel, dtype=np.int32))
    if a.shape != (L_t, k):
        raise ValueError(f"selection must be [{L_t}][{k}], got {a.shape}")
    return a


def _dtype_of(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return KVB_BF16
    if t.dtype == torch.float32:
        return KVB_F32
    raise ValueError(f"unsupported dtype {t.dtype}")


class Ctx:
    """Handle of a kvb_ctx plus the geometry it was created with."""

    def __init__(self, handle, src, tgt, top_k, max_pos, device):
        self.handle = handle
        self.src, self.tgt = src, tgt
        self.L_s, self.L_t = src.n_layers, tgt.n_layers
        self.H, self.d, self.k = src.n_kv_heads, src.head_dim, top_k
        self.max_pos, self.device = max_pos, device

    def __del__(self):
        if getattr(self, "handle", None) and _lib is not None:
            _lib.kvb_ctx_destroy(self.handle)
            self.handle = None


# ------------------------------------------------------------------ calls

def kvb_version() -> int:
    return load_library().kvb_version()


def kvb_ctx_create(src, tgt, top_k: int, max_pos: int, device: int = 0) -> Ctx:
    lib = load_library()
    s, t = _spec(src), _spec(tgt)
    h = ctypes.c_void_p()
    _check(lib.kvb_ctx_create(ctypes.byref(s), ctypes.byref(t), int(top_k), int(max_pos), int(device),
                              ctypes.byref(h)))
    return Ctx(h, s, t, int(top_k), int(max_pos), int(device))


def kvb_ctx_destroy(ctx: Ctx):
    if ctx.handle:
        _check(load_library().kvb_ctx_destroy(ctx.handle))
        ctx.handle = None


def kvb_ctx_reserve(ctx: Ctx, T: int):
    _check(load_library().kvb_ctx_reserve(ctx.handle, int(T)))


def kvb_ctx_check(ctx: Ctx, stream=None):
    _check(load_library().kvb_ctx_check(ctx.handle, _stream(stream)))


def kvb_profile_enable(ctx: Ctx, on: bool = True):
    _check(load_library().kvb_profile_enable(ctx.handle, 1 if on else 0))


def kvb_profile_read(ctx: Ctx) -> dict:
    """{kernel name: (launches, total_ms)} since the last read."""
    buf = (kvb_kernel_time * 16)()
    n = ctypes.c_int32()
    _check(load_library().kvb_profile_read(ctx.handle, buf, 16, ctypes.byref(n)))
    return {buf[i].name.decode(): (int(buf[i].launches), float(buf[i].total_ms)) for i in range(n.value)}


def kvb_map_apply(ctx: Ctx, src_k, src_v, positions, sel_k, sel_v, W_k, W_v, b_k, b_v, out_k, out_v,
                  stream=None):
    """Target caches out_k/out_v [L_t][H][T][d] from source caches [L_s][H][T][d].

    W_* are [L_t][H*d][k*H*d] (output-major), b_* float32 [L_t][H*d],
    positions int32 [T] on the device, sel_* [L_t][k] (host or CPU tensor).
    """
    T = int(src_k.shape[2])
    sk = _host_sel(sel_k, ctx.L_t, ctx.k)
    sv = _host_sel(sel_v, ctx.L_t, ctx.k)
    _check(load_library().kvb_map_apply(
        ctx.handle, _dtype_of(src_k), _dev(src_k), _dev(src_v), _dev(positions), T,
        sk.ctypes.data_as(_I32P), sv.ctypes.data_as(_I32P), _dev(W_k), _dev(W_v), _dev(b_k), _dev(b_v),
        _dev(out_k), _dev(out_v), _stream(stream)))


def kvb_map_apply_noalloc(src, tgt, top_k: int, max_pos: int, src_k, src_v, positions, sel_k, sel_v, W_k, W_v,
                          b_k, b_v, out_k, out_v, stream=None):
    """kvb_map_apply without a context and without any device allocation.

    For callers that may not allocate device memory (e.g. inside another
    framework's memory pool): the scratch lives in a fixed 64 MiB array of the
    library.  Calls share that array, so they must not overlap on the GPU.
    """
    s, t = _spec(src), _spec(tgt)
    L_t = t.n_layers
    T = int(src_k.shape[2])
    sk = _host_sel(sel_k, L_t, int(top_k))
    sv = _host_sel(sel_v, L_t, int(top_k))
    _check(load_library().kvb_map_apply_noalloc(
        ctypes.byref(s), ctypes.byref(t), int(top_k), int(max_pos), _dev(src_k), _dev(src_v), _dev(positions), T,
        sk.ctypes.data_as(_I32P), sv.ctypes.data_as(_I32P), _dev(W_k), _dev(W_v), _dev(b_k), _dev(b_v),
        _dev(out_k), _dev(out_v), _stream(stream)))


class Stats:
    def __init__(self, handle, ctx, dtype):
        self.handle, self.ctx, self.dtype = handle, ctx, dtype

    def __del__(self):
        if getattr(self, "handle", None) and _lib is not None:
            _lib.kvb_stats_destroy(self.handle)
            self.handle = None


def kvb_stats_create(ctx: Ctx, dtype: int, max_batch_tokens: int) -> Stats:
    h = ctypes.c_void_p()
    _check(load_library().kvb_stats_create(ctx.handle, int(dtype), int(max_batch_tokens), ctypes.byref(h)))
    return Stats(h, ctx, int(dtype))


def kvb_stats_create_block(ctx: Ctx, dtype: int, max_batch_tokens: int, t_begin: int, t_end: int) -> Stats:
    """Statistics of target layers [t_begin, t_end) only (bounded memory; one calibration pass per block)."""
    h = ctypes.c_void_p()
    _check(load_library().kvb_stats_create_block(ctx.handle, int(dtype), int(max_batch_tokens), int(t_begin),
                                                 int(t_end), ctypes.byref(h)))
    return Stats(h, ctx, int(dtype))


def kvb_stats_destroy(st: Stats):
    if st.handle:
        _check(load_library().kvb_stats_destroy(st.handle))
        st.handle = None


def kvb_stats_reset(st: Stats, stream=None):
    _check(load_library().kvb_stats_reset(st.handle, _stream(stream)))


def kvb_stats_accumulate(ctx: Ctx, st: Stats, src_k, src_v, tgt_k, tgt_v, positions, stride: int = 4,
                         stream=None):
    T = int(src_k.shape[2])
    _check(load_library().kvb_stats_accumulate(ctx.handle, st.handle, _dev(src_k), _dev(src_v), _dev(tgt_k),
                                               _dev(tgt_v), _dev(positions), T, int(stride), _stream(stream)))


def kvb_stats_count(st: Stats, stream=None) -> int:
    n = ctypes.c_int64()
    _check(load_library().kvb_stats_count(st.handle, ctypes.byref(n), _stream(stream)))
    return int(n.value)


def kvb_stats_export(st: Stats, kv: int, mean_x=None, mean_y=None, gram=None, cross=None, syy=None,
                     stream=None) -> int:
    """Copy one kv's statistics into the given float32 CUDA tensors; returns n."""
    n = ctypes.c_int64()
    _check(load_library().kvb_stats_export(st.handle, int(kv), ctypes.byref(n), _dev(mean_x), _dev(mean_y),
                                           _dev(gram), _dev(cross), _dev(syy), _stream(stream)))
    return int(n.value)


def kvb_stats_import(st: Stats, kv: int, n_obs: int, mean_x, mean_y, gram, cross, syy, stream=None):
    _check(load_library().kvb_stats_import(st.handle, int(kv), int(n_obs), _dev(mean_x), _dev(mean_y), _dev(gram),
                                           _dev(cross), _dev(syy), _stream(stream)))


def kvb_layer_select(ctx: Ctx, st: Stats, lam: float = 0.01, r2=None, stream=None, sel_k=None, sel_v=None):
    """Returns (sel_k, sel_v) as int32 numpy arrays [L_t][k]; fills r2 [2][L_t][L_s] if given.

    With block statistics only the block's rows are written: pass the arrays of
    earlier blocks as sel_k / sel_v (int32, [L_t][k], C-contiguous) to fill them in place.
    """
    sk = np.zeros((ctx.L_t, ctx.k), dtype=np.int32) if sel_k is None else sel_k
    sv = np.zeros((ctx.L_t, ctx.k), dtype=np.int32) if sel_v is None else sel_v
    for a in (sk, sv):
        if a.dtype != np.int32 or a.shape != (ctx.L_t, ctx.k) or not a.flags.c_contiguous:
            raise ValueError(f"selection arrays must be C-contiguous int32 [{ctx.L_t}][{ctx.k}]")
    _check(load_library().kvb_layer_select(ctx.handle, st.handle, float(lam), sk.ctypes.data_as(_I32P),
                                           sv.ctypes.data_as(_I32P), _dev(r2), _stream(stream)))
    return sk, sv


def kvb_ridge_solve(ctx: Ctx, st: Stats, sel_k, sel_v, lam, W_k, W_v, b_k, b_v, stream=None):
    sk = _host_sel(sel_k, ctx.L_t, ctx.k)
    sv = _host_sel(sel_v, ctx.L_t, ctx.k)
    _check(load_library().kvb_ridge_solve(ctx.handle, st.handle, sk.ctypes.data_as(_I32P),
                                          sv.ctypes.data_as(_I32P), float(lam), _dtype_of(W_k), _dev(W_k),
                                          _dev(W_v), _dev(b_k), _dev(b_v), _stream(stream)))


def kvb_attention_cosine(ctx: Ctx, q, q_pos, k_a, v_a, k_b, v_b, kv_pos, cos_out, stream=None):
    """cos_out [L_t][Hq][Tq] = cosine of the attention outputs with caches a and b.

    q [L_t][Hq][Tq][d], caches [L_t][H][T][d] (same dtype), q_pos int32 [Tq]
    and kv_pos int32 [T] on the device; key j is visible to query i iff
    kv_pos[j] <= q_pos[i].
    """
    _check(load_library().kvb_attention_cosine(
        ctx.handle, _dtype_of(q), _dev(q), int(q.shape[1]), _dev(q_pos), int(q.shape[2]), _dev(k_a), _dev(v_a),
        _dev(k_b), _dev(v_b), _dev(kv_pos), int(k_a.shape[2]), _dev(cos_out), _stream(stream)))
