"""kvb_attention_cosine against the float64 oracle's attention_output /
attention_cosine: grouped-query heads, causal-by-position masks, ragged key
tiles, suffix and unsorted positions, empty inputs, and the Qwen3-32B target
shape sampled."""
import numpy as np
import pytest

import oracle as O
import synth
from cases import TOL_COS, spec, to_host64

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


class Case:
    """Target queries and two caches (b = a + noise) on the device, with their exact host values."""

    def __init__(self, seed, L, H, g, d, T, Tq, dtype, q_pos=None, kv_pos=None, noise=0.3):
        self.L, self.H, self.Hq, self.d = L, H, H * g, d
        q = synth.content(seed, L, H * g, Tq, d, 0.5)
        ka = synth.content(seed + 1, L, H, T, d, 0.5)
        va = synth.content(seed + 2, L, H, T, d, 0.5)
        kb = ka + noise * synth.noise(seed + 3, ka.shape)
        vb = va + noise * synth.noise(seed + 4, va.shape)
        dev = lambda a: torch.from_numpy(a).to(dtype).cuda().contiguous()
        self.q, self.ka, self.va, self.kb, self.vb = (dev(a) for a in (q, ka, va, kb, vb))
        self.h = [to_host64(t) for t in (self.q, self.ka, self.va, self.kb, self.vb)]
        self.q_pos = np.arange(T - Tq, T, dtype=np.int32) if q_pos is None else np.asarray(q_pos, np.int32)
        self.kv_pos = np.arange(T, dtype=np.int32) if kv_pos is None else np.asarray(kv_pos, np.int32)

    def gpu(self, kvb, ctx):
        out = torch.full((self.L, self.Hq, self.q.shape[2]), float("nan"), dtype=torch.float32, device="cuda")
        qp = torch.from_numpy(self.q_pos).cuda()
        kp = torch.from_numpy(self.kv_pos).cuda()
        kvb.kvb_attention_cosine(ctx, self.q, qp, self.ka, self.va, self.kb, self.vb, kp, out)
        torch.cuda.synchronize()
        kvb.kvb_ctx_check(ctx)
        return out.cpu().numpy().astype(np.float64)

    def oracle(self, layers=None, kv_heads=None):
        """Oracle cosines [len(layers)][len(kv_heads) * g][Tq] (all when None)."""
        q, ka, va, kb, vb = self.h
        layers = range(self.L) if layers is None else layers
        kv_heads = range(self.H) if kv_heads is None else kv_heads
        g = self.Hq // self.H
        out = []
        for l in layers:
            rows = []
            for kh in kv_heads:
                sl = slice(kh * g, (kh + 1) * g)
                one = lambda a: a[l:l + 1, kh:kh + 1]
                rows.append(O.attention_cosine(q[l:l + 1, sl], self.q_pos, one(ka), one(va), one(kb), one(vb),
                                               self.kv_pos)[0])
            out.append(np.concatenate(rows))
        return np.stack(out)

    def select(self, c, layers, kv_heads):
        g = self.Hq // self.H
        idx = np.concatenate([np.arange(kh * g, (kh + 1) * g) for kh in kv_heads])
        return c[np.asarray(layers)][:, idx]


def _ctx(kvb, L, H, d):
    return kvb.kvb_ctx_create(spec(1, H, d, 1e6), spec(L, H, d, 1e6), 1, 64)


def test_fp32_causal_gqa_ragged_tiles(kvb):
    c = Case(80, L=2, H=2, g=3, d=64, T=77, Tq=77, dtype=torch.float32)
    got = c.gpu(kvb, _ctx(kvb, 2, 2, 64))
    ref = c.oracle()
    assert np.abs(got - ref).max() <= TOL_COS
    assert 0.2 < ref.mean() < 0.999  # the two caches differ, the outputs still agree in direction


@pytest.mark.parametrize("d", [16, 32, 64, 128])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_head_dims_and_dtypes(kvb, d, dtype):
    c = Case(81 + d, L=2, H=2, g=2, d=d, T=100, Tq=100, dtype=dtype)
    got = c.gpu(kvb, _ctx(kvb, 2, 2, d))
    assert np.abs(got - c.oracle()).max() <= TOL_COS


def test_suffix_queries_over_a_long_prefix(kvb):
    # held-out continuation: the last 50 positions query a 1000-token cache
    c = Case(90, L=1, H=2, g=4, d=128, T=1000, Tq=50, dtype=torch.bfloat16)
    got = c.gpu(kvb, _ctx(kvb, 1, 2, 128))
    assert np.abs(got - c.oracle()).max() <= TOL_COS


def test_unsorted_positions_mask_by_position_not_index(kvb):
    rng = np.random.default_rng(91)
    kv_pos = rng.permutation(300)
    q_pos = rng.integers(-3, 320, size=45)  # includes queries that see nothing or everything
    c = Case(91, L=2, H=1, g=2, d=32, T=300, Tq=45, dtype=torch.float32, q_pos=q_pos, kv_pos=kv_pos)
    got = c.gpu(kvb, _ctx(kvb, 2, 1, 32))
    ref = c.oracle()
    assert np.abs(got - ref).max() <= TOL_COS
    assert np.all(got[:, :, q_pos < 0] == 0)


def test_tensor_core_unsorted_positions_partial_row_blocks(kvb):
    # bf16, head_dim 128 (tensor-core kernel): permuted key positions over three key
    # tiles (the last partial), queries that see nothing, part or all of the keys, and
    # 3 x 45 = 135 query rows (a second, almost empty row block)
    rng = np.random.default_rng(98)
    kv_pos = rng.permutation(300)
    q_pos = np.concatenate([[-5, 0, 299, 1000], rng.integers(0, 300, size=41)])
    c = Case(98, L=2, H=2, g=3, d=128, T=300, Tq=45, dtype=torch.bfloat16, q_pos=q_pos, kv_pos=kv_pos)
    got = c.gpu(kvb, _ctx(kvb, 2, 2, 128))
    ref = c.oracle()
    assert np.abs(got - ref).max() <= TOL_COS
    assert np.all(got[:, :, q_pos < 0] == 0)


def test_tensor_core_rising_maxima_over_many_key_tiles(kvb):
    # tensor-core kernel against the oracle: row maxima that rise by more than 2^8
    # (base 2) several times across 9 key tiles, so that O is rescaled in TMEM, a
    # ragged last tile, a partial row block, and causal suffix queries that see 1 to
    # 9 tiles
    T = 1100
    q_pos = np.concatenate([np.arange(T - 70, T), [0, 1, 127, 128, 129, 500]])
    c = Case(99, L=2, H=2, g=2, d=128, T=T, Tq=76, dtype=torch.bfloat16, q_pos=q_pos)
    ramp = torch.linspace(0.2, 24.0, T, device="cuda").to(torch.bfloat16)[None, None, :, None]
    c.ka = (c.ka * ramp).contiguous()  # later keys score higher: the reference maximum rises
    c.kb = (c.kb * ramp).contiguous()
    c.h[1], c.h[3] = to_host64(c.ka), to_host64(c.kb)
    got = c.gpu(kvb, _ctx(kvb, 2, 2, 128))
    assert np.abs(got - c.oracle()).max() <= TOL_COS


def test_identical_caches_give_one(kvb):
    c = Case(92, L=1, H=2, g=2, d=128, T=130, Tq=130, dtype=torch.bfloat16, noise=0.0)
    got = c.gpu(kvb, _ctx(kvb, 1, 2, 128))
    assert np.abs(got - 1).max() <= 1e-6


def test_empty_inputs(kvb):
    ctx = _ctx(kvb, 1, 2, 16)
    # no keys: every output is zero, so every cosine is 0
    c = Case(93, L=1, H=2, g=1, d=16, T=0, Tq=5, dtype=torch.float32, q_pos=np.arange(5))
    assert np.all(c.gpu(kvb, ctx) == 0)
    # no queries: nothing to write, no error
    c = Case(94, L=1, H=2, g=1, d=16, T=8, Tq=0, dtype=torch.float32, q_pos=np.zeros(0))
    assert c.gpu(kvb, ctx).shape == (1, 2, 0)


def test_rejects_bad_arguments(kvb):
    ctx = _ctx(kvb, 1, 2, 16)
    c = Case(95, L=1, H=2, g=1, d=16, T=8, Tq=8, dtype=torch.float32)
    out = torch.zeros((1, 2, 8), device="cuda")
    qp = torch.from_numpy(c.q_pos).cuda()
    kp = torch.from_numpy(c.kv_pos).cuda()
    bad_q = torch.zeros((1, 3, 8, 16), device="cuda")  # 3 query heads over 2 KV heads
    with pytest.raises(kvb.KvbError):
        kvb.kvb_attention_cosine(ctx, bad_q, qp, c.ka, c.va, c.kb, c.vb, kp, out)
    ctx96 = _ctx(kvb, 1, 2, 96)
    q96 = torch.zeros((1, 2, 8, 96), device="cuda")
    kv96 = torch.zeros((1, 2, 8, 96), device="cuda")
    with pytest.raises(kvb.KvbError):
        kvb.kvb_attention_cosine(ctx96, q96, qp, kv96, kv96, kv96, kv96, kp, out)


def test_qwen3_32b_target_shape_sampled(kvb):
    # 64 layers, 64 query heads over 8 KV heads, head_dim 128: one 256-token
    # held-out sequence, every position a query; oracle on sampled layers/heads
    c = Case(96, L=64, H=8, g=8, d=128, T=256, Tq=256, dtype=torch.bfloat16)
    got = c.gpu(kvb, _ctx(kvb, 64, 8, 128))
    assert np.isfinite(got).all()
    layers, heads = [0, 31, 63], [0, 5, 7]
    assert np.abs(c.select(got, layers, heads) - c.oracle(layers, heads)).max() <= TOL_COS


def test_long_context_suffix_sampled(kvb):
    # 4096-token cache, last 64 positions as queries, 8 layers of the 32B shape
    c = Case(97, L=8, H=8, g=8, d=128, T=4096, Tq=64, dtype=torch.bfloat16)
    got = c.gpu(kvb, _ctx(kvb, 8, 8, 128))
    layers, heads = [2, 7], [3]
    assert np.abs(c.select(got, layers, heads) - c.oracle(layers, heads)).max() <= TOL_COS
