"""GPU parity of the nested KV4/KV8 cache (BitNest paper, Section 3.4, Appendix A.2)
through the C ABI: quantise-on-write code for code against the oracle (both decide in
fp32), and decode attention in both views and under the Recent-N policy against the
oracle's fp64 attention (relative L2 <= 1e-3, every element within 1e-2 * rms)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from nested_bit_quantized_gb300 import nest  # noqa: E402
from oracle import nest_oracle as O  # noqa: E402
from tests.helpers import parity  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


def _planes(cache, L):
    H, Lmax = cache.H, cache.Lmax
    b = cache.base.cpu().numpy().reshape(H, Lmax, 64)[:, :L]
    r = cache.ref.cpu().numpy().reshape(H, Lmax, 64)[:, :L]
    lo = lambda a: (a & 15).astype(np.int8) - 8
    hi = lambda a: (a >> 4).astype(np.int8) - 8
    q4 = np.stack([lo(b), hi(b)], axis=-1).reshape(H, L, 128)
    qr = np.stack([lo(r), hi(r)], axis=-1).reshape(H, L, 128)
    s = cache.scale.cpu().numpy().view(np.float16).reshape(H, Lmax)[:, :L]
    return q4, qr, s


@pytest.mark.parametrize("bf16", [False, True])
def test_kv_write_matches_oracle(dev, bf16):
    H, Lmax, T = 8, 96, 37
    rng = np.random.default_rng(3)
    x = (rng.normal(size=(T, H, 128)) * rng.uniform(0.05, 8, size=(T, H, 1))).astype(np.float32)
    x[5, 2] = 0.0                                        # a zero vector
    xt = torch.from_numpy(x).to(dev)
    if bf16:
        xt = xt.to(torch.bfloat16)
        x = xt.float().cpu().numpy()
    cache = nest.KVCache(H, Lmax, dev)
    nest.kv_write(cache, xt[:20], 0)
    nest.kv_write(cache, xt[20:], 20)                    # appended in a second call
    q4, qr, s = _planes(cache, T)
    rq4, rqr, rs = O.kv_quantize(np.transpose(x, (1, 0, 2)))
    assert np.array_equal(s.view(np.uint16), rs.view(np.uint16))
    assert np.array_equal(q4, rq4)
    assert np.array_equal(qr, rqr)
    nest.error_check()


@pytest.mark.parametrize("T,Hq,Hkv,L", [(1, 8, 4, 300), (1, 64, 32, 1000), (16, 4, 2, 700), (5, 6, 6, 77),
                                        (3, 32, 2, 2600)])
def test_kv_attention_views_and_recent_n(dev, T, Hq, Hkv, L):
    rng = np.random.default_rng(T * 1000 + L)
    Lmax = L + 16
    kx = rng.normal(size=(L, Hkv, 128)).astype(np.float32)
    vx = rng.normal(size=(L, Hkv, 128)).astype(np.float32)
    kc, vc = nest.KVCache(Hkv, Lmax, dev), nest.KVCache(Hkv, Lmax, dev)
    nest.kv_write(kc, torch.from_numpy(kx).to(dev), 0)
    nest.kv_write(vc, torch.from_numpy(vx).to(dev), 0)
    k = O.kv_quantize(np.transpose(kx, (1, 0, 2)))
    v = O.kv_quantize(np.transpose(vx, (1, 0, 2)))
    q = rng.normal(size=(T, Hq, 128)).astype(np.float32) * 2
    qt = torch.from_numpy(q).to(dev)
    for view, rn in ((8, 0), (4, 0), (4, 64), (4, L)):
        got = nest.kv_attention(qt, kc, vc, L, view, rn).cpu().numpy()
        ref = O.kv_attention(q, k, v, L, view, rn)
        parity(got.reshape(T * Hq, 128), ref.reshape(T * Hq, 128))
    nest.error_check()


def test_kv_attention_bf16_queries_and_long_context(dev):
    T, Hq, Hkv, L = 2, 16, 8, 9000
    rng = np.random.default_rng(11)
    kx = rng.normal(size=(L, Hkv, 128)).astype(np.float32)
    vx = rng.normal(size=(L, Hkv, 128)).astype(np.float32)
    kc, vc = nest.KVCache(Hkv, L, dev), nest.KVCache(Hkv, L, dev)
    nest.kv_write(kc, torch.from_numpy(kx).to(dev), 0)
    nest.kv_write(vc, torch.from_numpy(vx).to(dev), 0)
    qt = (torch.from_numpy(rng.normal(size=(T, Hq, 128)).astype(np.float32)) * 3).to(dev).to(torch.bfloat16)
    q = qt.float().cpu().numpy()
    k = O.kv_quantize(np.transpose(kx, (1, 0, 2)))
    v = O.kv_quantize(np.transpose(vx, (1, 0, 2)))
    for view in (4, 8):
        got = nest.kv_attention(qt, kc, vc, L, view, 128).cpu().numpy()
        parity(got.reshape(-1, 128), O.kv_attention(q, k, v, L, view, 128).reshape(-1, 128))
    nest.error_check()


@pytest.mark.parametrize("impl", ["cuda", "tc", "tc16"])
def test_kv_attention_both_kernels(dev, impl, monkeypatch):
    """The tensor-core kernels (default: 8- and 16-row CTAs, paired 32-row CTAs above 16
    rows), the tensor-core kernel with 16-row CTAs only, and the CUDA-core kernel on the
    same cache, rows per KV head from 1 to 40 (one and several tiles)."""
    monkeypatch.setenv("NEST_KV_IMPL", impl)
    rng = np.random.default_rng(21)
    Hkv, L = 3, 500
    kx = rng.normal(size=(L, Hkv, 128)).astype(np.float32)
    vx = rng.normal(size=(L, Hkv, 128)).astype(np.float32)
    kc, vc = nest.KVCache(Hkv, L, dev), nest.KVCache(Hkv, L, dev)
    nest.kv_write(kc, torch.from_numpy(kx).to(dev), 0)
    nest.kv_write(vc, torch.from_numpy(vx).to(dev), 0)
    k = O.kv_quantize(np.transpose(kx, (1, 0, 2)))
    v = O.kv_quantize(np.transpose(vx, (1, 0, 2)))
    for T, G in ((1, 1), (3, 3), (9, 1), (5, 8), (17, 2), (16, 3)):
        q = rng.normal(size=(T, Hkv * G, 128)).astype(np.float32)
        for view, rn in ((8, 0), (4, 17)):
            got = nest.kv_attention(torch.from_numpy(q).to(dev), kc, vc, L, view, rn).cpu().numpy()
            parity(got.reshape(-1, 128), O.kv_attention(q, k, v, L, view, rn).reshape(-1, 128))
    monkeypatch.delenv("NEST_KV_IMPL")
    nest.error_check()


@pytest.mark.parametrize("view", [4, 8])
def test_kv_attention_growing_and_falling_scores(dev, view):
    """Key norms that ramp up over the context (the running max grows at every block) and
    then down again (it never grows): both branches of the online-softmax rescale."""
    rng = np.random.default_rng(31 + view)
    T, Hq, Hkv, L = 4, 8, 2, 3000
    ramp = np.concatenate([np.linspace(0.2, 3.0, L // 2), np.linspace(3.0, 0.2, L - L // 2)])
    direction = rng.normal(size=(Hkv, 128))
    kx = (ramp[:, None, None] * (direction[None] + 0.3 * rng.normal(size=(L, Hkv, 128)))).astype(np.float32)
    vx = rng.normal(size=(L, Hkv, 128)).astype(np.float32)
    kc, vc = nest.KVCache(Hkv, L, dev), nest.KVCache(Hkv, L, dev)
    nest.kv_write(kc, torch.from_numpy(kx).to(dev), 0)
    nest.kv_write(vc, torch.from_numpy(vx).to(dev), 0)
    k = O.kv_quantize(np.transpose(kx, (1, 0, 2)))
    v = O.kv_quantize(np.transpose(vx, (1, 0, 2)))
    G = Hq // Hkv
    q = (np.repeat(direction, G, axis=0)[None] * 0.4 + 0.1 * rng.normal(size=(T, Hq, 128))).astype(np.float32)
    got = nest.kv_attention(torch.from_numpy(q).to(dev), kc, vc, L, view, 0).cpu().numpy()
    parity(got.reshape(-1, 128), O.kv_attention(q, k, v, L, view, 0).reshape(-1, 128))
    nest.error_check()
