"""Host-side argument checks of the Python binding.

The library takes raw device pointers and cannot see how large a buffer is, so
the binding checks every caller-provided buffer (size, dtype, contiguity, device)
before its pointer is passed on.  Here the checks run on CPU tensors: with the
device requirement switched off, each short or mistyped buffer must be refused
with a ValueError naming it; with the requirement on, a host tensor is refused.
No call here reaches a kernel.
"""
import pytest

torch = pytest.importorskip("torch")

from nested_bit_quantized_gb300 import nest  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def lib():
    import __graft_entry__
    __graft_entry__.build()
    return nest.load()


@pytest.fixture
def no_device_check(monkeypatch):
    monkeypatch.setattr(nest, "_require_cuda", lambda t, name: None)


def _layer(M=256, K=512, bits=7):
    return nest.Layer(M, K, bits, torch.zeros(nest.base_bytes(M, K), dtype=torch.uint8),
                      torch.zeros(nest.resid_bytes(M, K, bits), dtype=torch.uint8),
                      torch.ones(M, dtype=torch.int8), torch.ones(K, dtype=torch.int8))


def _xop(K, T, short=False):
    n = nest.xop_bytes(K, T) // 2
    return torch.zeros(n - 1 if short else n, dtype=torch.int16)


def test_host_tensor_is_refused():
    L, T = _layer(), 4
    with pytest.raises(ValueError, match="x_op must be a CUDA tensor"):
        nest.gemm(L, _xop(L.K, T), T, True, z=torch.zeros((T, L.M)))
    with pytest.raises(ValueError, match="x must be a CUDA tensor"):
        nest.linear(L, torch.zeros((T, L.K), dtype=torch.bfloat16), True)


def test_gemm_buffers(no_device_check):
    L, T = _layer(), 16
    with pytest.raises(ValueError, match="x_op holds"):
        nest.gemm(L, _xop(L.K, T, short=True), T, True, z=torch.zeros((T, L.M)))
    with pytest.raises(ValueError, match="z must be torch.float32"):
        nest.gemm(L, _xop(L.K, T), T, True, z=torch.zeros((T, L.M), dtype=torch.float64))
    with pytest.raises(ValueError, match="z holds"):
        nest.gemm(L, _xop(L.K, T), T, True, z=torch.zeros((T - 1, L.M)))
    with pytest.raises(ValueError, match="z must be contiguous"):
        nest.gemm(L, _xop(L.K, T), T, True, z=torch.zeros((L.M, T)).t())
    with pytest.raises(ValueError, match="one operand and one accumulator"):
        nest.gemm_group([L, L], [_xop(L.K, T)], T, True, zs=[torch.zeros((T, L.M))] * 2)
    with pytest.raises(ValueError, match="x_op holds"):
        nest.gemm_group([L, L], [_xop(L.K, T), _xop(L.K, T, short=True)], T, True,
                        zs=[torch.zeros((T, L.M))] * 2)


def test_linear_buffers(no_device_check):
    L, T = _layer(), 8
    x = torch.zeros((T, L.K), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match=r"x must be a \[8\]\[512\] tensor"):
        nest.linear(L, torch.zeros((T, L.K + 128), dtype=torch.bfloat16), True)
    with pytest.raises(ValueError, match="float32 or bfloat16"):
        nest.linear(L, torch.zeros((T, L.K), dtype=torch.float16), True)
    with pytest.raises(ValueError, match="y holds"):
        nest.linear(L, x, True, y=torch.zeros((T, L.M - 1)))
    need = nest.linear_scratch_bytes(L.M, L.K, T)
    assert need > 0
    with pytest.raises(ValueError, match="scratch holds"):
        nest.linear(L, x, True, y=torch.zeros((T, L.M)), scratch=torch.zeros(need - 1, dtype=torch.uint8))
    with pytest.raises(ValueError, match="share one dtype"):
        nest.linear_group([L, L], [x, x.float()], True)
    with pytest.raises(ValueError, match="scratch holds"):
        nest.linear_group([L, L], [x, x], True, scratch=torch.zeros(16, dtype=torch.uint8))


def test_rotation_buffers(no_device_check):
    T, n = 3, 1024
    x = torch.zeros((T, n), dtype=torch.bfloat16)
    s = torch.ones(n, dtype=torch.int8)
    with pytest.raises(ValueError, match="signs holds"):
        nest.rotate(x, s[:-1], 0, y=torch.zeros((T, n)))
    with pytest.raises(ValueError, match="signs must be torch.int8"):
        nest.rotate(x, s.float(), 0, y=torch.zeros((T, n)))
    with pytest.raises(ValueError, match="y holds"):
        nest.rotate(x, s, 0, y=torch.zeros((T, n - 1)))
    with pytest.raises(ValueError, match="x_op holds"):
        nest.rotate(x, s, 0, x_op=_xop(n, T, short=True))
    with pytest.raises(ValueError, match="one sign vector"):
        nest.rotate_group([x, x], [s], 0, x_ops=[_xop(n, T)] * 2)
    with pytest.raises(ValueError, match="zero must be torch.float32"):
        nest.rotate_group([x], [s], 0, x_ops=[_xop(n, T)], zero=[torch.zeros(8, dtype=torch.float64)])


def test_quantize_and_pack_buffers(no_device_check, monkeypatch):
    M, K = 256, 512
    W = torch.zeros((M, K))
    so, si = torch.ones(M, dtype=torch.int8), torch.ones(K, dtype=torch.int8)
    monkeypatch.setattr(nest, "_dev", lambda t, dtype, name: t)   # W's own device check
    with pytest.raises(ValueError, match="work holds"):
        nest.quantize(W, so, si, 7, work=torch.zeros((M, K - 1), dtype=torch.float64))
    with pytest.raises(ValueError, match="sign_in holds"):
        nest.quantize(W, so, si[:-1], 7)
    codes = torch.zeros((M, K), dtype=torch.uint8)
    scales = torch.zeros((M, K // 128), dtype=torch.int16)
    with pytest.raises(ValueError, match="resid_codes holds"):
        nest.pack(codes, scales, torch.zeros((M, K - 1), dtype=torch.int8), scales, 7, so, si)
    with pytest.raises(ValueError, match="base_scales holds"):
        nest.pack(codes, scales[:, :-1].contiguous(), None, None, 0, so, si)


def test_kv_buffers(no_device_check):
    cache = nest.KVCache.__new__(nest.KVCache)          # shape only: no device planes needed
    cache.H, cache.Lmax = 4, 64
    with pytest.raises(ValueError, match=r"x must be \[T\]\[4\]\[128\]"):
        nest.kv_write(cache, torch.zeros((3, 2, 128)), 0)
    with pytest.raises(ValueError, match=r"q must be \[T\]\[Hq\]\[128\]"):
        nest.kv_attention(torch.zeros((1, 8, 64)), cache, cache, 16, 8)
    with pytest.raises(ValueError, match="out holds"):
        nest.kv_attention(torch.zeros((1, 8, 128)), cache, cache, 16, 8, out=torch.zeros((1, 8, 127)))


def test_chain_buffers(no_device_check):
    from nested_bit_quantized_gb300 import chain
    M, T = 512, 4
    za, sa = torch.zeros((T, M)), torch.ones(M, dtype=torch.int8)
    work = torch.zeros(chain.chain_work_bytes(M, T) // 4)
    nxt = [nest.Layer(256, M, 0, torch.zeros(16, dtype=torch.uint8), None, sa, sa)]
    with pytest.raises(ValueError, match="work holds"):
        chain.chain(za, sa, None, None, T, work[:-1], None, nxt, [_xop(M, T)], None)
    with pytest.raises(ValueError, match="z_b and s_b"):
        chain.chain(za, sa, za.clone(), None, T, work, None, nxt, [_xop(M, T)], None)
    with pytest.raises(ValueError, match="x_op holds"):
        chain.chain(za, sa, None, None, T, work, None, nxt, [_xop(M, T, short=True)], None)
    with pytest.raises(ValueError, match="one operand"):
        chain.chain(za, sa, None, None, T, work, None, nxt, [], None)
    with pytest.raises(ValueError, match="reads 1024 features"):
        bad = [nest.Layer(256, 2 * M, 0, torch.zeros(16, dtype=torch.uint8), None, sa, sa)]
        chain.chain(za, sa, None, None, T, work, None, bad, [_xop(M, T)], None)
    with pytest.raises(ValueError, match="z_next holds"):
        chain.chain(za, sa, None, None, T, work, None, nxt, [_xop(M, T)], [torch.zeros((T, 255))])
