"""The rotation kernel's three paths against the oracle.

nest_rotate computes x' = H S x (mode 0) or y = S H z (mode 1) with blocks of
b = the largest power of two dividing n, at most 4096 (feedman.me/posts/wZBTJ,
POC recipe steps 1 and 4).  The kernel picks, per vector set, the register
path (b <= 512, n % 8 == 0, 16-byte aligned x and y), the segment path
(b >= 1024, 16-byte aligned y) or the shared-memory tile path.  Here every
shape runs once with aligned buffers and once with x and y views 4 bytes off a
16-byte boundary (which sends it to the tile path); both must match the oracle,
for both modes, both input types and the operand output.  The grouped call's
clearing is checked with counts that do and do not allow 16-byte stores and
with more clearing than rotation work.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from nested_bit_quantized_gb300 import nest, synth  # noqa: E402
from oracle import nest_oracle as O  # noqa: E402
from tests.helpers import decode_xop, to_dev  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


def _view(vals, dtype, dev, offset_bytes):
    """A [T][n] device tensor of `vals` in `dtype`, starting offset_bytes past a 512-byte
    aligned allocation."""
    T, n = vals.shape
    t = torch.from_numpy(np.ascontiguousarray(vals)).to(dtype)
    esz = t.element_size()
    assert offset_bytes % esz == 0
    k = offset_bytes // esz
    raw = torch.zeros(T * n + k + 8, dtype=dtype, device=dev)
    raw[k:k + T * n] = t.reshape(-1).to(dev)
    v = raw[k:k + T * n].view(T, n)
    assert v.data_ptr() % 16 == offset_bytes % 16
    return v


def _out(T, n, dev, offset_bytes):
    raw = torch.full((T * n + 8,), float("nan"), dtype=torch.float32, device=dev)
    k = offset_bytes // 4
    return raw[k:k + T * n].view(T, n)


def _close(got, ref, tol=1e-5):
    ref = np.asarray(ref, np.float64)
    assert np.max(np.abs(np.asarray(got, np.float64) - ref)) <= tol * max(1.0, np.max(np.abs(ref)))


# n: b = 256 (register, 256-element chunks), 512 x 3 (register, 512-element chunks),
# 1024 x 5, 2048 x 3, 4096 x 2, 4096 x 3 + 1024 (segment, ragged last segment), 96 (b = 32)
@pytest.mark.parametrize("n", [256, 1536, 5120, 6144, 8192, 13312, 96])
@pytest.mark.parametrize("T", [1, 5, 16])
def test_rotation_paths_match_oracle(dev, n, T):
    s = synth.signs(n, 900 + n)
    sd = to_dev(s, torch, dev)
    xb, xv = synth.activations(T, n, 901 + T)
    z = np.random.default_rng(n + T).normal(size=(T, n)).astype(np.float32)
    ref_in = O.rotate_activations(xv, s)
    ref_in32 = O.rotate_activations(z, s)
    ref_out = O.unrotate_outputs(z, s)
    for off in (0, 4):                                   # aligned, then 4 bytes off
        x16 = _view(xv, torch.bfloat16, dev, off)
        x32 = _view(z, torch.float32, dev, off)
        y = _out(T, n, dev, off)
        xop = nest.new_xop(n, T, dev) if n % 128 == 0 else None
        nest.rotate(x16, sd, 0, y=y, x_op=xop)
        _close(y.cpu().numpy(), ref_in)
        if xop is not None:
            h = decode_xop(xop.cpu().numpy(), n, T).astype(np.float64)
            assert np.max(np.abs(h - ref_in) / np.maximum(np.abs(ref_in), 6.2e-5)) <= 2.0 ** -10
        y = _out(T, n, dev, off)
        nest.rotate(x32, sd, 0, y=y)
        _close(y.cpu().numpy(), ref_in32)
        y = _out(T, n, dev, off)
        nest.rotate(x32, sd, 1, y=y)
        _close(y.cpu().numpy(), ref_out)
        # output side from a bf16 input
        y = _out(T, n, dev, off)
        nest.rotate(x16, sd, 1, y=y)
        _close(y.cpu().numpy(), O.unrotate_outputs(xv, s))
    nest.error_check()


@pytest.mark.parametrize("count", [1, 7, 8192, 8193, 100_000])
def test_grouped_rotation_clears(dev, count):
    """Clearing alongside a small rotation: scalar and 16-byte stores, and (100 000 floats
    beside one 256-element vector) CTAs that only clear."""
    n, T = 256, 1
    s = synth.signs(n, 77)
    xb, xv = synth.activations(T, n, 78)
    x = torch.from_numpy(xb.view(np.int16)).to(dev).view(torch.bfloat16)
    for off in (0, 4):
        raw = torch.full((count + 16,), 5.0, dtype=torch.float32, device=dev)
        k = off // 4
        zc = raw[k:k + count]
        ops = [nest.new_xop(n, T, dev)]
        nest.rotate_group([x], [to_dev(s, torch, dev)], 0, x_ops=ops, zero=[zc])
        assert torch.count_nonzero(zc).item() == 0
        assert torch.all(raw[:k] == 5.0) and torch.all(raw[k + count:] == 5.0)   # nothing past the range
        h = decode_xop(ops[0].cpu().numpy(), n, T).astype(np.float64)
        ref = O.rotate_activations(xv, s)
        assert np.max(np.abs(h - ref) / np.maximum(np.abs(ref), 6.2e-5)) <= 2.0 ** -10
    nest.error_check()
