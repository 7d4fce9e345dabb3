"""The GEMM pipeline under maximal launch overlap.

Back-to-back GEMM launches captured in a CUDA graph start each CTA while the
previous launch is still running (programmatic dependent launch), so the
weight-copy, decode and MMA stages of one CTA run at full speed against
heavy memory traffic and copies can land out of issue order.  A barrier phase
taken out of order then shows up as a wrong sum.  Every configuration of the
weight ring (odd and even stage counts, two and three activation slots) runs
here on a 21504 x 5376 linear, 20+ units per CTA, and every replay must equal
an eager launch up to the order of the fp32 reductions; the eager launch is
checked against the oracle on sampled row tiles.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from nested_bit_quantized_gb300 import nest, synth  # noqa: E402
from oracle import nest_oracle as O  # noqa: E402
from tests.helpers import parity, to_dev  # noqa: E402

pytestmark = pytest.mark.gpu

M, K = 21504, 5376
LAUNCHES = 8
REPLAYS = 4


@pytest.fixture(scope="module")
def dev():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


_LAYERS = {}


def _layer(bits, dev):
    if bits not in _LAYERS:
        bc, bs, rc, rs = synth.uniform_codes(M, K, bits, 900 + bits)
        s_o, s_i = synth.sign_pair(M, K, 910 + bits)
        layer = nest.pack(to_dev(bc, torch, dev), to_dev(bs, torch, dev), to_dev(rc, torch, dev),
                          to_dev(rs, torch, dev), bits, to_dev(s_o, torch, dev), to_dev(s_i, torch, dev))
        _LAYERS[bits] = (layer, bc, bs, rc, rs, s_i)
    return _LAYERS[bits]


def _close(a, b, rel=1e-6):
    """Equal up to the order of the fp32 additions of the split K range."""
    scale = np.sqrt(np.mean(np.asarray(b, np.float64) ** 2))
    err = np.max(np.abs(np.asarray(a, np.float64) - b))
    assert err <= rel * 64 * scale, f"max |diff| {err} vs rms {scale}"


@pytest.mark.parametrize("bits", [6, 7, 8])
@pytest.mark.parametrize("T", [16, 32, 40, 64])
def test_back_to_back_launches_in_graph(dev, bits, T):
    layer, bc, bs, rc, rs, s_i = _layer(bits, dev)
    xb, xv = synth.activations(T, K, 920 + T)
    x = torch.from_numpy(xb.view(np.int16)).to(dev).view(torch.bfloat16)
    xop = nest.new_xop(K, T, dev)
    nest.rotate(x, layer.sign_in, 0, x_op=xop)
    for verify in (False, True):
        ref = nest.gemm(layer, xop, T, verify).cpu().numpy()
        xr = O.rotate_activations(xv, s_i)
        for tile in (0, 97, M // 128 - 1):
            rows = np.arange(tile * 128, tile * 128 + 128)
            sub = {"base_codes": bc[rows], "base_scales": bs[rows].view(np.float16),
                   "resid_codes": rc[rows], "resid_scales": rs[rows].view(np.float16)}
            parity(ref[:, rows], O.forward_rows(sub, xr, verify))

        zs = [torch.zeros((T, M), dtype=torch.float32, device=dev) for _ in range(LAUNCHES)]
        stream = torch.cuda.Stream(device=dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                for z in zs:
                    nest.gemm(layer, xop, T, verify, z=z)
        torch.cuda.synchronize()
        for _ in range(REPLAYS):
            for z in zs:
                z.zero_()
            torch.cuda.synchronize()
            g.replay()
            torch.cuda.synchronize()
            for z in zs:
                _close(z.cpu().numpy(), ref)
        nest.error_check()
