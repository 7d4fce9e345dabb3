"""GPU parity of the BitNest W4/W8 codec (BitNest paper, Section 3.2-3.3 and Appendix A.1)
through the C ABI, against the CPU oracle: packing bit for bit, the quantizer code for code
(up to fp64 rounding-order ties), and the draft (W4) and verify (W8) GEMMs and whole
linears within the GEMM gate (relative L2 <= 1e-3, every element within 1e-2 * rms)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from nested_bit_quantized_gb300 import nest, synth  # noqa: E402
from oracle import nest_oracle as O  # noqa: E402
from oracle import pack as P  # noqa: E402
from tests.helpers import parity, to_dev  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


def _codes(M, K, seed):
    """Random admissible codes, q4 = -8 included (with the refinement clipped to [0, 7] there)."""
    rng = np.random.default_rng(seed)
    q4 = rng.integers(-8, 8, size=(M, K)).astype(np.int8)
    qr = rng.integers(-8, 8, size=(M, K)).astype(np.int8)
    qr = np.where(q4 == -8, np.abs(qr) % 8, qr).astype(np.int8)
    s4 = np.exp(rng.uniform(np.log(1e-3), np.log(5e-2), size=(M, K // 128))).astype(np.float16)
    return q4, s4, qr


def _layer(q4, s4, qr, s_o, s_i, dev):
    return nest.pack_w4w8(to_dev(q4, torch, dev), to_dev(s4.view(np.int16), torch, dev),
                          to_dev(qr, torch, dev) if qr is not None else None,
                          to_dev(s_o, torch, dev), to_dev(s_i, torch, dev))


@pytest.mark.parametrize("M,K", [(128, 128), (200, 384), (1, 256), (300, 1024)])
def test_pack_bit_exact(dev, M, K):
    q4, s4, qr = _codes(M, K, M + K)
    s_o, s_i = synth.sign_pair(M, K, 3)
    L = _layer(q4, s4, qr, s_o, s_i, dev)
    base, ref = P.pack_w4w8(q4, s4, qr)
    assert np.array_equal(L.base.cpu().numpy(), base)
    assert np.array_equal(L.resid.cpu().numpy(), ref)
    back = nest.unpack_w4w8(L)
    assert np.array_equal(back["q4"].cpu().numpy(), q4)
    assert np.array_equal(back["qr"].cpu().numpy(), qr)
    assert np.array_equal(back["s4"].cpu().numpy().view(np.uint16), s4.view(np.uint16))
    L0 = _layer(q4, s4, None, s_o, s_i, dev)
    assert L0.resid is None and np.array_equal(L0.base.cpu().numpy(), base)


@pytest.mark.parametrize("M,K", [(256, 512), (200, 1024), (96, 384)])
def test_quantizer_matches_oracle(dev, M, K):
    W = synth.weights(M, K, 17 + M, "entries")
    s_o, s_i = synth.sign_pair(M, K, 19)
    ref = O.quantize_layer_w4w8(W, s_o, s_i)
    got = nest.quantize_w4w8(to_dev(W.astype(np.float32), torch, dev), to_dev(s_o, torch, dev),
                             to_dev(s_i, torch, dev))
    s4 = got["s4"].cpu().numpy().view(np.float16)
    assert np.array_equal(s4.view(np.uint16), ref["s4"].view(np.uint16))
    q4, qr = got["q4"].cpu().numpy(), got["qr"].cpu().numpy()
    # codes agree except where W' sits within rounding-order distance of a decision point
    Wr = ref["Wr"]
    s = np.repeat(ref["s4"].astype(np.float64), 128, axis=1)
    near4 = np.abs(np.abs(Wr / np.where(s > 0, s, 1)) % 1 - 0.5) < 1e-9
    assert np.all((q4 == ref["q4"]) | near4)
    dW = Wr - O.dequant_w4(q4, ref["s4"])
    sref = s / 16
    near_r = np.abs(np.abs(dW / np.where(sref > 0, sref, 1)) % 1 - 0.5) < 1e-8
    ok = (qr == ref["qr"]) | near_r | (q4 != ref["q4"])
    assert np.all(ok)
    assert (q4 != ref["q4"]).sum() <= 2 and (~(qr == ref["qr"])).sum() <= 4


SHAPES = [(128, 128), (200, 384), (1280, 1024), (129, 256), (384, 2560)]


@pytest.mark.parametrize("M,K", SHAPES)
def test_gemm_parity(dev, M, K):
    W = synth.weights(M, K, 31 + M, "entries")
    s_o, s_i = synth.sign_pair(M, K, 37)
    lay = O.quantize_layer_w4w8(W, s_o, s_i)
    L = _layer(lay["q4"], lay["s4"], lay["qr"], s_o, s_i, dev)
    for T in (1, 5, 16, 17, 33, 64):
        xb, xv = synth.activations(T, K, 40 + T)
        x = torch.from_numpy(xb.view(np.int16)).to(dev).view(torch.bfloat16)
        xop = nest.new_xop(K, T, dev)
        nest.rotate(x, L.sign_in, 0, x_op=xop)
        for verify in (False, True):
            z = nest.gemm(L, xop, T, verify).cpu().numpy()
            parity(z, O.forward_w4w8(lay, s_o, s_i, xv, verify)["z"])
    nest.error_check()


def test_edge_codes_and_linear(dev):
    """Random admissible codes including q4 = -8 (refinement in [0, 7]), every code value,
    through the whole linear (rotate in, GEMM, rotate out), grouped with a second layer."""
    shapes = [(640, 1536), (384, 1536)]
    layers, refs = [], []
    for i, (M, K) in enumerate(shapes):
        q4, s4, qr = _codes(M, K, 50 + i)
        s_o, s_i = synth.sign_pair(M, K, 60 + i)
        layers.append(_layer(q4, s4, qr, s_o, s_i, dev))
        refs.append(({"q4": q4, "s4": s4, "qr": qr}, s_o, s_i))
    for T in (1, 16, 40):
        xb, xv = synth.activations(T, 1536, 70 + T)
        x = torch.from_numpy(xb.view(np.int16)).to(dev).view(torch.bfloat16)
        for verify in (False, True):
            y = nest.linear(layers[0], x, verify).cpu().numpy()
            parity(y, O.forward_w4w8(refs[0][0], refs[0][1], refs[0][2], xv, verify)["y"])
            ys = nest.linear_group(layers, [x, x], verify)
            for (lay, s_o, s_i), yg in zip(refs, ys):
                parity(yg.cpu().numpy(), O.forward_w4w8(lay, s_o, s_i, xv, verify)["y"])
    nest.error_check()


def test_draft_register_fragment_and_tcgen05_paths(dev, monkeypatch):
    """The W4 draft on both GEMM kernels: the register-fragment (mma.sync) kernel that
    serves T <= 8 by default, forced up to T = 32, and the tcgen05 kernel forced down to
    T = 1; random admissible codes (every q4 value), each against the oracle."""
    M, K = 1280, 2560
    q4, s4, qr = _codes(M, K, 90)
    s_o, s_i = synth.sign_pair(M, K, 91)
    L = _layer(q4, s4, qr, s_o, s_i, dev)
    lay = {"q4": q4, "s4": s4, "qr": qr}
    for T in (1, 3, 8, 9, 16, 17, 32):
        xb, xv = synth.activations(T, K, 92 + T)
        x = torch.from_numpy(xb.view(np.int16)).to(dev).view(torch.bfloat16)
        xop = nest.new_xop(K, T, dev)
        nest.rotate(x, L.sign_in, 0, x_op=xop)
        ref = O.forward_w4w8(lay, s_o, s_i, xv, False)["z"]
        for path in ("rf", "tc"):
            monkeypatch.setenv("NEST_GEMM_PATH", path)
            parity(nest.gemm(L, xop, T, False).cpu().numpy(), ref)
    monkeypatch.delenv("NEST_GEMM_PATH")
    nest.error_check()


def test_draft_is_exact_subset(dev):
    """With a zero refinement the W8 target decodes to 16 q4 s4 / 16: the draft's values."""
    M, K = 512, 1024
    q4, s4, qr = _codes(M, K, 80)
    qr[:] = 0
    s_o, s_i = synth.sign_pair(M, K, 81)
    L = _layer(q4, s4, qr, s_o, s_i, dev)
    xb, _ = synth.activations(16, K, 82)
    x = torch.from_numpy(xb.view(np.int16)).to(dev).view(torch.bfloat16)
    xop = nest.new_xop(K, 16, dev)
    nest.rotate(x, L.sign_in, 0, x_op=xop)
    a = nest.gemm(L, xop, 16, False).cpu().numpy().astype(np.float64)
    b = nest.gemm(L, xop, 16, True).cpu().numpy().astype(np.float64)
    scale = np.sqrt(np.mean(a * a))
    assert np.max(np.abs(a - b)) <= 1e-6 * 64 * scale


def test_w4w8_prefill(dev):
    M, K = 640, 1024
    q4, s4, qr = _codes(M, K, 90)
    s_o, s_i = synth.sign_pair(M, K, 91)
    L = _layer(q4, s4, qr, s_o, s_i, dev)
    lay = {"q4": q4, "s4": s4, "qr": qr}
    for T in (128, 256):
        xb, xv = synth.activations(T, K, 92 + T)
        x = torch.from_numpy(xb.view(np.int16)).to(dev).view(torch.bfloat16)
        for verify in (False, True):
            parity(nest.linear(L, x, verify).cpu().numpy(), O.forward_w4w8(lay, s_o, s_i, xv, verify)["y"])
    nest.error_check()
