"""GPU parity of the chained-layer path: nest_chain and a chained decoder layer.

Tolerance of chained outputs, derived from the arithmetic.  Each intermediate
is cast to bf16 (8 significant bits, relative ulp 2^-8..2^-7).  The GPU's fp32
intermediates differ from the oracle's fp64 ones by the fp16-operand GEMM
error (relative ~3e-4), so their bf16 roundings land on neighbouring values for
part of the elements: each cast re-injects a relative difference of order
ulp/sqrt(6) ~ 1e-3.  The gate * up product adds the relative differences of
its two factors, once per layer, so the difference grows about linearly with
depth.  The gate for an output reached through c bf16 casts is relative
L2 <= 1.5e-3 * c, every element within 6e-2 * rms.  Outputs with no cast on
their path (k, v of the first layer) and the nest_chain kernel itself keep the
GEMM gate (1e-3, 1e-2).
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from nested_bit_quantized_gb300 import chain, nest, synth  # noqa: E402
from oracle import nest_oracle as O  # noqa: E402
from tests.helpers import decode_xop, parity, to_dev  # noqa: E402

pytestmark = pytest.mark.gpu


def chained(got, ref, casts):
    parity(got, ref, 1.5e-3 * casts, 6e-2)


@pytest.fixture(scope="module")
def dev():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


@pytest.mark.parametrize("M,T,product", [(512, 1, False), (5376, 17, True), (3840, 64, False), (8192, 5, True)])
def test_chain_kernel(dev, M, T, product):
    rng = np.random.default_rng(M + T)
    za = rng.normal(size=(T, M)).astype(np.float32)
    zb = rng.normal(size=(T, M)).astype(np.float32) if product else None
    sa, sb = synth.signs(M, 1), synth.signs(M, 2)
    nxt = [synth.signs(M, 3 + j) for j in range(2)]
    y = torch.empty((T, M), dtype=torch.float32, device=dev)
    # two next linears reading h (their descriptors only need K == M and S_i)
    dummy = torch.zeros(16, dtype=torch.uint8, device=dev)
    layers = [nest.Layer(128, M, 0, dummy, None, to_dev(sa, torch, dev), to_dev(s, torch, dev)) for s in nxt]
    xops = [nest.new_xop(M, T, dev) for _ in nxt]
    zn = [torch.full((T, 128), 7.0, device=dev) for _ in nxt]
    chain.chain(to_dev(za, torch, dev), to_dev(sa, torch, dev), to_dev(zb, torch, dev) if product else None,
                to_dev(sb, torch, dev) if product else None, T, y, layers, xops, zn)
    ya = O.unrotate_outputs(za, sa)
    yref = ya * O.unrotate_outputs(zb, sb) if product else ya
    parity(y.cpu().numpy(), yref)
    h = O.chain_glue(ya, O.unrotate_outputs(zb, sb) if product else None)
    for s, xop in zip(nxt, xops):
        parity(decode_xop(xop.cpu().numpy(), M, T).astype(np.float64), O.rotate_activations(h, s))
    for z in zn:
        assert torch.count_nonzero(z).item() == 0


SMALL = dict(hidden=512, inter=1024, q=512, kv=256)


def _small_layer(l, bits):
    shapes = [("q", SMALL["q"], SMALL["hidden"]), ("k", SMALL["kv"], SMALL["hidden"]), ("v", SMALL["kv"], SMALL["hidden"]),
              ("o", SMALL["hidden"], SMALL["q"]), ("gate", SMALL["inter"], SMALL["hidden"]),
              ("up", SMALL["inter"], SMALL["hidden"]), ("down", SMALL["hidden"], SMALL["inter"])]
    out = {}
    for i, (n, M, K) in enumerate(shapes):
        W = synth.weights(M, K, 700 + 16 * l + i, "entries")
        s_o, s_i = synth.sign_pair(M, K, 7000 + 32 * l + 2 * i)
        out[n] = (O.quantize_layer(W, s_o, s_i, bits), s_o, s_i)
    return out


def _dev_layer(q, bits, s_o, s_i, dev):
    return nest.pack(to_dev(q["base_codes"], torch, dev), to_dev(q["base_scales"], torch, dev),
                     to_dev(q["resid_codes"], torch, dev), to_dev(q["resid_scales"], torch, dev), bits,
                     to_dev(s_o, torch, dev), to_dev(s_i, torch, dev))


@pytest.mark.parametrize("T", [1, 16, 64])
def test_two_chained_decoder_layers(dev, T):
    bits = 8
    ref = [_small_layer(l, bits) for l in range(2)]
    lin = [{n: _dev_layer(q, bits, so, si, dev) for n, (q, so, si) in r.items()} for r in ref]
    xb, xv = synth.activations(T, SMALL["hidden"], 77)
    x = torch.from_numpy(xb.view(np.int16)).to(dev).view(torch.bfloat16)
    for verify in (False, True):
        bufs = [chain.LayerBuffers(l, T, dev) for l in lin]
        chain.layer_input(lin[0], x, bufs[0])
        chain.layer_forward(lin[0], bufs[0], verify, lin[1], bufs[1])
        chain.layer_forward(lin[1], bufs[1], verify)
        o0 = O.decoder_layer_forward(ref[0], xv, verify)
        o1 = O.decoder_layer_forward(ref[1], o0["next"], verify)
        parity(bufs[0].y["k"].cpu().numpy(), o0["k"])                 # no cast on the path: GEMM gate
        parity(bufs[0].y["v"].cpu().numpy(), o0["v"])
        chained(bufs[0].y["down"].cpu().numpy(), o0["down"], 3)       # q->o, o->gate/up, gate*up->down
        chained(bufs[1].y["k"].cpu().numpy(), o1["k"], 4)              # + down -> next layer
        chained(bufs[1].y["down"].cpu().numpy(), o1["down"], 7)
    nest.error_check()
