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
GEMM gate (1e-3, 1e-2).  That end-to-end gate is an extra check only: the
stage-wise test holds every stage of the chain (each GEMM, each glue) to the GEMM
gate, each fed the GPU's own intermediate.
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


@pytest.mark.parametrize("M,T,product,in_place,n_next", [
    (512, 1, False, False, 2), (5376, 17, True, False, 2), (3840, 64, False, True, 2), (8192, 5, True, True, 1),
    (21504, 3, True, False, 1), (300, 4, True, False, 0), (4096, 2, False, True, 3), (5376, 160, True, False, 2),
    (8192, 3, True, "odd", 2), (21504, 2, False, "odd", 1), (2560, 4, True, "odd", 1)])
def test_chain_kernel(dev, M, T, product, in_place, n_next):
    """Out-rotation (+ product), RMS rescale, bf16 cast and next in-rotations; ragged last
    4096-element segments (5376, 21504), a segment shorter than one (300, 3840), h in place,
    and h written to a y 4 bytes off a 16-byte boundary ("odd": the shared-memory tile path
    instead of the register path for b <= 512 or the segment path for b >= 1024)."""
    rng = np.random.default_rng(M + T)
    za = rng.normal(size=(T, M)).astype(np.float32)
    zb = rng.normal(size=(T, M)).astype(np.float32) if product else None
    sa, sb = synth.signs(M, 1), synth.signs(M, 2)
    nxt = [synth.signs(M, 3 + j) for j in range(n_next)]
    za_d = to_dev(za, torch, dev)
    if in_place == "odd":
        y = torch.empty(T * M + 4, dtype=torch.float32, device=dev)[1:1 + T * M].view(T, M)
        assert y.data_ptr() % 16 == 4
        in_place = False
    else:
        y = None if in_place else torch.empty((T, M), dtype=torch.float32, device=dev)
    # next linears reading h (their descriptors only need K == M and S_i)
    dummy = torch.zeros(16, dtype=torch.uint8, device=dev)
    layers = [nest.Layer(1000 + 24 * j, M, 0, dummy, None, to_dev(sa, torch, dev), to_dev(s, torch, dev))
              for j, s in enumerate(nxt)]
    xops = [nest.new_xop(M, T, dev) for _ in nxt]
    zn = [torch.full((T, L.M), 7.0, device=dev) for L in layers]
    work = torch.full((chain.chain_work_bytes(M, T) // 4,), float("nan"), device=dev)
    chain.chain(za_d, to_dev(sa, torch, dev), to_dev(zb, torch, dev) if product else None,
                to_dev(sb, torch, dev) if product else None, T, work, y, layers, xops, zn)
    ya = O.unrotate_outputs(za, sa)
    yref = ya * O.unrotate_outputs(zb, sb) if product else ya
    parity((za_d if in_place else y).cpu().numpy(), yref)
    h = O.chain_glue(ya, O.unrotate_outputs(zb, sb) if product else None)
    for s, xop in zip(nxt, xops):
        parity(decode_xop(xop.cpu().numpy(), M, T).astype(np.float64), O.rotate_activations(h, s))
    for z in zn:
        assert torch.count_nonzero(z).item() == 0
    nest.error_check()


@pytest.mark.parametrize("M,T,product,side_ms", [
    (8192, 1, False, (4096, 4096)), (8192, 16, False, (4096, 5376)), (5376, 1, True, (512, 2560)),
    (5376, 17, False, (4096, 768)), (300, 4, False, (256,)), (21504, 3, True, (1024, 8192))])
def test_chain_side_rotations(dev, M, T, product, side_ms):
    """Output rotations of other linears handed to nest_chain (the k and v outputs beside
    the q glue): those whose block size puts them on the glue's path run as extra CTAs of
    its first launch, the others in a launch of their own; either way y = S_o H_o z against
    the oracle, and the glue's own results are those without side tasks."""
    rng = np.random.default_rng(M + 7 * T)
    za = rng.normal(size=(T, M)).astype(np.float32)
    zb = rng.normal(size=(T, M)).astype(np.float32) if product else None
    sa, sb, sn = synth.signs(M, 11), synth.signs(M, 12), synth.signs(M, 13)
    dummy = torch.zeros(16, dtype=torch.uint8, device=dev)
    layers = [nest.Layer(640, M, 0, dummy, None, to_dev(sa, torch, dev), to_dev(sn, torch, dev))] if M % 128 == 0 \
        else []
    zs = [rng.normal(size=(T, m)).astype(np.float32) for m in side_ms]
    ss = [synth.signs(m, 20 + i) for i, m in enumerate(side_ms)]
    ys = [torch.full((T, m), float("nan"), device=dev) for m in side_ms]
    side = [(to_dev(z, torch, dev), to_dev(sg, torch, dev), y) for z, sg, y in zip(zs, ss, ys)]
    runs = []
    for with_side in (True, False):
        xops = [nest.new_xop(M, T, dev) for _ in layers]
        y = torch.empty((T, M), dtype=torch.float32, device=dev)
        work = torch.full((chain.chain_work_bytes(M, T) // 4,), float("nan"), device=dev)
        chain.chain(to_dev(za, torch, dev), to_dev(sa, torch, dev), to_dev(zb, torch, dev) if product else None,
                    to_dev(sb, torch, dev) if product else None, T, work, y, layers, xops, None,
                    side=side if with_side else None)
        runs.append((y.cpu().numpy(), [decode_xop(x.cpu().numpy(), M, T) for x in xops]))
    for z, sg, yd in zip(zs, ss, ys):
        parity(yd.cpu().numpy(), O.unrotate_outputs(z, sg))
    assert np.array_equal(runs[0][0], runs[1][0])
    for a, b in zip(runs[0][1], runs[1][1]):
        assert np.array_equal(a, b)
    ya = O.unrotate_outputs(za, sa)
    parity(runs[0][0], ya * O.unrotate_outputs(zb, sb) if product else ya)
    nest.error_check()


@pytest.mark.parametrize("M,product", [(5376, False), (8192, True), (21504, True)])
def test_chain_zero_token(dev, M, product):
    """A token whose glue input is all zero (RMS 0): the rescale gives zeros, so its rows of
    every next operand are zero, while the other tokens are unaffected; on the register path
    (blocks of 256) and the segment path (one 4096 block per segment, and 1024-blocks over
    six segments)."""
    T = 3
    rng = np.random.default_rng(M)
    za = rng.normal(size=(T, M)).astype(np.float32)
    za[1] = 0.0
    zb = rng.normal(size=(T, M)).astype(np.float32) if product else None
    sa, sb = synth.signs(M, 1), synth.signs(M, 2)
    nxt = [synth.signs(M, 3)]
    dummy = torch.zeros(16, dtype=torch.uint8, device=dev)
    layers = [nest.Layer(640, M, 0, dummy, None, to_dev(sa, torch, dev), to_dev(nxt[0], torch, dev))]
    xops = [nest.new_xop(M, T, dev)]
    y = torch.empty((T, M), dtype=torch.float32, device=dev)
    work = torch.full((chain.chain_work_bytes(M, T) // 4,), float("nan"), device=dev)
    chain.chain(to_dev(za, torch, dev), to_dev(sa, torch, dev), to_dev(zb, torch, dev) if product else None,
                to_dev(sb, torch, dev) if product else None, T, work, y, layers, xops, None)
    ya = O.unrotate_outputs(za, sa)
    h = O.chain_glue(ya * O.unrotate_outputs(zb, sb) if product else ya)
    assert np.all(h[1] == 0)
    got = decode_xop(xops[0].cpu().numpy(), M, T).astype(np.float64)
    assert np.all(got[1] == 0) and np.all(y.cpu().numpy()[1] == 0)
    parity(got, O.rotate_activations(h, nxt[0]))
    nest.error_check()


def test_rotate_group_matches_single_calls(dev):
    """nest_rotate_group: three operands of one input plus cleared accumulators, and two
    output rotations, each equal to the single-call result."""
    T, K = 9, 5376
    xb, xv = synth.activations(T, K, 5)
    x = torch.from_numpy(xb.view(np.int16)).to(dev).view(torch.bfloat16)
    signs = [to_dev(synth.signs(K, 40 + j), torch, dev) for j in range(3)]
    ops = [nest.new_xop(K, T, dev).zero_() for _ in range(3)]          # padding tokens stay 0
    zs = [torch.full((T, 777 + j), 3.0, device=dev) for j in range(3)]
    nest.rotate_group([x] * 3, signs, 0, x_ops=ops, zero=zs)
    for s, op, z in zip(signs, ops, zs):
        one = nest.new_xop(K, T, dev).zero_()
        nest.rotate(x, s, 0, x_op=one)
        assert torch.equal(op[:one.numel()], one)
        assert torch.count_nonzero(z).item() == 0
    M = [8192, 3840]
    zin = [torch.randn((T, m), device=dev) for m in M]
    so = [to_dev(synth.signs(m, 50 + j), torch, dev) for j, m in enumerate(M)]
    ys = [torch.empty((T, m), device=dev) for m in M]
    nest.rotate_group(zin, so, 1, ys=ys)
    for z, s, y in zip(zin, so, ys):
        ref = torch.empty_like(y)
        nest.rotate(z, s, 1, y=ref)
        assert torch.equal(y, ref)
    nest.error_check()


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


@pytest.mark.parametrize("T", [1, 16, 64])
def test_chained_layers_stagewise(dev, T):
    """Every stage of two chained layers at the GEMM gate (relative L2 <= 1e-3, every element
    within 1e-2 * rms), each stage fed the GPU's own intermediate.  After layer_forward the
    in-place glue calls leave y_q, y_o and y_gate * y_up (fp32, rotated back) in z_q, z_o and
    z_gate; z_up and z_down keep the rotated-basis accumulators; y_down is written apart.
    The oracle's glue (unit RMS in fp64, bf16 cast) applied to a GPU intermediate gives the
    next stage's input, so no stage inherits an earlier stage's rounding differences; the
    operands the glue kernel wrote are checked against the same glue, rotated."""
    bits = 8
    ref = [_small_layer(l, bits) for l in range(2)]
    lin = [{n: _dev_layer(q, bits, so, si, dev) for n, (q, so, si) in r.items()} for r in ref]
    xb, xv = synth.activations(T, SMALL["hidden"], 78)
    x = torch.from_numpy(xb.view(np.int16)).to(dev).view(torch.bfloat16)
    host = lambda t: t.cpu().numpy().astype(np.float64)
    for verify in (False, True):
        bufs = [chain.LayerBuffers(l, T, dev) for l in lin]
        chain.layer_input(lin[0], x, bufs[0])
        chain.layer_forward(lin[0], bufs[0], verify, lin[1], bufs[1])
        chain.layer_forward(lin[1], bufs[1], verify)
        torch.cuda.synchronize()
        fwd = lambda r, n, xin: O.forward(r[n][0], r[n][1], r[n][2], xin, verify)
        xin = xv
        for l in range(2):
            r, b = ref[l], bufs[l]
            y_q = host(b.z["q"])
            parity(y_q, fwd(r, "q", xin)["y"])
            parity(host(b.y["k"]), fwd(r, "k", xin)["y"])
            parity(host(b.y["v"]), fwd(r, "v", xin)["y"])
            h_q = O.chain_glue(y_q)
            parity(decode_xop(b.xop["o"].cpu().numpy(), SMALL["q"], T).astype(np.float64),
                   O.rotate_activations(h_q, r["o"][2]))
            y_o = host(b.z["o"])
            parity(y_o, fwd(r, "o", h_q)["y"])
            h_o = O.chain_glue(y_o)
            for n in ("gate", "up"):
                parity(decode_xop(b.xop[n].cpu().numpy(), SMALL["hidden"], T).astype(np.float64),
                       O.rotate_activations(h_o, r[n][2]))
            parity(host(b.z["up"]), fwd(r, "up", h_o)["z"])
            y_up_gpu = O.unrotate_outputs(host(b.z["up"]), r["up"][1])
            prod = host(b.z["gate"])
            parity(prod, fwd(r, "gate", h_o)["y"] * y_up_gpu)
            h_gu = O.chain_glue(prod)
            parity(decode_xop(b.xop["down"].cpu().numpy(), SMALL["inter"], T).astype(np.float64),
                   O.rotate_activations(h_gu, r["down"][2]))
            y_down = host(b.y["down"])
            parity(host(b.z["down"]), fwd(r, "down", h_gu)["z"])
            parity(y_down, fwd(r, "down", h_gu)["y"])
            xin = O.chain_glue(y_down)
            if l == 0:
                for n in ("q", "k", "v"):
                    parity(decode_xop(bufs[1].xop[n].cpu().numpy(), SMALL["hidden"], T).astype(np.float64),
                           O.rotate_activations(xin, ref[1][n][2]))
    nest.error_check()
