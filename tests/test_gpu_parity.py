"""GPU parity: the CUDA library (through its C-ABI binding) against the CPU oracle.

Integer work (packing, codes, scales) must match bit for bit; floating-point
outputs must pass the gate of the workload definition: relative L2 <= 1e-3
and every element within 1e-2 * rms(reference).
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from nested_bit_quantized_gb300 import nest, synth  # noqa: E402
from oracle import nest_oracle as O  # noqa: E402
from oracle import pack as P  # noqa: E402
from tests.helpers import decode_xop, parity, to_dev  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


_CACHE = {}


def ref_layer(M, K, bits, seed=1, outliers="entries"):
    key = (M, K, bits, seed, outliers)
    if key not in _CACHE:
        W = synth.weights(M, K, seed, outliers)
        s_o, s_i = synth.sign_pair(M, K, seed + 7)
        _CACHE[key] = (W, s_o, s_i, O.quantize_layer(W, s_o, s_i, bits))
    return _CACHE[key]


def dev_layer(q, bits, s_o, s_i, dev):
    return nest.pack(to_dev(q["base_codes"], torch, dev), to_dev(q["base_scales"], torch, dev),
                     to_dev(q["resid_codes"], torch, dev) if bits else None,
                     to_dev(q["resid_scales"], torch, dev) if bits else None, bits,
                     to_dev(s_o, torch, dev), to_dev(s_i, torch, dev))


def bf16_x(T, K, seed, dev):
    bits, vals = synth.activations(T, K, seed)
    return torch.from_numpy(bits.view(np.int16)).to(dev).view(torch.bfloat16), vals


def run_gemm(layer, x, verify, dev):
    T = x.shape[0]
    xop = nest.new_xop(layer.K, T, dev)
    nest.rotate(x, layer.sign_in, 0, x_op=xop)
    return nest.gemm(layer, xop, T, verify).cpu().numpy()


# ----------------------------------------------------------------------------
# packing and quantisation: bit-exact
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("M,K,bits", [(128, 128, 8), (200, 256, 7), (77, 384, 6), (1, 128, 8), (300, 1024, 7)])
def test_pack_bit_exact(dev, M, K, bits):
    bc, bs, rc, rs = synth.uniform_codes(M, K, bits, 23)
    layer = nest.pack(to_dev(bc, torch, dev), to_dev(bs, torch, dev), to_dev(rc, torch, dev),
                      to_dev(rs, torch, dev), bits, torch.ones(M, dtype=torch.int8, device=dev),
                      torch.ones(K, dtype=torch.int8, device=dev))
    assert np.array_equal(layer.base.cpu().numpy()[:P.base_bytes(M, K)], P.pack_base(bc, bs))
    assert np.array_equal(layer.resid.cpu().numpy()[:P.resid_bytes(M, K, bits)], P.pack_resid(rc, rs, bits))
    u = nest.unpack(layer)
    assert np.array_equal(u["base_codes"].cpu().numpy(), bc)
    assert np.array_equal(u["base_scales"].cpu().numpy().view(np.uint16), bs)
    assert np.array_equal(u["resid_codes"].cpu().numpy(), rc)
    assert np.array_equal(u["resid_scales"].cpu().numpy().view(np.uint16), rs)


def _boundary_ok(q, mism_b, mism_r, bits):
    """Code differences are allowed only where the oracle's value sits on a decision boundary."""
    Wr = q["Wr"]
    s = np.repeat(q["base_scales"].astype(np.float64), 128, axis=1)
    t = O.base_threshold()
    u = np.abs(Wr[mism_b] / s[mism_b])
    assert np.all(np.abs(u - t) <= 1e-9 * t), "base code mismatch away from the decision point"
    if bits:
        R = Wr - O.dequant_base(q["base_codes"], q["base_scales"])
        sr = np.repeat(q["resid_scales"].astype(np.float64), 128, axis=1)
        v = R[mism_r] / sr[mism_r]
        assert np.all(np.abs(np.abs(v - np.floor(v)) - 0.5) <= 1e-9 * np.maximum(1, np.abs(v))), \
            "residual code mismatch away from a rounding tie"


@pytest.mark.parametrize("M,K,bits,outl", [(256, 512, 8, "columns"), (200, 384, 7, "entries"), (96, 1024, 6, None),
                                           (512, 2560, 7, "entries"), (33, 128, 0, None)])
def test_quantize_matches_oracle(dev, M, K, bits, outl):
    W, s_o, s_i, q = ref_layer(M, K, bits or 8, seed=5, outliers=outl)
    g = nest.quantize(to_dev(W, torch, dev), to_dev(s_o, torch, dev), to_dev(s_i, torch, dev), bits)
    assert np.array_equal(g["base_scales"].cpu().numpy().view(np.uint16), q["base_scales"].view(np.uint16))
    mb = g["base_codes"].cpu().numpy() != q["base_codes"]
    mr = np.zeros_like(mb)
    if bits:
        assert np.array_equal(g["resid_scales"].cpu().numpy().view(np.uint16), q["resid_scales"].view(np.uint16))
        mr = g["resid_codes"].cpu().numpy() != q["resid_codes"]
    _boundary_ok(q, mb, mr, bits)


def test_degenerate_weights_and_tokens(dev):
    """The method's degenerate cases on the GPU path.  One output Hadamard block of W all
    zero (M = 384, blocks of 128 rows): its rotated rows are zero, so every group there
    takes base scale 0 and code 2, residual scale 0 and code 0; the GPU quantiser must give
    exactly those.  All-zero activation tokens (the first and, at T = 17, the last): their
    z and y rows are zero.  The draft and verify GEMMs (T = 1 on the look-up kernel, T = 17
    on the tensor cores) and the whole linear against the oracle, zeros exactly."""
    M, K, bits = 384, 512, 7
    W = synth.weights(M, K, 41, "entries")
    W[128:256] = 0.0
    s_o, s_i = synth.sign_pair(M, K, 42)
    q = O.quantize_layer(W, s_o, s_i, bits)
    assert np.all(q["base_scales"][128:256] == 0) and np.all(q["base_codes"][128:256] == 2)
    assert np.all(q["resid_scales"][128:256] == 0) and np.all(q["resid_codes"][128:256] == 0)
    g = nest.quantize(to_dev(W, torch, dev), to_dev(s_o, torch, dev), to_dev(s_i, torch, dev), bits)
    for key in ("base_scales", "resid_scales"):
        assert np.array_equal(g[key].cpu().numpy().view(np.uint16), q[key].view(np.uint16))
    assert np.all(g["base_codes"].cpu().numpy()[128:256] == 2)
    assert np.all(g["resid_codes"].cpu().numpy()[128:256] == 0)
    layer = dev_layer(q, bits, s_o, s_i, dev)
    for T in (1, 17):
        xb, xv = synth.activations(T, K, 43 + T)
        xb, xv = xb.copy(), xv.copy()
        for t in {0, T - 1}:
            xb[t] = 0
            xv[t] = 0.0
        x = torch.from_numpy(xb.view(np.int16)).to(dev).view(torch.bfloat16)
        for verify in (False, True):
            ref = O.forward(q, s_o, s_i, xv, verify)
            z = run_gemm(layer, x, verify, dev)
            parity(z, ref["z"])
            assert np.all(z[[0, T - 1]] == 0) and np.all(z[:, 128:256] == 0)
            y = nest.linear(layer, x, verify).cpu().numpy()
            parity(y, ref["y"])
            assert np.all(y[[0, T - 1]] == 0) and np.all(y[:, 128:256] == 0)
    nest.error_check()


# ----------------------------------------------------------------------------
# rotation
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("n,T", [(128, 1), (384, 3), (2560, 16), (4096, 17), (5376, 5), (8192, 2), (96, 4),
                                 (200, 3), (7, 2), (15360, 1), (1024, 64), (1000, 3), (12, 5), (9728, 16)])
def test_rotate_matches_oracle(dev, n, T):
    s = synth.signs(n, 31)
    xb, xv = synth.activations(T, n, 32)
    x = torch.from_numpy(xb.view(np.int16)).to(dev).view(torch.bfloat16)
    y = torch.empty((T, n), dtype=torch.float32, device=dev)
    xop = nest.new_xop(n, T, dev) if n % 128 == 0 else None
    nest.rotate(x, to_dev(s, torch, dev), 0, y=y, x_op=xop)
    ref = O.rotate_activations(xv, s)
    got = y.cpu().numpy()
    assert np.max(np.abs(got - ref)) <= 1e-5 * max(1.0, np.max(np.abs(ref)))
    if xop is not None:
        h = decode_xop(xop.cpu().numpy(), n, T).astype(np.float64)
        assert np.max(np.abs(h - ref) / np.maximum(np.abs(ref), 6.2e-5)) <= 2.0 ** -10
    # output side from fp32 input
    z = np.random.default_rng(n).normal(size=(T, n)).astype(np.float32)
    yo = torch.empty((T, n), dtype=torch.float32, device=dev)
    nest.rotate(torch.from_numpy(z).to(dev), to_dev(s, torch, dev), 1, y=yo)
    refo = O.unrotate_outputs(z, s)
    assert np.max(np.abs(yo.cpu().numpy() - refo)) <= 1e-5 * max(1.0, np.max(np.abs(refo)))
    # input side from fp32 input
    yi = torch.empty((T, n), dtype=torch.float32, device=dev)
    nest.rotate(torch.from_numpy(z).to(dev), to_dev(s, torch, dev), 0, y=yi)
    refi = O.rotate_activations(z, s)
    assert np.max(np.abs(yi.cpu().numpy() - refi)) <= 1e-5 * max(1.0, np.max(np.abs(refi)))


# ----------------------------------------------------------------------------
# draft / verify GEMMs
# ----------------------------------------------------------------------------

SHAPES = [(128, 128), (256, 512), (200, 384), (1280, 1024), (384, 9728), (1, 128), (129, 256)]


@pytest.mark.parametrize("M,K", SHAPES)
@pytest.mark.parametrize("bits", [6, 7, 8])
def test_gemm_parity_small(dev, M, K, bits):
    W, s_o, s_i, q = ref_layer(M, K, bits)
    layer = dev_layer(q, bits, s_o, s_i, dev)
    for T in (1, 2, 16, 17, 33, 64):
        x, xv = bf16_x(T, K, 40 + T, dev)
        for verify in (False, True):
            z = run_gemm(layer, x, verify, dev)
            ref = O.forward(q, s_o, s_i, xv, verify)["z"]
            parity(z, ref)


@pytest.mark.parametrize("bits", [6, 7, 8])
def test_linear_parity(dev, bits):
    M, K = 640, 1536
    W, s_o, s_i, q = ref_layer(M, K, bits, seed=3)
    layer = dev_layer(q, bits, s_o, s_i, dev)
    for T in (1, 9, 16, 64):
        x, xv = bf16_x(T, K, 50 + T, dev)
        for verify in (False, True):
            y = nest.linear(layer, x, verify).cpu().numpy()
            parity(y, O.forward(q, s_o, s_i, xv, verify)["y"])


@pytest.mark.parametrize("bits", [7, 8])
def test_grouped_gemm_and_linear_parity(dev, bits):
    shapes = [(384, 512), (200, 1024), (1280, 384)]          # ragged M, different K per linear
    refs = [ref_layer(M, K, bits, seed=11 + i) for i, (M, K) in enumerate(shapes)]
    layers = [dev_layer(q, bits, so, si, dev) for (W, so, si, q) in refs]
    for T in (1, 16, 40):
        xs = [bf16_x(T, K, 60 + i + T, dev) for i, (M, K) in enumerate(shapes)]
        xops = []
        for L, (x, _) in zip(layers, xs):
            xop = nest.new_xop(L.K, T, dev)
            nest.rotate(x, L.sign_in, 0, x_op=xop)
            xops.append(xop)
        for verify in (False, True):
            zs = nest.gemm_group(layers, xops, T, verify)
            for (W, so, si, q), (x, xv), z in zip(refs, xs, zs):
                parity(z.cpu().numpy(), O.forward(q, so, si, xv, verify)["z"])
            ys = nest.linear_group(layers, [x for x, _ in xs], verify)
            for (W, so, si, q), (x, xv), y in zip(refs, xs, ys):
                parity(y.cpu().numpy(), O.forward(q, so, si, xv, verify)["y"])


@pytest.mark.parametrize("bits", [0, 6, 7, 8])
def test_register_fragment_and_tcgen05_paths(dev, bits, monkeypatch):
    """Both GEMM kernels on the same inputs: the register-fragment (mma.sync) kernel that
    serves T <= 16 by default, forced up to T = 32, and the tcgen05 kernel forced down to
    T = 1; each against the oracle."""
    M, K = 1280, 2560
    W, s_o, s_i, q = ref_layer(M, K, bits or 7, seed=5)
    layer = dev_layer(q, bits or 7, s_o, s_i, dev)
    verify = bits != 0
    for T in (1, 3, 8, 9, 16, 17, 32):
        x, xv = bf16_x(T, K, 90 + T, dev)
        ref = O.forward(q, s_o, s_i, xv, verify)["z"]
        for path in ("rf", "tc"):
            monkeypatch.setenv("NEST_GEMM_PATH", path)
            parity(run_gemm(layer, x, verify, dev), ref)
    monkeypatch.delenv("NEST_GEMM_PATH")
    nest.error_check()


def test_draft_grouped_many_units(dev):
    """The draft with several stages per CTA and stages that meet the boundary of two
    linears: gate and up of the MLP triplet's shape (2 x 9728x2560, 3040 units) in one
    grouped launch, random 2-bit codes and scales, T from 1 to 8."""
    M, K, G = 9728, 2560, 2560 // 128
    rng = np.random.default_rng(77)
    layers, refs = [], []
    for i in range(2):
        q = {"base_codes": rng.integers(0, 4, size=(M, K)).astype(np.uint8),
             "base_scales": np.exp(rng.uniform(np.log(1e-3), np.log(3e-2), size=(M, G))).astype(np.float16),
             "resid_codes": np.zeros((M, K), np.int8), "resid_scales": np.zeros((M, G), np.float16)}
        s_o, s_i = synth.sign_pair(M, K, 78 + i)
        layers.append(dev_layer(q, 0, s_o, s_i, dev))
        refs.append((q, s_o, s_i))
    for T in (1, 5, 8):
        x, xv = bf16_x(T, K, 80 + T, dev)
        xops = []
        for L in layers:
            xop = nest.new_xop(K, T, dev)
            nest.rotate(x, L.sign_in, 0, x_op=xop)
            xops.append(xop)
        zs = nest.gemm_group(layers, xops, T, False)
        for (q, s_o, s_i), z in zip(refs, zs):
            parity(z.cpu().numpy(), O.forward(q, s_o, s_i, xv, False)["z"])
    nest.error_check()


@pytest.mark.parametrize("shape", [None, "16x2x1", "8x2x2"])
def test_draft_lookup_kernel_grouped(dev, monkeypatch, shape):
    """The one-token draft's table look-up kernel on a grouped launch large enough that
    each CTA's range wraps its stage and table rings and crosses task boundaries: seven
    4096x4096 linears and a ragged 4296x4096 one (its last row block has two tiles, the
    last tile 72 rows), random 2-bit codes and scales; against the oracle, and against the
    register-fragment kernel forced on the same inputs.  Every compiled shape of the
    kernel (row warps x rows per lane x CTAs per SM) is run."""
    if shape is not None:
        monkeypatch.setenv("NEST_LUT_SHAPE", shape)
    rng = np.random.default_rng(91)
    shapes = [(4096, 4096)] * 7 + [(4296, 4096)]
    layers, refs, xops = [], [], []
    x, xv = bf16_x(1, 4096, 92, dev)
    for i, (M, K) in enumerate(shapes):
        G = K // 128
        q = {"base_codes": rng.integers(0, 4, size=(M, K)).astype(np.uint8),
             "base_scales": np.exp(rng.uniform(np.log(1e-3), np.log(3e-2), size=(M, G))).astype(np.float16),
             "resid_codes": np.zeros((M, K), np.int8), "resid_scales": np.zeros((M, G), np.float16)}
        s_o, s_i = synth.sign_pair(M, K, 93 + i)
        L = dev_layer(q, 0, s_o, s_i, dev)
        xop = nest.new_xop(K, 1, dev)
        nest.rotate(x, L.sign_in, 0, x_op=xop)
        layers.append(L)
        refs.append((q, s_o, s_i))
        xops.append(xop)
    zs = nest.gemm_group(layers, xops, 1, False)
    monkeypatch.setenv("NEST_GEMM_PATH", "rf")
    zr = nest.gemm_group(layers, xops, 1, False)
    monkeypatch.delenv("NEST_GEMM_PATH")
    for (q, s_o, s_i), z, r in zip(refs, zs, zr):
        ref = O.forward(q, s_o, s_i, xv, False)["z"]
        parity(z.cpu().numpy(), ref)
        parity(r.cpu().numpy(), ref)
    nest.error_check()


def _close(a, b, rel=1e-6):
    """Equal up to the order of the fp32 additions of the split K range."""
    scale = np.sqrt(np.mean(np.asarray(b, np.float64) ** 2))
    assert np.max(np.abs(np.asarray(a, np.float64) - b)) <= rel * 64 * scale


def test_draft_is_subset_of_verify(dev):
    # with a zero residual the verify kernel decodes the same fp16 weights as the draft
    M, K, bits = 512, 1024, 7
    W, s_o, s_i, q = ref_layer(M, K, bits)
    q0 = dict(q)
    q0["resid_codes"] = np.zeros_like(q["resid_codes"])
    lv = dev_layer(q0, bits, s_o, s_i, dev)
    x, _ = bf16_x(16, K, 7, dev)
    _close(run_gemm(lv, x, True, dev), run_gemm(lv, x, False, dev))


def test_gemm_accumulates_into_z(dev):
    M, K, bits = 256, 512, 8
    W, s_o, s_i, q = ref_layer(M, K, bits)
    layer = dev_layer(q, bits, s_o, s_i, dev)
    x, xv = bf16_x(4, K, 9, dev)
    xop = nest.new_xop(K, 4, dev)
    nest.rotate(x, layer.sign_in, 0, x_op=xop)
    z0 = torch.full((4, M), 0.5, dtype=torch.float32, device=dev)
    z = nest.gemm(layer, xop, 4, True, z=z0.clone())
    ref = O.forward(q, s_o, s_i, xv, True)["z"]
    parity(z.cpu().numpy() - 0.5, ref)


def test_repeatable_and_token_independent(dev):
    M, K, bits = 1024, 2560, 7
    W, s_o, s_i, q = ref_layer(M, K, bits)
    layer = dev_layer(q, bits, s_o, s_i, dev)
    x, xv = bf16_x(16, K, 8, dev)
    a = run_gemm(layer, x, True, dev)
    b = run_gemm(layer, x, True, dev)
    _close(a, b)
    for t in (0, 5, 15):
        one = run_gemm(layer, x[t:t + 1].contiguous(), True, dev)
        parity(one[0], a[t])
    nest.error_check()


# ----------------------------------------------------------------------------
# full sizes of the workloads
# ----------------------------------------------------------------------------

def _full_layer(wl, lin, bits):
    W = synth.weights(lin.M, lin.K, lin.w_seed, lin.outliers)
    s_o, s_i = synth.sign_pair(lin.M, lin.K, lin.sign_seed)
    return W, s_o, s_i, O.quantize_layer(W, s_o, s_i, bits)


@pytest.mark.slow
def test_full_single_4096(dev):
    wl = synth.WORKLOADS["single_4096"]
    lin = wl.linears[0]
    W, s_o, s_i, q = _full_layer(wl, lin, 8)
    layer = dev_layer(q, 8, s_o, s_i, dev)
    for T in wl.T:
        x, xv = bf16_x(T, lin.K, wl.x_seed, dev)
        for verify in (False, True):
            ref = O.forward(q, s_o, s_i, xv, verify)
            parity(run_gemm(layer, x, verify, dev), ref["z"])
            parity(nest.linear(layer, x, verify).cpu().numpy(), ref["y"])


@pytest.mark.slow
def test_full_mlp_triplet(dev):
    wl = synth.WORKLOADS["mlp_triplet_4b"]
    for lin in wl.linears:
        W, s_o, s_i, q = _full_layer(wl, lin, 7)
        layer = dev_layer(q, 7, s_o, s_i, dev)
        for T in (1, 16, 32):
            x, xv = bf16_x(T, lin.K, wl.x_seed, dev)
            for verify in (False, True):
                parity(nest.linear(layer, x, verify).cpu().numpy(), O.forward(q, s_o, s_i, xv, verify)["y"])


@pytest.mark.slow
@pytest.mark.parametrize("name,idx,T", [("decoder_31b", 4, 64), ("decoder_31b", 6, 1), ("decoder_12b", 6, 16)])
def test_full_size_sampled_rows(dev, name, idx, T):
    """Full-size shapes of the 31B/12B workloads with uniformly drawn codes: every
    output row of 3 sampled tiles and every token, against the oracle's dequantised rows."""
    lin = synth.WORKLOADS[name].linears[idx]
    M, K = lin.M, lin.K
    bc, bs, rc, rs = synth.uniform_codes(M, K, 8, lin.w_seed)
    s_o, s_i = synth.sign_pair(M, K, lin.sign_seed)
    layer = nest.pack(to_dev(bc, torch, dev), to_dev(bs, torch, dev), to_dev(rc, torch, dev), to_dev(rs, torch, dev),
                      8, to_dev(s_o, torch, dev), to_dev(s_i, torch, dev))
    x, xv = bf16_x(T, K, 77, dev)
    xr = O.rotate_activations(xv, s_i)
    tiles = [0, (M // 128) // 2, (M - 1) // 128]
    rows = np.concatenate([np.arange(t * 128, min(M, t * 128 + 128)) for t in tiles])
    for verify in (False, True):
        z = run_gemm(layer, x, verify, dev)
        sub = {"base_codes": bc[rows], "base_scales": bs[rows].view(np.float16),
               "resid_codes": rc[rows], "resid_scales": rs[rows].view(np.float16)}
        parity(z[:, rows], O.forward_rows(sub, xr, verify))


@pytest.mark.slow
def test_grouped_launch_as_benched(dev):
    """The default bench line's launches at full size and in its launch configuration: 32
    distinct packed copies of the 4096x4096 linear (b = 8) in one grouped gemm_group call
    sharing one activation operand, as the bench graphs them: verify at T = 16 (the line's
    value) and T = 1, and the draft at T = 1 (the look-up kernel).  Every token of every row
    of three tiles of three copies against the oracle's rows; codes drawn uniformly over
    their stored ranges, so the check does not go through any quantiser."""
    lin = synth.WORKLOADS["single_4096"].linears[0]
    M, K, C, bits = lin.M, lin.K, 32, 8
    picked = (0, 13, 31)
    tiles = (0, 16, 31)
    rows = np.concatenate([np.arange(t * 128, t * 128 + 128) for t in tiles])
    layers, subs = [], {}
    for c in range(C):
        bc, bs, rc, rs = synth.uniform_codes(M, K, bits, 500 + c)
        s_o, s_i = synth.sign_pair(M, K, 600 + c)
        layers.append(nest.pack(to_dev(bc, torch, dev), to_dev(bs, torch, dev), to_dev(rc, torch, dev),
                                to_dev(rs, torch, dev), bits, to_dev(s_o, torch, dev), to_dev(s_i, torch, dev)))
        if c in picked:
            subs[c] = {"base_codes": bc[rows], "base_scales": bs[rows].view(np.float16),
                       "resid_codes": rc[rows], "resid_scales": rs[rows].view(np.float16)}
        if c == 0:
            s_i0 = s_i
    for T, verify in ((16, True), (1, True), (1, False)):
        x, xv = bf16_x(T, K, 900 + T, dev)
        xop = nest.new_xop(K, T, dev)
        nest.rotate(x, layers[0].sign_in, 0, x_op=xop)
        zs = nest.gemm_group(layers, [xop] * C, T, verify)
        xr = O.rotate_activations(xv, s_i0)
        for c in picked:
            parity(zs[c].cpu().numpy()[:, rows], O.forward_rows(subs[c], xr, verify))
        del zs
    nest.error_check()


def test_concurrent_streams(dev):
    """The one-token look-up draft and the 16-token tensor-core verify launched on two
    streams at once, ten times each, so their CTAs share the SMs: every result against the
    oracle (the kernels share no state but the error flags)."""
    M, K, bits = 1280, 1024, 8
    W, s_o, s_i, q = ref_layer(M, K, bits, seed=61)
    layer = dev_layer(q, bits, s_o, s_i, dev)
    x1, xv1 = bf16_x(1, K, 62, dev)
    x16, xv16 = bf16_x(16, K, 63, dev)
    op1, op16 = nest.new_xop(K, 1, dev), nest.new_xop(K, 16, dev)
    nest.rotate(x1, layer.sign_in, 0, x_op=op1)
    nest.rotate(x16, layer.sign_in, 0, x_op=op16)
    torch.cuda.synchronize()
    sa, sb = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    za = [torch.zeros((1, M), device=dev) for _ in range(10)]
    zb = [torch.zeros((16, M), device=dev) for _ in range(10)]
    torch.cuda.synchronize()                 # the cleared accumulators before either stream starts
    for i in range(10):
        with torch.cuda.stream(sa):
            nest.gemm(layer, op1, 1, False, z=za[i])
        with torch.cuda.stream(sb):
            nest.gemm(layer, op16, 16, True, z=zb[i])
    torch.cuda.synchronize()
    ra = O.forward(q, s_o, s_i, xv1, False)["z"]
    rb = O.forward(q, s_o, s_i, xv16, True)["z"]
    for i in range(10):
        parity(za[i].cpu().numpy(), ra)
        parity(zb[i].cpu().numpy(), rb)
    nest.error_check()


def test_error_flag_clear(dev):
    nest.error_check()


# ----------------------------------------------------------------------------
# prefill-size token counts (65..256): one CTA per SM, N up to 256 per MMA
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("M,K,bits", [(200, 384, 7), (1280, 1024, 8), (129, 256, 6)])
def test_gemm_parity_prefill(dev, M, K, bits):
    W, s_o, s_i, q = ref_layer(M, K, bits, seed=13)
    layer = dev_layer(q, bits, s_o, s_i, dev)
    for T in (65, 100, 128, 129, 200, 256):
        x, xv = bf16_x(T, K, 110 + T, dev)
        for verify in (False, True):
            z = run_gemm(layer, x, verify, dev)
            parity(z, O.forward(q, s_o, s_i, xv, verify)["z"])
    nest.error_check()


def test_linear_group_of_64(dev):
    """nest_linear_group at its largest count: 64 independent linears of mixed shapes (ragged
    row tiles; input widths with Hadamard blocks of 128 and 1024, so the grouped rotation in
    mixes its register and segment paths) in three launches, draft at T = 1 and verify at
    T = 16, against the oracle."""
    shapes = [(128, 256), (200, 384), (384, 1024), (72, 128)]
    refs = [ref_layer(*shapes[i % 4], 8, seed=300 + i % 8) for i in range(64)]
    layers = [dev_layer(q, 8, so, si, dev) for (W, so, si, q) in refs]
    for T, verify in ((1, False), (16, True)):
        xs = [bf16_x(T, L.K, 400 + i, dev) for i, L in enumerate(layers)]
        ys = nest.linear_group(layers, [x for x, _ in xs], verify)
        for (W, so, si, q), (x, xv), y in zip(refs, xs, ys):
            parity(y.cpu().numpy(), O.forward(q, so, si, xv, verify)["y"])
    nest.error_check()


def test_linear_and_group_prefill(dev):
    shapes = [(384, 512), (200, 1024)]
    refs = [ref_layer(M, K, 7, seed=21 + i) for i, (M, K) in enumerate(shapes)]
    layers = [dev_layer(q, 7, so, si, dev) for (W, so, si, q) in refs]
    for T in (96, 256):
        xs = [bf16_x(T, K, 130 + i + T, dev) for i, (M, K) in enumerate(shapes)]
        for verify in (False, True):
            ys = nest.linear_group(layers, [x for x, _ in xs], verify)
            for (W, so, si, q), (x, xv), y in zip(refs, xs, ys):
                parity(y.cpu().numpy(), O.forward(q, so, si, xv, verify)["y"])
    nest.error_check()


@pytest.mark.parametrize("M,K,T,bits", [(384, 512, 1, 8), (200, 1024, 16, 7), (1280, 384, 40, 6)])
def test_gemm_from_fp32_rotated_operand(dev, M, K, T, bits):
    """A caller holding x' = H_i S_i x in fp32 (the oracle's own x') lays it out with
    nest_operand and calls the GEMMs: draft and verify against the oracle's z, and the
    operand equals fp16(x') element for element (padding tokens zero)."""
    W, s_o, s_i, q = ref_layer(M, K, bits, seed=71)
    layer = dev_layer(q, bits, s_o, s_i, dev)
    _, xv = bf16_x(T, K, 72, dev)
    xr = O.rotate_activations(xv, s_i)
    x_op = nest.new_xop(K, T, dev).fill_(0x7E00)                       # NaN bits: every byte is written
    nest.operand(torch.from_numpy(xr.astype(np.float32)).to(dev), x_op=x_op)
    got = decode_xop(x_op.cpu().numpy(), K, T)
    assert np.array_equal(got.view(np.uint16), xr.astype(np.float32).astype(np.float16).view(np.uint16))
    Np = nest.xop_bytes(K, T) // (2 * K)
    if Np > T:
        assert not np.isnan(x_op.cpu().numpy().view(np.float16)).any()
    for verify in (False, True):
        parity(nest.gemm(layer, x_op, T, verify).cpu().numpy(), O.forward(q, s_o, s_i, xv, verify)["z"])
    nest.error_check()
