"""Whole linears across the shapes of the rotations' blocks.

nest_linear and nest_linear_group compute y = S_o H_o (Q (H_i S_i x))
(feedman.me/posts/wZBTJ, POC recipe steps 1 and 4), H_i and H_o block-diagonal
with blocks of b = the largest power of two dividing K (or M), at most 4096.
These cases cover b_in from 128 to 4096 and b_out from 1 to 4096 (ragged last
tiles, a block spanning 32 row tiles), fp32 and bf16 inputs, a bf16 input off
a 16-byte boundary, both GEMM kernels and every epilogue split, scratch that
starts as garbage and is reused by calls of other T, outputs that start as NaN
(every element written), and grouped calls of many row tiles with one
128-column group each.  Each output is checked against the oracle with the
workload's parity gate.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from nested_bit_quantized_gb300 import nest, synth  # noqa: E402
from oracle import nest_oracle as O  # noqa: E402
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


def _layer(q, bits, s_o, s_i, dev):
    return nest.pack(to_dev(q["base_codes"], torch, dev), to_dev(q["base_scales"], torch, dev),
                     to_dev(q["resid_codes"], torch, dev), to_dev(q["resid_scales"], torch, dev), bits,
                     to_dev(s_o, torch, dev), to_dev(s_i, torch, dev))


def _bf16_x(T, K, seed, dev):
    bits, vals = synth.activations(T, K, seed)
    return torch.from_numpy(bits.view(np.int16)).to(dev).view(torch.bfloat16), vals


def _random_codes(M, K, bits, seed):
    """Uniformly drawn codes and scales in the stored ranges (no quantisation run)."""
    bc, bs, rc, rs = synth.uniform_codes(M, K, bits, seed)
    return {"base_codes": bc, "base_scales": bs.view(np.float16), "resid_codes": rc,
            "resid_scales": rs.view(np.float16)}


# (M, K): b_out / b_in = 4096 / 256 (a block of 32 row tiles), 1024 / 128, 512 / 256,
# 128 / 512, 8 / 128 with a ragged last tile, 32 / 256 inside one partial tile, 1 / 128
# (M = 1), 128 / 1024 and 256 / 4096
SHAPES = [(4096, 256), (1024, 384), (1536, 256), (640, 512), (200, 128), (96, 256), (1, 128), (384, 1024),
          (256, 4096)]


@pytest.mark.parametrize("M,K", SHAPES)
def test_linear_rotates_every_block(dev, M, K):
    bits = 7
    W = synth.weights(M, K, 5 + M, "entries")
    s_o, s_i = synth.sign_pair(M, K, 6 + M)
    q = O.quantize_layer(W, s_o, s_i, bits)
    layer = _layer(q, bits, s_o, s_i, dev)
    # one scratch of garbage bytes for every T (each call clears what it needs)
    scratch = torch.full((nest.linear_scratch_bytes(M, K, 130),), 0xFF, dtype=torch.uint8, device=dev)
    for T in (1, 3, 16, 17, 32, 33, 64, 130, 2):
        x, xv = _bf16_x(T, K, 40 + T, dev)
        for verify in (False, True):
            ref = O.forward(q, s_o, s_i, xv, verify)["y"]
            y = torch.full((T, M), float("nan"), dtype=torch.float32, device=dev)
            nest.linear(layer, x, verify, y=y, scratch=scratch)
            parity(y.cpu().numpy(), ref)
    nest.error_check()


@pytest.mark.parametrize("T", [1, 16])
def test_linear_fp32_and_misaligned_inputs(dev, T):
    """fp32 activations, and a bf16 input 2 bytes off a 16-byte boundary."""
    M, K, bits = 640, 1536, 8
    W = synth.weights(M, K, 31, "entries")
    s_o, s_i = synth.sign_pair(M, K, 32)
    q = O.quantize_layer(W, s_o, s_i, bits)
    layer = _layer(q, bits, s_o, s_i, dev)
    xb, xv = synth.activations(T, K, 33)
    x32 = torch.from_numpy(xv.astype(np.float32)).to(dev)
    raw = torch.zeros(T * K + 1, dtype=torch.int16, device=dev)
    raw[1:] = torch.from_numpy(xb.view(np.int16).ravel()).to(dev)
    x_off = raw[1:].view(T, K).view(torch.bfloat16)
    assert x_off.data_ptr() % 16 == 2
    for verify in (False, True):
        ref = O.forward(q, s_o, s_i, xv, verify)["y"]
        parity(nest.linear(layer, x32, verify).cpu().numpy(), ref)
        parity(nest.linear(layer, x_off, verify).cpu().numpy(), ref)
    nest.error_check()


@pytest.mark.parametrize("ntasks,T", [(2, 1), (2, 16), (4, 1), (4, 16), (4, 130)])
def test_group_many_tiles_one_group_each(dev, ntasks, T):
    """K = 128 (one group per row tile) and 200 row tiles per linear: every CTA of the
    GEMM covers units of several row tiles and linears."""
    bits, M, K = 7, 25600, 128
    layers, refs = [], []
    for i in range(ntasks):
        q = _random_codes(M, K, bits, 300 + i)
        s_o, s_i = synth.sign_pair(M, K, 310 + i)
        layers.append(_layer(q, bits, s_o, s_i, dev))
        refs.append((q, s_o, s_i))
    xs = [_bf16_x(T, K, 320 + i, dev) for i in range(ntasks)]
    for verify in (False, True):
        ys = [torch.full((T, M), float("nan"), dtype=torch.float32, device=dev) for _ in range(ntasks)]
        nest.linear_group(layers, [x for x, _ in xs], verify, ys=ys)
        for (q, s_o, s_i), (x, xv), y in zip(refs, xs, ys):
            parity(y.cpu().numpy(), O.forward(q, s_o, s_i, xv, verify)["y"])
    nest.error_check()


def test_group_mixed_block_sizes_shared_scratch(dev):
    """Three linears with different b_out in one grouped call, the same scratch used by
    calls of different T in turn."""
    bits = 8
    shapes = [(4096, 128), (200, 256), (1280, 384)]       # b_out 4096, 8, 256
    layers, refs = [], []
    for i, (M, K) in enumerate(shapes):
        q = _random_codes(M, K, bits, 400 + i)
        s_o, s_i = synth.sign_pair(M, K, 410 + i)
        layers.append(_layer(q, bits, s_o, s_i, dev))
        refs.append((q, s_o, s_i))
    scratch = torch.zeros(max(nest.linear_group_scratch_bytes(layers, T) for T in (1, 16, 96)), dtype=torch.uint8,
                          device=dev)
    for T in (16, 1, 96, 16):
        xs = [_bf16_x(T, K, 420 + i + T, dev) for i, (M, K) in enumerate(shapes)]
        for verify in (True, False):
            ys = nest.linear_group(layers, [x for x, _ in xs], verify, scratch=scratch)
            for (q, s_o, s_i), (x, xv), y in zip(refs, xs, ys):
                parity(y.cpu().numpy(), O.forward(q, s_o, s_i, xv, verify)["y"])
    nest.error_check()
