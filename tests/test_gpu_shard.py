"""The row-sharded split on one GPU: every rank's part of the data path through the
library (shard views of the packed buffers, the GEMM on a rank's rows into its block,
nest_shard_gather, the output rotation), the ranks emulated one after another with the
all-gather replaced by placing each rank's block in one buffer, against the oracle.
Ranks that wait on one another are never run as kernels on one GPU; the collective
itself is covered by the gloo test on the CPU."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from nested_bit_quantized_gb300 import nest, shard, synth  # noqa: E402
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


def _layer(M, K, bits, seed, dev):
    W = synth.weights(M, K, seed, "entries")
    s_o, s_i = synth.sign_pair(M, K, seed + 1)
    q = O.quantize_layer(W, s_o, s_i, bits)
    L = nest.pack(to_dev(q["base_codes"], torch, dev), to_dev(q["base_scales"], torch, dev),
                  to_dev(q["resid_codes"], torch, dev), to_dev(q["resid_scales"], torch, dev), bits,
                  to_dev(s_o, torch, dev), to_dev(s_i, torch, dev))
    return q, s_o, s_i, L


@pytest.mark.parametrize("M,K,bits,world,T", [(1000, 512, 8, 3, 16), (4096, 1024, 7, 2, 1), (640, 256, 6, 4, 5),
                                              (5376, 768, 8, 8, 3)])
def test_emulated_ranks_match_oracle(dev, M, K, bits, world, T):
    q, s_o, s_i, L = _layer(M, K, bits, 31, dev)
    xb, xv = synth.activations(T, K, 32)
    x = torch.from_numpy(xb.view(np.int16)).to(dev).view(torch.bfloat16)
    plan = shard.RowPlan(M, world)
    for verify in (False, True):
        gathered = torch.full((world * T * plan.Mp,), float("nan"), device=dev)
        for r in range(world):
            flat = gathered[r * T * plan.Mp:(r + 1) * T * plan.Mp]
            flat.zero_()
            x_op = nest.new_xop(K, T, dev)
            nest.rotate(x, L.sign_in, 0, x_op=x_op)
            local = shard.shard_layer(L, plan, r)
            if local is not None:
                nest.gemm(local, x_op, T, verify, z=shard.block(flat, plan, r, T))
        z = nest.shard_gather(gathered, world, T, plan.Mp, M)
        ref = O.forward(q, s_o, s_i, xv, verify)
        parity(z.cpu().numpy(), ref["z"])
        y = torch.empty((T, M), dtype=torch.float32, device=dev)
        nest.rotate(z, L.sign_out, 1, y=y)
        parity(y.cpu().numpy(), ref["y"])
    nest.error_check()


def test_one_rank_sharded_linear(dev):
    M, K, T = 1280, 1536, 9
    q, s_o, s_i, L = _layer(M, K, 8, 41, dev)
    xb, xv = synth.activations(T, K, 42)
    x = torch.from_numpy(xb.view(np.int16)).to(dev).view(torch.bfloat16)
    lin = shard.RowShardedLinear(L, 1, 0)
    for verify in (False, True):
        y = lin.forward(x, verify)
        parity(y.cpu().numpy(), O.forward(q, s_o, s_i, xv, verify)["y"])
    nest.error_check()


@pytest.mark.parametrize("world,T,Mp,M", [(3, 4, 384, 1000), (1, 2, 256, 200), (4, 1, 128, 300)])
def test_shard_gather_layout(dev, world, T, Mp, M):
    """The reorder alone, bit for bit: rank r's [T][M_r] block at the start of its T * Mp floats."""
    g = torch.randn(world * T * Mp, device=dev)
    z = nest.shard_gather(g, world, T, Mp, M).cpu().numpy()
    h = g.cpu().numpy()
    ref = np.zeros((T, M), np.float32)
    for r in range(world):
        Mr = max(0, min(Mp, M - r * Mp))
        ref[:, r * Mp:r * Mp + Mr] = h[r * T * Mp:r * T * Mp + T * Mr].reshape(T, Mr)
    assert np.array_equal(z, ref)
    nest.error_check()
