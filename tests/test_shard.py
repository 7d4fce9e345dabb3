"""The row-sharded split of one linear over several ranks, on the CPU: the partition,
the shard views of the packed buffers, and the one all-gather, run as gloo ranks.

Each rank's rows of z are computed by the oracle (its rows of the dense dequantised
W_v times x'), written into the rank's block in the layout the library's reorder
reads, and exchanged with the same all-gather helper the GPU path uses; the rows put
back token-major and rotated back must equal the oracle's one-device forward."""
import os
import socket
import sys

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

from nested_bit_quantized_gb300 import nest, shard, synth  # noqa: E402
from oracle import nest_oracle as O  # noqa: E402
from oracle import pack as P  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("M,world", [(4096, 2), (5376, 4), (1000, 3), (128, 4), (129, 2), (21504, 8), (77, 1)])
def test_row_plan_partitions_whole_tiles(M, world):
    plan = shard.RowPlan(M, world)
    covered = []
    for r in range(world):
        m0, m1 = plan.rows(r)
        assert m0 % 128 == 0 and m0 <= m1 and m1 - m0 <= plan.Mp
        assert m1 - m0 == plan.count(r)
        covered.extend(range(m0, m1))
        if r > 0:
            assert m0 == plan.rows(r - 1)[1]          # contiguous, in rank order
    assert covered == list(range(M))
    assert plan.Mp % 128 == 0 and world * plan.Mp >= M


def _packed_cpu_layer(q, bits, s_o, s_i):
    """A packed layer on the host, by the oracle's packer (the shard views only slice it)."""
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))
    base = P.pack_base(q["base_codes"], q["base_scales"].view(np.uint16))
    resid = P.pack_resid(q["resid_codes"], q["resid_scales"].view(np.uint16), bits)
    M, K = q["base_codes"].shape
    return nest.Layer(M, K, bits, t(base), t(resid), t(s_o), t(s_i))


@pytest.mark.parametrize("M,K,bits,world", [(1000, 256, 7, 3), (512, 384, 8, 2), (300, 128, 6, 4)])
def test_shard_views_are_the_packing_of_their_rows(M, K, bits, world):
    """A rank's view of the packed buffers equals, byte for byte, the oracle packer's
    output for that rank's rows alone (the units are tile-major, shards start on tiles)."""
    W = synth.weights(M, K, 3, "entries")
    s_o, s_i = synth.sign_pair(M, K, 4)
    q = O.quantize_layer(W, s_o, s_i, bits)
    full = _packed_cpu_layer(q, bits, s_o, s_i)
    plan = shard.RowPlan(M, world)
    for r in range(world):
        m0, m1 = plan.rows(r)
        v = shard.shard_layer(full, plan, r)
        if m1 == m0:
            assert v is None
            continue
        sub = {k: q[k][m0:m1] for k in ("base_codes", "base_scales", "resid_codes", "resid_scales")}
        ref = _packed_cpu_layer(sub, bits, s_o[m0:m1], s_i)
        assert v.M == m1 - m0 and v.K == K
        assert torch.equal(v.base, ref.base) and torch.equal(v.resid, ref.resid)
        assert torch.equal(v.sign_out, ref.sign_out)


def _reorder(gathered, world, T, Mp, M):
    """Token-major z from the gathered blocks, as the library's reorder documents it."""
    z = np.zeros((T, M))
    for r in range(world):
        Mr = max(0, min(Mp, M - r * Mp))
        z[:, r * Mp:r * Mp + Mr] = gathered[r * T * Mp:r * T * Mp + T * Mr].reshape(T, Mr)
    return z


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, M, K, bits, T, verify, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        W = synth.weights(M, K, 11, "entries")
        s_o, s_i = synth.sign_pair(M, K, 12)
        q = O.quantize_layer(W, s_o, s_i, bits)
        _, x = synth.activations(T, K, 13)
        plan = shard.RowPlan(M, world)
        m0, m1 = plan.rows(rank)
        xr = O.rotate_activations(x, s_i)                       # every rank rotates x itself
        rows = {k: q[k][m0:m1] for k in ("base_codes", "base_scales", "resid_codes", "resid_scales")}
        flat = torch.zeros(T * plan.Mp, dtype=torch.float64)
        if m1 > m0:
            shard.block(flat, plan, rank, T).copy_(torch.from_numpy(O.forward_rows(rows, xr, verify)))
        gathered = shard.all_gather_blocks(flat, plan, T).numpy()
        y = O.unrotate_outputs(_reorder(gathered, world, T, plan.Mp, M), s_o)
        ref = O.forward(q, s_o, s_i, x, verify)["y"]
        out[rank] = float(np.max(np.abs(y - ref)) / np.sqrt(np.mean(ref ** 2)))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("M,K,bits,world,T,verify", [(1000, 256, 8, 2, 5, True), (1000, 256, 7, 3, 1, False),
                                                      (640, 384, 6, 3, 16, True)])
def test_gloo_ranks_gather_the_oracle_forward(M, K, bits, world, T, verify):
    out = mp.Manager().dict()
    mp.spawn(_rank, args=(world, _free_port(), M, K, bits, T, verify, out), nprocs=world, join=True)
    assert sorted(out.keys()) == list(range(world))
    for r in range(world):
        assert out[r] < 1e-12, f"rank {r}: max error {out[r]:.3e} of rms"
