"""Row-sharded linear over several GPUs: the output rows split by whole 128-row tiles.

Each of `world` ranks holds the packed units of its row tiles (a contiguous slice of
the base and residual buffers, which are tile-major), rotates the replicated input
itself, and runs the draft or verify GEMM on its rows.  One all-gather of the ranks'
rotated-basis output blocks is the only exchange; nest_shard_gather puts the blocks
back token-major and the output rotation (nest_rotate, mode 1) runs on every rank,
since each output block of the rotation spans rows of several ranks.  No page has a
counterpart: the pages run one device.  This module partitions, slices and sequences
library calls; all arithmetic runs in libnest, the collective in torch.distributed.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional, Tuple

import torch

from . import nest

ROWS = 128


@dataclass(frozen=True)
class RowPlan:
    """Partition of M output rows over `world` ranks: rank r owns tiles
    [r * tiles_per_rank, (r + 1) * tiles_per_rank) clipped to the layer, i.e. rows
    [r * Mp, min((r + 1) * Mp, M)); trailing ranks may own none."""
    M: int
    world: int

    @property
    def tiles(self) -> int:
        return (self.M + ROWS - 1) // ROWS

    @property
    def tiles_per_rank(self) -> int:
        return (self.tiles + self.world - 1) // self.world

    @property
    def Mp(self) -> int:
        """Rows of one rank's block (the largest share)."""
        return ROWS * self.tiles_per_rank

    def tile_range(self, rank: int) -> Tuple[int, int]:
        t0 = min(rank * self.tiles_per_rank, self.tiles)
        return t0, min(t0 + self.tiles_per_rank, self.tiles)

    def rows(self, rank: int) -> Tuple[int, int]:
        t0, t1 = self.tile_range(rank)
        return min(ROWS * t0, self.M), min(ROWS * t1, self.M)

    def count(self, rank: int) -> int:
        m0, m1 = self.rows(rank)
        return m1 - m0


def _unit_bytes(layer: nest.Layer) -> Tuple[int, int]:
    """Bytes of one (tile, group) unit of the base and the second buffer."""
    G = layer.K // ROWS
    tiles = (layer.M + ROWS - 1) // ROWS
    base = layer.base.numel() // (tiles * G)
    second = layer.resid.numel() // (tiles * G) if layer.resid is not None else 0
    return base, second


def shard_layer(layer: nest.Layer, plan: RowPlan, rank: int) -> Optional[nest.Layer]:
    """Rank `rank`'s rows of a packed layer as views of its buffers (no copy), or None
    when the rank owns no rows.  The views start on unit boundaries, so they keep the
    buffers' 16-byte alignment."""
    if plan.M != layer.M:
        raise ValueError(f"plan is for {plan.M} rows, the layer has {layer.M}")
    t0, t1 = plan.tile_range(rank)
    if t1 <= t0:
        return None
    m0, m1 = plan.rows(rank)
    G = layer.K // ROWS
    ub, ur = _unit_bytes(layer)
    base = layer.base[t0 * G * ub:t1 * G * ub]
    resid = layer.resid[t0 * G * ur:t1 * G * ur] if layer.resid is not None else None
    return nest.Layer(m1 - m0, layer.K, layer.bits, base, resid, layer.sign_out[m0:m1], layer.sign_in,
                      layer.codec)


def block(flat: torch.Tensor, plan: RowPlan, rank: int, T: int) -> torch.Tensor:
    """Rank `rank`'s [T][M_r] output rows inside its block of T * Mp floats (the first
    T * M_r of them), the layout nest_shard_gather reads."""
    Mr = plan.count(rank)
    return flat[:T * Mr].view(T, Mr)


def all_gather_blocks(local: torch.Tensor, plan: RowPlan, T: int, group=None,
                      out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """The one exchange: every rank's T * Mp block, concatenated in rank order."""
    import torch.distributed as dist
    if local.numel() != T * plan.Mp:
        raise ValueError(f"block holds {local.numel()} floats, needs T * Mp = {T * plan.Mp}")
    if plan.world == 1:
        return local
    if out is None:
        out = torch.empty(plan.world * T * plan.Mp, dtype=local.dtype, device=local.device)
    dist.all_gather_into_tensor(out, local, group=group)
    return out


class RowShardedLinear:
    """One linear split over the ranks of `group` by output rows.

    full: the packed layer (only its tile range of this rank is read: the rank may hold
    the whole packed buffers or just its views, see shard_layer).  Every rank gets the
    whole output y [T][M]."""

    def __init__(self, full: nest.Layer, world: int, rank: int, group=None):
        self.plan = RowPlan(full.M, world)
        self.rank, self.group = rank, group
        self.M, self.K = full.M, full.K
        self.sign_out, self.sign_in = full.sign_out, full.sign_in
        self.local = shard_layer(full, self.plan, rank)
        self._bufs = {}

    def _buffers(self, T: int):
        """This rank's block, the operand, the gathered blocks and z for T tokens, kept
        between calls (so a call allocates nothing after the first at each T)."""
        if T not in self._bufs:
            dev, Mp, W = self.sign_in.device, self.plan.Mp, self.plan.world
            self._bufs[T] = (torch.empty(T * Mp, dtype=torch.float32, device=dev), nest.new_xop(self.K, T, dev),
                             torch.empty(W * T * Mp, dtype=torch.float32, device=dev) if W > 1 else None,
                             torch.empty((T, self.M), dtype=torch.float32, device=dev))
        return self._bufs[T]

    def forward(self, x: torch.Tensor, verify: bool, y: Optional[torch.Tensor] = None) -> torch.Tensor:
        """y = S_o H_o (W_v (H_i S_i x)) for x [T][K] (bf16 or fp32), on torch's current
        stream (the collective runs there too).  Buffers are reused between calls, so calls
        of one instance must not overlap on the GPU."""
        T = x.shape[0]
        flat, x_op, gathered, z = self._buffers(T)
        # x' = H_i S_i x on every rank; the same launch clears this rank's block
        nest.rotate_group([x], [self.sign_in], 0, x_ops=[x_op], zero=[flat])
        if self.local is not None:
            nest.gemm(self.local, x_op, T, verify, z=block(flat, self.plan, self.rank, T))
        gathered = all_gather_blocks(flat, self.plan, T, self.group, out=gathered)
        nest.shard_gather(gathered, self.plan.world, T, self.plan.Mp, self.M, z=z)
        if y is None:
            y = torch.empty((T, self.M), dtype=torch.float32, device=x.device)
        nest.rotate(z, self.sign_out, 1, y=y)
        return y
