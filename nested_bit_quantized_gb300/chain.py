"""Chained decoder layer on the device: the order of library calls only.

A layer of seven linears (q, k, v, o, gate, up, down) is run as grouped GEMMs
joined by nest_chain, which fuses each output rotation, the unit-RMS rescale
and bf16 cast standing in for the normalisation between linears, and the next
linears' input rotations.  q, k, v read the layer input; o reads q's output;
gate and up read o's output; down reads gate * up; the next layer reads down's
output.  The k and v outputs are rotated back and kept (the KV-cache stand-in).
Every step runs in libnest; this module only allocates buffers and sequences
the calls.
"""
from __future__ import annotations

from typing import Dict, List, Optional

import torch

from . import nest

NAMES = ("q", "k", "v", "o", "gate", "up", "down")


class LayerBuffers:
    """Operands, accumulators, outputs and glue work space of one layer for a fixed T."""

    def __init__(self, lin: Dict[str, nest.Layer], T: int, device):
        self.T = T
        self.xop = {n: nest.new_xop(lin[n].K, T, device) for n in NAMES}
        self.z = {n: torch.zeros((T, lin[n].M), dtype=torch.float32, device=device) for n in NAMES}
        self.y = {n: torch.empty((T, lin[n].M), dtype=torch.float32, device=device) for n in ("k", "v", "down")}
        wb = max(chain_work_bytes(lin[n].M, T) for n in NAMES)
        self.work = torch.empty(wb // 4, dtype=torch.float32, device=device)


def chain_work_bytes(M: int, T: int) -> int:
    return int(nest.load().nest_chain_work_bytes(M, T))


def chain(z_a, s_a, z_b, s_b, T: int, work: torch.Tensor, y=None, nexts: Optional[List[nest.Layer]] = None,
          x_ops=None, z_next=None, stream=None, side=None):
    """nest_chain (see include/nest.h).  Without y, the glue output overwrites z_a.  side: up to
    two (z, sign_out, y) output rotations of other linears run in the glue's first launch."""
    lib = nest.load()
    nexts = nexts or []
    x_ops = x_ops or []
    z_next = z_next or []
    side = side or []
    M = z_a.shape[1]
    nest._buf(z_a, "z_a", 4 * T * M, torch.float32)
    nest._buf(s_a, "s_a", M, torch.int8)
    if (z_b is None) != (s_b is None):
        raise ValueError("z_b and s_b go together")
    if z_b is not None:
        nest._buf(z_b, "z_b", 4 * T * M, torch.float32)
        nest._buf(s_b, "s_b", M, torch.int8)
    if y is not None:
        nest._buf(y, "y", 4 * T * M, torch.float32)
    nest._buf(work, "work", chain_work_bytes(M, T))
    if len(x_ops) != len(nexts) or (z_next and len(z_next) != len(nexts)):
        raise ValueError("one operand (and one accumulator, if any) per next linear")
    for L, xo in zip(nexts, x_ops):
        if L.K != M:
            raise ValueError(f"a next linear reads {L.K} features, the glue writes {M}")
        nest._buf(L.sign_in, "sign_in", M, torch.int8)
        nest._buf(xo, "x_op", nest.xop_bytes(M, T))
    for L, zn in zip(nexts, z_next):
        nest._buf(zn, "z_next", 4 * T * L.M, torch.float32)
    sd = (nest.RotateTask * len(side))() if side else None
    for i, (zs, ss, ys) in enumerate(side):
        n = zs.shape[1]
        nest._buf(zs, "side z", 4 * T * n, torch.float32)
        nest._buf(ss, "side sign_out", n, torch.int8)
        nest._buf(ys, "side y", 4 * T * n, torch.float32)
        sd[i] = nest.RotateTask(zs.data_ptr(), ss.data_ptr(), n, ys.data_ptr(), None, None, 0)
    arr = nest._layers(nexts) if nexts else None
    xo = nest._ptrs(x_ops) if nexts else None
    zn = nest._ptrs(z_next) if z_next else None
    st = lib.nest_chain(nest._ptr(z_a), nest._ptr(s_a), nest._ptr(z_b), nest._ptr(s_b), M, T, nest._ptr(y),
                        arr, len(nexts), xo, zn, nest._ptr(work), sd, len(side), nest._stream(stream))
    nest._check(st, "nest_chain")


def layer_input(lin: Dict[str, nest.Layer], x: torch.Tensor, buf: LayerBuffers, stream=None):
    """Rotate the layer input into the q, k, v operands and clear their accumulators (one launch)."""
    names = ("q", "k", "v")
    nest.rotate_group([x] * 3, [lin[n].sign_in for n in names], 0, x_ops=[buf.xop[n] for n in names],
                      zero=[buf.z[n] for n in names], stream=stream)


def layer_forward(lin: Dict[str, nest.Layer], buf: LayerBuffers, verify: bool,
                  next_lin: Optional[Dict[str, nest.Layer]] = None, next_buf: Optional[LayerBuffers] = None,
                  stream=None):
    """One layer from prepared q/k/v operands.  Feeds next_lin's q/k/v operands, or writes
    buf.y['down'] when this is the last layer."""
    T = buf.T
    g = lambda names: nest.gemm_group([lin[n] for n in names], [buf.xop[n] for n in names], T, verify,
                                      zs=[buf.z[n] for n in names], stream=stream)
    g(("q", "k", "v"))
    # the k and v outputs are rotated back by extra CTAs of the q glue's first launch
    chain(buf.z["q"], lin["q"].sign_out, None, None, T, buf.work, None, [lin["o"]], [buf.xop["o"]], [buf.z["o"]],
          stream, side=[(buf.z["k"], lin["k"].sign_out, buf.y["k"]), (buf.z["v"], lin["v"].sign_out, buf.y["v"])])
    g(("o",))
    chain(buf.z["o"], lin["o"].sign_out, None, None, T, buf.work, None, [lin["gate"], lin["up"]],
          [buf.xop["gate"], buf.xop["up"]], [buf.z["gate"], buf.z["up"]], stream)
    g(("gate", "up"))
    chain(buf.z["gate"], lin["gate"].sign_out, buf.z["up"], lin["up"].sign_out, T, buf.work, None, [lin["down"]],
          [buf.xop["down"]], [buf.z["down"]], stream)
    g(("down",))
    if next_lin is None:
        chain(buf.z["down"], lin["down"].sign_out, None, None, T, buf.work, buf.y["down"], stream=stream)
    else:
        chain(buf.z["down"], lin["down"].sign_out, None, None, T, buf.work, buf.y["down"],
              [next_lin[n] for n in ("q", "k", "v")], [next_buf.xop[n] for n in ("q", "k", "v")],
              [next_buf.z[n] for n in ("q", "k", "v")], stream)
