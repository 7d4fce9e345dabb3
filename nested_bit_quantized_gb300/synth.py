"""Seeded synthetic inputs for the nested-bit quantized linear layer.

This module only draws random numbers and holds the workload shapes.  It
contains none of the method's arithmetic (no rotation, no quantisation, no
packing): both the CPU oracle and the CUDA path take their inputs from here,
and nothing here depends on either of them.

Workloads stand in for the real models the source pages measured on (Qwen-4B,
Gemma-12B and a 31B dense model): the shapes are those models' decoder-layer
linears, the values are synthetic.

Recipes
-------
* Weights ``W`` (M x K, float32): i.i.d. N(0, 0.02^2).
  - ``outliers="columns"``: round(0.01*K) distinct input columns, chosen with
    the same generator, are multiplied by 8 (the single-layer workload).
  - ``outliers="entries"``: round(0.005*M*K) distinct entries, chosen
    uniformly, are replaced by 0.02 * t_4 (Student-t with 4 degrees of
    freedom).  The pages give no outlier scale; 0.02 (the weight sigma) is
    the plain reading.
* Activations ``x`` (T x K): N(0, 1) drawn in float32, rounded to bfloat16
  (round to nearest even), returned as the bf16 bit patterns and as float32.
* Sign vectors: the +-1 vectors S_o (seed) and S_i (seed + 1) are drawn with
  ``torch.Generator().manual_seed(seed)`` and ``randint(0, 2) * 2 - 1``, the
  generator the 2-bit-base post names in its POC recipe, step 1 (Rotation).
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Tuple

import numpy as np


# ----------------------------------------------------------------------------
# random draws
# ----------------------------------------------------------------------------

def weights(M: int, K: int, seed: int, outliers: str | None = None) -> np.ndarray:
    """float32 [M][K] synthetic weight matrix (see the module docstring)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    W = rng.normal(0.0, 0.02, size=(M, K))
    if outliers == "columns":
        n = int(round(0.01 * K))
        cols = rng.choice(K, size=n, replace=False)
        W[:, cols] *= 8.0
    elif outliers == "entries":
        n = int(round(0.005 * M * K))
        idx = rng.choice(M * K, size=n, replace=False)
        W.reshape(-1)[idx] = 0.02 * rng.standard_t(4.0, size=n)
    elif outliers is not None:
        raise ValueError(f"unknown outlier recipe {outliers!r}")
    return W.astype(np.float32)


def weights_device(M: int, K: int, seed: int, outliers: str | None, device) -> "torch.Tensor":
    """Same recipe as :func:`weights`, drawn on ``device`` with torch's
    generator (for workloads too large to draw on the host in seconds).  The
    values are not the same draws as :func:`weights`."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    W = torch.randn((M, K), generator=g, device=device, dtype=torch.float32) * 0.02
    if outliers == "columns":
        n = int(round(0.01 * K))
        cols = torch.randperm(K, generator=g, device=device)[:n]
        W[:, cols] *= 8.0
    elif outliers == "entries":
        n = int(round(0.005 * M * K))
        idx = torch.randint(0, M * K, (n,), generator=g, device=device)
        # Student-t(4) = N / sqrt(chi2_4 / 4); chi2_4 = -2 log(U1 U2)
        nrm = torch.randn((n,), generator=g, device=device, dtype=torch.float64)
        u = torch.rand((2, n), generator=g, device=device, dtype=torch.float64).clamp_min(1e-300)
        chi2 = -2.0 * torch.log(u[0] * u[1])
        t4 = nrm / torch.sqrt(chi2 / 4.0)
        W.view(-1)[idx] = (0.02 * t4).to(torch.float32)
    elif outliers is not None:
        raise ValueError(f"unknown outlier recipe {outliers!r}")
    return W


def activations(T: int, K: int, seed: int) -> Tuple[np.ndarray, np.ndarray]:
    """bf16 N(0,1) activations [T][K]: (bit patterns as uint16, values as float32)."""
    import torch
    rng = np.random.Generator(np.random.PCG64(seed))
    x32 = rng.standard_normal(size=(T, K)).astype(np.float32)
    xb = torch.from_numpy(x32).to(torch.bfloat16)
    bits = xb.view(torch.int16).numpy().view(np.uint16).copy()
    vals = xb.to(torch.float32).numpy().copy()
    return bits, vals


def signs(n: int, seed: int) -> np.ndarray:
    """int8 +-1 vector of length n from torch's CPU generator seeded with ``seed``."""
    import torch
    g = torch.Generator().manual_seed(int(seed))
    s = torch.randint(0, 2, (n,), generator=g) * 2 - 1
    return s.to(torch.int8).numpy().copy()


def sign_pair(M: int, K: int, seed: int) -> Tuple[np.ndarray, np.ndarray]:
    """(S_o of length M from ``seed``, S_i of length K from ``seed + 1``)."""
    return signs(M, seed), signs(K, seed + 1)


def uniform_codes(M: int, K: int, bits: int, seed: int):
    """Random codes and fp16 scales in the stored ranges (edge-case tests):
    base codes 0..3, residual codes in [-(2^(bits-1)-1), 2^(bits-1)-1],
    scales drawn log-uniformly in [1e-3, 1e-1] and rounded to fp16."""
    rng = np.random.Generator(np.random.PCG64(seed))
    qm = (1 << (bits - 1)) - 1
    bc = rng.integers(0, 4, size=(M, K), dtype=np.uint8)
    rc = rng.integers(-qm, qm + 1, size=(M, K)).astype(np.int8)
    G = K // 128
    bs = np.exp(rng.uniform(np.log(1e-3), np.log(1e-1), size=(M, G))).astype(np.float16)
    rs = (bs.astype(np.float64) / (4 * qm)).astype(np.float16)
    return bc, bs.view(np.uint16).copy(), rc, rs.view(np.uint16).copy()


# ----------------------------------------------------------------------------
# workloads
# ----------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class Linear:
    name: str
    M: int          # d_out
    K: int          # d_in
    w_seed: int
    sign_seed: int  # S_o uses sign_seed, S_i uses sign_seed + 1
    outliers: str | None


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    linears: Tuple[Linear, ...]
    bits: Tuple[int, ...]
    T: Tuple[int, ...]
    x_seed: int
    description: str


def _decoder(prefix: str, hidden: int, inter: int, q: int, kv: int, base: int,
             layer: int = 0) -> Tuple[Linear, ...]:
    shapes = [("q", q, hidden), ("k", kv, hidden), ("v", kv, hidden), ("o", hidden, q),
              ("gate", inter, hidden), ("up", inter, hidden), ("down", hidden, inter)]
    out = []
    for i, (n, M, K) in enumerate(shapes):
        idx = 16 * layer + i
        out.append(Linear(f"{prefix}{n}", M, K, base + idx, 10 * base + 2 * idx, "entries"))
    return tuple(out)


WORKLOADS: Dict[str, Workload] = {
    "single_4096": Workload(
        "single_4096",
        (Linear("w", 4096, 4096, 0, 0, "columns"),),
        bits=(8,), T=(1, 16), x_seed=2,
        description="single linear 4096x4096, N(0,0.02^2) with 1% columns x8, "
                    "8-bit residual, bf16 N(0,1) activations"),
    "mlp_triplet_4b": Workload(
        "mlp_triplet_4b",
        (Linear("gate", 9728, 2560, 200_000, 2_000_000, "entries"),
         Linear("up", 9728, 2560, 200_001, 2_000_002, "entries"),
         Linear("down", 2560, 9728, 200_002, 2_000_004, "entries")),
        bits=(7,), T=(1, 4, 8, 16, 32), x_seed=299_999,
        description="Qwen-4B-like MLP triplet gate/up 9728x2560, down 2560x9728, "
                    "7-bit residual, N(0,0.02^2) + 0.5% t4 outliers"),
    "decoder_12b": Workload(
        "decoder_12b",
        _decoder("", 3840, 15360, 4096, 2048, 300_000),
        bits=(6, 7, 8), T=(16,), x_seed=399_999,
        description="Gemma-12B-like decoder linears (hidden 3840, intermediate 15360), "
                    "residual 6/7/8 bits, T=16"),
    "decoder_31b": Workload(
        "decoder_31b",
        _decoder("", 5376, 21504, 8192, 4096, 400_000),
        bits=(8,), T=(1, 64), x_seed=499_999,
        description="31B-class decoder linears (hidden 5376, intermediate 21504), "
                    "8-bit residual, draft T=1, verify T=64, chained"),
}


def stack_31b(n_layers: int = 60) -> List[Tuple[Linear, ...]]:
    """The 60-layer 31B-class stack: per-layer linears of decoder_31b's shapes."""
    return [_decoder(f"L{l}.", 5376, 21504, 8192, 4096, 500_000, layer=l)
            for l in range(n_layers)]
