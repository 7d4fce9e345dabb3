"""CPU oracle for the nested-bit quantized linear layer.  TEST INFRASTRUCTURE.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module.  The product path (the CUDA library and
its Python binding) never imports or calls it, and the oracle imports nothing
from the product package except the seeded input generators.

Everything is numpy float64 and written as the pages state it, one step at a
time, with no blocking or fusion beyond what the definitions themselves say:

* rotation -- randomized Hadamard transform, Sylvester construction,
  block-diagonal, two-sided:  W~ = H_o S_o W S_i H_i,  x' = H_i S_i x,
  y = S_o H_o z.  Source: feedman.me/posts/wZBTJ ("2-bit base in VRAM,
  residual in RAM" post), POC recipe, step 1 "Rotation".  The block-diagonal
  H is applied as an explicit dense H_b per block (a matrix product is the
  library step).
* 2-bit base -- per (output row, 128-column group) scale = RMS of the block
  rounded to fp16; code = nearest of the 4 Lloyd-Max levels.  Same post, POC
  recipe step 2 (RTN variant: the GPTQ/LDLQ error feedback needs calibration
  data and is not part of this path).
* residual -- R~ = W~ - Q_base in the rotated basis; uniform symmetric b-bit,
  levels -qm..qm with qm = 2^(b-1) - 1 (printed garbled as "2b-1 - 1"),
  scale = max|block| / qm per (row, 128-group) in fp16.  POC recipe step 3
  (RTN variant).
* forward -- x' = H_i S_i x; draft z = Q_base x'; verify z = (Q_base +
  Q_resid) x'; y = S_o H_o z.  POC recipe step 4 ("the draft forward is the
  same but without y_r").  The split between GPU and CPU in that step is
  prior art; the oracle computes the plain sum.

Readings where the pages are silent:
* nearest-level ties: |u| exactly at the midpoint of the inner and outer
  level goes to the inner level; u == 0 takes the positive inner level.
* zero groups: scale 0 gives code 2 (+inner level) and a zero base; a zero
  residual scale gives residual code 0.
* residual rounding is round-half-to-even (numpy ``rint``).
* levels are exactly +-0.4528 and +-1.5104 (the workload definition), the
  Gaussian 4-level Lloyd-Max quantizer; the post's own fitted sets
  (+-0.4535/+-1.5066, +-0.4511/+-1.5021) are reproduced by ``lloyd_max_fit``
  as a check, not used.

Parity status: every function here is pinned by tests under ``tests/``
(closed forms, printed values, invariants and brute force); the GEMM output
values themselves have no worked example on the pages and are pinned only
through those invariants.
"""
from __future__ import annotations

import math
from typing import Dict, Tuple

import numpy as np

GROUP = 128
HAD_CAP = 4096
LEVELS = np.array([-1.5104, -0.4528, 0.4528, 1.5104], dtype=np.float64)


# ----------------------------------------------------------------------------
# 1. Randomized Hadamard rotation
# ----------------------------------------------------------------------------

def hadamard_block_size(n: int) -> int:
    """Largest power of two dividing n, capped at 4096 (POC recipe step 1)."""
    if n <= 0:
        raise ValueError("n must be positive")
    b = 1
    while n % (2 * b) == 0 and 2 * b <= HAD_CAP:
        b *= 2
    return b


def sylvester_unnormalised(b: int) -> np.ndarray:
    """Sylvester +-1 matrix: start from [1], repeat H <- [[H, H], [H, -H]]."""
    if b < 1 or (b & (b - 1)) != 0:
        raise ValueError("block size must be a power of two")
    H = np.ones((1, 1), dtype=np.float64)
    while H.shape[0] < b:
        H = np.block([[H, H], [H, -H]])
    return H


def sylvester(b: int) -> np.ndarray:
    """Normalised Sylvester Hadamard H_b = (+-1 matrix) / sqrt(b)."""
    return sylvester_unnormalised(b) / math.sqrt(b)


def block_hadamard_left(A: np.ndarray) -> np.ndarray:
    """H_n @ A for the block-diagonal H_n = diag(H_b, ..., H_b), b = block size of n.

    A has n rows.  Each band of b rows is multiplied by the dense H_b."""
    n = A.shape[0]
    b = hadamard_block_size(n)
    H = sylvester(b)
    out = np.empty_like(A, dtype=np.float64)
    for j in range(n // b):
        out[j * b:(j + 1) * b] = H @ A[j * b:(j + 1) * b]
    return out


def rotate_weights(W: np.ndarray, s_o: np.ndarray, s_i: np.ndarray) -> np.ndarray:
    """W~ = H_o . S_o . W . S_i . H_i   (S = diag of the sign vector)."""
    W = np.asarray(W, dtype=np.float64)
    WS = W * s_i.astype(np.float64)[None, :]              # W . S_i
    WSH = block_hadamard_left(WS.T).T                      # (H_i (W S_i)^T)^T = W S_i H_i, H_i symmetric
    SWSH = s_o.astype(np.float64)[:, None] * WSH           # S_o . (...)
    return block_hadamard_left(SWSH)                       # H_o . (...)


def unrotate_weights(Wr: np.ndarray, s_o: np.ndarray, s_i: np.ndarray) -> np.ndarray:
    """W = S_o . H_o . W~ . H_i . S_i  (the exact inverse)."""
    A = s_o.astype(np.float64)[:, None] * block_hadamard_left(np.asarray(Wr, np.float64))
    AH = block_hadamard_left(A.T).T
    return AH * s_i.astype(np.float64)[None, :]


def rotate_activations(x: np.ndarray, s_i: np.ndarray) -> np.ndarray:
    """x' = H_i . S_i . x for every token.  x is [T][K] (one row per token)."""
    x = np.asarray(x, dtype=np.float64)
    Sx = s_i.astype(np.float64)[:, None] * x.T             # [K][T]: S_i x_t as columns
    return block_hadamard_left(Sx).T


def unrotate_outputs(z: np.ndarray, s_o: np.ndarray) -> np.ndarray:
    """y = S_o . H_o . z for every token.  z is [T][M]."""
    Hz = block_hadamard_left(np.asarray(z, np.float64).T)  # [M][T]
    return (s_o.astype(np.float64)[:, None] * Hz).T


# ----------------------------------------------------------------------------
# 2. 2-bit base (RTN, 4 Lloyd-Max levels, fp16 RMS group scale)
# ----------------------------------------------------------------------------

def to_fp16(a) -> np.ndarray:
    """Round float64 values to fp16 (round to nearest even, numpy's conversion)."""
    return np.asarray(a, dtype=np.float64).astype(np.float16)


def base_threshold(levels: np.ndarray = LEVELS) -> float:
    """Decision point between the inner and the outer positive level."""
    return float((levels[2] + levels[3]) / 2.0)


def quantize_base(Wr: np.ndarray, levels: np.ndarray = LEVELS, group: int = GROUP) -> Tuple[np.ndarray, np.ndarray]:
    """Per (row, group of `group` columns, 128 in the format): s = fp16(RMS of the block);
    code = nearest level of W~/s.

    Returns (codes uint8 [M][K] in 0..3 indexing ``levels`` ascending,
             scales float16 [M][K/group])."""
    Wr = np.asarray(Wr, dtype=np.float64)
    M, K = Wr.shape
    if K % group:
        raise ValueError(f"K must be a multiple of the group ({group})")
    G = K // group
    blocks = Wr.reshape(M, G, group)
    rms = np.sqrt(np.mean(blocks * blocks, axis=2))
    s16 = to_fp16(rms)
    s = s16.astype(np.float64)
    t = base_threshold(levels)
    codes = np.full((M, G, group), 2, dtype=np.uint8)
    nz = s > 0
    with np.errstate(divide="ignore", invalid="ignore"):
        u = blocks / s[:, :, None]
    outer = np.abs(u) > t
    neg = u < 0
    c = np.where(neg, np.where(outer, 0, 1), np.where(outer, 3, 2)).astype(np.uint8)
    codes[nz] = c[nz]
    return codes.reshape(M, K), s16


def dequant_base(codes: np.ndarray, scales16: np.ndarray, levels: np.ndarray = LEVELS) -> np.ndarray:
    """Q_base = L[code] * s  (float64 [M][K]); the group is K / (scales per row)."""
    M, K = codes.shape
    G = scales16.shape[1]
    L = levels[codes.reshape(M, G, K // G)]
    return (L * scales16.astype(np.float64)[:, :, None]).reshape(M, K)


# ----------------------------------------------------------------------------
# 3. b-bit uniform residual
# ----------------------------------------------------------------------------

def qmax(bits: int) -> int:
    """Largest residual level: 2^(bits-1) - 1."""
    return (1 << (bits - 1)) - 1


def quantize_residual(R: np.ndarray, bits: int, group: int = GROUP) -> Tuple[np.ndarray, np.ndarray]:
    """Per (row, group of `group` columns): s = fp16(max|R| / qm); q = clip(rint(R/s), -qm, qm).

    Returns (codes int8 [M][K], scales float16 [M][K/group])."""
    R = np.asarray(R, dtype=np.float64)
    M, K = R.shape
    G = K // group
    qm = qmax(bits)
    blocks = R.reshape(M, G, group)
    amax = np.max(np.abs(blocks), axis=2)
    s16 = to_fp16(amax / qm)
    s = s16.astype(np.float64)
    q = np.zeros((M, G, group), dtype=np.int64)
    nz = s > 0
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.rint(blocks / s[:, :, None])
    r = np.clip(r, -qm, qm)
    q[nz] = r[nz].astype(np.int64)
    return q.reshape(M, K).astype(np.int8), s16


def dequant_residual(codes: np.ndarray, scales16: np.ndarray) -> np.ndarray:
    """Q_resid = q * s (float64 [M][K]); the group is K / (scales per row)."""
    M, K = codes.shape
    G = scales16.shape[1]
    q = codes.reshape(M, G, K // G).astype(np.float64)
    return (q * scales16.astype(np.float64)[:, :, None]).reshape(M, K)


# ----------------------------------------------------------------------------
# offline pipeline and forward passes
# ----------------------------------------------------------------------------

def quantize_layer(W: np.ndarray, s_o: np.ndarray, s_i: np.ndarray, bits: int,
                   group: int = GROUP) -> Dict[str, np.ndarray]:
    """Rotate, fit the base, quantize the residual.  Returns codes, scales and W~.  The
    storage format's group is 128 columns; other groups serve the oracle's own checks."""
    Wr = rotate_weights(W, s_o, s_i)
    bc, bs = quantize_base(Wr, group=group)
    R = Wr - dequant_base(bc, bs)
    rc, rs = quantize_residual(R, bits, group=group)
    return {"Wr": Wr, "base_codes": bc, "base_scales": bs,
            "resid_codes": rc, "resid_scales": rs}


def dense_rotated(layer: Dict[str, np.ndarray], verify: bool) -> np.ndarray:
    """W_v = Q_base (+ Q_resid) in the rotated basis (float64 [M][K])."""
    Wv = dequant_base(layer["base_codes"], layer["base_scales"])
    if verify:
        Wv = Wv + dequant_residual(layer["resid_codes"], layer["resid_scales"])
    return Wv


def forward(layer: Dict[str, np.ndarray], s_o: np.ndarray, s_i: np.ndarray,
            x: np.ndarray, verify: bool) -> Dict[str, np.ndarray]:
    """x' = H_i S_i x; z = W_v x' (rotated basis); y = S_o H_o z.

    x is [T][K] (float values of the bf16 activations); returns x', z, y as
    float64 [T][K], [T][M], [T][M]."""
    xr = rotate_activations(x, s_i)
    Wv = dense_rotated(layer, verify)
    z = xr @ Wv.T
    y = unrotate_outputs(z, s_o)
    return {"x_rot": xr, "z": z, "y": y}


def forward_rows(layer_rows: Dict[str, np.ndarray], xr: np.ndarray, verify: bool) -> np.ndarray:
    """z for a subset of output rows, given x' (used for sampled checks at full size)."""
    Wv = dequant_base(layer_rows["base_codes"], layer_rows["base_scales"])
    if verify:
        Wv = Wv + dequant_residual(layer_rows["resid_codes"], layer_rows["resid_scales"])
    return np.asarray(xr, np.float64) @ Wv.T


# ----------------------------------------------------------------------------
# level fitting (checks on the level constants)
# ----------------------------------------------------------------------------

def lloyd_max_fit(samples: np.ndarray, iters: int = 60) -> np.ndarray:
    """4-level scalar Lloyd-Max fit as the post describes it: start from the
    0.125/0.375/0.625/0.875 quantiles, alternate nearest-level assignment and
    centroid update for ``iters`` iterations, then make the set symmetric."""
    v = np.sort(np.asarray(samples, dtype=np.float64).ravel())
    L = np.quantile(v, [0.125, 0.375, 0.625, 0.875])
    for _ in range(iters):
        edges = (L[:-1] + L[1:]) / 2.0
        cut = np.searchsorted(v, edges)
        parts = np.split(v, cut)
        L = np.array([p.mean() if p.size else L[i] for i, p in enumerate(parts)])
    inner = (L[2] - L[1]) / 2.0
    outer = (L[3] - L[0]) / 2.0
    return np.array([-outer, -inner, inner, outer])


def gaussian_lloyd_max_4(iters: int = 200) -> Tuple[float, float, float]:
    """Fixed point of the centroid conditions of the 4-level quantizer for a
    standard normal: inner = E[X | 0 < X < t], outer = E[X | X > t],
    t = (inner + outer) / 2.  Returns (inner, outer, t)."""
    phi = lambda a: math.exp(-a * a / 2.0) / math.sqrt(2.0 * math.pi)
    Phi = lambda a: 0.5 * (1.0 + math.erf(a / math.sqrt(2.0)))
    inner, outer = 0.5, 1.5
    for _ in range(iters):
        t = (inner + outer) / 2.0
        inner = (phi(0.0) - phi(t)) / (Phi(t) - 0.5)
        outer = phi(t) / (1.0 - Phi(t))
    return inner, outer, (inner + outer) / 2.0


# ----------------------------------------------------------------------------
# storage accounting
# ----------------------------------------------------------------------------

def bits_per_weight(base: bool, resid_bits: int | None) -> float:
    """Storage bits per weight: 2 code bits (+ b residual bits) and one fp16
    scale per 128 weights for each part."""
    bpw = 0.0
    if base:
        bpw += 2 + 16 / GROUP
    if resid_bits:
        bpw += resid_bits + 16 / GROUP
    return bpw


# ----------------------------------------------------------------------------
# chained decoder layer (the chained-layer workload's reading; not on the pages)
# ----------------------------------------------------------------------------

def round_bf16(a) -> np.ndarray:
    """Round float64 values to bfloat16 (8 significant bits, round half to even)."""
    a = np.asarray(a, dtype=np.float64)
    m, e = np.frexp(a)                        # a = m * 2**e, 0.5 <= |m| < 1
    return np.ldexp(np.rint(m * 256.0) / 256.0, e)


def chain_glue(y_a: np.ndarray, y_b: np.ndarray | None = None) -> np.ndarray:
    """Input of the next linear: h = y_a (or y_a * y_b, e.g. gate * up), rescaled to unit
    RMS per token (row) as a stand-in for the normalisation between linears, then cast to
    bf16.  Returns the bf16 values as float64 [T][M]."""
    h = np.asarray(y_a, np.float64) if y_b is None else np.asarray(y_a, np.float64) * np.asarray(y_b, np.float64)
    rms = np.sqrt(np.mean(h * h, axis=1, keepdims=True))
    with np.errstate(divide="ignore", invalid="ignore"):
        h = np.where(rms > 0, h / rms, 0.0)
    return round_bf16(h)


def decoder_layer_forward(lin: Dict[str, tuple], x: np.ndarray, verify: bool) -> Dict[str, np.ndarray]:
    """One chained decoder layer.  lin maps q, k, v, o, gate, up, down to
    (quantized layer dict, S_o, S_i).  q, k, v read x; o reads q's output; gate and up
    read o's output; down reads gate * up; every intermediate goes through chain_glue.
    Returns each linear's y and the next layer's input."""
    out = {}
    fwd = lambda name, xin: forward(lin[name][0], lin[name][1], lin[name][2], xin, verify)["y"]
    for n in ("q", "k", "v"):
        out[n] = fwd(n, x)
    out["o"] = fwd("o", chain_glue(out["q"]))
    xg = chain_glue(out["o"])
    out["gate"] = fwd("gate", xg)
    out["up"] = fwd("up", xg)
    out["down"] = fwd("down", chain_glue(out["gate"], out["up"]))
    out["next"] = chain_glue(out["down"])
    return out


# ----------------------------------------------------------------------------
# BitNest W4/W8 nested weights (BitNest: Bit-Nested Speculative Decoding for
# Memory-Efficient LLM Inference Acceleration, Section 3.2 and Appendix A.1,
# Eq. (5)-(10); dual-plane storage, Section 3.3)
# ----------------------------------------------------------------------------

W4_QMIN, W4_QMAX = -8, 7


def quantize_w4(Wr: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """W4 base, Eq. (5): group-wise (g = 128) signed 4-bit codes q4 in [-8, 7]
    and a scale s4 per (row, group), so that W_draft = q4 * s4 (Eq. (6)).

    The paper builds the base with GPTQ, which needs calibration data; the RTN
    base is taken instead (a reading): s4 = fp16(max|W'| / 7), the symmetric
    rule the paper states for its KV cache (Eq. (11)), and q4 = clip(rint(W'/s4),
    -8, 7) with round-half-to-even.  A zero group gets s4 = 0 and q4 = 0.

    Returns (q4 int8 [M][K], s4 float16 [M][K/128])."""
    Wr = np.asarray(Wr, dtype=np.float64)
    M, K = Wr.shape
    if K % GROUP:
        raise ValueError("K must be a multiple of 128")
    G = K // GROUP
    blocks = Wr.reshape(M, G, GROUP)
    amax = np.max(np.abs(blocks), axis=2)
    s16 = to_fp16(amax / 7.0)
    s = s16.astype(np.float64)
    q = np.zeros((M, G, GROUP), dtype=np.int64)
    nz = s > 0
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.clip(np.rint(blocks / s[:, :, None]), W4_QMIN, W4_QMAX)
    q[nz] = r[nz].astype(np.int64)
    return q.reshape(M, K).astype(np.int8), s16


def refine_w4w8(Wr: np.ndarray, q4: np.ndarray, s4: np.ndarray) -> np.ndarray:
    """Fixed-base refinement, Eq. (7)-(9): dW = W' - q4 s4 (Eq. (7)),
    s_ref = s4 / 16 (Eq. (8)), and

        q_r = clip(round(dW / s_ref), 0, 7)    where q4 == -8,
        q_r = clip(round(dW / s_ref), -8, 7)   elsewhere             (Eq. (9)),

    so that 16 q4 + q_r never leaves the signed 8-bit range.  round is
    round-half-to-even (a reading); s_ref = 0 gives q_r = 0.

    Returns q_r int8 [M][K]."""
    Wr = np.asarray(Wr, dtype=np.float64)
    M, K = Wr.shape
    G = K // GROUP
    dW = Wr - dequant_w4(q4, s4)
    s_ref = (s4.astype(np.float64) / 16.0)[:, :, None]
    lo = np.where(q4.reshape(M, G, GROUP) == W4_QMIN, 0, -8)
    q = np.zeros((M, G, GROUP), dtype=np.int64)
    nz = np.broadcast_to(s_ref > 0, (M, G, GROUP))
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.rint(dW.reshape(M, G, GROUP) / s_ref)
    r = np.minimum(np.maximum(r, lo), 7)
    q[nz] = r[nz].astype(np.int64)
    return q.reshape(M, K).astype(np.int8)


def dequant_w4(q4: np.ndarray, s4: np.ndarray) -> np.ndarray:
    """W_draft = q4 * s4, Eq. (6) (float64 [M][K])."""
    M, K = q4.shape
    G = K // GROUP
    return (q4.reshape(M, G, GROUP).astype(np.float64) * s4.astype(np.float64)[:, :, None]).reshape(M, K)


def dequant_w8(q4: np.ndarray, s4: np.ndarray, qr: np.ndarray) -> np.ndarray:
    """W_target = (16 q4 + q_r) s_ref with s_ref = s4 / 16, Eq. (10) (float64 [M][K])."""
    M, K = q4.shape
    G = K // GROUP
    c8 = 16 * q4.reshape(M, G, GROUP).astype(np.int64) + qr.reshape(M, G, GROUP).astype(np.int64)
    return (c8.astype(np.float64) * (s4.astype(np.float64) / 16.0)[:, :, None]).reshape(M, K)


def quantize_layer_w4w8(W: np.ndarray, s_o: np.ndarray, s_i: np.ndarray) -> Dict[str, np.ndarray]:
    """Rotate (the same two-sided randomized Hadamard rotation as the 2-bit path,
    standing in for the paper's folded function-preserving rotations), then the
    W4 base and its fixed-base 4-bit refinement."""
    Wr = rotate_weights(W, s_o, s_i)
    q4, s4 = quantize_w4(Wr)
    qr = refine_w4w8(Wr, q4, s4)
    return {"Wr": Wr, "q4": q4, "s4": s4, "qr": qr}


def forward_w4w8(layer: Dict[str, np.ndarray], s_o: np.ndarray, s_i: np.ndarray,
                 x: np.ndarray, verify: bool) -> Dict[str, np.ndarray]:
    """x' = H_i S_i x; draft z = W_draft x', verify z = W_target x' (rotated basis);
    y = S_o H_o z.  The draft reads the base plane only (Section 3.3)."""
    xr = rotate_activations(x, s_i)
    W = dequant_w8(layer["q4"], layer["s4"], layer["qr"]) if verify else dequant_w4(layer["q4"], layer["s4"])
    z = xr @ W.T
    return {"x_rot": xr, "z": z, "y": unrotate_outputs(z, s_o)}


def forward_rows_w4w8(rows: Dict[str, np.ndarray], xr: np.ndarray, verify: bool) -> np.ndarray:
    """z for a subset of output rows, given x'."""
    W = dequant_w8(rows["q4"], rows["s4"], rows["qr"]) if verify else dequant_w4(rows["q4"], rows["s4"])
    return np.asarray(xr, np.float64) @ W.T


def bits_per_weight_w4w8(verify: bool) -> float:
    """Dual-plane storage (Section 3.3): the base plane holds 4 bits per weight plus
    the fp16 group scale; the refinement plane 4 bits per weight and no scale
    (s_ref is derived from s4)."""
    return 4 + 16 / GROUP + (4 if verify else 0)


# ----------------------------------------------------------------------------
# Nested KV4/KV8 cache (BitNest paper, Section 3.4 and Appendix A.2, Eq. (11)-(14))
# ----------------------------------------------------------------------------

KV_DIM = 128


def kv_quantize(x: np.ndarray) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Online per-token, per-KV-head symmetric RTN of vectors x[..., d] (d = 128):

        s = max_i |x_i| / 7,  q4 = clip(round(x / s), -8, 7)                         (Eq. (11))
        q_r = clip(round((x - q4 s) / (s / 16)), -8, 7)                                (Eq. (13))

    Readings: s is stored as fp16 and used as that fp16 value; round is half-to-even;
    the decisions are taken in fp32 (the pages fix no precision; fp32 is the kernel's),
    each operation rounded on its own (no fused multiply-add).  A zero vector gets s = 0
    and zero codes.

    Returns (q4 int8 [..., d], q_r int8 [..., d], s float16 [...])."""
    x32 = np.asarray(x, dtype=np.float32)
    amax = np.max(np.abs(x32), axis=-1)
    s16 = (amax / np.float32(7.0)).astype(np.float32).astype(np.float16)
    s = s16.astype(np.float32)[..., None]
    nz = s > 0
    with np.errstate(divide="ignore", invalid="ignore"):
        q4 = np.where(nz, np.clip(np.rint(x32 / s), -8, 7), 0).astype(np.float32)
        sref = s / np.float32(16.0)
        res = (x32 - (q4 * s).astype(np.float32)).astype(np.float32)
        qr = np.where(nz, np.clip(np.rint(res / sref), -8, 7), 0)
    return q4.astype(np.int8), qr.astype(np.int8), s16


def kv_dequant(q4: np.ndarray, qr: np.ndarray, s16: np.ndarray, view: int) -> np.ndarray:
    """KV4 view q4 s (Eq. (12)) or KV8 view (16 q4 + q_r) s / 16 (Eq. (14)), float64."""
    s = s16.astype(np.float64)[..., None]
    if view == 4:
        return q4.astype(np.float64) * s
    return (16 * q4.astype(np.int64) + qr.astype(np.int64)).astype(np.float64) * (s / 16.0)


def kv_attention(q: np.ndarray, k: Tuple[np.ndarray, np.ndarray, np.ndarray],
                 v: Tuple[np.ndarray, np.ndarray, np.ndarray], L: int, view: int, recent_n: int) -> np.ndarray:
    """Decode attention over a nested cache, float64.

    q: [T][Hq][d] queries of the T newest tokens (already written at positions L-T..L-1);
    k, v: (q4, q_r, s) with q4/q_r [Hkv][Lmax][d] and s [Hkv][Lmax].  Query head h reads
    KV head h // (Hq / Hkv) (grouped-query attention).  Query t sees positions
    [0, L - T + t + 1) (causal), with scores q.k / sqrt(d) and a softmax over them.
    View 8 reads KV8 everywhere (verification); view 4 reads the KV4 base (drafting)
    except the newest recent_n positions of the cache, j >= L - recent_n, which are read
    at KV8 (the Recent-N policy of Appendix A.2).

    Returns out [T][Hq][d]."""
    q = np.asarray(q, dtype=np.float64)
    T, Hq, d = q.shape
    Hkv = k[0].shape[0]
    G = Hq // Hkv
    K8 = kv_dequant(k[0][:, :L], k[1][:, :L], k[2][:, :L], 8)
    V8 = kv_dequant(v[0][:, :L], v[1][:, :L], v[2][:, :L], 8)
    if view == 4:
        K4 = kv_dequant(k[0][:, :L], k[1][:, :L], k[2][:, :L], 4)
        V4 = kv_dequant(v[0][:, :L], v[1][:, :L], v[2][:, :L], 4)
        hi = np.arange(L) >= L - recent_n
        Kv = np.where(hi[None, :, None], K8, K4)
        Vv = np.where(hi[None, :, None], V8, V4)
    else:
        Kv, Vv = K8, V8
    out = np.zeros((T, Hq, d))
    for t in range(T):
        n = L - T + t + 1
        for h in range(Hq):
            kh = h // G
            sc = Kv[kh, :n] @ q[t, h] / math.sqrt(d)
            p = np.exp(sc - sc.max())
            out[t, h] = (p / p.sum()) @ Vv[kh, :n]
    return out
