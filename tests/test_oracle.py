"""Pins for the CPU oracle: printed values, closed forms, invariants, brute force.

Each test pins the oracle to something other than itself, chosen so that a
plausible slip (a dropped term, a wrong sign or index, a transposed operand,
a wrong rounding) fails at least one of them.
"""
import math
import os

import numpy as np
import pytest
import scipy.linalg

from oracle import nest_oracle as O
from oracle import pack as P
from nested_bit_quantized_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    out = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                out.append(line.split())
    return out


# ----------------------------------------------------------------------------
# rotation
# ----------------------------------------------------------------------------

def test_block_size_printed_examples():
    for n, b, nb in _rows("block_sizes.txt"):
        n, b, nb = int(n), int(b), int(nb)
        assert O.hadamard_block_size(n) == b
        assert n // O.hadamard_block_size(n) == nb


def test_block_size_rule_small():
    # largest power of two dividing n, capped at 4096: odd n -> 1, 2^20 -> 4096
    assert O.hadamard_block_size(1) == 1
    assert O.hadamard_block_size(6) == 2
    assert O.hadamard_block_size(96) == 32
    assert O.hadamard_block_size(1 << 20) == 4096
    assert O.hadamard_block_size(3 * 8192) == 4096


@pytest.mark.parametrize("b", [1, 2, 4, 8, 16, 64, 256, 1024, 4096])
def test_sylvester_is_textbook_walsh_hadamard(b):
    # scipy.linalg.hadamard is the Sylvester construction (natural order)
    assert np.array_equal(O.sylvester_unnormalised(b), scipy.linalg.hadamard(b).astype(np.float64))


@pytest.mark.parametrize("b", [2, 8, 128, 512, 2048])
def test_hadamard_orthonormal_symmetric_self_inverse(b):
    Hu = O.sylvester_unnormalised(b)
    assert np.array_equal(Hu @ Hu.T, b * np.eye(b))
    H = O.sylvester(b)
    assert np.array_equal(H, H.T)
    assert np.allclose(H @ H, np.eye(b), atol=1e-12)


def _dense_blockdiag(n):
    b = O.hadamard_block_size(n)
    Hb = scipy.linalg.hadamard(b) / math.sqrt(b)
    return scipy.linalg.block_diag(*([Hb] * (n // b)))


@pytest.mark.parametrize("M,K", [(64, 128), (48, 96), (24, 40), (16, 384)])
def test_rotate_weights_matches_dense_formula(M, K):
    rng = np.random.default_rng(1)
    W = rng.normal(size=(M, K))
    s_o = rng.choice([-1, 1], size=M).astype(np.int8)
    s_i = rng.choice([-1, 1], size=K).astype(np.int8)
    Ho, Hi = _dense_blockdiag(M), _dense_blockdiag(K)
    ref = Ho @ np.diag(s_o.astype(float)) @ W @ np.diag(s_i.astype(float)) @ Hi
    assert np.allclose(O.rotate_weights(W, s_o, s_i), ref, atol=1e-12)


def test_rotation_exact_inverse_and_norm():
    rng = np.random.default_rng(2)
    M, K = 96, 256
    W = rng.normal(size=(M, K))
    s_o, s_i = synth.sign_pair(M, K, 11)
    Wr = O.rotate_weights(W, s_o, s_i)
    assert np.allclose(O.unrotate_weights(Wr, s_o, s_i), W, atol=1e-12)
    assert math.isclose(np.linalg.norm(Wr), np.linalg.norm(W), rel_tol=1e-12)
    # the rotation does change the matrix (signs and mixing are applied)
    assert not np.allclose(Wr, W)


def test_activation_rotation_dense_and_norm():
    rng = np.random.default_rng(3)
    T, K = 5, 384
    x = rng.normal(size=(T, K))
    s_i = synth.signs(K, 9)
    Hi = _dense_blockdiag(K)
    ref = (Hi @ np.diag(s_i.astype(float)) @ x.T).T
    xr = O.rotate_activations(x, s_i)
    assert np.allclose(xr, ref, atol=1e-12)
    assert np.allclose(np.linalg.norm(xr, axis=1), np.linalg.norm(x, axis=1), rtol=1e-12)
    # outputs: y = S_o H_o z is the inverse of z = H_o S_o y
    z = rng.normal(size=(T, 96))
    s_o = synth.signs(96, 4)
    Ho = _dense_blockdiag(96)
    assert np.allclose(O.unrotate_outputs(z, s_o), (np.diag(s_o.astype(float)) @ Ho @ z.T).T, atol=1e-12)


def test_rotated_product_equals_plain_product():
    # unquantized: S_o H_o (W~ x') == W x, which ties the activation rotation to the weight rotation
    rng = np.random.default_rng(4)
    M, K, T = 128, 512, 3
    W = rng.normal(size=(M, K))
    x = rng.normal(size=(T, K))
    s_o, s_i = synth.sign_pair(M, K, 21)
    Wr = O.rotate_weights(W, s_o, s_i)
    y = O.unrotate_outputs(O.rotate_activations(x, s_i) @ Wr.T, s_o)
    assert np.allclose(y, x @ W.T, atol=1e-10)


# ----------------------------------------------------------------------------
# levels
# ----------------------------------------------------------------------------

def test_gaussian_lloyd_max_closed_form_gives_levels():
    inner, outer, t = O.gaussian_lloyd_max_4()
    gold = {r[0]: (float(r[1]), float(r[2])) for r in _rows("levels.txt")}
    assert round(inner, 4) == gold["gaussian"][0] == O.LEVELS[2]
    assert round(outer, 4) == gold["gaussian"][1] == O.LEVELS[3]
    assert O.LEVELS[0] == -O.LEVELS[3] and O.LEVELS[1] == -O.LEVELS[2]
    assert abs(t - 0.9816) < 1e-3


def test_lloyd_fit_on_rotated_weights_near_printed_fits():
    # ~2M rotated weights normalised by their group RMS, quantile init, 60 iterations, symmetrised
    M, K = 1024, 2048
    W = synth.weights(M, K, 5, "entries").astype(np.float64)
    s_o, s_i = synth.sign_pair(M, K, 5)
    Wr = O.rotate_weights(W, s_o, s_i).reshape(M, K // 128, 128)
    u = Wr / np.sqrt(np.mean(Wr * Wr, axis=2, keepdims=True))
    L = O.lloyd_max_fit(u.ravel(), iters=60)
    gold = {r[0]: (float(r[1]), float(r[2])) for r in _rows("levels.txt")}
    for key in ("fitted_12b", "fitted_31b"):
        gi, go = gold[key]
        assert abs(L[2] - gi) / gi < 0.01
        assert abs(L[3] - go) / go < 0.01
    assert np.allclose(L, -L[::-1])


# ----------------------------------------------------------------------------
# 2-bit base
# ----------------------------------------------------------------------------

def _layer(M, K, bits, seed=7, outliers="entries"):
    W = synth.weights(M, K, seed, outliers)
    s_o, s_i = synth.sign_pair(M, K, seed + 100)
    return W, s_o, s_i, O.quantize_layer(W, s_o, s_i, bits)


def test_base_codes_bruteforce_nearest_level():
    M, K = 32, 256
    _, _, _, q = _layer(M, K, 8)
    Wr, codes, s = q["Wr"], q["base_codes"], q["base_scales"].astype(np.float64)
    for m in range(M):
        for g in range(K // 128):
            sc = s[m, g]
            # scale: the fp16 value nearest the RMS (no fp16 value is closer)
            blk = Wr[m, g * 128:(g + 1) * 128]
            rms = math.sqrt(sum(v * v for v in blk) / 128.0)
            s16 = np.float16(sc)
            up = float(np.nextafter(s16, np.float16(np.inf)))
            dn = float(np.nextafter(s16, np.float16(-np.inf)))
            assert abs(sc - rms) <= abs(up - rms) and abs(sc - rms) <= abs(dn - rms)
            for j in range(128):
                w = blk[j]
                dist = [abs(w - lv * sc) for lv in O.LEVELS]
                assert codes[m, g * 128 + j] == int(np.argmin(dist))


def test_base_relative_mse_is_gaussian_lloyd_max_distortion():
    # textbook: the 4-level Lloyd-Max quantizer of a unit Gaussian has MSE 0.1175
    M, K = 512, 4096
    W = synth.weights(M, K, 8, None).astype(np.float64)
    s_o, s_i = synth.sign_pair(M, K, 8)
    Wr = O.rotate_weights(W, s_o, s_i)
    c, s = O.quantize_base(Wr)
    err = Wr - O.dequant_base(c, s)
    rel = np.sum(err ** 2) / np.sum(Wr ** 2)
    assert abs(rel - 0.1175) < 0.003


def test_base_ties_and_zero_groups():
    t = O.base_threshold()
    Wr = np.zeros((2, 128))
    Wr[1, :] = 1.0                      # RMS 1 -> scale 1.0 exactly
    Wr[1, 0] = 0.0                      # u == 0 -> positive inner
    Wr[1, 1] = -t                       # |u| == threshold -> inner level
    Wr[1, 2] = np.nextafter(t, 2.0)     # just past it -> outer level
    Wr[1, 3] = -5.0
    # RMS is no longer 1 once entries change; compute what the scale must be
    c, s = O.quantize_base(Wr)
    assert s[0, 0] == 0 and np.all(c[0] == 2)            # zero group: code 2, zero base
    assert np.all(O.dequant_base(c, s)[0] == 0.0)
    sc = float(s[1, 0])
    u = Wr[1] / sc
    assert c[1, 0] == 2
    assert c[1, 3] == 0
    exp = np.where(u < 0, np.where(np.abs(u) > t, 0, 1), np.where(np.abs(u) > t, 3, 2))
    assert np.array_equal(c[1], exp)


# ----------------------------------------------------------------------------
# residual
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("bits", [6, 7, 8])
def test_residual_bruteforce_and_bound(bits):
    M, K = 16, 256
    _, _, _, q = _layer(M, K, bits, seed=9)
    R = q["Wr"] - O.dequant_base(q["base_codes"], q["base_scales"])
    rc, rs = q["resid_codes"], q["resid_scales"].astype(np.float64)
    qm = (1 << (bits - 1)) - 1
    levels = np.arange(-qm, qm + 1)
    for m in range(M):
        for g in range(K // 128):
            sc = rs[m, g]
            blk = R[m, g * 128:(g + 1) * 128]
            assert np.max(np.abs(rc[m, g * 128:(g + 1) * 128])) == qm   # the block max maps to +-qm
            for j in range(128):
                d = np.abs(blk[j] - levels * sc)
                assert abs(int(rc[m, g * 128 + j]) - levels[np.argmin(d)]) == 0 or \
                    math.isclose(d.min(), d[int(rc[m, g * 128 + j]) + qm], rel_tol=1e-12)
    E = R - O.dequant_residual(rc, q["resid_scales"])
    half = np.repeat(rs, 128, axis=1) / 2.0
    assert np.all(np.abs(E) <= half * (1 + 1e-12))


def test_residual_zero_scale_gives_zero_codes():
    R = np.zeros((1, 128))
    q, s = O.quantize_residual(R, 7)
    assert np.all(q == 0) and s[0, 0] == 0


def test_residual_scale_is_fp16_of_absmax_over_qm():
    rng = np.random.default_rng(5)
    R = rng.normal(size=(3, 256)) * 1e-3
    for bits in (6, 7, 8):
        q, s = O.quantize_residual(R, bits)
        qm = (1 << (bits - 1)) - 1
        for m in range(3):
            for g in range(2):
                amax = max(abs(v) for v in R[m, g * 128:(g + 1) * 128])
                assert s[m, g] == np.float16(amax / qm)


def test_small_group_quantizers_and_forward_by_scalar_loops():
    # A group of 8 columns on an 8 x 16 layer, every step redone by scalar loops from
    # the post's POC recipe (steps 2-4): RMS scale, nearest level, absmax residual scale,
    # rounding, and z = sum_k (Q_base + Q_resid)[m][k] x'[k].  Pins the group index
    # arithmetic (a slip that mixes up groups shows only when a row has many of them).
    M, K, G, bits, T = 8, 16, 8, 7, 3
    rng = np.random.default_rng(21)
    W = rng.normal(size=(M, K))
    s_o = rng.choice([-1, 1], size=M).astype(np.int8)
    s_i = rng.choice([-1, 1], size=K).astype(np.int8)
    x = rng.normal(size=(T, K))
    q = O.quantize_layer(W, s_o, s_i, bits, group=G)
    Wr = q["Wr"]
    levels = [-1.5104, -0.4528, 0.4528, 1.5104]
    t = (0.4528 + 1.5104) / 2
    qm = (1 << (bits - 1)) - 1
    Wv = [[0.0] * K for _ in range(M)]
    for m in range(M):
        for g in range(K // G):
            cols = range(g * G, (g + 1) * G)
            sb = float(np.float16(math.sqrt(sum(Wr[m, k] ** 2 for k in cols) / G)))
            assert float(q["base_scales"][m, g]) == sb
            base = {}
            for k in cols:
                if sb == 0:
                    c = 2
                else:
                    u = Wr[m, k] / sb
                    c = (3 if abs(u) > t else 2) if u >= 0 else (0 if abs(u) > t else 1)
                assert q["base_codes"][m, k] == c
                base[k] = levels[c] * sb
            sr = float(np.float16(max(abs(Wr[m, k] - base[k]) for k in cols) / qm))
            assert float(q["resid_scales"][m, g]) == sr
            for k in cols:
                r = 0 if sr == 0 else int(np.clip(np.rint((Wr[m, k] - base[k]) / sr), -qm, qm))
                assert q["resid_codes"][m, k] == r
                Wv[m][k] = base[k] + r * sr
    xr = O.rotate_activations(x, s_i)
    z = O.forward(q, s_o, s_i, x, verify=True)["z"]
    for tt in range(T):
        for m in range(M):
            ref = sum(Wv[m][k] * xr[tt, k] for k in range(K))
            assert math.isclose(z[tt, m], ref, rel_tol=1e-12, abs_tol=1e-12)
    # the group changes the fit: one group per row gives other scales and codes
    q16 = O.quantize_layer(W, s_o, s_i, bits, group=K)
    assert q16["base_scales"].shape == (M, 1) and not np.array_equal(q16["base_codes"], q["base_codes"])


# ----------------------------------------------------------------------------
# forward passes
# ----------------------------------------------------------------------------

def test_draft_is_exact_subset_of_verify():
    M, K, T = 64, 256, 4
    W, s_o, s_i, q = _layer(M, K, 8)
    _, x = synth.activations(T, K, 3)
    q0 = dict(q)
    q0["resid_codes"] = np.zeros_like(q["resid_codes"])
    a = O.forward(q0, s_o, s_i, x, verify=True)
    b = O.forward(q, s_o, s_i, x, verify=False)
    assert np.array_equal(a["z"], b["z"]) and np.array_equal(a["y"], b["y"])


@pytest.mark.parametrize("bits", [6, 8])
def test_verify_matches_plain_product_within_residual_error(bits):
    M, K, T = 256, 1024, 8
    W, s_o, s_i, q = _layer(M, K, bits)
    _, x = synth.activations(T, K, 4)
    yv = O.forward(q, s_o, s_i, x, verify=True)["y"]
    yd = O.forward(q, s_o, s_i, x, verify=False)["y"]
    y = x.astype(np.float64) @ W.astype(np.float64).T
    E = q["Wr"] - O.dense_rotated(q, verify=True)
    bound = np.linalg.norm(E, 2) * np.linalg.norm(x, axis=1)
    assert np.all(np.linalg.norm(yv - y, axis=1) <= bound * (1 + 1e-9))
    # errors of the expected size: verify ~ residual rounding, draft ~ base distortion
    ev = np.linalg.norm(yv - y) / np.linalg.norm(y)
    ed = np.linalg.norm(yd - y) / np.linalg.norm(y)
    qm = (1 << (bits - 1)) - 1
    assert ev < 0.05 * 127 / qm / 10
    assert 0.25 < ed < 0.45                     # sqrt(0.1175) = 0.343 for Gaussianised weights
    assert ev < ed / 10


def test_token_columns_are_independent():
    M, K, T = 128, 512, 6
    W, s_o, s_i, q = _layer(M, K, 7)
    _, x = synth.activations(T, K, 6)
    full = O.forward(q, s_o, s_i, x, verify=True)
    for t in range(T):
        one = O.forward(q, s_o, s_i, x[t:t + 1], verify=True)
        assert np.allclose(one["y"][0], full["y"][t], rtol=1e-12, atol=1e-14)


def test_bruteforce_tiny_forward():
    # y[t][m] by explicit loops over the dense dequantised matrix and dense H.D
    M, K, T = 16, 128, 2
    W, s_o, s_i, q = _layer(M, K, 8, seed=12, outliers=None)
    _, x = synth.activations(T, K, 13)
    Wv = O.dense_rotated(q, verify=True)
    Ho, Hi = _dense_blockdiag(M), _dense_blockdiag(K)
    y = np.zeros((T, M))
    for t in range(T):
        xr = [sum(Hi[k, kk] * s_i[kk] * float(x[t, kk]) for kk in range(K)) for k in range(K)]
        z = [sum(Wv[m, k] * xr[k] for k in range(K)) for m in range(M)]
        for m in range(M):
            y[t, m] = s_o[m] * sum(Ho[m, mm] * z[mm] for mm in range(M))
    assert np.allclose(O.forward(q, s_o, s_i, x, verify=True)["y"], y, atol=1e-12)


# ----------------------------------------------------------------------------
# storage accounting and packing
# ----------------------------------------------------------------------------

def test_bits_per_weight_printed():
    for label, bits, group, bpw in _rows("bits_per_weight.txt"):
        bits, group, bpw = int(bits), int(group), float(bpw)
        assert bits + 16 / group == bpw
    assert O.bits_per_weight(True, None) == 2.125
    for b, v in ((6, 6.125), (7, 7.125), (8, 8.125)):
        assert O.bits_per_weight(False, b) == v
    assert O.bits_per_weight(True, 8) == 10.25


@pytest.mark.parametrize("bits", [6, 7, 8])
def test_packed_sizes_match_accounting(bits):
    M, K = 256, 512
    assert P.base_bytes(M, K) * 8 / (M * K) == O.bits_per_weight(True, None)
    assert P.resid_bytes(M, K, bits) * 8 / (M * K) == O.bits_per_weight(False, bits)


def test_storage_printed_approximately():
    for name, layers, gb in _rows("storage_gb.txt"):
        wl = synth.WORKLOADS[name]
        n = sum(l.M * l.K for l in wl.linears) * int(layers)
        est = n * O.bits_per_weight(True, None) / 8 / 1e9
        assert abs(est - float(gb)) / float(gb) < 0.03


@pytest.mark.parametrize("M,K,bits", [(128, 128, 8), (200, 256, 7), (77, 384, 6), (1, 128, 8)])
def test_pack_roundtrip(M, K, bits):
    bc, bs, rc, rs = synth.uniform_codes(M, K, bits, 17)
    pb = P.pack_base(bc, bs)
    pr = P.pack_resid(rc, rs, bits)
    c2, s2 = P.unpack_base(pb, M, K)
    r2, t2 = P.unpack_resid(pr, M, K, bits)
    assert np.array_equal(c2, bc) and np.array_equal(s2, bs)
    assert np.array_equal(r2, rc) and np.array_equal(t2, rs)


def _word(buf, unit_off, r, w):
    off = unit_off + ((w // 4) * 128 + r) * 16 + (w % 4) * 4
    return int.from_bytes(bytes(buf[off:off + 4]), "little")


def test_pack_hand_worked_examples():
    # base: column j holds code j % 4.  Column 16w + 4p + q sits at bits 8q + 2p, so byte q of
    # every word holds the code q four times: bytes 00 55 AA FF, word 0xFFAA5500.
    M, K = 1, 128
    bc = (np.arange(K) % 4).astype(np.uint8)[None, :]
    bs = np.array([[0x3C00]], dtype=np.uint16)               # fp16 1.0
    pb = P.pack_base(bc, bs)
    assert pb.size == 4352
    for w in range(8):
        assert _word(pb, 0, 0, w) == 0xFFAA5500
    assert pb[4096] == 0x00 and pb[4097] == 0x3C
    assert not pb[16:2048].any()                              # rows 1..127 of chunk 0 are padding
    # residual b = 8: q_j = j - 64 stored as u = j + 64, column 4w + q in byte q of word w
    rc = (np.arange(K) - 64).astype(np.int8)[None, :]
    pr = P.pack_resid(rc, np.array([[0x1234]], np.uint16), 8)
    for w in range(32):
        assert _word(pr, 0, 0, w) == sum((4 * w + q + 64) << (8 * q) for q in range(4))
    assert pr[16384] == 0x34 and pr[16385] == 0x12
    # rows past M store q = 0 (u = 128) and scale 0
    assert _word(pr, 0, 1, 0) == 0x80808080
    # residual b = 7: all q = 0 (u = 64 = 0b1000000) except column 5 with q = 63 (u = 127)
    rc = np.zeros((1, K), np.int8)
    rc[0, 5] = 63
    pr = P.pack_resid(rc, np.array([[0]], np.uint16), 7)
    # column 5 = 8*0 + 4*1 + 1: low nibble 15 at bits 8*1 + 4 = 12..15 of word 0
    assert _word(pr, 0, 0, 0) == 0x0000F000
    assert all(_word(pr, 0, 0, w) == 0 for w in range(1, 16))
    # column 5 = 16*0 + 4*1 + 1: middle pair 3 at bits 8*1 + 2*1 = 10..11 of word 16
    assert _word(pr, 0, 0, 16) == 0x00000C00
    assert all(_word(pr, 0, 0, w) == 0 for w in range(17, 24))
    # bit 6 of u is 1 for every column (u = 64 and u = 127): words 24..27 all ones
    assert all(_word(pr, 0, 0, w) == 0xFFFFFFFF for w in range(24, 28))


# ----------------------------------------------------------------------------
# chained-layer glue
# ----------------------------------------------------------------------------

def test_round_bf16_matches_library_conversion():
    import torch
    rng = np.random.default_rng(30)
    a = (rng.standard_normal(20000) * np.exp(rng.uniform(-20, 20, 20000))).astype(np.float32).astype(np.float64)
    a[:4] = [0.0, -0.0, 1.0, 1.0 + 2.0 ** -8]          # exact tie rounds to even
    ref = torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16).double().numpy()
    assert np.array_equal(O.round_bf16(a), ref)


def test_chain_glue_unit_rms_and_product():
    rng = np.random.default_rng(31)
    ya, yb = rng.normal(size=(3, 256)) * 5.0, rng.normal(size=(3, 256))
    h = O.chain_glue(ya)
    assert np.allclose(np.sqrt(np.mean(h * h, axis=1)), 1.0, atol=4e-3)      # bf16 rounding only
    hp = O.chain_glue(ya, yb)
    p = ya * yb
    assert np.allclose(hp, p / np.sqrt(np.mean(p * p, axis=1, keepdims=True)), rtol=2 ** -8, atol=0)
    assert np.array_equal(O.chain_glue(np.zeros((1, 128))), np.zeros((1, 128)))


# ----------------------------------------------------------------------------
# BitNest W4/W8 nested weights (BitNest paper, Section 3.2-3.3, Appendix A.1)
# ----------------------------------------------------------------------------

def _rotated(M, K, seed):
    W = synth.weights(M, K, seed, "entries")
    s_o, s_i = synth.sign_pair(M, K, seed + 1)
    return O.rotate_weights(W, s_o, s_i)


def test_w4_base_is_nearest_of_the_16_levels():
    """Eq. (5): brute force over all 16 codes; the scale makes max|W'| land on +-7."""
    Wr = _rotated(24, 256, 901)
    q4, s4 = O.quantize_w4(Wr)
    M, K = Wr.shape
    s = np.repeat(s4.astype(np.float64), 128, axis=1)
    cand = np.arange(-8, 8)[None, None, :] * s[:, :, None]
    err = np.abs(Wr[:, :, None] - cand)
    best = err.min(axis=2)
    got = np.abs(Wr - q4.astype(np.float64) * s)
    assert np.allclose(got, best, rtol=0, atol=1e-15)
    amax = np.abs(Wr).reshape(M, 2, 128).max(axis=2)
    assert np.all(np.abs(s4.astype(np.float64) * 7 - amax) <= amax * 2.0 ** -11)
    assert q4.min() >= -7 and q4.max() <= 7        # symmetric RTN never needs -8
    top = np.abs(Wr).reshape(M, 2, 128).argmax(axis=2)
    assert np.all(np.abs(np.take_along_axis(q4.reshape(M, 2, 128).astype(int), top[:, :, None], 2)) == 7)


def test_w4w8_refinement_is_nearest_allowed_code():
    """Eq. (7)-(9): brute force over the allowed refinement codes, s_ref = s4 / 16."""
    Wr = _rotated(16, 384, 903)
    q4, s4 = O.quantize_w4(Wr)
    qr = O.refine_w4w8(Wr, q4, s4)
    dW = Wr - O.dequant_w4(q4, s4)
    sref = np.repeat(s4.astype(np.float64) / 16, 128, axis=1)
    cand = np.arange(-8, 8)[None, None, :] * sref[:, :, None]
    best = np.abs(dW[:, :, None] - cand).min(axis=2)
    assert np.allclose(np.abs(dW - qr * sref), best, rtol=0, atol=1e-15)
    # the error is at most s_ref, and at most s_ref / 2 where no clip at +7 happened
    E = np.abs(Wr - O.dequant_w8(q4, s4, qr))
    assert np.all(E <= sref * (1 + 1e-12))
    unclipped = dW / sref < 7.5
    assert np.all(E[unclipped] <= sref[unclipped] / 2 * (1 + 1e-12))


def test_w4w8_asymmetric_clip_at_minus_eight():
    """Eq. (9): where q4 = -8 the refinement is clipped to [0, 7], so 16 q4 + q_r >= -128."""
    s4 = np.full((1, 1), 0.5, dtype=np.float16)          # s_ref = 1/32
    q4 = np.full((1, 128), -7, dtype=np.int8)
    q4[0, :64] = -8
    Wr = q4.astype(np.float64) * 0.5 - 3.2 / 32           # dW / s_ref = -3.2 everywhere
    Wr[0, 10] = -8 * 0.5 + 5.4 / 32                       # dW / s_ref = +5.4 under q4 = -8
    qr = O.refine_w4w8(Wr, q4, s4)
    assert np.all(qr[0, :64][np.arange(64) != 10] == 0)    # clipped at 0
    assert qr[0, 10] == 5
    assert np.all(qr[0, 64:] == -3)                       # q4 > -8: ordinary rounding
    # every admissible (q4, q_r) pair composes to a signed 8-bit code; the unclipped rule would not
    codes = [16 * a + b for a in range(-8, 8) for b in (range(0, 8) if a == -8 else range(-8, 8))]
    assert min(codes) == -128 and max(codes) == 119 and len(set(codes)) == len(codes)
    assert 16 * -8 + -8 < -128


def test_w8_target_identity_and_exact_subset():
    """Eq. (10): q4 s4 + q_r s_ref == (16 q4 + q_r) s_ref exactly; q_r = 0 gives the draft."""
    Wr = _rotated(8, 256, 905)
    q4, s4 = O.quantize_w4(Wr)
    qr = O.refine_w4w8(Wr, q4, s4)
    sref = np.repeat(s4.astype(np.float64) / 16, 128, axis=1)
    two_terms = O.dequant_w4(q4, s4) + qr.astype(np.float64) * sref
    assert np.array_equal(two_terms, O.dequant_w8(q4, s4, qr))
    assert np.array_equal(O.dequant_w8(q4, s4, np.zeros_like(qr)), O.dequant_w4(q4, s4))


def test_w4w8_zero_group_and_storage():
    Wr = _rotated(4, 256, 907)
    Wr[1, 128:] = 0.0
    q4, s4 = O.quantize_w4(Wr)
    qr = O.refine_w4w8(Wr, q4, s4)
    assert s4[1, 1] == 0 and np.all(q4[1, 128:] == 0) and np.all(qr[1, 128:] == 0)
    # dual-plane storage (Section 3.3): N/2 bytes per plane, the scale only on the base
    assert O.bits_per_weight_w4w8(False) == 4.125 and O.bits_per_weight_w4w8(True) == 8.125


def test_w4w8_forward_bruteforce_and_error_order():
    """Triple loop on a tiny case against the dense path, and the target's output error
    is about 1/16 of the draft's (one extra 4-bit refinement of the same scale)."""
    M, K, T = 16, 128, 3
    W = synth.weights(M, K, 909, "entries")
    s_o, s_i = synth.sign_pair(M, K, 910)
    lay = O.quantize_layer_w4w8(W, s_o, s_i)
    _, x = synth.activations(T, K, 911)
    for verify in (False, True):
        out = O.forward_w4w8(lay, s_o, s_i, x, verify)
        Wd = O.dequant_w8(lay["q4"], lay["s4"], lay["qr"]) if verify else O.dequant_w4(lay["q4"], lay["s4"])
        z = np.zeros((T, M))
        for t in range(T):
            for m in range(M):
                z[t, m] = sum(Wd[m, k] * out["x_rot"][t, k] for k in range(K))
        assert np.allclose(out["z"], z, rtol=1e-12, atol=1e-12)
    M, K = 64, 512
    W = synth.weights(M, K, 913, "entries")
    s_o, s_i = synth.sign_pair(M, K, 914)
    lay = O.quantize_layer_w4w8(W, s_o, s_i)
    _, x = synth.activations(8, K, 915)
    ref = x @ W.T
    e4 = np.linalg.norm(O.forward_w4w8(lay, s_o, s_i, x, False)["y"] - ref)
    e8 = np.linalg.norm(O.forward_w4w8(lay, s_o, s_i, x, True)["y"] - ref)
    assert 8 < e4 / e8 < 32


@pytest.mark.parametrize("M,K", [(128, 128), (200, 384), (1, 256)])
def test_w4w8_pack_roundtrip(M, K):
    rng = np.random.default_rng(M + K)
    q4 = rng.integers(-8, 8, size=(M, K)).astype(np.int8)
    qr = rng.integers(-8, 8, size=(M, K)).astype(np.int8)
    s4 = rng.uniform(1e-3, 1e-1, size=(M, K // 128)).astype(np.float16)
    base, ref = P.pack_w4w8(q4, s4, qr)
    tiles = (M + 127) // 128
    assert base.size == tiles * (K // 128) * 8448 and ref.size == tiles * (K // 128) * 8192
    u4, us, ur = P.unpack_w4w8(base, ref, M, K)
    assert np.array_equal(u4, q4) and np.array_equal(ur, qr) and np.array_equal(us, s4.view(np.uint16))
    b2, r2 = P.pack_w4w8(q4, s4, None)
    assert r2 is None and np.array_equal(b2, base)


def test_w4w8_pack_hand_worked_examples():
    """Nibble positions written out by hand from the layout description."""
    M, K = 2, 128
    q4 = np.zeros((M, K), dtype=np.int8)
    qr = np.zeros((M, K), dtype=np.int8)
    q4[0, 0] = 3        # u = 11: row 0, word 0, bits 0..3    -> byte 0 low nibble
    q4[0, 4] = -2       # u = 6:  row 0, word 0, bits 4..7    -> byte 0 high nibble
    q4[1, 9] = -8       # u = 0:  row 1, word 1, bits 8..11   -> byte (0*128+1)*16 + 4 + 1, low nibble
    q4[0, 127] = 7      # u = 15: row 0, word 15 (chunk 3, word 3), bits 28..31 -> byte (3*128)*16 + 12 + 3
    qr[1, 33] = 5       # u = 13: row 1, word 4 (chunk 1, word 0), bits 8..11 -> byte (128+1)*16 + 1
    s4 = np.zeros((M, 1), dtype=np.float16)
    s4[1, 0] = 1.0      # 0x3C00 at 8192 + 2
    base, ref = P.pack_w4w8(q4, s4, qr)
    assert base[0] == 0x6B
    assert base[16 + 5] & 0x0F == 0x0 and base[16 + 5] >> 4 == 0x8
    assert base[3 * 128 * 16 + 15] >> 4 == 0xF
    assert ref[(128 + 1) * 16 + 1] & 0x0F == 0xD
    assert base[8192 + 2] == 0x00 and base[8192 + 3] == 0x3C
    assert base[17] == 0x88                      # untouched columns hold q = 0 (u = 8)


# ----------------------------------------------------------------------------
# nested KV4/KV8 cache (BitNest paper, Section 3.4, Appendix A.2)
# ----------------------------------------------------------------------------

def test_kv_quantize_nearest_codes_and_views():
    """Eq. (11)-(14): the base is the nearest of 16 levels of s, the refinement the nearest
    of 16 levels of s/16 around it; KV8 = (16 q4 + q_r) s/16 exactly equals q4 s + q_r s/16."""
    rng = np.random.default_rng(5)
    x = rng.normal(size=(6, 4, 128)).astype(np.float32) * rng.uniform(0.1, 4, size=(6, 4, 1)).astype(np.float32)
    q4, qr, s16 = O.kv_quantize(x)
    s = s16.astype(np.float64)[..., None]
    amax = np.abs(x).max(axis=-1)
    assert np.all(np.abs(s16.astype(np.float64) * 7 - amax) <= amax * 2.0 ** -10)
    levels = np.arange(-8, 8)
    e4 = np.abs(x[..., None] - levels * s[..., None])
    assert np.allclose(np.abs(x - q4 * s), e4.min(axis=-1), rtol=0, atol=1e-6 * amax.max())
    r = x - q4 * s
    er = np.abs(r[..., None] - levels * (s / 16)[..., None])
    assert np.allclose(np.abs(r - qr * s / 16), er.min(axis=-1), rtol=0, atol=1e-6 * amax.max())
    k8 = O.kv_dequant(q4, qr, s16, 8)
    assert np.array_equal(k8, O.kv_dequant(q4, qr, s16, 4) + qr * (s / 16))
    assert np.all(np.abs(x - k8) <= s / 16 * (1 + 1e-6))                 # <= s_ref (clip at +7), ~s_ref/2 typical
    assert np.abs(x - k8).mean() < np.abs(x - O.kv_dequant(q4, qr, s16, 4)).mean() / 8
    assert q4.min() >= -7                                                  # s = max/7 never needs -8
    z = np.zeros((1, 128), np.float32)
    zq4, zqr, zs = O.kv_quantize(z)
    assert zs[0] == 0 and not zq4.any() and not zqr.any()


def test_kv_attention_bruteforce_and_policies():
    """Causal GQA decode attention against explicit loops; Recent-N = 0 is the pure KV4 view,
    Recent-N >= L the pure KV8 view; a one-position window reduces to that value."""
    rng = np.random.default_rng(7)
    Hkv, G, L, T, d = 2, 3, 11, 3, 128
    kx = rng.normal(size=(Hkv, 16, d)).astype(np.float32)
    vx = rng.normal(size=(Hkv, 16, d)).astype(np.float32)
    k = O.kv_quantize(kx)
    v = O.kv_quantize(vx)
    q = rng.normal(size=(T, Hkv * G, d))
    out = O.kv_attention(q, k, v, L, 8, 0)
    K8 = O.kv_dequant(*k, 8)
    V8 = O.kv_dequant(*v, 8)
    for t in range(T):
        for h in range(Hkv * G):
            n = L - T + t + 1
            w = [math.exp(sum(K8[h // G, j, i] * q[t, h, i] for i in range(d)) / math.sqrt(d)) for j in range(n)]
            ref = sum(w[j] * V8[h // G, j] for j in range(n)) / sum(w)
            assert np.allclose(out[t, h], ref, rtol=1e-10, atol=1e-12)
    assert np.allclose(O.kv_attention(q, k, v, L, 4, L), out, rtol=0, atol=1e-14)
    o4 = O.kv_attention(q, k, v, L, 4, 0)
    K4 = O.kv_dequant(*k, 4)
    V4 = O.kv_dequant(*v, 4)
    sc = K4[0, :L - T + 1] @ q[0, 0] / math.sqrt(d)
    p = np.exp(sc - sc.max())
    assert np.allclose(o4[0, 0], p / p.sum() @ V4[0, :L - T + 1], rtol=1e-12)
    one = O.kv_attention(q[:1], k, v, 1, 4, 0)
    assert np.allclose(one[0, 0], V4[0, 0], rtol=1e-12)
    mixed = O.kv_attention(q, k, v, L, 4, 3)
    assert not np.allclose(mixed, o4) and not np.allclose(mixed, out)


# ----------------------------------------------------------------------------
# sampled-row forwards and the chained decoder layer
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("verify", [False, True])
def test_forward_rows_equals_triple_loop_and_rows_of_forward(verify):
    """forward_rows (used for sampled checks at full size) on a subset of rows equals a
    triple loop over the hand-dequantised rows, and the same rows of forward's z."""
    M, K, T = 40, 256, 3
    _, s_o, s_i, q = _layer(M, K, 7, seed=21)
    _, x = synth.activations(T, K, 22)
    full = O.forward(q, s_o, s_i, x, verify)
    rows = np.array([0, 3, 17, 39, 20])
    sub = {k: q[k][rows] for k in ("base_codes", "base_scales", "resid_codes", "resid_scales")}
    z = O.forward_rows(sub, full["x_rot"], verify)
    lv = [-1.5104, -0.4528, 0.4528, 1.5104]
    ref = np.zeros((T, rows.size))
    for t in range(T):
        for j, m in enumerate(rows):
            acc = 0.0
            for k in range(K):
                w = lv[q["base_codes"][m, k]] * float(q["base_scales"][m, k // 128])
                if verify:
                    w += float(q["resid_codes"][m, k]) * float(q["resid_scales"][m, k // 128])
                acc += w * full["x_rot"][t, k]
            ref[t, j] = acc
    assert np.allclose(z, ref, rtol=1e-12, atol=1e-13)
    assert np.allclose(z, full["z"][:, rows], rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("verify", [False, True])
def test_forward_rows_w4w8_equals_triple_loop_and_rows_of_forward(verify):
    """forward_rows_w4w8 on a subset of rows equals a triple loop over q4 s4 (draft,
    Eq. (6)) or (16 q4 + q_r) s4 / 16 (target, Eq. (10)), and forward_w4w8's rows."""
    M, K, T = 24, 256, 2
    W = synth.weights(M, K, 930, "entries")
    s_o, s_i = synth.sign_pair(M, K, 931)
    lay = O.quantize_layer_w4w8(W, s_o, s_i)
    _, x = synth.activations(T, K, 932)
    full = O.forward_w4w8(lay, s_o, s_i, x, verify)
    rows = np.array([1, 0, 23, 11])
    sub = {k: lay[k][rows] for k in ("q4", "s4", "qr")}
    z = O.forward_rows_w4w8(sub, full["x_rot"], verify)
    ref = np.zeros((T, rows.size))
    for t in range(T):
        for j, m in enumerate(rows):
            for k in range(K):
                s = float(lay["s4"][m, k // 128])
                c = 16 * int(lay["q4"][m, k]) + int(lay["qr"][m, k]) if verify else int(lay["q4"][m, k])
                ref[t, j] += c * (s / 16 if verify else s) * full["x_rot"][t, k]
    assert np.allclose(z, ref, rtol=1e-12, atol=1e-13)
    assert np.allclose(z, full["z"][:, rows], rtol=1e-12, atol=1e-13)


def _bf16_bits(a):
    """Round float64 to bfloat16 (8 significant bits, ties to even) on the IEEE bit pattern:
    keep the top 7 of the 52 stored mantissa bits, round on the 45 dropped ones.  Normal
    numbers only (the glue's values are O(1))."""
    a = np.asarray(a, np.float64)
    u = a.view(np.uint64)
    lsb = (u >> np.uint64(45)) & np.uint64(1)
    u = (u + np.uint64((1 << 44) - 1) + lsb) & ~np.uint64((1 << 45) - 1)
    return u.view(np.float64)


def test_decoder_layer_routing_against_dense_composition():
    """decoder_layer_forward against an independently written composition of the chained
    layer: each linear is the explicit dense matrix S_o H_o W_v H_i S_i (scipy's Hadamard
    blocks, W_v dequantised by hand), each glue the unit-RMS rescale per token followed by
    a bit-level bf16 rounding.  q, k, v read x; o reads glue(q); gate and up read glue(o);
    down reads glue(gate * up); the next layer reads glue(down).  Distinct widths (hidden
    256, q 128, intermediate 384) and the mis-routed variants checked at the end make a
    wrong routing fail."""
    hidden, qd, kvd, inter, bits = 256, 128, 128, 384, 8
    shapes = {"q": (qd, hidden), "k": (kvd, hidden), "v": (kvd, hidden), "o": (hidden, qd),
              "gate": (inter, hidden), "up": (inter, hidden), "down": (hidden, inter)}
    lin = {}
    for i, (n, (M, K)) in enumerate(shapes.items()):
        W = synth.weights(M, K, 940 + i, "entries")
        s_o, s_i = synth.sign_pair(M, K, 960 + 2 * i)
        lin[n] = (O.quantize_layer(W, s_o, s_i, bits), s_o, s_i)
    _, x = synth.activations(3, hidden, 980)
    lv = np.array([-1.5104, -0.4528, 0.4528, 1.5104])

    def dense(n, verify):
        q, s_o, s_i = lin[n]
        M, K = shapes[n]
        sb = np.repeat(q["base_scales"].astype(np.float64), 128, axis=1)
        Wv = lv[q["base_codes"]] * sb
        if verify:
            Wv = Wv + q["resid_codes"].astype(np.float64) * np.repeat(q["resid_scales"].astype(np.float64), 128, axis=1)
        return np.diag(s_o.astype(np.float64)) @ _dense_blockdiag(M) @ Wv @ _dense_blockdiag(K) @ np.diag(
            s_i.astype(np.float64))

    def glue(h):
        rms = np.sqrt(np.sum(h * h, axis=1, keepdims=True) / h.shape[1])
        return _bf16_bits(h / rms)

    for verify in (False, True):
        Wd = {n: dense(n, verify) for n in shapes}
        f = lambda n, xin: xin @ Wd[n].T
        ref = {n: f(n, x) for n in ("q", "k", "v")}
        ref["o"] = f("o", glue(ref["q"]))
        xg = glue(ref["o"])
        ref["gate"], ref["up"] = f("gate", xg), f("up", xg)
        ref["down"] = f("down", glue(ref["gate"] * ref["up"]))
        ref["next"] = glue(ref["down"])
        got = O.decoder_layer_forward(lin, x, verify)
        for n in ref:
            assert got[n].shape == ref[n].shape, n
            assert np.allclose(got[n], ref[n], rtol=1e-9, atol=1e-12), n
        # the composition has the power to see a mis-routed layer
        wrong_down = f("down", glue(ref["gate"]))                    # down reading gate alone
        assert not np.allclose(got["down"], wrong_down, rtol=1e-3, atol=1e-6)
        wrong_up = f("up", glue(f("o", glue(ref["k"]))))             # o reading k instead of q
        assert not np.allclose(got["up"], wrong_up, rtol=1e-3, atol=1e-6)
