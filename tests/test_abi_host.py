"""Host-only checks of the C-ABI library: it loads, exports every declared
symbol, computes sizes, and rejects bad arguments before any device work.
No call here touches a GPU (all rejected cases fail validation first)."""
import ctypes
import os
import re

import pytest

from nested_bit_quantized_gb300 import build as nb
from nested_bit_quantized_gb300 import nest
from oracle import pack as P

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    nb.build()
    return nest.load()


def _declared():
    src = open(os.path.join(ROOT, "include", "nest.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(nest_[a-z_0-9]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert len(names) >= 14
    so = ctypes.CDLL(nb.LIB)
    for n in names:
        assert hasattr(so, n), f"{n} declared in nest.h but not exported"


def test_status_strings(lib):
    for s in range(6):
        assert lib.nest_status_string(s)


def test_hadamard_block_sizes(lib):
    for n, b in [(4096, 4096), (8192, 4096), (15360, 1024), (3840, 256), (5376, 256), (7, 1), (96, 32), (0, 0)]:
        assert nest.hadamard_block(n) == b


@pytest.mark.parametrize("M,K,bits", [(128, 128, 8), (200, 256, 7), (77, 384, 6), (9728, 2560, 7), (1, 128, 8)])
def test_sizes_match_reference_packer(lib, M, K, bits):
    assert nest.base_bytes(M, K) == P.base_bytes(M, K)
    assert nest.resid_bytes(M, K, bits) == P.resid_bytes(M, K, bits)


def test_sizes_reject_bad_shapes(lib):
    assert nest.base_bytes(128, 100) == 0
    assert nest.resid_bytes(128, 128, 5) == 0
    assert nest.xop_bytes(128, 257) == 0
    assert nest.xop_bytes(128, 65) == 256 * 128 and nest.xop_bytes(256, 200) == 2 * 256 * 256
    assert nest.xop_bytes(256, 1) == 2 * 256 * 16
    assert nest.xop_bytes(256, 17) == 2 * 256 * 32
    assert nest.linear_scratch_bytes(128, 128, 0) == 0
    assert nest.linear_scratch_bytes(4096, 4096, 16) == nest.xop_bytes(4096, 16) + 16 * 4096 * 4


def _layer(M=256, K=512, bits=8, base=0x10000, resid=0x20000):
    return nest._Layer(M, K, bits, base, resid, 0x30000, 0x40000)


def test_gemm_argument_validation(lib):
    L = _layer()
    ok = ctypes.c_void_p(0x50000)
    f = lib.nest_verify_gemm
    assert f(None, ok, ok, 16, None) == 1                              # null layer
    assert f(ctypes.byref(L), None, ok, 16, None) == 1                 # null operand
    assert f(ctypes.byref(L), ok, ok, 0, None) == 1                    # T < 1
    assert f(ctypes.byref(L), ok, ok, 257, None) == 2                  # T > 256
    assert f(ctypes.byref(_layer(K=200)), ok, ok, 4, None) == 2         # K % 128
    assert f(ctypes.byref(_layer(bits=5)), ok, ok, 4, None) == 2        # bit width
    assert f(ctypes.byref(_layer(bits=0)), ok, ok, 4, None) == 1        # verify needs a residual
    assert f(ctypes.byref(_layer(base=0x10001)), ok, ok, 4, None) == 3  # misaligned base
    assert f(ctypes.byref(L), ctypes.c_void_p(0x50008), ok, 4, None) == 3
    assert f(ctypes.byref(_layer(M=0)), ok, ok, 4, None) == 1
    d = lib.nest_draft_gemv
    assert d(ctypes.byref(_layer(bits=0, resid=0)), ok, ok, 70, None) == 2
    arr = (nest._Layer * 2)(_layer(), _layer(bits=7))
    ptrs = (ctypes.c_void_p * 2)(0x50000, 0x60000)
    g = lib.nest_verify_gemm_group
    assert g(arr, 0, ptrs, ptrs, 4, None) == 1                        # empty group
    assert g(arr, 65, ptrs, ptrs, 4, None) == 2                       # more than 64 linears
    assert g(arr, 2, ptrs, ptrs, 4, None) == 1                        # mixed residual widths
    assert g(None, 2, ptrs, ptrs, 4, None) == 1
    assert d(ctypes.byref(_layer(bits=0, resid=0)), ok, None, 4, None) == 1


def test_rotate_pack_quantize_validation(lib):
    ok = ctypes.c_void_p(0x50000)
    r = lib.nest_rotate
    assert r(None, 1, ok, 128, 4, 0, ok, None, None) == 1
    assert r(ok, 2, ok, 128, 4, 0, ok, None, None) == 1          # dtype
    assert r(ok, 1, ok, 128, 4, 2, ok, None, None) == 1          # mode
    assert r(ok, 1, ok, 128, 4, 0, None, None, None) == 1        # no output
    assert r(ok, 1, ok, 100, 4, 0, None, ok, None) == 2          # operand needs n % 128
    assert r(ok, 1, ok, 128, 257, 0, None, ok, None) == 2        # operand needs T <= 256
    assert r(ok, 1, ok, 128, 4, 1, None, ok, None) == 1          # operand only on the input side
    assert r(ok, 1, ok, 128, 4, 0, None, ctypes.c_void_p(0x50002), None) == 3
    p = lib.nest_pack
    assert p(None, ok, None, None, 128, 128, 0, ok, None, None) == 1
    assert p(ok, ok, None, None, 128, 100, 0, ok, None, None) == 2
    assert p(ok, ok, None, None, 128, 128, 7, ok, None, None) == 1   # residual pointers missing
    assert p(ok, ok, ok, ok, 128, 128, 9, ok, ok, None) == 2
    q = lib.nest_quantize
    assert q(ok, ok, ok, 128, 100, 8, ok, ok, ok, ok, ok, None) == 2
    assert q(ok, ok, ok, 128, 128, 8, ok, ok, ok, None, ok, None) == 1
    assert q(ctypes.c_void_p(0x50004), ok, ok, 128, 128, 8, ok, ok, ok, ok, ok, None) == 3


def test_chain_and_rotate_group_validation(lib):
    ok = ctypes.c_void_p(0x50000)
    # one fp32 partial per (token, 256-element chunk) or per (token, 4096-element segment),
    # whichever is more, rounded up to 256 bytes
    assert lib.nest_chain_work_bytes(5376, 64) == 256 * ((64 * 21 * 4 + 255) // 256)
    assert lib.nest_chain_work_bytes(300, 3) == 256 * ((3 * 2 * 4 + 255) // 256)
    assert lib.nest_chain_work_bytes(21504, 64) == 64 * 6 * 4
    assert lib.nest_chain_work_bytes(100, 257) == 0
    L = nest._Layer(256, 512, 0, 0x50000, None, 0x50000, 0x50000)
    nx = (nest._Layer * 1)(L)
    xo = (ctypes.c_void_p * 1)(0x50000)
    c = lib.nest_chain
    assert c(ok, ok, None, None, 512, 4, None, nx, 1, xo, None, None, None, 0, None) == 1       # work missing
    assert c(ok, ok, ok, None, 512, 4, None, nx, 1, xo, None, ok, None, 0, None) == 1         # partner sign missing
    assert c(ok, ok, ok, ok, 512, 4, None, nx, 1, xo, None, ok, None, 0, None) == 1           # z_b aliases z_a
    assert c(ok, ok, None, None, 512, 257, None, nx, 1, xo, None, ok, None, 0, None) == 2     # T > 256
    assert c(ok, ok, None, None, 640, 4, None, nx, 1, xo, None, ok, None, 0, None) == 1       # next K != M
    assert c(ok, ok, None, None, 500, 4, None, nx, 1, xo, None, ok, None, 0, None) == 2       # operand needs M % 128
    assert c(ok, ok, None, None, 512, 4, None, nx, 4, xo, None, ok, None, 0, None) == 2       # more than 3 next
    assert c(ok, ok, None, None, 512, 4, None, nx, 1, xo, None, ctypes.c_void_p(0x50002), None, 0, None) == 3
    # side output rotations: at most two, plain z -> y tasks on buffers of their own
    R = nest.RotateTask
    sd = lambda *t: (R * len(t))(*t)
    good = R(0x60000, 0x60000, 256, 0x68000, None, None, 0)
    assert c(ok, ok, None, None, 512, 4, None, nx, 1, xo, None, ok, None, 1, None) == 1          # side missing
    assert c(ok, ok, None, None, 512, 4, None, nx, 1, xo, None, ok, sd(good, good, good), 3, None) == 2
    assert c(ok, ok, None, None, 512, 4, None, nx, 1, xo, None, ok,
             sd(R(0x60000, 0x60000, 256, None, None, None, 0)), 1, None) == 1                       # no y
    assert c(ok, ok, None, None, 512, 4, None, nx, 1, xo, None, ok,
             sd(R(0x60000, 0x60000, 256, 0x68000, 0x69000, None, 0)), 1, None) == 1                 # operand
    assert c(ok, ok, None, None, 512, 4, None, nx, 1, xo, None, ok,
             sd(R(0x60000, 0x60000, 256, 0x50000, None, None, 0)), 1, None) == 1                    # y is z_a
    assert c(ok, ok, None, None, 512, 4, None, nx, 1, xo, None, ok, sd(good, good), 2, None) == 1  # overlap
    assert c(ok, ok, None, None, 512, 4, None, nx, 1, xo, None, ok,
             sd(R(0x60000, 0x60000, 256, 0x68002, None, None, 0)), 1, None) == 3                    # misaligned
    T = nest.RotateTask
    one = (T * 1)(T(0x50000, 0x50000, 128, 0x50000, None, None, 0))
    g = lib.nest_rotate_group
    assert g(one, 0, 1, 4, 0, None) == 1
    assert g(one, 65, 1, 4, 0, None) == 2
    assert g(one, 1, 2, 4, 0, None) == 1                                                # dtype
    bad = (T * 1)(T(0x50000, 0x50000, 128, 0x50000, None, None, 16))
    assert g(bad, 1, 1, 4, 0, None) == 1                                                # zero_count without buffer
    opr = (T * 1)(T(0x50000, 0x50000, 100, None, 0x50000, None, 0))
    assert g(opr, 1, 1, 4, 0, None) == 2                                                # operand needs n % 128
    mis = (T * 1)(T(0x50000, 0x50000, 128, None, 0x50008, None, 0))
    assert g(mis, 1, 1, 4, 0, None) == 3


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(nest, "_lib", None)
    monkeypatch.setattr(nest._build, "LIB", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError):
        nest.load()


def test_w4w8_sizes_and_validation(lib):
    for M, K in [(128, 128), (200, 384), (1, 256), (21504, 5376)]:
        assert lib.nest_w4_base_bytes(M, K) == P.w4_bytes(M, K)
        assert lib.nest_w4_ref_bytes(M, K) == P.w4ref_bytes(M, K)
    assert lib.nest_w4_base_bytes(128, 100) == 0
    ok = ctypes.c_void_p(0x50000)
    q = lib.nest_quantize_w4w8
    assert q(None, ok, ok, 128, 128, ok, ok, ok, ok, None) == 1
    assert q(ok, ok, ok, 128, 100, ok, ok, ok, ok, None) == 2
    assert q(ok, ok, ok, 128, 128, ok, ok, ctypes.c_void_p(0x50001), ok, None) == 3
    p = lib.nest_pack_w4w8
    assert p(ok, ok, ok, 128, 128, ok, None, None) == 1              # refinement codes without a plane
    assert p(ok, ok, None, 128, 100, ok, None, None) == 2
    assert p(ok, ok, None, 128, 128, ctypes.c_void_p(0x50008), None, None) == 3
    # layer validation: codec and refinement width
    xo = (ctypes.c_void_p * 1)(0x50000)
    zs = (ctypes.c_void_p * 1)(0x60000)
    bad = (nest._Layer * 1)(nest._Layer(256, 512, 6, 0x50000, 0x50000, 0x30000, 0x40000, nest.CODEC_W4W8))
    assert lib.nest_verify_gemm_group(bad, 1, xo, zs, 4, None) == 2
    nocodec = (nest._Layer * 1)(nest._Layer(256, 512, 4, 0x50000, 0x50000, 0x30000, 0x40000, 7))
    assert lib.nest_draft_gemv_group(nocodec, 1, xo, zs, 4, None) == 2
    noref = (nest._Layer * 1)(nest._Layer(256, 512, 0, 0x50000, None, 0x30000, 0x40000, nest.CODEC_W4W8))
    assert lib.nest_verify_gemm_group(noref, 1, xo, zs, 4, None) == 1
    mixed = (nest._Layer * 2)(nest._Layer(256, 512, 4, 0x50000, 0x50000, 0x30000, 0x40000, nest.CODEC_W4W8),
                              nest._Layer(256, 512, 0, 0x50000, None, 0x30000, 0x40000, nest.CODEC_L2))
    xo2 = (ctypes.c_void_p * 2)(0x50000, 0x50000)
    zs2 = (ctypes.c_void_p * 2)(0x60000, 0x60000)
    assert lib.nest_draft_gemv_group(mixed, 2, xo2, zs2, 4, None) == 1
    u = lib.nest_unpack_w4w8
    assert u(ctypes.byref(nest._Layer(256, 512, 4, 0x50000, 0x50000, 0x30000, 0x40000, nest.CODEC_L2)),
             ok, ok, ok, None) == 1


def test_kv_cache_validation(lib):
    assert lib.nest_kv_plane_bytes(8, 100) == 8 * 100 * 64 and lib.nest_kv_plane_bytes(0, 4) == 0
    C = nest._KvCache(0x50000, 0x60000, 0x70000, 4, 64)
    w = lib.nest_kv_write
    ok = ctypes.c_void_p(0x50000)
    assert w(ok, 0, 8, ctypes.byref(C), 60, None) == 1                    # past Lmax
    assert w(ok, 2, 8, ctypes.byref(C), 0, None) == 1                     # dtype
    assert w(ctypes.c_void_p(0x50002), 0, 8, ctypes.byref(C), 0, None) == 3
    bad = nest._KvCache(0x50008, 0x60000, 0x70000, 4, 64)
    assert w(ok, 0, 8, ctypes.byref(bad), 0, None) == 3
    huge = nest._KvCache(0x50000, 0x60000, 0x70000, 64, 1 << 20)         # a plane of 4 GiB
    assert w(ok, 0, 8, ctypes.byref(huge), 0, None) == 2
    a = lib.nest_kv_attention
    V = nest._KvCache(0x50000, 0x60000, 0x70000, 4, 64)
    assert a(ok, 0, 2, 6, ctypes.byref(C), ctypes.byref(V), 32, 8, 0, ok, ok, None) == 1   # Hq % Hkv
    assert a(ok, 0, 2, 8, ctypes.byref(C), ctypes.byref(V), 32, 5, 0, ok, ok, None) == 1   # view
    assert a(ok, 0, 2, 8, ctypes.byref(C), ctypes.byref(V), 1, 8, 0, ok, ok, None) == 1    # L < T
    assert a(ok, 0, 2, 8, ctypes.byref(C), ctypes.byref(V), 65, 8, 0, ok, ok, None) == 1   # L > Lmax
    assert a(ok, 0, 2, 8, ctypes.byref(C), ctypes.byref(V), 32, 4, -1, ok, ok, None) == 1  # recent_n


def test_shard_gather_rejects_bad_arguments(lib):
    """Validation before any device work: null pointers, sizes, a layout that cannot hold M rows."""
    p = ctypes.c_void_p(16)
    assert lib.nest_shard_gather(None, p, 2, 1, 128, 200, None) == 1
    assert lib.nest_shard_gather(p, None, 2, 1, 128, 200, None) == 1
    assert lib.nest_shard_gather(p, p, 0, 1, 128, 200, None) == 1
    assert lib.nest_shard_gather(p, p, 2, 0, 128, 200, None) == 1
    assert lib.nest_shard_gather(p, p, 1, 1, 128, 200, None) == 1          # 1 x 128 < 200 rows
    assert lib.nest_shard_gather(p, p, 1 << 12, 1 << 10, 1 << 10, 200, None) == 2
    assert lib.nest_shard_gather(ctypes.c_void_p(18), p, 2, 1, 128, 200, None) == 3


def test_operand_rejects_bad_arguments(lib):
    p = ctypes.c_void_p(16)
    assert lib.nest_operand(None, 128, 1, p, None) == 1
    assert lib.nest_operand(p, 128, 0, p, None) == 1
    assert lib.nest_operand(p, 100, 1, p, None) == 2          # K % 128
    assert lib.nest_operand(p, 128, 257, p, None) == 2        # T > 256
    assert lib.nest_operand(p, 128, 1, ctypes.c_void_p(24), None) == 3


def test_group_other_than_128_is_refused(lib):
    """The descriptor's group: 0 or 128 pass validation, any other size is refused before a launch
    (the storage format has one group size, 128 columns)."""
    z = ctypes.c_void_p(0x60000)
    xop = ctypes.c_void_p(0x50000)
    for g in (8, 64, 256, -1):
        L = nest._Layer(256, 512, 8, 0x10000, 0x20000, 0x30000, 0x40000, 0, g)
        assert lib.nest_verify_gemm(ctypes.byref(L), xop, z, 4, None) == 2
        assert lib.nest_draft_gemv(ctypes.byref(L), xop, z, 4, None) == 2
    bad = (nest._Layer * 1)(nest._Layer(256, 512, 8, 0x10000, 0x20000, 0x30000, 0x40000, 0, 32))
    assert lib.nest_chain(z, ctypes.c_void_p(0x30000), None, None, 512, 1, None, bad, 1,
                          (nest._P * 1)(0x70000), None, z, None, 0, None) == 2


def test_wait_selftest_rejects_unknown_kernel_family(lib):
    # 0 (GEMM kernels) and 1 (look-up kernel) launch; anything else is refused before any launch
    for which in (-1, 2, 7):
        assert lib.nest_wait_selftest(which, None) == 1
