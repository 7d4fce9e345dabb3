"""ctypes front end of the reference packer in ``pack_ref.c``.  TEST INFRASTRUCTURE.

``build()`` compiles the C file with the host gcc into ``oracle/_build``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pack_ref.c")
_OUT = os.path.join(_HERE, "_build", "libpackref.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile pack_ref.c into a shared library (plain C, portable flags)."""
    if force or not os.path.exists(_OUT) or os.path.getmtime(_OUT) < os.path.getmtime(_SRC):
        os.makedirs(os.path.dirname(_OUT), exist_ok=True)
        tmp = _OUT + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", _SRC, "-o", tmp])
        os.replace(tmp, _OUT)
    return _OUT


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        lib.ref_base_bytes.argtypes, lib.ref_base_bytes.restype = [I, I], S
        lib.ref_resid_bytes.argtypes, lib.ref_resid_bytes.restype = [I, I, I], S
        lib.ref_pack_base.argtypes, lib.ref_pack_base.restype = [P, P, I, I, P], None
        lib.ref_unpack_base.argtypes, lib.ref_unpack_base.restype = [P, I, I, P, P], None
        lib.ref_pack_resid.argtypes, lib.ref_pack_resid.restype = [P, P, I, I, I, P], I
        lib.ref_unpack_resid.argtypes, lib.ref_unpack_resid.restype = [P, I, I, I, P, P], I
        lib.ref_w4_bytes.argtypes, lib.ref_w4_bytes.restype = [I, I], S
        lib.ref_w4ref_bytes.argtypes, lib.ref_w4ref_bytes.restype = [I, I], S
        lib.ref_pack_w4w8.argtypes, lib.ref_pack_w4w8.restype = [P, P, P, I, I, P, P], None
        lib.ref_unpack_w4w8.argtypes, lib.ref_unpack_w4w8.restype = [P, P, I, I, P, P, P], None
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def base_bytes(M: int, K: int) -> int:
    return int(_load().ref_base_bytes(M, K))


def resid_bytes(M: int, K: int, bits: int) -> int:
    return int(_load().ref_resid_bytes(M, K, bits))


def pack_base(codes: np.ndarray, scales16: np.ndarray) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    sc = np.ascontiguousarray(np.asarray(scales16).view(np.uint16))
    M, K = codes.shape
    out = np.empty(base_bytes(M, K), dtype=np.uint8)
    _load().ref_pack_base(_ptr(codes), _ptr(sc), M, K, _ptr(out))
    return out


def unpack_base(packed: np.ndarray, M: int, K: int):
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    codes = np.zeros((M, K), dtype=np.uint8)
    sc = np.zeros((M, K // 128), dtype=np.uint16)
    _load().ref_unpack_base(_ptr(packed), M, K, _ptr(codes), _ptr(sc))
    return codes, sc


def pack_resid(codes: np.ndarray, scales16: np.ndarray, bits: int) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.int8)
    sc = np.ascontiguousarray(np.asarray(scales16).view(np.uint16))
    M, K = codes.shape
    out = np.empty(resid_bytes(M, K, bits), dtype=np.uint8)
    if _load().ref_pack_resid(_ptr(codes), _ptr(sc), M, K, bits, _ptr(out)):
        raise ValueError("bits must be 6, 7 or 8")
    return out


def unpack_resid(packed: np.ndarray, M: int, K: int, bits: int):
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    codes = np.zeros((M, K), dtype=np.int8)
    sc = np.zeros((M, K // 128), dtype=np.uint16)
    if _load().ref_unpack_resid(_ptr(packed), M, K, bits, _ptr(codes), _ptr(sc)):
        raise ValueError("bits must be 6, 7 or 8")
    return codes, sc


def w4_bytes(M: int, K: int) -> int:
    return int(_load().ref_w4_bytes(M, K))


def w4ref_bytes(M: int, K: int) -> int:
    return int(_load().ref_w4ref_bytes(M, K))


def pack_w4w8(q4: np.ndarray, s4: np.ndarray, qr: np.ndarray | None):
    """Dual-plane W4/W8 packing: returns (base plane bytes, refinement plane bytes or None)."""
    q4 = np.ascontiguousarray(q4, dtype=np.int8)
    sc = np.ascontiguousarray(np.asarray(s4).view(np.uint16))
    M, K = q4.shape
    base = np.empty(w4_bytes(M, K), dtype=np.uint8)
    ref = None
    qrp = None
    if qr is not None:
        qrp = np.ascontiguousarray(qr, dtype=np.int8)
        ref = np.empty(w4ref_bytes(M, K), dtype=np.uint8)
    _load().ref_pack_w4w8(_ptr(q4), _ptr(sc), _ptr(qrp) if qrp is not None else None, M, K, _ptr(base),
                          _ptr(ref) if ref is not None else None)
    return base, ref


def unpack_w4w8(base: np.ndarray, ref: np.ndarray | None, M: int, K: int):
    base = np.ascontiguousarray(base, dtype=np.uint8)
    q4 = np.zeros((M, K), dtype=np.int8)
    qr = np.zeros((M, K), dtype=np.int8)
    sc = np.zeros((M, K // 128), dtype=np.uint16)
    refp = np.ascontiguousarray(ref, dtype=np.uint8) if ref is not None else None
    _load().ref_unpack_w4w8(_ptr(base), _ptr(refp) if refp is not None else None, M, K, _ptr(q4), _ptr(sc),
                            _ptr(qr))
    return q4, sc, (qr if ref is not None else None)
