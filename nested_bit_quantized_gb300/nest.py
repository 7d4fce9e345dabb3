"""Python binding of libnest (include/nest.h): argument marshalling only.

Every step runs in the CUDA library; this module only checks tensor
properties, passes ``data_ptr()`` values and the current CUDA stream through
ctypes, and turns status codes into exceptions.  PyTorch is used for device
memory and streams.  There is no CPU path: if the library is not built, or
the device is not sm_103a, the calls raise.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass, field
from typing import Optional

import torch

from . import build as _build

_P, _I32, _SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t

STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "misaligned", 4: "CUDA error", 5: "timeout"}


class NestError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {STATUS.get(status, status)} (status {status})")
        self.status = status


CODEC_L2, CODEC_W4W8 = 0, 1     # nest_layer.codec (include/nest.h)


class _KvCache(ctypes.Structure):
    _fields_ = [("base", _P), ("ref", _P), ("scale", _P), ("H", _I32), ("Lmax", _I32)]


class _Layer(ctypes.Structure):
    _fields_ = [("M", _I32), ("K", _I32), ("resid_bits", _I32),
                ("base", _P), ("resid", _P), ("sign_out", _P), ("sign_in", _P), ("codec", _I32), ("group", _I32)]


class RotateTask(ctypes.Structure):
    """nest_rotate_task: one set of vectors of a grouped rotation."""
    _fields_ = [("x", _P), ("signs", _P), ("n", _I32), ("y", _P), ("x_op", _P), ("zero_out", _P),
                ("zero_count", ctypes.c_int64)]


_lib = None


def library_path() -> str:
    return _build.LIB


def load() -> ctypes.CDLL:
    """Load the built library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_build.LIB):
        raise RuntimeError(f"libnest is not built ({_build.LIB} missing); run nested_bit_quantized_gb300.build.build()")
    lib = ctypes.CDLL(_build.LIB)
    sig = {
        "nest_status_string": ([_I32], ctypes.c_char_p),
        "nest_hadamard_block": ([_I32], _I32),
        "nest_base_bytes": ([_I32, _I32], _SZ),
        "nest_resid_bytes": ([_I32, _I32, _I32], _SZ),
        "nest_xop_bytes": ([_I32, _I32], _SZ),
        "nest_linear_scratch_bytes": ([_I32, _I32, _I32], _SZ),
        "nest_quantize": ([_P, _P, _P, _I32, _I32, _I32, _P, _P, _P, _P, _P, _P], _I32),
        "nest_pack": ([_P, _P, _P, _P, _I32, _I32, _I32, _P, _P, _P], _I32),
        "nest_unpack": ([ctypes.POINTER(_Layer), _P, _P, _P, _P, _P], _I32),
        "nest_rotate": ([_P, _I32, _P, _I32, _I32, _I32, _P, _P, _P], _I32),
        "nest_draft_gemv": ([ctypes.POINTER(_Layer), _P, _P, _I32, _P], _I32),
        "nest_verify_gemm": ([ctypes.POINTER(_Layer), _P, _P, _I32, _P], _I32),
        "nest_linear": ([ctypes.POINTER(_Layer), _I32, _P, _I32, _I32, _P, _P, _P], _I32),
        "nest_draft_gemv_group": ([ctypes.POINTER(_Layer), _I32, ctypes.POINTER(_P), ctypes.POINTER(_P), _I32, _P], _I32),
        "nest_verify_gemm_group": ([ctypes.POINTER(_Layer), _I32, ctypes.POINTER(_P), ctypes.POINTER(_P), _I32, _P], _I32),
        "nest_linear_group_scratch_bytes": ([ctypes.POINTER(_Layer), _I32, _I32], _SZ),
        "nest_linear_group": ([ctypes.POINTER(_Layer), _I32, _I32, ctypes.POINTER(_P), _I32, _I32,
                               ctypes.POINTER(_P), _P, _P], _I32),
        "nest_chain_work_bytes": ([_I32, _I32], _SZ),
        "nest_w4_base_bytes": ([_I32, _I32], _SZ),
        "nest_w4_ref_bytes": ([_I32, _I32], _SZ),
        "nest_quantize_w4w8": ([_P, _P, _P, _I32, _I32, _P, _P, _P, _P, _P], _I32),
        "nest_pack_w4w8": ([_P, _P, _P, _I32, _I32, _P, _P, _P], _I32),
        "nest_unpack_w4w8": ([ctypes.POINTER(_Layer), _P, _P, _P, _P], _I32),
        "nest_chain": ([_P, _P, _P, _P, _I32, _I32, _P, ctypes.POINTER(_Layer), _I32, ctypes.POINTER(_P),
                        ctypes.POINTER(_P), _P, ctypes.POINTER(RotateTask), _I32, _P], _I32),
        "nest_rotate_group": ([ctypes.POINTER(RotateTask), _I32, _I32, _I32, _I32, _P], _I32),
        "nest_kv_plane_bytes": ([_I32, _I32], _SZ),
        "nest_kv_write": ([_P, _I32, _I32, ctypes.POINTER(_KvCache), _I32, _P], _I32),
        "nest_kv_attention_work_bytes": ([_I32, _I32, _I32, _I32], _SZ),
        "nest_kv_attention": ([_P, _I32, _I32, _I32, ctypes.POINTER(_KvCache), ctypes.POINTER(_KvCache), _I32, _I32,
                               _I32, _P, _P, _P], _I32),
        "nest_shard_gather": ([_P, _P, _I32, _I32, _I32, _I32, _P], _I32),
        "nest_operand": ([_P, _I32, _I32, _P, _P], _I32),
        "nest_error_check": ([_P], _I32),
        "nest_wait_selftest": ([_I32, _P], _I32),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes, fn.restype = args, res
    _lib = lib
    return lib


def _check(st: int, what: str):
    if st != 0:
        raise NestError(st, what)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dev(t: torch.Tensor, dtype, name: str):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _buf(t, name: str, nbytes: int = 0, dtype=None):
    """Check a tensor whose pointer goes to the library: contiguous, of `dtype` when given,
    at least `nbytes` bytes, on the device.  The library sees only the pointer, so a short
    or host buffer would be read or written out of bounds by a kernel.  The size is checked
    before the device, so the checks can be exercised without a GPU."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    have = t.numel() * t.element_size()
    if have < nbytes:
        raise ValueError(f"{name} holds {have} bytes, needs {nbytes}")
    _require_cuda(t, name)
    return t


def _require_cuda(t: torch.Tensor, name: str):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")


def _act(x, name: str, T: int, K: int):
    """An activation block [T][K] of bf16 or fp32; returns the library's dtype code."""
    if not isinstance(x, torch.Tensor) or x.dim() != 2 or x.shape[0] != T or x.shape[1] != K:
        raise ValueError(f"{name} must be a [{T}][{K}] tensor, got {tuple(getattr(x, 'shape', ()))}")
    if x.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError(f"{name} must be float32 or bfloat16")
    _buf(x, name)
    return 1 if x.dtype == torch.bfloat16 else 0


# ---------------------------------------------------------------------------
# sizes
# ---------------------------------------------------------------------------

def hadamard_block(n: int) -> int:
    return int(load().nest_hadamard_block(n))


def base_bytes(M: int, K: int) -> int:
    return int(load().nest_base_bytes(M, K))


def resid_bytes(M: int, K: int, bits: int) -> int:
    return int(load().nest_resid_bytes(M, K, bits))


def xop_bytes(K: int, T: int) -> int:
    return int(load().nest_xop_bytes(K, T))


def linear_scratch_bytes(M: int, K: int, T: int) -> int:
    return int(load().nest_linear_scratch_bytes(M, K, T))


def _u8(n: int, device) -> torch.Tensor:
    # 16-byte aligned byte buffer (the caching allocator returns 512-byte aligned blocks)
    return torch.empty(max(n, 16), dtype=torch.uint8, device=device)


# ---------------------------------------------------------------------------
# offline: quantize, pack, unpack
# ---------------------------------------------------------------------------

def quantize(W: torch.Tensor, sign_out: torch.Tensor, sign_in: torch.Tensor, bits: int,
             work: Optional[torch.Tensor] = None, stream=None) -> dict:
    """RTN quantizer on the device (nest_quantize).  Returns codes and fp16 scale bits."""
    _dev(W, torch.float32, "W")
    M, K = W.shape
    _buf(sign_out, "sign_out", M, torch.int8)
    _buf(sign_in, "sign_in", K, torch.int8)
    dev = W.device
    if work is None:
        work = torch.empty((M, K), dtype=torch.float64, device=dev)
    _buf(work, "work", 8 * M * K, torch.float64)
    out = {
        "base_codes": torch.empty((M, K), dtype=torch.uint8, device=dev),
        "base_scales": torch.empty((M, K // 128), dtype=torch.int16, device=dev),
        "resid_codes": torch.empty((M, K), dtype=torch.int8, device=dev) if bits else None,
        "resid_scales": torch.empty((M, K // 128), dtype=torch.int16, device=dev) if bits else None,
    }
    st = load().nest_quantize(_ptr(W), _ptr(sign_out), _ptr(sign_in), M, K, bits, _ptr(work),
                              _ptr(out["base_codes"]), _ptr(out["base_scales"]),
                              _ptr(out["resid_codes"]), _ptr(out["resid_scales"]), _stream(stream))
    _check(st, "nest_quantize")
    return out


@dataclass
class Layer:
    """A packed layer resident on the device (owns its buffers)."""
    M: int
    K: int
    bits: int
    base: torch.Tensor
    resid: Optional[torch.Tensor]
    sign_out: torch.Tensor
    sign_in: torch.Tensor
    codec: int = CODEC_L2
    _cs: Optional[_Layer] = field(default=None, init=False, repr=False, compare=False)

    def c_struct(self) -> _Layer:
        """The C descriptor (built once: the layer's buffers do not move)."""
        if self._cs is None:
            self._cs = _Layer(self.M, self.K, self.bits, self.base.data_ptr(),
                              self.resid.data_ptr() if self.resid is not None else None,
                              self.sign_out.data_ptr(), self.sign_in.data_ptr(), self.codec, 128)
        return self._cs

    @property
    def weight_bytes(self) -> int:
        return self.base.numel() + (self.resid.numel() if self.resid is not None else 0)


def pack(base_codes: torch.Tensor, base_scales: torch.Tensor, resid_codes: Optional[torch.Tensor],
         resid_scales: Optional[torch.Tensor], bits: int, sign_out: torch.Tensor, sign_in: torch.Tensor,
         stream=None) -> Layer:
    """Pack device codes/scales into the unit format (nest_pack)."""
    _dev(base_codes, torch.uint8, "base_codes")
    M, K = base_codes.shape
    _buf(base_scales, "base_scales", 2 * M * (K // 128))
    if bits:
        _buf(resid_codes, "resid_codes", M * K)
        _buf(resid_scales, "resid_scales", 2 * M * (K // 128))
    _buf(sign_out, "sign_out", M, torch.int8)
    _buf(sign_in, "sign_in", K, torch.int8)
    dev = base_codes.device
    base = _u8(base_bytes(M, K), dev)
    resid = _u8(resid_bytes(M, K, bits), dev) if bits else None
    st = load().nest_pack(_ptr(base_codes), _ptr(base_scales), _ptr(resid_codes), _ptr(resid_scales),
                          M, K, bits, _ptr(base), _ptr(resid), _stream(stream))
    _check(st, "nest_pack")
    return Layer(M, K, bits, base, resid, sign_out, sign_in)


def quantize_w4w8(W: torch.Tensor, sign_out: torch.Tensor, sign_in: torch.Tensor, refine: bool = True,
                  work: Optional[torch.Tensor] = None, stream=None) -> dict:
    """BitNest W4/W8 quantizer on the device (nest_quantize_w4w8): q4, s4 (fp16 bits), q_r."""
    _dev(W, torch.float32, "W")
    M, K = W.shape
    _buf(sign_out, "sign_out", M, torch.int8)
    _buf(sign_in, "sign_in", K, torch.int8)
    dev = W.device
    if work is None:
        work = torch.empty((M, K), dtype=torch.float64, device=dev)
    _buf(work, "work", 8 * M * K, torch.float64)
    out = {"q4": torch.empty((M, K), dtype=torch.int8, device=dev),
           "s4": torch.empty((M, K // 128), dtype=torch.int16, device=dev),
           "qr": torch.empty((M, K), dtype=torch.int8, device=dev) if refine else None}
    st = load().nest_quantize_w4w8(_ptr(W), _ptr(sign_out), _ptr(sign_in), M, K, _ptr(work), _ptr(out["q4"]),
                                   _ptr(out["s4"]), _ptr(out["qr"]), _stream(stream))
    _check(st, "nest_quantize_w4w8")
    return out


def pack_w4w8(q4: torch.Tensor, s4: torch.Tensor, qr: Optional[torch.Tensor], sign_out: torch.Tensor,
              sign_in: torch.Tensor, stream=None) -> Layer:
    """Dual-plane packing (nest_pack_w4w8); a layer of codec W4W8 (resid_bits 4, or 0 without q_r)."""
    _dev(q4, torch.int8, "q4")
    M, K = q4.shape
    _buf(s4, "s4", 2 * M * (K // 128))
    if qr is not None:
        _buf(qr, "qr", M * K)
    _buf(sign_out, "sign_out", M, torch.int8)
    _buf(sign_in, "sign_in", K, torch.int8)
    dev = q4.device
    lib = load()
    base = _u8(int(lib.nest_w4_base_bytes(M, K)), dev)
    ref = _u8(int(lib.nest_w4_ref_bytes(M, K)), dev) if qr is not None else None
    st = lib.nest_pack_w4w8(_ptr(q4), _ptr(s4), _ptr(qr), M, K, _ptr(base), _ptr(ref), _stream(stream))
    _check(st, "nest_pack_w4w8")
    return Layer(M, K, 4 if qr is not None else 0, base, ref, sign_out, sign_in, CODEC_W4W8)


def unpack_w4w8(layer: Layer, stream=None) -> dict:
    """Inverse of pack_w4w8 (nest_unpack_w4w8)."""
    dev = layer.base.device
    out = {"q4": torch.empty((layer.M, layer.K), dtype=torch.int8, device=dev),
           "s4": torch.empty((layer.M, layer.K // 128), dtype=torch.int16, device=dev),
           "qr": torch.empty((layer.M, layer.K), dtype=torch.int8, device=dev) if layer.resid is not None else None}
    L = layer.c_struct()
    st = load().nest_unpack_w4w8(ctypes.byref(L), _ptr(out["q4"]), _ptr(out["s4"]), _ptr(out["qr"]),
                                 _stream(stream))
    _check(st, "nest_unpack_w4w8")
    return out


def unpack(layer: Layer, stream=None) -> dict:
    M, K, dev = layer.M, layer.K, layer.base.device
    out = {
        "base_codes": torch.empty((M, K), dtype=torch.uint8, device=dev),
        "base_scales": torch.empty((M, K // 128), dtype=torch.int16, device=dev),
        "resid_codes": torch.empty((M, K), dtype=torch.int8, device=dev) if layer.bits else None,
        "resid_scales": torch.empty((M, K // 128), dtype=torch.int16, device=dev) if layer.bits else None,
    }
    L = layer.c_struct()
    st = load().nest_unpack(ctypes.byref(L), _ptr(out["base_codes"]), _ptr(out["base_scales"]),
                            _ptr(out["resid_codes"]), _ptr(out["resid_scales"]), _stream(stream))
    _check(st, "nest_unpack")
    return out


def quantize_and_pack(W: torch.Tensor, sign_out: torch.Tensor, sign_in: torch.Tensor, bits: int,
                      stream=None) -> Layer:
    q = quantize(W, sign_out, sign_in, bits, stream=stream)
    return pack(q["base_codes"], q["base_scales"], q["resid_codes"], q["resid_scales"], bits,
                sign_out, sign_in, stream=stream)


# ---------------------------------------------------------------------------
# forward kernels
# ---------------------------------------------------------------------------

def rotate(x: torch.Tensor, signs: torch.Tensor, mode: int, y: Optional[torch.Tensor] = None,
           x_op: Optional[torch.Tensor] = None, stream=None):
    """nest_rotate: mode 0 -> H S x (optionally into the GEMM operand), mode 1 -> S H x."""
    if not isinstance(x, torch.Tensor) or x.dim() != 2:
        raise ValueError("x must be a [T][n] tensor")
    T, n = x.shape
    dt = _act(x, "x", T, n)
    _rot_bufs(signs, y, x_op, T, n)
    st = load().nest_rotate(_ptr(x), dt, _ptr(signs), n, T, mode, _ptr(y), _ptr(x_op), _stream(stream))
    _check(st, "nest_rotate")
    return y, x_op


def _rot_bufs(signs, y, x_op, T: int, n: int):
    _buf(signs, "signs", n, torch.int8)
    if y is not None:
        _buf(y, "y", 4 * T * n, torch.float32)
    if x_op is not None:
        _buf(x_op, "x_op", xop_bytes(n, T))


def rotate_group(xs, signs, mode: int, ys=None, x_ops=None, zero=None, stream=None):
    """nest_rotate_group: up to 64 rotations (same dtype, T and mode) in one launch.
    xs, signs: lists; ys / x_ops: lists (entries may be None) or None; zero: list of
    fp32 tensors (or None entries) cleared by the same launch."""
    n_t = len(xs)
    ys = ys or [None] * n_t
    x_ops = x_ops or [None] * n_t
    zero = zero or [None] * n_t
    dt = 1 if xs[0].dtype == torch.bfloat16 else 0
    T = xs[0].shape[0]
    arr = (RotateTask * n_t)()
    if not (len(signs) == len(ys) == len(x_ops) == len(zero) == n_t):
        raise ValueError("one sign vector (and output / operand / clear entry) per input")
    for i, (x, s, y, xo, z) in enumerate(zip(xs, signs, ys, x_ops, zero)):
        if x.dtype != xs[0].dtype or x.dim() != 2 or x.shape[0] != T:
            raise ValueError("all inputs of a grouped rotation are [T][n] and share dtype and T")
        _act(x, "x", T, x.shape[1])
        _rot_bufs(s, y, xo, T, x.shape[1])
        if z is not None:
            _buf(z, "zero", 0, torch.float32)
        arr[i] = RotateTask(_ptr(x), _ptr(s), x.shape[1], _ptr(y), _ptr(xo), _ptr(z), 0 if z is None else z.numel())
    st = load().nest_rotate_group(arr, n_t, dt, T, mode, _stream(stream))
    _check(st, "nest_rotate_group")


def operand(x_rot: torch.Tensor, x_op: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """nest_operand: the GEMM operand from an already-rotated fp32 x' [T][K]."""
    if not isinstance(x_rot, torch.Tensor) or x_rot.dim() != 2:
        raise ValueError("x_rot must be a [T][K] tensor")
    T, K = x_rot.shape
    _buf(x_rot, "x_rot", 4 * T * K, torch.float32)
    if x_op is None:
        x_op = new_xop(K, T, x_rot.device)
    _buf(x_op, "x_op", xop_bytes(K, T))
    _check(load().nest_operand(_ptr(x_rot), K, T, _ptr(x_op), _stream(stream)), "nest_operand")
    return x_op


def new_xop(K: int, T: int, device="cuda") -> torch.Tensor:
    return torch.empty(xop_bytes(K, T) // 2, dtype=torch.int16, device=device)


def gemm(layer: Layer, x_op: torch.Tensor, T: int, verify: bool, z: Optional[torch.Tensor] = None,
         stream=None) -> torch.Tensor:
    """nest_verify_gemm (verify=True) or nest_draft_gemv: z [T][M] fp32 in the rotated basis.

    The library ACCUMULATES into z; a new z is zero-filled, a given z is added to."""
    dev = layer.base.device
    _buf(x_op, "x_op", xop_bytes(layer.K, T))
    if z is None:
        z = torch.zeros((T, layer.M), dtype=torch.float32, device=dev)
    _buf(z, "z", 4 * T * layer.M, torch.float32)
    L = layer.c_struct()
    fn = load().nest_verify_gemm if verify else load().nest_draft_gemv
    st = fn(ctypes.byref(L), _ptr(x_op), _ptr(z), T, _stream(stream))
    _check(st, "nest_verify_gemm" if verify else "nest_draft_gemv")
    return z


def linear(layer: Layer, x: torch.Tensor, verify: bool, y: Optional[torch.Tensor] = None,
           scratch: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """nest_linear: y = S_o H_o (Q (H_i S_i x)) for x [T][K] (bf16 or fp32)."""
    T = x.shape[0]
    dt = _act(x, "x", T, layer.K)
    dev = layer.base.device
    if y is None:
        y = torch.empty((T, layer.M), dtype=torch.float32, device=dev)
    _buf(y, "y", 4 * T * layer.M, torch.float32)
    need = linear_scratch_bytes(layer.M, layer.K, T)
    if scratch is None:
        scratch = torch.empty(need, dtype=torch.uint8, device=dev)
    _buf(scratch, "scratch", need)
    L = layer.c_struct()
    st = load().nest_linear(ctypes.byref(L), int(verify), _ptr(x), dt, T, _ptr(y), _ptr(scratch), _stream(stream))
    _check(st, "nest_linear")
    return y


def shard_gather(gathered: torch.Tensor, world: int, T: int, Mp: int, M: int, z: Optional[torch.Tensor] = None,
                 stream=None) -> torch.Tensor:
    """nest_shard_gather: the all-gathered [world][T][Mp] row-shard blocks -> z [T][M]."""
    _buf(gathered, "gathered", 4 * world * T * Mp, torch.float32)
    if z is None:
        z = torch.empty((T, M), dtype=torch.float32, device=gathered.device)
    _buf(z, "z", 4 * T * M, torch.float32)
    _check(load().nest_shard_gather(_ptr(gathered), _ptr(z), world, T, Mp, M, _stream(stream)), "nest_shard_gather")
    return z


def error_check(stream=None) -> None:
    _check(load().nest_error_check(_stream(stream)), "nest_error_check")


def wait_selftest(which: int = 0, stream=None) -> None:
    """Launch the bounded-wait give-up check (nest_wait_selftest) of the GEMM kernels
    (which=0) or of the one-token look-up kernel (which=1); the next error_check raises
    NestError with status 5 (timeout)."""
    _check(load().nest_wait_selftest(int(which), _stream(stream)), "nest_wait_selftest")


# ---------------------------------------------------------------------------
# grouped launches (independent linears in one launch)
# ---------------------------------------------------------------------------

def _layers(layers):
    arr = (_Layer * len(layers))()
    for i, L in enumerate(layers):
        arr[i] = L.c_struct()
    return arr


def _ptrs(ts):
    return (_P * len(ts))(*[t.data_ptr() for t in ts])


def gemm_group(layers, x_ops, T: int, verify: bool, zs=None, stream=None):
    """nest_verify_gemm_group / nest_draft_gemv_group: one launch over up to 64 linears.
    Accumulates into zs (new zs are zero-filled)."""
    dev = layers[0].base.device
    if zs is None:
        zs = [torch.zeros((T, L.M), dtype=torch.float32, device=dev) for L in layers]
    if not (len(x_ops) == len(zs) == len(layers)):
        raise ValueError("one operand and one accumulator per layer")
    for L, xo, z in zip(layers, x_ops, zs):
        _buf(xo, "x_op", xop_bytes(L.K, T))
        _buf(z, "z", 4 * T * L.M, torch.float32)
    arr = _layers(layers)
    fn = load().nest_verify_gemm_group if verify else load().nest_draft_gemv_group
    st = fn(arr, len(layers), _ptrs(x_ops), _ptrs(zs), T, _stream(stream))
    _check(st, "nest_verify_gemm_group" if verify else "nest_draft_gemv_group")
    return zs


def linear_group_scratch_bytes(layers, T: int, arr=None) -> int:
    arr = _layers(layers) if arr is None else arr
    return int(load().nest_linear_group_scratch_bytes(arr, len(layers), T))


def linear_group(layers, xs, verify: bool, ys=None, scratch: Optional[torch.Tensor] = None, stream=None):
    """nest_linear_group: y_k = S_o H_o (Q_k (H_i S_i x_k)) for up to 64 linears in 3 launches."""
    T = xs[0].shape[0]
    dev = layers[0].base.device
    if ys is None:
        ys = [torch.empty((T, L.M), dtype=torch.float32, device=dev) for L in layers]
    if not (len(xs) == len(ys) == len(layers)):
        raise ValueError("one input and one output per layer")
    dt = _act(xs[0], "x", T, layers[0].K)
    for L, x, y in zip(layers, xs, ys):
        if _act(x, "x", T, L.K) != dt:
            raise ValueError("all inputs of a grouped linear share one dtype")
        _buf(y, "y", 4 * T * L.M, torch.float32)
    arr = _layers(layers)
    need = linear_group_scratch_bytes(layers, T, arr)
    if scratch is None:
        scratch = torch.empty(need, dtype=torch.uint8, device=dev)
    _buf(scratch, "scratch", need)
    st = load().nest_linear_group(arr, len(layers), int(verify), _ptrs(xs), dt, T, _ptrs(ys),
                                  _ptr(scratch), _stream(stream))
    _check(st, "nest_linear_group")
    return ys


# ----------------------------------------------------------------------------
# nested KV4/KV8 cache
# ----------------------------------------------------------------------------

class KVCache:
    """One nested cache (keys or values): base and refinement nibble planes and fp16 scales
    for H heads x Lmax positions of dimension 128 (nest_kv_cache)."""

    def __init__(self, H: int, Lmax: int, device="cuda"):
        n = int(load().nest_kv_plane_bytes(H, Lmax))
        if n == 0:
            raise ValueError("bad cache shape")
        self.H, self.Lmax = H, Lmax
        self.base = torch.zeros(n, dtype=torch.uint8, device=device)
        self.ref = torch.zeros(n, dtype=torch.uint8, device=device)
        self.scale = torch.zeros(H * Lmax, dtype=torch.int16, device=device)

    def c_struct(self) -> _KvCache:
        return _KvCache(self.base.data_ptr(), self.ref.data_ptr(), self.scale.data_ptr(), self.H, self.Lmax)


def kv_write(cache: KVCache, x: torch.Tensor, pos0: int, stream=None):
    """nest_kv_write: store x [T][H][128] (fp32 or bf16) at positions pos0 .. pos0+T-1."""
    if x.dim() != 3 or x.shape[1] != cache.H or x.shape[2] != 128:
        raise ValueError(f"x must be [T][{cache.H}][128], got {tuple(x.shape)}")
    if x.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("x must be float32 or bfloat16")
    dt = 1 if x.dtype == torch.bfloat16 else 0
    _buf(x, "x")
    C = cache.c_struct()
    st = load().nest_kv_write(_ptr(x), dt, x.shape[0], ctypes.byref(C), pos0, _stream(stream))
    _check(st, "nest_kv_write")


def kv_attention(q: torch.Tensor, k: KVCache, v: KVCache, L: int, view: int, recent_n: int = 0,
                 out: Optional[torch.Tensor] = None, work: Optional[torch.Tensor] = None, stream=None):
    """nest_kv_attention: q [T][Hq][128] -> out [T][Hq][128] fp32."""
    if q.dim() != 3 or q.shape[2] != 128:
        raise ValueError(f"q must be [T][Hq][128], got {tuple(q.shape)}")
    if q.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("q must be float32 or bfloat16")
    T, Hq, d = q.shape
    dt = 1 if q.dtype == torch.bfloat16 else 0
    _buf(q, "q")
    lib = load()
    if out is None:
        out = torch.empty((T, Hq, d), dtype=torch.float32, device=q.device)
    _buf(out, "out", 4 * T * Hq * d, torch.float32)
    need = int(lib.nest_kv_attention_work_bytes(T, Hq, k.H, L))
    if work is None:
        work = torch.empty(need // 4 + 1, dtype=torch.float32, device=q.device)
    _buf(work, "work", need)
    K, V = k.c_struct(), v.c_struct()
    st = lib.nest_kv_attention(_ptr(q), dt, T, Hq, ctypes.byref(K), ctypes.byref(V), L, view, recent_n, _ptr(out),
                               _ptr(work), _stream(stream))
    _check(st, "nest_kv_attention")
    return out
