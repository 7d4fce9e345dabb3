"""nest_linear_static: the whole-linear call that allocates nothing.

Some callers cannot allocate device memory for the linear's intermediate
buffers: processes whose memory pool is fixed at start-up, plain C callers
without an allocator, loops that cannot afford cudaMalloc's implicit
synchronisation.  nest_linear_static keeps those buffers in a fixed array in
the library's own device memory.  This test calls it through the C ABI and
checks that two calls in a row give the result of nest_linear with caller
scratch, within the parity tolerance the other GPU tests use, that a call after
the first changes the device's free memory by nothing, and that shapes whose
buffers exceed the array are refused before any launch.

The file is named so that pytest collects it after every other test.
"""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from nested_bit_quantized_gb300 import nest, synth  # noqa: E402
from oracle import nest_oracle as O  # noqa: E402
from tests.helpers import parity, to_dev  # noqa: E402

pytestmark = pytest.mark.gpu


def _static_fn():
    lib = nest.load()
    fn = lib.nest_linear_static
    fn.argtypes = [ctypes.POINTER(nest._Layer), ctypes.c_int32, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                   ctypes.c_void_p, ctypes.c_void_p]
    fn.restype = ctypes.c_int32
    return fn


def test_static_scratch_linear_matches_caller_scratch_linear():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "this test needs a CUDA device"
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    fn = _static_fn()

    M, K, T, bits = 640, 1536, 16, 7
    W = synth.weights(M, K, 21, "entries")
    s_o, s_i = synth.sign_pair(M, K, 22)
    q = O.quantize_layer(W, s_o, s_i, bits)
    layer = nest.pack(to_dev(q["base_codes"], torch, dev), to_dev(q["base_scales"], torch, dev),
                      to_dev(q["resid_codes"], torch, dev), to_dev(q["resid_scales"], torch, dev), bits,
                      to_dev(s_o, torch, dev), to_dev(s_i, torch, dev))
    xb, _ = synth.activations(T, K, 23)
    x = torch.from_numpy(xb.view(np.int16)).to(dev).view(torch.bfloat16)
    L = layer.c_struct()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    ys = [torch.empty((T, M), dtype=torch.float32, device=dev) for _ in range(2)]
    for verify in (False, True):
        ref = nest.linear(layer, x, verify).cpu().numpy()
        for i, y in enumerate(ys):                             # the second call reuses the array
            y.fill_(float("nan"))
            torch.cuda.synchronize()
            free_before = torch.cuda.mem_get_info(dev)[0]
            st = fn(ctypes.byref(L), int(verify), ctypes.c_void_p(x.data_ptr()), 1, T,
                    ctypes.c_void_p(y.data_ptr()), stream)
            assert st == 0, f"nest_linear_static returned {st}"
            torch.cuda.synchronize()
            if i == 1 or verify:                               # after the first call loaded the module
                assert torch.cuda.mem_get_info(dev)[0] == free_before, "the call changed free device memory"
            parity(y.cpu().numpy(), ref)

    # shapes whose operand + accumulator exceed the fixed array are refused without a launch
    big = nest._Layer(100_000, 4096, 8, layer.base.data_ptr(), layer.resid.data_ptr(),
                      layer.sign_out.data_ptr(), layer.sign_in.data_ptr())
    assert fn(ctypes.byref(big), 1, ctypes.c_void_p(x.data_ptr()), 1, 64, ctypes.c_void_p(ys[0].data_ptr()),
              stream) == 2
    nest.error_check()
