"""The kernels' bounded waits give up cleanly.

Every pipeline wait of the GEMM kernels (and of the one-token look-up kernel) is
bounded by %globaltimer; when it runs out the kernel raises a device error flag,
returns, and nest_error_check reports
NEST_ERR_TIMEOUT.  nest_wait_selftest runs that wait on a barrier nothing ever
arrives on (no fault, no trap: the wait itself ends), so the give-up path runs
for real.  Afterwards the flag is clear and the same context still computes a
verify GEMM that passes the parity gate against the oracle.
"""
import time

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from nested_bit_quantized_gb300 import nest, synth  # noqa: E402
from oracle import nest_oracle as O  # noqa: E402
from tests.helpers import parity, to_dev  # noqa: E402

pytestmark = pytest.mark.gpu

WAIT_LIMIT_S = 2.0      # the kernels' wait limit


@pytest.fixture(scope="module")
def dev():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


@pytest.mark.parametrize("which", [0, 1])
def test_wait_gives_up_and_context_stays_usable(dev, which):
    """which = 0: the wait of the tensor-core and register-fragment GEMM kernels; 1: the
    wait of the one-token look-up kernel (its own error flag)."""
    nest.error_check()                                   # no flag left over
    torch.cuda.synchronize()
    t0 = time.monotonic()
    nest.wait_selftest(which)
    with pytest.raises(nest.NestError) as err:
        nest.error_check()                               # synchronises
    waited = time.monotonic() - t0
    assert err.value.status == 5                         # NEST_ERR_TIMEOUT
    assert WAIT_LIMIT_S * 0.9 <= waited <= WAIT_LIMIT_S + 30.0, waited
    nest.error_check()                                   # the check cleared the flag

    M, K, bits, T = 256, 512, 7, 16
    W = synth.weights(M, K, 31, "entries")
    s_o, s_i = synth.sign_pair(M, K, 38)
    q = O.quantize_layer(W, s_o, s_i, bits)
    layer = nest.pack(to_dev(q["base_codes"], torch, dev), to_dev(q["base_scales"], torch, dev),
                      to_dev(q["resid_codes"], torch, dev), to_dev(q["resid_scales"], torch, dev), bits,
                      to_dev(s_o, torch, dev), to_dev(s_i, torch, dev))
    xb, xv = synth.activations(T, K, 39)
    x = torch.from_numpy(xb.view(np.int16)).to(dev).view(torch.bfloat16)
    xop = nest.new_xop(K, T, dev)
    nest.rotate(x, layer.sign_in, 0, x_op=xop)
    z = nest.gemm(layer, xop, T, True)
    parity(z.cpu().numpy(), O.forward(q, s_o, s_i, xv, True)["z"])
    # and the one-token draft (the look-up kernel)
    x1 = x[:1].contiguous()
    xop1 = nest.new_xop(K, 1, dev)
    nest.rotate(x1, layer.sign_in, 0, x_op=xop1)
    z1 = nest.gemm(layer, xop1, 1, False)
    parity(z1.cpu().numpy(), O.forward(q, s_o, s_i, xv[:1], False)["z"])
    nest.error_check()
