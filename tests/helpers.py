"""Shared test helpers: tensor marshalling, the activation-operand decoder and the parity gate."""
import numpy as np

# parity gate for floating-point outputs: relative L2 <= 1e-3 and every element within 1e-2 * rms(ref)
REL_L2 = 1e-3
ELEM_RMS = 1e-2


def parity(got, ref, rel_l2=REL_L2, elem_rms=ELEM_RMS):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), "non-finite output"
    rms = np.sqrt(np.mean(ref ** 2))
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)
    worst = np.max(np.abs(got - ref)) / max(rms, 1e-300)
    assert rel <= rel_l2 and worst <= elem_rms, f"parity: rel L2 {rel:.3e} (<= {rel_l2}), worst/rms {worst:.3e} (<= {elem_rms})"
    return rel, worst


def to_dev(a, torch, dev):
    """numpy -> torch on device; fp16 arrays travel as their int16 bit patterns."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16 or a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).to(dev)


def n_pad(T):
    return next(n for n in (16, 32, 64, 128, 256) if T <= n)


def decode_xop(buf, K, T):
    """Activation operand bytes -> fp16 array [T][K] (layout of include/nest.h)."""
    Np = n_pad(T)
    NB = Np // 8
    h = np.asarray(buf).view(np.uint8).view(np.float16)
    out = np.zeros((T, K), np.float16)
    for g in range(K // 128):
        blk = h[g * 128 * Np:(g + 1) * 128 * Np]
        for c in range(16):
            for t in range(T):
                off = ((c * NB + t // 8) * 8 + t % 8) * 8
                out[t, g * 128 + 8 * c:g * 128 + 8 * c + 8] = blk[off:off + 8]
    return out
