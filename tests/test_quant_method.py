"""Checks, without a GPU, the arithmetic identities the CUDA quantizer relies
on to avoid a division per scale (no CUDA code is imported here).

For a bf16 absmax a = M * 2^k (8-bit significand M in [128, 255]), scaling by
a power of two commutes with rounding while the result stays normal, so
    fl32(a / 127)     == fl32(M / 127) * 2^k
    fl32(1 / s)       == fl32(1 / fl32(M / 127)) * 2^-k.
The kernels use two 128-entry tables of fl32(M / 127) and its reciprocal for
exponent fields 8..250 and IEEE division elsewhere."""
import numpy as np


def test_scale_table_identity_exhaustive():
    bits = np.arange(0x0080, 0x7F80, dtype=np.uint32)  # every positive normal finite bf16
    a = (bits << 16).view(np.float32)
    with np.errstate(over="ignore", divide="ignore"):
        s = a / np.float32(127)
        inv = np.float32(1) / s
    f = (bits & 0x7F).astype(np.int64)
    ef = ((bits >> 7) & 0xFF).astype(np.int64)
    T = (np.arange(128, 256, dtype=np.float32) / np.float32(127)).astype(np.float32)
    R = (np.float32(1) / T).astype(np.float32)
    k = ef - 134
    sb = T.view(np.uint32).astype(np.int64)[f] + (k << 23)
    ib = R.view(np.uint32).astype(np.int64)[f] - (k << 23)
    used = (ef >= 8) & (ef <= 250)
    assert used.sum() > 30000
    assert np.array_equal(sb[used].astype(np.uint32), s.view(np.uint32)[used])
    assert np.array_equal(ib[used].astype(np.uint32), inv.view(np.uint32)[used])


def test_fma_rounding_constant():
    """fl(P + 1.5 * 2^23) rounds P to the nearest integer, ties to even, and its
    low byte is that integer in two's complement (|P| < 2^22)."""
    magic = np.float32(12582912.0)
    P = np.array([-127.0, -126.5, -2.5, -1.5, -0.5, 0.0, 0.5, 1.5, 2.5, 3.49, 126.5, 127.0], np.float32)
    big = (P + magic).astype(np.float32)
    low = (big.view(np.uint32) & 0xFF).astype(np.uint8).view(np.int8)
    assert list(low) == [-127, -126, -2, -2, 0, 0, 0, 2, 2, 3, 126, 127]
