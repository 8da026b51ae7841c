"""Shared helpers of the GPU parity tests."""
import numpy as np
import torch


def bits(t):
    """bf16 CUDA/CPU tensor -> numpy uint16 bit patterns."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def bf16_ulp_distance(a, b):
    """Distance in bf16 units in the last place between two bf16 bit arrays,
    with +0 and -0 equal (ordered-integer mapping of the bit patterns)."""
    def ordered(u):
        u = np.asarray(u, np.int32)
        mag = u & 0x7FFF
        return np.where(u & 0x8000, -mag, mag)
    return np.abs(ordered(a) - ordered(b))


def assert_bf16_close(got, want, max_ulp=1):
    d = bf16_ulp_distance(got, want)
    assert d.max(initial=0) <= max_ulp, f"max bf16 ulp distance {d.max()} at {np.unravel_index(d.argmax(), d.shape)}"
    return d


def edge_indices(n, tile, extra, rng):
    """Every first/last index of every `tile`-wide tile, the last index, and
    `extra` random ones."""
    idx = set()
    for t0 in range(0, n, tile):
        idx.add(t0)
        idx.add(min(t0 + tile - 1, n - 1))
    idx.add(n - 1)
    if n > 0:
        idx.update(rng.integers(0, n, extra).tolist())
    return np.array(sorted(idx), dtype=np.int64)
