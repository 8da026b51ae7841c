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


def bf16_values(u16):
    """bf16 bit patterns -> float64 values."""
    return (np.asarray(u16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def assert_quant_follows_plain(oracle, Yk, Yp, qk, sk, qp, sp, group, max_frac=2e-3, err_bound=None,
                               max_frac_beyond_ulp=0.0):
    """Tolerance check of a fused "bf16 value, then quantization" kernel
    against the plain-definition oracle.

    Yk, Yp: the kernel's and the plain oracle's bf16 values (uint16 [M, K]);
    qk / qp: their int8 codes [M, K]; sk / sp: fp32 scales [M, K / group]
    (group = K for per-token scales, 128 for 1x128 blocks).
      - every bf16 value within 1 ulp, or, where err_bound (an array of
        absolute error bounds of the kernel's arithmetic, same shape) is
        given, within that bound; at most max_frac of the values differ at
        all and at most max_frac_beyond_ulp by more than 1 ulp;
      - the kernel's codes and scales are the plain quantization of the
        kernel's own bf16 values, bit for bit;
      - where a group's bf16 inputs are identical on both sides, its codes
        and scale are identical too; where only some differ and the scale is
        the same, the codes of the identical values are identical.
    Returns the number of groups with any differing value."""
    Yk = np.asarray(Yk)
    Yp = np.asarray(Yp)
    M, K = Yk.shape
    d = bf16_ulp_distance(Yk, Yp)
    beyond = d > 1
    if err_bound is not None:
        within = np.abs(bf16_values(Yk) - bf16_values(Yp)) <= np.asarray(err_bound)
        assert np.all(within | ~beyond), f"{(beyond & ~within).sum()} values beyond 1 ulp and the error bound"
        assert beyond.sum() <= max(1, max_frac_beyond_ulp * d.size), f"{beyond.sum()} values beyond 1 ulp"
    else:
        assert d.max(initial=0) <= 1, f"max bf16 ulp distance {d.max()}"
    assert (d > 0).sum() <= max(2, max_frac * d.size), f"{(d > 0).sum()} of {d.size} values differ"
    mode = oracle.PER_ROW if group == K else oracle.BLOCK
    q2, s2 = oracle.quantize_act(Yk, mode)
    assert np.array_equal(qk, q2), "codes are not the quantization of the kernel's values"
    assert np.array_equal(np.asarray(sk).view(np.uint32).reshape(s2.shape), s2.view(np.uint32)), \
        "scales are not those of the kernel's values"
    G = K // group
    same_val = (d == 0).reshape(M, G, group)
    same_group = same_val.all(axis=2)
    sk_ = np.asarray(sk).reshape(M, G).view(np.uint32)
    sp_ = np.asarray(sp).reshape(M, G).view(np.uint32)
    assert np.array_equal(sk_[same_group], sp_[same_group])
    qk3 = np.asarray(qk).reshape(M, G, group)
    qp3 = np.asarray(qp).reshape(M, G, group)
    same_scale = (sk_ == sp_)[:, :, None]
    mask = same_val & same_scale
    assert np.array_equal(qk3[mask], qp3[mask])
    return int((~same_group).sum())


def norm_error_bound(X, gamma, beta, eps, layer):
    """Absolute error bound of a binary32 evaluation of RMSNorm / LayerNorm
    whose statistics are sums of at most L = 7 + log2(K / 8) rounded
    additions per element (8-element chunks, then a pairwise tree), against
    the exact value (first order in u = 2^-24):
      mean:      |d mu| <= L u mean|x| + u |mu|
      x - mu:    |d d|  <= |d mu| + u |x - mu|
      variance:  relative L u + 4 u (the mean's error enters at second
                 order, sum (x - mu) = 0), so r = 1/sqrt(v + eps) within
                 (L / 2 + 3) u,
      y = ((d r) g) + b:  |d y| <= r |g| |d mu| + (L / 2 + 6) u |d r g| + u |y|.
    Returned doubled for the rounding of y to bf16 and of the plain value."""
    u = 2.0 ** -24
    x = bf16_values(X)
    K = x.shape[1]
    L = 7 + int(np.ceil(np.log2(max(1, K // 8))))
    mu = x.mean(axis=1, keepdims=True) if layer else np.zeros((x.shape[0], 1))
    d = x - mu
    r = 1.0 / np.sqrt((d * d).mean(axis=1, keepdims=True) + float(np.float32(eps)))
    g = np.ones(K) if gamma is None else bf16_values(gamma)
    b = np.zeros(K) if beta is None else bf16_values(beta)
    y = d * r * g + b
    dmu = L * u * np.abs(x).mean(axis=1, keepdims=True) + u * np.abs(mu)
    return 2.0 * (r * np.abs(g) * dmu + (L / 2 + 6) * u * np.abs(d * r * g) + u * np.abs(y))
