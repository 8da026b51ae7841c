"""Pins of the CPU oracle to facts outside itself (no GPU).

Each test ties one oracle function to something it does not compute itself:
hand-derived tie cases, exact rational arithmetic, a library routine for a
special case, a closed form, or brute force on tiny inputs.  A plausible
mistake (a dropped term, a wrong sign or index, a transposed operand, a
multiplication by 127/absmax instead of a division by the scale, a missing
bias, an ascending/descending fold order) fails at least one of them.
"""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

HERE = os.path.dirname(os.path.abspath(__file__))


# ----------------------------------------------------------------- helpers
def f32_exact(z: Fraction) -> Fraction:
    """Round a rational to the nearest binary32 value, ties to even (exact)."""
    if z == 0:
        return Fraction(0)
    sign = -1 if z < 0 else 1
    a = abs(z)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    elif Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, -126)  # subnormals share the exponent of the smallest normal
    ulp = Fraction(2) ** (e - 23)
    m = a / ulp
    r = round(m)  # Fraction.__round__ rounds half to even
    return sign * r * ulp


def q_exact(x: float, s: Fraction) -> int:
    if s == 0:
        return 0
    v = f32_exact(Fraction(x) / s)
    q = round(v)  # half to even
    return max(-127, min(127, q))


def bf16_bits_of(values):
    t = torch.tensor(values, dtype=torch.float32).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bits_to_f32(bits):
    return (np.asarray(bits, np.uint32) << 16).view(np.float32)


def rand_bf16(rng, shape, scale=1.0):
    return bf16_bits_of((rng.standard_normal(shape) * scale).astype(np.float32))


# ----------------------------------------------------------------- bf16 conversion
def test_bf16_round_matches_torch(oracle):
    """bf16 rounding (nearest, ties to even) against torch's conversion."""
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * 100,
        (rng.standard_normal(2000) * 1e-38).astype(np.float32),
        np.array([0.0, -0.0, 1.0, -1.0, 3.4e38, -3.4e38, 1e-45, np.inf, -np.inf], np.float32),
    ])
    # exact halfway cases: low 16 bits == 0x8000, both parities of bit 16
    base = rng.integers(0x3F800000, 0x47000000, 2000, dtype=np.uint32) & 0xFFFF0000
    ties = np.concatenate([base | 0x8000, (base | 0x10000) | 0x8000]).view(np.float32)
    x = np.concatenate([x, ties])
    got = oracle.bf16_from_f32(x)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)
    assert np.array_equal(oracle.f32_from_bf16(got), bits_to_f32(got))


# ----------------------------------------------------------------- quantizer
def load_ties():
    rows = []
    with open(os.path.join(HERE, "golden", "quant_ties.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            a, x, q = line.split()
            rows.append((float(a), float(x), int(q)))
    return rows


def test_quant_hand_ties(oracle):
    cases = load_ties()
    assert len(cases) >= 20
    X = np.zeros((len(cases), 16), np.float32)
    for i, (a, x, _) in enumerate(cases):
        X[i, 0] = a
        X[i, 1] = x
    Xq, sx = oracle.quantize_act(bf16_bits_of(X), oracle.PER_ROW)
    for i, (a, x, q) in enumerate(cases):
        assert sx[i] == np.float32(a) / np.float32(127), (a, sx[i])
        assert Xq[i, 1] == q, (a, x, Xq[i, 1], q)
        assert Xq[i, 0] == 127


def test_quant_matches_exact_rational(oracle):
    """Per-row and 1x128 quantization against exact rational arithmetic:
    s = fl32(absmax/127), q = rne(fl32(x/s)) clamped; includes rows built so
    that many x/s land on or next to half-integers."""
    rng = np.random.default_rng(1)
    rows = [rng.standard_normal(256).astype(np.float32) * 3]
    # s = 1: x = k + 0.5 exact ties and their bf16 neighbours
    t = (np.arange(-120, 120) + 0.5).astype(np.float32)
    rows.append(np.concatenate([[127.0], t, np.zeros(15)]).astype(np.float32))
    # absmax not a nice number: x/s close to half-integers
    a = np.float32(3.7)
    s = np.float32(a / np.float32(127))
    near = ((np.arange(-100, 100) + 0.5) * s).astype(np.float32)
    rows.append(np.concatenate([[a], near, np.zeros(55)]).astype(np.float32))
    rows.append(np.zeros(256, np.float32))                       # all zero
    rows.append((rng.standard_normal(256) * 1e-37).astype(np.float32))  # tiny scale
    X = bf16_bits_of(np.stack([r[:256] for r in rows]))
    xf = bits_to_f32(X)
    for mode, group in ((oracle.PER_ROW, 256), (oracle.BLOCK, 128)):
        Xq, sx = oracle.quantize_act(X, mode)
        sx = sx.reshape(len(rows), -1)
        for i in range(len(rows)):
            for g in range(256 // group):
                seg = xf[i, g * group:(g + 1) * group]
                amax = max(abs(Fraction(float(v))) for v in seg)
                s_ex = f32_exact(amax / 127)
                assert Fraction(float(sx[i, g])) == s_ex
                for k in range(group):
                    assert Xq[i, g * group + k] == q_exact(float(seg[k]), s_ex)


def test_quant_invariants(oracle):
    rng = np.random.default_rng(2)
    X = rand_bf16(rng, (64, 512))
    Xq, sx = oracle.quantize_act(X, oracle.PER_ROW)
    xf = bits_to_f32(X)
    # the absmax element maps to +-127 with its sign; |q| <= 127; never -128
    am = np.argmax(np.abs(xf), axis=1)
    assert np.all(np.abs(Xq[np.arange(64), am]) == 127)
    assert np.all(np.sign(Xq[np.arange(64), am]) == np.sign(xf[np.arange(64), am]))
    assert Xq.min() >= -127 and Xq.max() <= 127
    # q has the sign of x (or is 0)
    assert np.all((Xq == 0) | (np.sign(Xq) == np.sign(xf)))
    # sign symmetry: Q(-x) == -Q(x)
    Xn = X ^ np.uint16(0x8000)
    Xqn, sxn = oracle.quantize_act(Xn, oracle.PER_ROW)
    assert np.array_equal(Xqn, -Xq) and np.array_equal(sxn, sx)
    # power-of-two scaling leaves q unchanged and scales s exactly
    for p in (-3, 5):
        Xp = bf16_bits_of(xf * np.float32(2.0 ** p))
        Xqp, sxp = oracle.quantize_act(Xp, oracle.PER_ROW)
        assert np.array_equal(Xqp, Xq)
        assert np.array_equal(sxp, sx * np.float32(2.0 ** p))
    # monotone in x within a row
    i = 3
    order = np.argsort(xf[i], kind="stable")
    assert np.all(np.diff(Xq[i, order].astype(np.int32)) >= 0)
    # dequantized values lie within s/2 of x (up to fp32 rounding of x/s)
    deq = Xq.astype(np.float64) * sx.astype(np.float64)[:, None]
    assert np.all(np.abs(deq - xf) <= sx[:, None] * (0.5 + 1e-5))


def test_weight_quant_modes(oracle):
    """Per-channel weight quant == per-token quant of W's rows; a 128x128 block
    equals the per-row quantizer applied with the block's absmax, and a
    partial last block uses only its own rows."""
    rng = np.random.default_rng(3)
    W = rand_bf16(rng, (300, 256), 0.02)
    Wq, sw = oracle.quantize_weight(W, oracle.PER_ROW)
    Xq, sx = oracle.quantize_act(W, oracle.PER_ROW)
    assert np.array_equal(Wq, Xq) and np.array_equal(sw, sx)
    Wqb, swb = oracle.quantize_weight(W, oracle.BLOCK)
    assert swb.shape == (3, 2)
    wf = bits_to_f32(W)
    for nb in range(3):
        for kb in range(2):
            blk = wf[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128]
            amax = np.abs(blk).max()
            assert swb[nb, kb] == np.float32(amax) / np.float32(127)
            s = Fraction(float(swb[nb, kb]))
            sub = Wqb[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128]
            for (r, c) in [(0, 0), (5, 77), (blk.shape[0] - 1, 127)]:
                assert sub[r, c] == q_exact(float(blk[r, c]), s)
            assert np.abs(sub).max() == 127
    assert Wqb.shape == (300, 256)


# ----------------------------------------------------------------- GEMM (int32)
def test_gemm_s32_brute_force_tiny(oracle):
    rng = np.random.default_rng(4)
    for M, N, K in [(1, 1, 16), (2, 3, 128), (3, 2, 256), (3, 3, 16)]:
        Xq = rng.integers(-127, 128, (M, K), dtype=np.int8)
        Wq = rng.integers(-127, 128, (N, K), dtype=np.int8)
        acc = oracle.gemm_s32(Xq, Wq)
        for m in range(M):
            for n in range(N):
                assert acc[m, n] == sum(int(Xq[m, k]) * int(Wq[n, k]) for k in range(K))


def test_gemm_s32_library_and_closed_forms(oracle):
    rng = np.random.default_rng(5)
    M, N, K = 37, 53, 400  # non-square: a transposed operand fails
    Xq = rng.integers(-127, 128, (M, K), dtype=np.int8)
    Wq = rng.integers(-127, 128, (N, K), dtype=np.int8)
    assert np.array_equal(oracle.gemm_s32(Xq, Wq), Xq.astype(np.int64) @ Wq.astype(np.int64).T)
    # all +-127 at K = 13824: |acc| = 16129 * K, the int32 worst case of the workloads
    K = 13824
    Xq = np.full((2, K), 127, np.int8)
    Xq[1] = -127
    Wq = np.full((3, K), 127, np.int8)
    Wq[1, ::2] = -127
    acc = oracle.gemm_s32(Xq, Wq)
    assert acc[0, 0] == 16129 * K and acc[1, 0] == -16129 * K
    assert acc[0, 1] == 0 and acc[1, 2] == -16129 * K


# ----------------------------------------------------------------- epilogues
def test_postscale_epilogue_special_cases(oracle):
    rng = np.random.default_rng(6)
    acc = rng.integers(-2**28, 2**28, (8, 24), dtype=np.int64).astype(np.int32)
    ones_m = np.ones(8, np.float32)
    ones_n = np.ones(24, np.float32)
    # unit scales, no bias: Y = bf16(float(acc)) (torch's conversions)
    Y = oracle.epilogue_postscale(acc, ones_m, ones_n, None)
    want = torch.from_numpy(acc).to(torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(Y, want)
    # power-of-two scales are exact: Y = bf16(acc * 2^a * 2^b)
    sx = np.float32(2.0) ** rng.integers(-8, 8, 8).astype(np.float32)
    sw = np.float32(2.0) ** rng.integers(-8, 8, 24).astype(np.float32)
    Y = oracle.epilogue_postscale(acc, sx, sw, None)
    exact = acc.astype(np.float64) * sx.astype(np.float64)[:, None] * sw.astype(np.float64)[None, :]
    want = torch.from_numpy(exact).to(torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(Y, want)
    # bias: zero acc gives Y == bias exactly; no bias gives +0
    z = np.zeros((2, 24), np.int32)
    b = bf16_bits_of(rng.standard_normal(24).astype(np.float32))
    assert np.array_equal(oracle.epilogue_postscale(z, ones_m[:2], ones_n, b), np.stack([b, b]))
    assert np.all(oracle.epilogue_postscale(z, ones_m[:2], ones_n, None) == 0)


def _bf16_ulp(y):
    y = np.abs(y.astype(np.float64))
    e = np.floor(np.log2(np.maximum(y, 2.0 ** -126)))
    return 2.0 ** (e - 7)


def test_postscale_linear_vs_fp64_dequant(oracle):
    """Y is within one bf16 ulp plus the fp32 epilogue error of the fp64
    dequantize-then-matmul closed form; with the bias dropped it is not."""
    rng = np.random.default_rng(7)
    M, N, K = 48, 40, 512
    X = rand_bf16(rng, (M, K))
    W = rand_bf16(rng, (N, K), 0.02)
    b = rand_bf16(rng, (N,), 0.01)
    r = oracle.linear_postscale(X, W, b)
    deq = (r["Xq"].astype(np.float64) * r["sx"].astype(np.float64)[:, None]) @ \
          (r["Wq"].astype(np.float64) * r["sw"].astype(np.float64)[:, None]).T
    y64 = deq + bits_to_f32(b).astype(np.float64)[None, :]
    Y = bits_to_f32(r["Y"]).astype(np.float64)
    bound = _bf16_ulp(y64) + 4 * 2.0 ** -24 * (np.abs(deq) + np.abs(y64)) + 1e-30
    assert np.all(np.abs(Y - y64) <= bound)
    # the int32 accumulator is the fp64 matmul of the int8 matrices
    assert np.array_equal(r["acc"].astype(np.float64), r["Xq"].astype(np.float64) @ r["Wq"].astype(np.float64).T)
    # a dropped bias is visible to this check
    r2 = oracle.linear_postscale(X, W, None)
    assert not np.all(np.abs(bits_to_f32(r2["Y"]) - y64) <= bound)
    # the quantized Linear approximates the bf16 Linear (sanity of the reading)
    ref = bits_to_f32(X).astype(np.float64) @ bits_to_f32(W).astype(np.float64).T + bits_to_f32(b)
    rel = np.linalg.norm(Y - ref) / np.linalg.norm(ref)
    assert rel < 0.02


def test_blockwise_closed_forms(oracle):
    rng = np.random.default_rng(8)
    M, N, K = 5, 200, 384
    Xq = rng.integers(-127, 128, (M, K), dtype=np.int8)
    Wq = rng.integers(-127, 128, (N, K), dtype=np.int8)
    kbs = K // 128
    # power-of-two scales, one per row and one per 128-row weight block
    # (the same for every k block): every product and partial sum is
    # exact in fp32 (|sum P| < 2^24), so acc is the exact scaled sum
    sx = np.repeat(np.float32(2.0) ** rng.integers(-6, 6, (M, 1)), kbs, axis=1).astype(np.float32)
    sw = np.repeat(np.float32(2.0) ** rng.integers(-6, 6, (2, 1)), kbs, axis=1).astype(np.float32)
    acc = oracle.gemm_blockwise_f32(Xq, sx, Wq, sw)
    exact = np.zeros((M, N))
    for kb in range(kbs):
        P = Xq[:, kb * 128:(kb + 1) * 128].astype(np.int64) @ Wq[:, kb * 128:(kb + 1) * 128].astype(np.int64).T
        exact += P * sx[:, kb][:, None].astype(np.float64) * sw[np.arange(N) // 128, kb][None, :].astype(np.float64)
    assert np.array_equal(acc.astype(np.float64), exact)
    # unit scales: blockwise == int32 GEMM (|acc| < 2^24 here, so exact in fp32)
    acc1 = oracle.gemm_blockwise_f32(Xq, np.ones((M, kbs), np.float32), Wq, np.ones((2, kbs), np.float32))
    assert np.array_equal(acc1, oracle.gemm_s32(Xq, Wq).astype(np.float32))
    # general scales: within the fp32 rounding bound of the fp64 sum
    sx = rng.random((M, kbs)).astype(np.float32) * 0.01
    sw = rng.random((2, kbs)).astype(np.float32) * 0.001
    acc = oracle.gemm_blockwise_f32(Xq, sx, Wq, sw).astype(np.float64)
    ex = np.zeros((M, N))
    mag = np.zeros((M, N))
    for kb in range(kbs):
        P = Xq[:, kb * 128:(kb + 1) * 128].astype(np.int64) @ Wq[:, kb * 128:(kb + 1) * 128].astype(np.int64).T
        t = P * sx[:, kb][:, None].astype(np.float64) * sw[np.arange(N) // 128, kb][None, :].astype(np.float64)
        ex += t
        mag += np.abs(t)
    assert np.all(np.abs(acc - ex) <= (kbs + 2) * 2.0 ** -23 * mag + 1e-30)


def test_blockwise_fold_order_is_ascending(oracle):
    """acc = ((0 + t0) + t1) + t2 in fp32, k blocks ascending: build t's where
    the order changes the fp32 result."""
    K = 384
    Xq = np.zeros((1, K), np.int8)
    Wq = np.zeros((1, K), np.int8)
    Xq[0, 0], Wq[0, 0] = 1, 1        # block 0: P = 1
    Xq[0, 128], Wq[0, 128] = 1, 1    # block 1: P = 1
    Xq[0, 256], Wq[0, 256] = 1, 1    # block 2: P = 1
    sw = np.ones((1, 3), np.float32)
    sx = np.array([[2.0 ** 24, 1.0, 1.0]], np.float32)
    # ascending: (2^24 + 1) -> 2^24 (tie to even), + 1 -> 2^24
    acc = oracle.gemm_blockwise_f32(Xq, sx, Wq, sw)
    assert acc[0, 0] == np.float32(2.0 ** 24)
    sx_rev = np.array([[1.0, 1.0, 2.0 ** 24]], np.float32)
    # ascending here: 1 + 1 = 2, 2 + 2^24 = 2^24 + 2 (exact)
    acc = oracle.gemm_blockwise_f32(Xq, sx_rev, Wq, sw)
    assert acc[0, 0] == np.float32(2.0 ** 24 + 2)


def test_blockwise_epilogue_bias(oracle):
    rng = np.random.default_rng(9)
    acc = (rng.standard_normal((4, 16)) * 10).astype(np.float32)
    b = bf16_bits_of(rng.standard_normal(16).astype(np.float32))
    Y = oracle.epilogue_blockwise(acc, b)
    want = (torch.from_numpy(acc) + torch.from_numpy(bits_to_f32(b))).to(torch.bfloat16)
    assert np.array_equal(Y, want.view(torch.int16).numpy().view(np.uint16))
    Y0 = oracle.epilogue_blockwise(acc, None)
    assert np.array_equal(Y0, torch.from_numpy(acc).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))


# ----------------------------------------------------------------- sampled evaluation
@pytest.mark.parametrize("mode", ["postscale", "blockwise"])
def test_sampled_matches_full(oracle, mode):
    rng = np.random.default_rng(10)
    M, N, K = 40, 300, 256
    X = rand_bf16(rng, (M, K))
    W = rand_bf16(rng, (N, K), 0.02)
    b = rand_bf16(rng, (N,), 0.01)
    if mode == "postscale":
        full = oracle.linear_postscale(X, W, b)
        md = oracle.PER_ROW
    else:
        full = oracle.linear_blockwise(X, W, b)
        md = oracle.BLOCK
    rows = np.array([0, 7, 39])
    cols = np.array([0, 127, 128, 255, 256, 299])
    Y, acc = oracle.linear_sampled(X, W, b, rows, cols, md)
    assert np.array_equal(Y, full["Y"][np.ix_(rows, cols)])
    assert np.array_equal(acc, full["acc"][np.ix_(rows, cols)])


# ----------------------------------------------------------------- GELU of the FFN up-projection
def _bf16_all(lo, hi):
    """Every finite bf16 value in [lo, hi] as (float32 array, uint16 bits)."""
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = (bits.astype(np.uint32) << 16).view(np.float32)
    keep = np.isfinite(vals) & (vals >= lo) & (vals <= hi)
    return vals[keep], bits[keep]


def _bf16_of_f64(v):
    """fp64 -> fp32 -> bf16 bits (round to nearest even both times), by torch."""
    t = torch.from_numpy(np.asarray(v, np.float64).astype(np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def test_gelu_matches_scipy_ndtr_on_every_bf16(oracle):
    """Against x * ndtr(x), ndtr being scipy's standard normal CDF (the Cephes
    routine, another implementation of Phi), rounded the same way: identical
    bits on every finite bf16 input."""
    sp = pytest.importorskip("scipy.special")
    x, h = _bf16_all(-np.inf, np.inf)
    G = oracle.gelu_bf16(h)
    xd = x.astype(np.float64)
    want = _bf16_of_f64(xd * sp.ndtr(xd))
    assert np.array_equal(G, want)


def test_gelu_correctly_rounded_against_mpmath(oracle):
    """Against x * Phi(x) in 40-digit arithmetic (mpmath.ncdf): the binary64
    evaluation rounds to the same bf16 on a sample of 4000 bf16 inputs
    spanning [-14, 14], where the result is neither x nor 0."""
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 40
    x, h = _bf16_all(-14.0, 14.0)
    sel = np.linspace(0, x.size - 1, 4000).astype(np.int64)
    x, h = x[sel], h[sel]
    exact = np.array([float(mpmath.mpf(float(v)) * mpmath.ncdf(mpmath.mpf(float(v)))) for v in x])
    assert np.array_equal(oracle.gelu_bf16(h), _bf16_of_f64(exact))


def test_gelu_normal_table_values(oracle):
    """Phi from a printed table of the standard normal distribution
    (Phi(0.5) = 0.6914624613, Phi(1) = 0.8413447461, Phi(2) = 0.9772498681,
    Phi(3) = 0.9986501020) and Phi(-x) = 1 - Phi(x)."""
    table = {0.5: 0.6914624613, 1.0: 0.8413447461, 2.0: 0.9772498681, 3.0: 0.9986501020}
    x = np.array(list(table) + [-v for v in table], np.float64)
    phi = np.array(list(table.values()) + [1.0 - v for v in table.values()])
    g = oracle.gelu_f64(x)
    assert np.all(np.abs(g - x * phi) <= 1e-10 * np.abs(x))


def test_gelu_tail_asymptotic_series(oracle):
    """For x <= -8, Phi(x) = phi(x) / |x| * (1 - 1/x^2 + 3/x^4 - 15/x^6 +
    105/x^8 - ...), phi the normal density; the truncated series is within
    its next term (945/x^10 < 1e-6).  This catches a 1 + erf(x / sqrt 2)
    evaluation, which loses all accuracy there."""
    x = -np.linspace(8.0, 37.0, 2901)
    x2 = x * x
    series = 1 - 1 / x2 + 3 / x2 ** 2 - 15 / x2 ** 3 + 105 / x2 ** 4
    phi = np.exp(-x2 / 2) / np.sqrt(2 * np.pi)
    want = x * phi / np.abs(x) * series
    g = oracle.gelu_f64(x)
    assert np.all(np.abs(g - want) <= 2e-6 * np.abs(want))


def test_gelu_special_values(oracle):
    g = oracle.gelu_f64(np.array([0.0, -0.0]))
    assert g[0] == 0 and not np.signbit(g[0])
    assert g[1] == 0 and np.signbit(g[1])       # -0 * Phi keeps the sign
    # Phi(x) + Phi(-x) = 1, so g(x) - g(-x) = x
    rng = np.random.default_rng(6)
    v = rng.normal(0, 3, 5000)
    assert np.all(np.abs(oracle.gelu_f64(v) - oracle.gelu_f64(-v) - v) <= 1e-15 * (1 + np.abs(v)))
    # the minimum of gelu sits where g'(x) = Phi(x) + x phi(x) = 0, found here
    # with scipy's ndtr and a bracketing root finder
    sp = pytest.importorskip("scipy.special")
    from scipy.optimize import brentq
    xm = brentq(lambda t: sp.ndtr(t) + t * np.exp(-t * t / 2) / np.sqrt(2 * np.pi), -1.0, -0.5, xtol=1e-14)
    xs = np.linspace(xm - 1e-3, xm + 1e-3, 20001)
    gs = oracle.gelu_f64(xs)
    assert abs(xs[np.argmin(gs)] - xm) <= 2e-7 and abs(gs.min() - xm * sp.ndtr(xm)) <= 1e-15
    # bf16: g = x from x = 4 up (Phi rounds away), -0 far below zero, x / 2 for tiny x
    x, h = _bf16_all(4.0, np.inf)
    assert np.array_equal(oracle.gelu_bf16(h), h)
    x, h = _bf16_all(-np.inf, -14.0)
    assert np.all(oracle.gelu_bf16(h) == 0x8000)
    x, h = _bf16_all(2.0 ** -120, 2.0 ** -12)
    assert np.array_equal(oracle.gelu_bf16(h), _bf16_of_f64(x.astype(np.float64) / 2))


def test_gelu_matches_torch_bf16(oracle):
    """torch.nn.functional.gelu (erf form, evaluated in fp32) rounded to bf16:
    identical on every bf16 |x| <= 3, never more than 1 ulp apart on
    -4 <= x <= 5.  (Further down torch's fp32 1 + erf(x / sqrt 2) has lost
    most of its relative accuracy: Phi(-4.4) is 5e-6, 85 units of fp32
    rounding near 1.)"""
    for lo, hi, max_ulp in ((-3.0, 3.0, 0), (-4.0, 5.0, 1)):
        x, h = _bf16_all(lo, hi)
        G = oracle.gelu_bf16(h)
        T = torch.nn.functional.gelu(torch.from_numpy(x)).to(torch.bfloat16)
        Tb = T.view(torch.int16).numpy().view(np.uint16)
        d = np.abs(_ordered(G) - _ordered(Tb))
        assert d.max() <= max_ulp


def test_ffn_up_gelu_quant_composition(oracle):
    """G is the GELU of the post-scale Linear's bf16 output, and (Gq, sg) its
    1x128 quantization: sg = absmax(|G| of the block) / 127 exactly, and
    Gq * sg reproduces G within half a step."""
    rng = np.random.default_rng(7)
    M, N, K = 5, 384, 256
    X = oracle.bf16_from_f32(rng.normal(0, 1, (M, K)).astype(np.float32))
    W = oracle.bf16_from_f32(rng.normal(0, 0.1, (N, K)).astype(np.float32))
    b = oracle.bf16_from_f32(rng.normal(0, 0.5, N).astype(np.float32))
    r = oracle.ffn_up_gelu_quant(X, W, b)
    lin = oracle.linear_postscale(X, W, b)
    assert np.array_equal(r["Y"], lin["Y"])
    assert np.array_equal(r["G"], oracle.gelu_bf16(lin["Y"]))
    G = oracle.f32_from_bf16(r["G"]).reshape(M, N // 128, 128)
    amax = np.abs(G).max(axis=2)
    assert np.array_equal(r["sg"], (amax / np.float32(127)).astype(np.float32))
    deq = r["Gq"].reshape(M, N // 128, 128).astype(np.float64) * r["sg"][:, :, None].astype(np.float64)
    assert np.all(np.abs(deq - G) <= 0.5 * r["sg"][:, :, None] * (1 + 1e-6))
    assert np.abs(r["Gq"]).max() == 127


# ----------------------------------------------------------------- normalization fused with quantization
def _ordered(u):
    u = np.asarray(u).astype(np.int64)
    return np.where(u & 0x8000, 0x8000 - (u & 0x7FFF), u + 0x8000)


NORMS = ("norm_quant", "norm_quant_fixed_order")


@pytest.mark.parametrize("fn", NORMS)
@pytest.mark.parametrize("K", [128, 4096, 5120])
def test_layer_norm_matches_torch(oracle, fn, K):
    """Against torch.nn.functional.layer_norm in fp32 (another summation
    order), rounded to bf16: within 1 ulp everywhere, identical almost
    everywhere; a missing beta or gamma skips exactly that operation."""
    rng = np.random.default_rng(K)
    Xf = (rng.normal(0.5, 2.0, (16, K)) * rng.choice([1.0, 30.0], (16, K), p=[0.99, 0.01])).astype(np.float32)
    X = oracle.bf16_from_f32(Xf)
    g = oracle.bf16_from_f32(rng.normal(1.0, 0.2, K).astype(np.float32))
    b = oracle.bf16_from_f32(rng.normal(0.0, 0.2, K).astype(np.float32))
    xt = torch.from_numpy(oracle.f32_from_bf16(X))
    for gg, bb in ((g, b), (g, None), (None, None)):
        Y, _, _ = getattr(oracle, fn)(X, gg, bb, 1e-5, oracle.LAYER_NORM)
        T = torch.nn.functional.layer_norm(
            xt, (K,), None if gg is None else torch.from_numpy(oracle.f32_from_bf16(gg)),
            None if bb is None else torch.from_numpy(oracle.f32_from_bf16(bb)), 1e-5)
        Tb = T.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        d = np.abs(_ordered(Y) - _ordered(Tb))
        assert d.max() <= 1 and (d > 0).mean() < 2e-3


@pytest.mark.parametrize("fn", NORMS)
@pytest.mark.parametrize("K", [256, 5120])
def test_rms_norm_matches_torch(oracle, fn, K):
    """Against torch.nn.functional.rms_norm in fp32, rounded to bf16; the
    codes are the per-token quantization of the bf16 output."""
    rng = np.random.default_rng(K + 1)
    X = oracle.bf16_from_f32(rng.normal(0.0, 3.0, (16, K)).astype(np.float32))
    g = oracle.bf16_from_f32(rng.normal(1.0, 0.2, K).astype(np.float32))
    Y, Xq, sx = getattr(oracle, fn)(X, g, None, 1e-6, oracle.RMS_NORM)
    T = torch.nn.functional.rms_norm(torch.from_numpy(oracle.f32_from_bf16(X)), (K,),
                                     torch.from_numpy(oracle.f32_from_bf16(g)), 1e-6)
    Tb = T.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    d = np.abs(_ordered(Y) - _ordered(Tb))
    assert d.max() <= 1 and (d > 0).mean() < 2e-3
    q2, s2 = oracle.quantize_act(Y, oracle.PER_ROW)
    assert np.array_equal(Xq, q2) and np.array_equal(sx, s2)


def _norm_exact(x, g, b, eps, layer, mpmath):
    """One row by exact rational statistics and a 50-digit square root."""
    xs = [Fraction(float(v)) for v in x]
    K = len(xs)
    mu = sum(xs, Fraction(0)) / K if layer else Fraction(0)
    var = sum(((v - mu) ** 2 for v in xs), Fraction(0)) / K
    den = mpmath.sqrt(mpmath.mpf(var.numerator) / var.denominator + mpmath.mpf(float(np.float32(eps))))
    out = []
    for i, v in enumerate(xs):
        y = (mpmath.mpf((v - mu).numerator) / (v - mu).denominator) / den
        if g is not None:
            y = y * float(g[i])
        if layer and b is not None:
            y = y + float(b[i])
        out.append(float(y))
    return np.array(out)


def test_norm_plain_against_exact_arithmetic(oracle):
    """The plain definition against exact rational mean and variance and a
    50-digit square root, rounded to fp32 and bf16: identical bits, for
    LayerNorm and RMSNorm, with and without gamma/beta, on random rows and on
    rows whose fp32 sums would cancel (2^24 + 1 + 1 - 2^24)."""
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 50
    rng = np.random.default_rng(11)
    rows = [rng.normal(0.3, 2.0, 24) for _ in range(12)]
    c = np.zeros(32)
    c[0], c[8], c[16], c[24] = 2.0 ** 24, 1.0, 1.0, -(2.0 ** 24)
    rows.append(c)
    rows.append(np.full(16, 1000.0) + rng.integers(-3, 4, 16) * 8.0)  # large mean, small spread
    for row in rows:
        K = len(row)
        X = oracle.bf16_from_f32(row.astype(np.float32)[None, :])
        x = oracle.f32_from_bf16(X)[0]
        g = oracle.bf16_from_f32(rng.normal(1.0, 0.3, K).astype(np.float32))
        b = oracle.bf16_from_f32(rng.normal(0.0, 0.3, K).astype(np.float32))
        for layer in (False, True):
            for gg, bb in ((None, None), (g, b)):
                Y, _, _ = oracle.norm_quant(X, gg, bb, 1e-5, oracle.LAYER_NORM if layer else oracle.RMS_NORM)
                want = _norm_exact(x, None if gg is None else oracle.f32_from_bf16(gg),
                                   None if bb is None else oracle.f32_from_bf16(bb), 1e-5, layer, mpmath)
                assert np.array_equal(Y[0], _bf16_of_f64(want))


def test_norm_closed_forms(oracle):
    K = 1024
    for fn in NORMS:
        f = getattr(oracle, fn)
        # constant row c, eps = 0: RMSNorm gives c / |c| = 1 exactly
        c = np.float32(1.5)
        X = oracle.bf16_from_f32(np.full((1, K), c, np.float32))
        Y, Xq, sx = f(X, None, None, 0.0, oracle.RMS_NORM)
        assert np.all(oracle.f32_from_bf16(Y) == 1.0)
        assert np.all(Xq == 127) and sx[0] == np.float32(1.0) / np.float32(127)
        # LayerNorm of a constant row: x - mu = 0, so y = beta exactly
        b = oracle.bf16_from_f32(np.linspace(-1, 1, K).astype(np.float32))
        Y, Xq, sx = f(X, None, b, 1e-5, oracle.LAYER_NORM)
        assert np.array_equal(Y[0], b)
        # +-a alternating: mean 0, variance a^2; with eps = 0 every |y| = 1
        a = np.float32(0.375)
        X2 = oracle.bf16_from_f32(np.tile(np.array([a, -a], np.float32), K // 2)[None, :])
        Y, Xq, sx = f(X2, None, None, 0.0, oracle.LAYER_NORM)
        assert np.array_equal(np.abs(oracle.f32_from_bf16(Y)), np.ones((1, K), np.float32))
        assert np.array_equal(Xq[0], np.tile(np.array([127, -127], np.int8), K // 2))


def test_norm_fixed_order_sum(oracle):
    """The fixed-order statement sums chunks of 8 and then a pairwise tree,
    not a left-to-right scan: on a row where the two orders give different
    binary32 sums it takes the tree's value, while the plain definition takes
    the exact one."""
    K = 32  # 4 chunks: tree ((s0 + s1) + (s2 + s3))
    x = np.zeros(K, np.float32)
    x[0] = 2.0 ** 24          # chunk 0
    x[8] = 1.0                # chunk 1: 2^24 + 1 rounds to 2^24 in a left-to-right scan ...
    x[16] = 1.0               # chunk 2: ... and again, while the tree adds 1 + 1 = 2 first
    x[24] = -(2.0 ** 24)      # chunk 3
    tree = ((np.float32(2.0 ** 24) + np.float32(1.0)) + (np.float32(1.0) + np.float32(-(2.0 ** 24))))
    scan = np.float32(0)
    for v in x:
        scan = np.float32(scan + v)
    assert tree != scan
    X = oracle.bf16_from_f32(x[None, :])
    mu_tree = np.float32(tree) / np.float32(K)
    Y, _, _ = oracle.norm_quant_fixed_order(X, None, None, 1.0, oracle.LAYER_NORM)
    y1 = oracle.f32_from_bf16(Y)[0, 1]     # an element equal to 0: -mu * r
    assert np.sign(y1) == -np.sign(mu_tree) or mu_tree == 0
    # exact mean 2 / 32 > 0: the plain definition gives y < 0 there
    Yp, _, _ = oracle.norm_quant(X, None, None, 1.0, oracle.LAYER_NORM)
    assert oracle.f32_from_bf16(Yp)[0, 1] < 0


def test_norm_fixed_order_within_one_ulp_of_plain(oracle):
    rng = np.random.default_rng(13)
    for K in (264, 5120):
        X = oracle.bf16_from_f32((rng.normal(0.75, 2.0, (32, K)) *
                                  rng.choice([1.0, 30.0], (32, K), p=[0.99, 0.01])).astype(np.float32))
        g = oracle.bf16_from_f32(rng.normal(1.0, 0.2, K).astype(np.float32))
        b = oracle.bf16_from_f32(rng.normal(0.0, 0.2, K).astype(np.float32))
        for kind, bb in ((oracle.RMS_NORM, None), (oracle.LAYER_NORM, b)):
            Yp, _, _ = oracle.norm_quant(X, g, bb, 1e-5, kind)
            Yf, _, _ = oracle.norm_quant_fixed_order(X, g, bb, 1e-5, kind)
            d = np.abs(_ordered(Yp) - _ordered(Yf))
            assert d.max() <= 1 and (d > 0).mean() < 2e-3
