"""Full-size workloads on the GPU, in the launch configuration the benchmark
times, checked against the oracle on sampled outputs: every first and last
row of every 128-row tile (and every first/last column of every 256-column
tile) in a sample of tiles, plus random points.  The oracle quantizes only
the X rows and W rows (or 128-row W blocks) those outputs depend on."""
import numpy as np
import pytest
import torch

from gpu_helpers import assert_bf16_close, assert_quant_follows_plain, bits, edge_indices
from w8a8_int8_linear_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
DEV = "cuda"


def sample(n, tile, rng, max_count):
    idx = edge_indices(n, tile, 16, rng)
    if len(idx) > max_count:
        keep = np.concatenate([idx[:4], idx[-4:], rng.choice(idx[4:-4], max_count - 8, replace=False)])
        idx = np.unique(keep)
    return idx


def run_case(w8a8, oracle, work, rows_max=96, cols_max=96):
    rng = np.random.default_rng(0)
    X = wl.make_x(work, DEV)
    W = wl.make_w(work, DEV)
    b = wl.make_bias(work, DEV)
    mode = w8a8.PER_ROW if work.mode == "postscale" else w8a8.BLOCK
    Wq, sw = w8a8.quantize_weight(W, mode)
    Xq, sx = w8a8.quantize_act(X, mode)
    if mode == w8a8.PER_ROW:
        Y = w8a8.gemm_postscale(Xq, sx, Wq, sw, b)
        Yf, sxf, _ = w8a8.linear_postscale(X, w8a8.pack_weight(Wq), sw, b)
    else:
        Y = w8a8.gemm_blockwise(Xq, sx, Wq, sw, b)
        Yf, sxf, _ = w8a8.linear_blockwise(X, w8a8.pack_weight(Wq), sw, b)
    torch.cuda.synchronize()
    # the fused Linear (the benchmark's step) gives the same bytes everywhere
    assert torch.equal(Yf, Y) and torch.equal(sxf, sx)
    assert w8a8.get_device_error() == (0, 0)
    rows = sample(work.M, 128, rng, rows_max)
    cols = sample(work.N, 256, rng, cols_max)
    Xs = bits(X[torch.from_numpy(rows).to(DEV)])
    # quantized rows: bit-exact against the oracle
    oq, osx = oracle.quantize_act(Xs, oracle.PER_ROW if mode == w8a8.PER_ROW else oracle.BLOCK)
    assert np.array_equal(Xq[torch.from_numpy(rows).to(DEV)].cpu().numpy(), oq)
    assert np.array_equal(sx[torch.from_numpy(rows).to(DEV)].cpu().numpy().view(np.uint32), osx.view(np.uint32))
    # outputs at the sampled points; the oracle gets the full bf16 X rows and W
    Wh = bits(W)
    bh = None if b is None else bits(b)
    Yo, _ = oracle.linear_sampled(Xs, Wh, bh, np.arange(len(rows)), cols,
                                  oracle.PER_ROW if mode == w8a8.PER_ROW else oracle.BLOCK)
    Yg = bits(Y[torch.from_numpy(rows).to(DEV)][:, torch.from_numpy(cols).to(DEV)])
    d = assert_bf16_close(Yg, Yo, 1)
    assert d.max() == 0
    # properties that hold everywhere: finite, and Y == 0 exactly only where
    # it may be (no uninitialized tiles)
    assert torch.isfinite(Y).all()


def test_square_4096(w8a8, oracle):
    run_case(w8a8, oracle, wl.SQUARE)


def test_ffn_up_32768x13824x5120(w8a8, oracle):
    run_case(w8a8, oracle, wl.FFN_UP, rows_max=64, cols_max=64)


def test_ffn_up_full_row_bands(w8a8, oracle):
    """Every output of two 128-row bands of the FFN up-projection (an
    interior band and the last one, each 128 x 13824) from the fused Linear
    the benchmark times, element by element against the oracle."""
    work = wl.FFN_UP
    X = wl.make_x(work, DEV)
    W = wl.make_w(work, DEV)
    b = wl.make_bias(work, DEV)
    Wq, sw = w8a8.quantize_weight(W)
    Y, sx, _ = w8a8.linear_postscale(X, w8a8.pack_weight(Wq), sw, b)
    torch.cuda.synchronize()
    assert w8a8.get_device_error() == (0, 0)
    Wh, bh = bits(W), bits(b)
    cols = np.arange(work.N)
    for r0 in (12800, work.M - 128):
        Xs = bits(X[r0:r0 + 128])
        Yo, _ = oracle.linear_sampled(Xs, Wh, bh, np.arange(128), cols, oracle.PER_ROW)
        d = assert_bf16_close(bits(Y[r0:r0 + 128]), Yo, 1)
        assert d.max() == 0


def test_ffn_down_blockwise_32768x5120x13824(w8a8, oracle):
    run_case(w8a8, oracle, wl.FFN_DOWN, rows_max=48, cols_max=48)


@pytest.mark.parametrize("M", wl.RAGGED_M)
@pytest.mark.parametrize("N", wl.RAGGED_N)
def test_ragged_sweep(w8a8, oracle, M, N):
    run_case(w8a8, oracle, wl.ragged(M, N), rows_max=24, cols_max=24)


def test_ffn_up_gelu_quant_full_size(w8a8, oracle):
    """The fused FFN up-projection (GELU + 1x128 quantization epilogue) at
    32768 x 13824 x 5120: codes and block scales of sampled rows and sampled
    128-column blocks (every edge block of the 256-wide tiles among them)
    against the plain oracle (erf GELU in fp64), with the tolerance rule of
    the small-size test (assert_quant_follows_plain)."""
    rng = np.random.default_rng(1)
    work = wl.FFN_UP
    X = wl.make_x(work, DEV)
    W = wl.make_w(work, DEV)
    b = wl.make_bias(work, DEV)
    Wq, sw = w8a8.quantize_weight(W)
    G, sg, sx, _ = w8a8.linear_postscale_gelu_quant(X, w8a8.pack_weight(Wq), sw, b)
    torch.cuda.synchronize()
    assert w8a8.get_device_error() == (0, 0)
    rows = sample(work.M, 128, rng, 40)
    blocks = sample(work.N // 128, 2, rng, 12)
    cols = (blocks[:, None] * 128 + np.arange(128)[None, :]).reshape(-1)
    Xs = bits(X[torch.from_numpy(rows).to(DEV)])
    Yo, _ = oracle.linear_sampled(Xs, bits(W), bits(b), np.arange(len(rows)), cols, oracle.PER_ROW)
    Gp = oracle.gelu_bf16(Yo)
    Gq_p, sg_p = oracle.quantize_act(Gp, oracle.BLOCK)
    Yd = torch.from_numpy(np.ascontiguousarray(Yo).view(np.int16)).view(torch.bfloat16).to(DEV)
    Gk = bits(w8a8.gelu_bf16(Yd))
    r = torch.from_numpy(rows).to(DEV)
    Gg = G[r][:, torch.from_numpy(cols).to(DEV)].float().cpu()
    sgg = sg[r][:, torch.from_numpy(blocks).to(DEV)].cpu().numpy()
    differing = assert_quant_follows_plain(oracle, Gk, Gp, Gg.to(torch.int8).numpy(), sgg, Gq_p, sg_p, 128)
    assert differing <= max(1, sg_p.size // 100)
    assert torch.isfinite(sg).all() and (G.abs() <= 127).all()
