"""Parity of the CUDA path against the CPU oracle, element by element, on
seeded inputs at sizes the oracle finishes in seconds (several tiles and a
ragged tail).  Integers (int8 codes, int32 accumulators) and fp32 scales and
blockwise accumulators must be bit-exact; bf16 outputs within 1 bf16 ulp."""
import numpy as np
import pytest
import torch

from gpu_helpers import (assert_bf16_close, assert_quant_follows_plain, bf16_ulp_distance, bits,
                         norm_error_bound)

pytestmark = pytest.mark.gpu

DEV = "cuda"


def rand_bf16(shape, seed, scale=1.0, outliers=0.0, oscale=1.0):
    g = torch.Generator(device="cpu").manual_seed(seed)
    x = torch.randn(shape, generator=g) * scale
    if outliers > 0:
        idx = torch.randperm(shape[-1], generator=g)[: max(1, int(round(outliers * shape[-1])))]
        x[..., idx] *= oscale
    return x.to(torch.bfloat16)


def special_rows(K):
    """Rows that hit the quantizer's edge cases."""
    rows = []
    r = torch.zeros(K)
    r[0] = 127.0
    r[1:min(K, 241)] = torch.arange(-120, 120)[: min(K, 241) - 1].float() + 0.5  # exact ties, s = 1
    rows.append(r)
    a = 3.7
    s = torch.tensor(a, dtype=torch.float32) / 127.0
    r = torch.zeros(K)
    r[0] = a
    n = min(K - 1, 200)
    r[1:1 + n] = (torch.arange(n).float() - n / 2 + 0.5) * s  # near-ties
    rows.append(r)
    rows.append(torch.zeros(K))                                  # all zero
    rows.append(-torch.zeros(K))                                 # all -0
    rows.append(torch.randn(K, generator=torch.Generator().manual_seed(5)) * 1e-38)  # subnormal scale
    rows.append(torch.randn(K, generator=torch.Generator().manual_seed(6)) * 1e30)
    r = torch.zeros(K)
    r[K - 1] = -1.0
    rows.append(r)                                               # single negative element
    return torch.stack(rows).to(torch.bfloat16)


# ----------------------------------------------------------------- quantization
@pytest.mark.parametrize("M,K", [(1, 16), (7, 256), (5, 1024), (9, 2048), (33, 4096), (300, 5120), (3, 6144),
                                 (2, 8192), (33, 13824), (5, 20480), (3, 131072)])
def test_quantize_act_per_token(w8a8, oracle, M, K):
    X = torch.cat([rand_bf16((M, K), seed=M + K, outliers=0.01, oscale=20.0), special_rows(K)])
    Xq, sx = w8a8.quantize_act(X.to(DEV), w8a8.PER_ROW)
    oq, os_ = oracle.quantize_act(bits(X), oracle.PER_ROW)
    assert np.array_equal(Xq.cpu().numpy(), oq)
    assert np.array_equal(sx.cpu().numpy().view(np.uint32), os_.view(np.uint32))


@pytest.mark.parametrize("M,K", [(6000, 2048), (1300, 8192), (3000, 5120), (2600, 8192), (2500, 13824)])
def test_quantize_act_per_token_streamed_many_units(w8a8, oracle, M, K):
    """Enough rows (at least 16 per SM from 2432 on) that the quantizer takes
    its many-row launch shapes: one 64-thread CTA per 5120-wide row, 128
    threads up to 8192, 256 up to 16384."""
    X = rand_bf16((M, K), seed=M, outliers=0.01, oscale=20.0)
    Xq, sx = w8a8.quantize_act(X.to(DEV), w8a8.PER_ROW)
    oq, os_ = oracle.quantize_act(bits(X), oracle.PER_ROW)
    assert np.array_equal(Xq.cpu().numpy(), oq)
    assert np.array_equal(sx.cpu().numpy().view(np.uint32), os_.view(np.uint32))
    assert w8a8.get_device_error() == (0, 0)


def test_scales_cover_every_absmax_mantissa(w8a8, oracle):
    """Rows whose absmax takes all 128 bf16 significands at several binary
    exponents (including ones that fall back to IEEE division), so every
    entry of the quantizer's scale tables is compared with the oracle."""
    rows = []
    for e in (-130, -126, -100, -20, -3, 0, 5, 40, 120, 126):
        for i in range(128):
            r = torch.zeros(256)
            r[7] = (128 + i) / 128.0 * 2.0 ** e
            r[100] = -(64 + i / 2) / 128.0 * 2.0 ** e
            rows.append(r)
    X = torch.stack(rows).to(torch.bfloat16)
    for mode in (w8a8.PER_ROW, w8a8.BLOCK):
        Xq, sx = w8a8.quantize_act(X.to(DEV), mode)
        oq, os_ = oracle.quantize_act(bits(X), mode)
        assert np.array_equal(Xq.cpu().numpy(), oq)
        assert np.array_equal(sx.cpu().numpy().view(np.uint32), os_.view(np.uint32))


@pytest.mark.parametrize("M,K", [(1, 128), (9, 256), (1000, 1408), (17, 13824), (4001, 4096)])
def test_quantize_act_block(w8a8, oracle, M, K):
    X = torch.cat([torch.nn.functional.gelu(rand_bf16((M, K), seed=K).float()).to(torch.bfloat16),
                   special_rows(K)])
    Xq, sx = w8a8.quantize_act(X.to(DEV), w8a8.BLOCK)
    oq, os_ = oracle.quantize_act(bits(X), oracle.BLOCK)
    assert np.array_equal(Xq.cpu().numpy(), oq)
    assert np.array_equal(sx.cpu().numpy().view(np.uint32), os_.view(np.uint32))


@pytest.mark.parametrize("N,K", [(128, 128), (300, 256), (1, 1024), (129, 13824)])
def test_quantize_weight_modes(w8a8, oracle, N, K):
    W = rand_bf16((N, K), seed=N * 7 + K, scale=0.02)
    for mode in (w8a8.PER_ROW, w8a8.BLOCK):
        Wq, sw = w8a8.quantize_weight(W.to(DEV), mode)
        oq, os_ = oracle.quantize_weight(bits(W), mode)
        assert np.array_equal(Wq.cpu().numpy(), oq)
        assert np.array_equal(sw.cpu().numpy().view(np.uint32), os_.view(np.uint32))


# ----------------------------------------------------------------- post-scale GEMM
@pytest.mark.parametrize("M,N,K,bias", [
    (64, 128, 256, True),      # the tiny workload shape
    (1, 8, 16, False),         # smallest legal shape
    (300, 520, 1040, True),    # ragged M and N, K not a multiple of 64
    (257, 600, 2048, False),   # two folds of 1024 K
    (129, 264, 4112, True),    # five folds, last one 16 K
    (77, 3072, 5120, False),
    (2048, 4096, 1024, True),  # selects 224-column tiles (2 full waves of CTA pairs)
    (2432, 1792, 768, False),  # selects 256-column tiles
])
def test_gemm_postscale(w8a8, oracle, M, N, K, bias):
    check_postscale(w8a8, oracle, M, N, K, bias)


# Few tokens, both routes.  The GEMM on int8 codes (gemm_postscale) runs the
# GEMV or the int8-operand kernels (gemm_s8.cu).  The fused Linear on a
# packed bf16 image (linear_postscale) runs, up to 256 tokens, the swapped
# tensor-core kernel on images: weights on the 256-row side, tokens on the
# narrow side, Y written transposed, K split into int32 partials summed by a
# second kernel.  The split counts S below are those of the swapped kernel.
@pytest.mark.parametrize("M,N,K,bias", [
    (1, 4096, 4096, True),     # one token: 32-token tiles, S = 4
    (16, 24, 128, False),      # fewer output columns than one store box, S = 1
    (32, 520, 1040, True),     # S = 4, the last split ends in a 16-wide K stage
    (33, 1000, 2048, False),   # 64-token tiles, S = 8
    (64, 776, 512, True),      # S = 2
    (65, 304, 1408, True),     # 128-token tiles, S = 5
    (128, 257, 256, False),    # N % 8 != 0: direct stores, S = 1
    (200, 1536, 3072, True),   # 256-token tiles, S = 8
    (256, 2048, 1024, False),  # the largest swapped M, S = 4
    (77, 9728, 1024, True),    # 38 weight tiles: no split, TMA stores
    (3, 10000, 256, False),    # 40 weight tiles, no split, ragged last tile
])
def test_gemm_postscale_few_tokens(w8a8, oracle, M, N, K, bias):
    check_postscale(w8a8, oracle, M, N, K, bias)
    check_linear_image(w8a8, oracle, M, N, K, bias)


# The int8-operand kernels at their boundaries: every token tile (16, 32, 64,
# 96 on the narrow kernel; 128, 160, 192, 224, 256 in two token parts and 288
# in three on the wide one), both sides of the split rule (at most 76 weight
# tiles and 256 K per split), a last stage of 16 K (zero-filled past K), and
# a last weight tile of one row.
@pytest.mark.parametrize("M,N,K,bias", [
    (5, 300, 5120, True),      # 16-token tile, 3 weight tiles: K split 8 ways
    (17, 1000, 1040, False),   # 32-token tile, 9 stages (the last 16 K): split 3 ways
    (96, 9728, 640, True),     # 96-token tile, 76 weight tiles: split 2 ways
    (97, 9856, 512, False),    # wide 128-token tile, 77 weight tiles: no split
    (64, 129, 16400, True),    # a last weight tile of one row, 129 stages, split 8 ways
    (128, 2048, 384, False),   # 6 stages of 64 K: too few to split
    (120, 700, 4096, True),    # wide 128-token tile, 6 weight tiles: split 8 ways
    (129, 300, 5120, True),    # 160-token tile (half 1 mostly zero rows): split 8 ways
    (160, 1000, 1040, False),  # 160 exactly, 17 stages of 64 K (the last 16 K): split 4 ways
    (193, 9728, 640, True),    # 224-token tile, 76 weight tiles, one SM each: no split
    (250, 2048, 384, False),   # 256-token tile, 6 stages: too few to split
    (257, 9856, 2048, False),  # 288-token tile, 77 weight tiles, two 1024-K chunks: no split
    (288, 129, 16400, True),   # 288 exactly, a last weight tile of one row, 257 stages: split 8 ways
    (200, 3072, 5120, True),   # 224-token tile at a model shape: 24 tiles, split 6 ways
    (77, 19200, 1024, True),   # 150 weight tiles: some CTAs take two units (narrow kernel)
    (200, 19200, 1040, False), # the same on the wide kernel: the region table carries over units
    (288, 20000, 2048, True),  # three token parts over two units, two chunks per unit
    (130, 64, 16, True),       # wide kernel, K shorter than one 64-K stage (zero-filled past K)
    (97, 1, 48, False),        # one weight row: the tile's other 127 rows past N
    (6, 1, 4096, True),        # the same on the narrow kernel, K split 8 ways
])
def test_gemm_postscale_int8_operands(w8a8, oracle, M, N, K, bias):
    check_postscale(w8a8, oracle, M, N, K, bias)


@pytest.mark.parametrize("M", [77, 200])
def test_int8_operands_repeatable_after_fresh_quantization(w8a8, M):
    """The int8-operand kernels right after the quantization kernels that
    produce their operands, on fresh inputs every time: two GEMMs on the same
    codes must agree bit for bit, 150 times over.  The narrow kernel's two
    converter warpgroups take alternate stages of an odd-length ring; with one
    full barrier per slot, a group could pass its wait while the other
    group's earlier copy into the slot was still landing (copies complete out
    of order), and convert a half-written stage -- a wrong tile, or a stall,
    a few times in a few hundred launches."""
    N, K = 13824, 5120
    g = torch.Generator(device=DEV).manual_seed(7)
    for _ in range(150):
        X = torch.randn((M, K), generator=g, device=DEV).to(torch.bfloat16)
        W = (0.02 * torch.randn((N, K), generator=g, device=DEV)).to(torch.bfloat16)
        Xq, sx = w8a8.quantize_act(X)
        Wq, sw = w8a8.quantize_weight(W)
        Y1 = w8a8.gemm_postscale(Xq, sx, Wq, sw)
        Y2 = w8a8.gemm_postscale(Xq, sx, Wq, sw)
        assert torch.equal(Y1, Y2)
    assert w8a8.get_device_error() == (0, 0)


# At most 4 tokens (M * K <= 131072): a CUDA-core GEMV on the int8 codes
# (dp4a), the activation codes staged in each CTA's shared memory by one bulk
# copy.  Warps own balanced ranges of weight-row groups (1 row for up to 2
# tokens, and for 3..4 with N <= 4096; else 2 rows) and walk each row in steps
# of 4 x 512 bytes, prefetching the next
# step.  The shapes cover every token count, K shorter than one slice, a
# partial last step, many steps per row, N below one group per warp, odd,
# and larger than the persistent grid's warp count, the shared-memory limit,
# and shapes past it; 5..8 tokens take the int8-operand tensor-core kernel
# (its 16-token tile).
@pytest.mark.parametrize("M,N,K,bias", [
    (1, 1, 16, True),          # one output, one 16-byte slice
    (2, 3, 48, False),
    (3, 7, 528, True),         # partial step
    (4, 33, 2064, False),
    (5, 300, 5120, True),
    (6, 1031, 1040, False),
    (7, 64, 16384, True),      # 16 steps per row
    (8, 777, 4112, True),      # the tensor-core kernel's 16-token tile, odd N
    (1, 3072, 5120, False),    # the decode shape
    (4, 4096, 5120, False),    # the largest N with one row per warp at 4 tokens
    (3, 4097, 528, True),      # odd N with 2-row groups, partial step
    (4, 9999, 256, False),     # more row groups than the grid's warps
    (4, 300, 32768, True),     # 128 KB of codes: the shared-memory limit
    (4, 100, 32784, False),    # past it: the tensor-core kernel
    (8, 300, 16384, True),
])
def test_gemm_postscale_gemv(w8a8, oracle, M, N, K, bias):
    check_postscale(w8a8, oracle, M, N, K, bias)


# The GEMV on long weight streams (N * K >= 2^22): several row groups per
# warp, an odd row count, K ending in a partial 512-byte slice.
@pytest.mark.parametrize("M,N,K,bias", [
    (1, 8192, 4096, True),
    (2, 4096, 4096, False),
    (3, 1031, 16384, True),
    (4, 2000, 2064, False),
])
def test_gemm_postscale_gemv_long(w8a8, oracle, M, N, K, bias):
    check_postscale(w8a8, oracle, M, N, K, bias)


@pytest.mark.parametrize("M,N,K", [(1, 24, 131072), (4, 40, 32768)])
def test_gemv_exactness_at_max_k(w8a8, oracle, M, N, K):
    """All-+-127 codes at the largest K the GEMV takes for this M: at one
    token |acc| reaches 127*127*131072 = 2,114,060,288, just inside int32."""
    g = torch.Generator().manual_seed(12)
    Xq = ((torch.randint(0, 2, (M, K), generator=g) * 2 - 1) * 127).to(torch.int8)
    Wq = ((torch.randint(0, 2, (N, K), generator=g) * 2 - 1) * 127).to(torch.int8)
    Xq[0] = 127
    Wq[0] = 127
    Wq[1] = -127
    assert w8a8.gemv_takes(M, K)
    ref = oracle.gemm_s32(Xq.numpy(), Wq.numpy())
    acc = w8a8.gemm_postscale_s32(Xq.to(DEV), Wq.to(DEV)).cpu().numpy()
    assert acc[0, 0] == 16129 * K and acc[0, 1] == -16129 * K
    assert np.array_equal(acc, ref)
    assert w8a8.get_device_error() == (0, 0)


def check_postscale(w8a8, oracle, M, N, K, bias):
    X = rand_bf16((M, K), seed=1 + M, outliers=0.01, oscale=20.0)
    W = rand_bf16((N, K), seed=2 + N, scale=0.02)
    b = rand_bf16((N,), seed=3, scale=0.01) if bias else None
    ref = oracle.linear_postscale(bits(X), bits(W), None if b is None else bits(b))
    Xq, sx = w8a8.quantize_act(X.to(DEV))
    Wq, sw = w8a8.quantize_weight(W.to(DEV))
    acc = w8a8.gemm_postscale_s32(Xq, Wq)
    Y = w8a8.gemm_postscale(Xq, sx, Wq, sw, None if b is None else b.to(DEV))
    assert np.array_equal(Xq.cpu().numpy(), ref["Xq"])
    assert np.array_equal(Wq.cpu().numpy(), ref["Wq"])
    assert np.array_equal(acc.cpu().numpy(), ref["acc"])
    d = assert_bf16_close(bits(Y), ref["Y"], 1)
    assert d.max() == 0  # same op order on both sides: expect bit-exact
    assert w8a8.get_device_error() == (0, 0)


@pytest.mark.parametrize("M", [16, 200])
def test_int8_operands_exactness_at_max_k(w8a8, oracle, M):
    """The int8-operand kernels at the largest K (131072, K split 8 ways)
    with all-+-127 codes: |acc| reaches 127*127*131072 = 2,114,060,288, just
    inside int32, and the split sums add up exactly; a ragged last weight
    tile (136 rows).  16 tokens: the narrow kernel (units of 16 exact fp32
    chunks); 200 tokens: the wide kernel, its token parts rotating through
    the accumulator regions over 2048 stages of 64 K."""
    N, K = 136, 131072
    g = torch.Generator().manual_seed(21)
    Xq = ((torch.randint(0, 2, (M, K), generator=g) * 2 - 1) * 127).to(torch.int8)
    Wq = ((torch.randint(0, 2, (N, K), generator=g) * 2 - 1) * 127).to(torch.int8)
    Xq[0] = 127
    Wq[0] = 127
    Wq[135] = -127
    ref = oracle.gemm_s32(Xq.numpy(), Wq.numpy())
    acc = w8a8.gemm_postscale_s32(Xq.to(DEV), Wq.to(DEV)).cpu().numpy()
    assert acc[0, 0] == 16129 * K and acc[0, 135] == -16129 * K
    assert np.array_equal(acc, ref)
    assert w8a8.get_device_error() == (0, 0)


@pytest.mark.parametrize("M", [16, 77, 130, 288, 520])  # int8-operand kernels (K split 8 ways) / regular
def test_gemm_exactness_adversary(w8a8, oracle, M):
    """All-+-127 operands at K = 13824: per-chunk partial sums reach
    127*127*1024 and the total 2.2e8, far past fp32's 2^24 integer range."""
    N, K = 260, 13824
    g = torch.Generator().manual_seed(11)
    sgn_x = torch.randint(0, 2, (M, K), generator=g) * 2 - 1
    sgn_w = torch.randint(0, 2, (N, K), generator=g) * 2 - 1
    Xq = (sgn_x * 127).to(torch.int8)
    Wq = (sgn_w * 127).to(torch.int8)
    Xq[0] = 127
    Wq[0] = 127          # acc[0,0] = 16129 * K
    Wq[1] = -127         # acc[0,1] = -16129 * K
    Xq[1, ::2] = -127
    Xq[1, 1::2] = 127    # row 1: alternating signs
    ref = oracle.gemm_s32(Xq.numpy(), Wq.numpy())
    acc = w8a8.gemm_postscale_s32(Xq.to(DEV), Wq.to(DEV)).cpu().numpy()
    assert acc[0, 0] == 16129 * K and acc[0, 1] == -16129 * K
    assert np.array_equal(acc, ref)
    # near 2^24 inside one chunk: values that a 24-bit accumulator would round
    Xq2 = torch.full((M, 1024), 127, dtype=torch.int8)
    Wq2 = torch.full((256, 1024), 127, dtype=torch.int8)
    Wq2[:, :7] = torch.arange(1, 8, dtype=torch.int8)  # odd offsets from the all-127 sum
    ref2 = oracle.gemm_s32(Xq2.numpy(), Wq2.numpy())
    acc2 = w8a8.gemm_postscale_s32(Xq2.to(DEV), Wq2.to(DEV)).cpu().numpy()
    assert np.array_equal(acc2, ref2)


def test_gemm_zero_and_degenerate(w8a8, oracle):
    # M = 0 and N = 0 launch nothing and succeed
    Xq = torch.zeros((0, 64), dtype=torch.int8, device=DEV)
    Wq = torch.zeros((16, 64), dtype=torch.int8, device=DEV)
    Y = w8a8.gemm_postscale(Xq, torch.zeros(0, device=DEV), Wq, torch.ones(16, device=DEV))
    assert Y.shape == (0, 16)
    # all-zero activations: Y == bias exactly, or +0 without bias
    X = torch.zeros((5, 64), dtype=torch.bfloat16)
    W = rand_bf16((16, 64), seed=9, scale=0.02)
    b = rand_bf16((16,), seed=10, scale=0.01)
    Xq, sx = w8a8.quantize_act(X.to(DEV))
    Wq, sw = w8a8.quantize_weight(W.to(DEV))
    assert torch.all(sx == 0)
    Y = w8a8.gemm_postscale(Xq, sx, Wq, sw, b.to(DEV))
    assert np.array_equal(bits(Y), np.stack([bits(b)] * 5))
    Y0 = w8a8.gemm_postscale(Xq, sx, Wq, sw, None)
    assert np.all(bits(Y0) == 0)


def test_gemm_rejects_bad_arguments(w8a8):
    Xq = torch.zeros((4, 24), dtype=torch.int8, device=DEV)
    Wq = torch.zeros((4, 24), dtype=torch.int8, device=DEV)
    with pytest.raises(w8a8.W8A8Error, match="SHAPE"):
        w8a8.gemm_postscale(Xq, torch.ones(4, device=DEV), Wq, torch.ones(4, device=DEV))
    Xq = torch.zeros((4, 33), dtype=torch.int8, device=DEV)[:, 1:]
    with pytest.raises(ValueError):
        w8a8.gemm_postscale(Xq, torch.ones(4, device=DEV), Wq, torch.ones(4, device=DEV))
    # more than 288 tokens: the bf16-image path, which needs the whole workspace
    with pytest.raises(w8a8.W8A8Error, match="WORKSPACE"):
        w8a8.gemm_postscale(torch.zeros((300, 32), dtype=torch.int8, device=DEV), torch.ones(300, device=DEV),
                            torch.zeros((4, 32), dtype=torch.int8, device=DEV), torch.ones(4, device=DEV),
                            workspace=torch.empty(16, dtype=torch.uint8, device=DEV))
    # 5..288 tokens stream the int8 codes and need only the fp16 image of Xq
    # (K too short to split): 16 x 32 x 2 bytes, rounded up to 256
    args = (torch.ones((16, 32), dtype=torch.int8, device=DEV), torch.ones(16, device=DEV),
            torch.ones((4, 32), dtype=torch.int8, device=DEV), torch.ones(4, device=DEV))
    with pytest.raises(w8a8.W8A8Error, match="WORKSPACE"):
        w8a8.gemm_postscale(*args, workspace=torch.empty(768, dtype=torch.uint8, device=DEV))
    Y = w8a8.gemm_postscale(*args, workspace=torch.empty(1024, dtype=torch.uint8, device=DEV))
    assert torch.all(Y.float() == 32.0)
    # up to 4 tokens the GEMV needs no workspace: a short one is fine
    Y = w8a8.gemm_postscale(torch.ones((4, 32), dtype=torch.int8, device=DEV), torch.ones(4, device=DEV),
                            torch.ones((4, 32), dtype=torch.int8, device=DEV), torch.ones(4, device=DEV),
                            workspace=torch.empty(16, dtype=torch.uint8, device=DEV))
    assert torch.all(Y.float() == 32.0)


# ----------------------------------------------------------------- blockwise GEMM
@pytest.mark.parametrize("M,N,K,bias", [
    (64, 256, 256, False),
    (300, 456, 1408, True),    # ragged N (456 = 3.6 weight blocks), 11 K blocks
    (129, 5120, 1024, False),
    (1, 130, 13824, False),    # 108 K blocks, M = 1, partial last weight block
])
def test_gemm_blockwise(w8a8, oracle, M, N, K, bias):
    X = torch.nn.functional.gelu(rand_bf16((M, K), seed=20 + M).float()).to(torch.bfloat16)
    W = rand_bf16((N, K), seed=21 + N, scale=0.01)
    b = rand_bf16((N,), seed=22, scale=0.01) if bias else None
    ref = oracle.linear_blockwise(bits(X), bits(W), None if b is None else bits(b))
    Xq, sx = w8a8.quantize_act(X.to(DEV), w8a8.BLOCK)
    Wq, sw = w8a8.quantize_weight(W.to(DEV), w8a8.BLOCK)
    acc = w8a8.gemm_blockwise_f32(Xq, sx, Wq, sw)
    Y = w8a8.gemm_blockwise(Xq, sx, Wq, sw, None if b is None else b.to(DEV))
    assert np.array_equal(sx.cpu().numpy().view(np.uint32), ref["sx"].view(np.uint32))
    assert np.array_equal(sw.cpu().numpy().view(np.uint32), ref["sw"].view(np.uint32))
    assert np.array_equal(acc.cpu().numpy().view(np.uint32), ref["acc"].view(np.uint32))
    d = assert_bf16_close(bits(Y), ref["Y"], 1)
    assert d.max() == 0
    assert w8a8.get_device_error() == (0, 0)


def test_blockwise_adversary(w8a8, oracle):
    """Every 128-K block partial at its extreme +-2,064,512 with unit scales:
    the fp32 fold of 108 such blocks rounds, identically on both sides."""
    M, N, K = 128, 256, 13824
    Xq = torch.full((M, K), 127, dtype=torch.int8)
    Wq = torch.full((N, K), 127, dtype=torch.int8)
    Wq[1::2, ::3] = -127
    kbs = K // 128
    sx = torch.ones((M, kbs)) * 1.0000001
    sw = torch.ones(((N + 127) // 128, kbs)) * 0.999999
    ref = oracle.gemm_blockwise_f32(Xq.numpy(), sx.numpy(), Wq.numpy(), sw.numpy())
    acc = w8a8.gemm_blockwise_f32(Xq.to(DEV), sx.to(DEV), Wq.to(DEV), sw.to(DEV)).cpu().numpy()
    assert np.array_equal(acc.view(np.uint32), ref.view(np.uint32))


# ----------------------------------------------------------------- fused Linear entry points
def test_pack_weight_is_exact_image(w8a8):
    g = torch.Generator().manual_seed(31)
    Wq = torch.randint(-127, 128, (300, 1040), generator=g, dtype=torch.int8)
    Wimg = w8a8.pack_weight(Wq.to(DEV))
    assert torch.equal(Wimg.cpu().float(), Wq.float())
    assert np.array_equal(bits(Wimg), bits(Wq.to(torch.bfloat16)))


@pytest.mark.parametrize("M,N,K,bias", [(64, 128, 256, True), (300, 520, 1040, True), (2048, 4096, 1024, False),
                                        (77, 3072, 5120, True), (5, 4096, 4096, False), (2500, 256, 5120, True),
                                        (2600, 136, 8192, False)])
def test_linear_postscale_fused(w8a8, oracle, M, N, K, bias):
    check_linear_image(w8a8, oracle, M, N, K, bias)


def check_linear_image(w8a8, oracle, M, N, K, bias):
    """The fused Linear on a packed weight image against the oracle."""
    X = rand_bf16((M, K), seed=40 + M, outliers=0.01, oscale=20.0)
    W = rand_bf16((N, K), seed=41 + N, scale=0.02)
    b = rand_bf16((N,), seed=42, scale=0.01) if bias else None
    ref = oracle.linear_postscale(bits(X), bits(W), None if b is None else bits(b))
    Wq, sw = w8a8.quantize_weight(W.to(DEV))
    Wimg = w8a8.pack_weight(Wq)
    Y, sx, Xq = w8a8.linear_postscale(X.to(DEV), Wimg, sw, None if b is None else b.to(DEV), codes=True)
    assert np.array_equal(Xq.cpu().numpy(), ref["Xq"])
    assert np.array_equal(sx.cpu().numpy().view(np.uint32), ref["sx"].view(np.uint32))
    d = assert_bf16_close(bits(Y), ref["Y"], 1)
    assert d.max() == 0
    # without codes requested: same output
    Y2, _, none = w8a8.linear_postscale(X.to(DEV), Wimg, sw, None if b is None else b.to(DEV))
    assert none is None and torch.equal(Y2, Y)
    assert w8a8.get_device_error() == (0, 0)


# The fused Linear on int8 weight codes: one GEMV kernel that quantizes X in
# every CTA for one or two tokens (M * K <= 131072); the quantization kernel
# and then the GEMV (weights read before its dependency wait) up to 4 tokens;
# else the quantization kernel and the int8-operand tensor-core kernels (up
# to 288 tokens) or operand images.
@pytest.mark.parametrize("M,N,K,bias", [(1, 3072, 5120, True), (2, 1000, 4096, False), (2, 7, 16, True),
                                        (3, 520, 1040, False), (8, 4096, 4096, True),
                                        (5, 1000, 16, True), (8, 520, 16384, False), (1, 300, 131072, True),
                                        (2, 300, 131072, False), (9, 600, 2048, True), (77, 3072, 5120, False),
                                        (6, 100, 32768, True), (2, 2048, 4112, True), (1, 4096, 2048, False),
                                        (257, 3072, 5120, True), (140, 13824, 1024, False),
                                        (288, 600, 32768, True), (300, 520, 1040, True)])
def test_linear_postscale_codes(w8a8, oracle, M, N, K, bias):
    X = rand_bf16((M, K), seed=45 + M, outliers=0.01, oscale=20.0)
    W = rand_bf16((N, K), seed=46 + N, scale=0.02)
    b = rand_bf16((N,), seed=47, scale=0.01) if bias else None
    ref = oracle.linear_postscale(bits(X), bits(W), None if b is None else bits(b))
    Wq, sw = w8a8.quantize_weight(W.to(DEV))
    bd = None if b is None else b.to(DEV)
    # scales buffer filled with NaN: no CTA may read a scale another CTA writes
    sx0 = torch.full((M,), float("nan"), device=DEV)
    Y, sx, Xq = w8a8.linear_postscale_codes(X.to(DEV), Wq, sw, bd, codes=True, sx_out=sx0)
    assert np.array_equal(Xq.cpu().numpy(), ref["Xq"])
    assert np.array_equal(sx.cpu().numpy().view(np.uint32), ref["sx"].view(np.uint32))
    d = assert_bf16_close(bits(Y), ref["Y"], 1)
    assert d.max() == 0
    # codes kept in the workspace instead: same output
    Y2, _, none = w8a8.linear_postscale_codes(X.to(DEV), Wq, sw, bd)
    assert none is None and torch.equal(Y2, Y)
    assert w8a8.get_device_error() == (0, 0)


def test_linear_postscale_codes_rejects_bad_arguments(w8a8):
    X = torch.zeros((4, 64), dtype=torch.bfloat16, device=DEV)
    Wq = torch.zeros((8, 64), dtype=torch.int8, device=DEV)
    sw = torch.ones(8, device=DEV)
    with pytest.raises(w8a8.W8A8Error, match="WORKSPACE"):
        w8a8.linear_postscale_codes(torch.zeros((16, 64), dtype=torch.bfloat16, device=DEV), Wq, sw,
                                    workspace=torch.empty(16, dtype=torch.uint8, device=DEV))
    with pytest.raises(w8a8.W8A8Error, match="SHAPE"):
        w8a8.linear_postscale_codes(torch.zeros((4, 24), dtype=torch.bfloat16, device=DEV),
                                    torch.zeros((8, 24), dtype=torch.int8, device=DEV), sw)
    Y, sx, _ = w8a8.linear_postscale_codes(torch.zeros((0, 64), dtype=torch.bfloat16, device=DEV), Wq, sw)
    assert Y.shape == (0, 8)
    # all-zero tokens: the output is the bias exactly
    b = rand_bf16((8,), seed=48).to(DEV)
    Y, sx, _ = w8a8.linear_postscale_codes(X, Wq, sw, b)
    assert torch.equal(Y, b.expand(4, 8)) and torch.all(sx == 0)


@pytest.mark.parametrize("M,N,K,bias", [(64, 256, 256, False), (300, 456, 1408, True), (1, 130, 13824, False)])
def test_linear_blockwise_fused(w8a8, oracle, M, N, K, bias):
    X = torch.nn.functional.gelu(rand_bf16((M, K), seed=50 + M).float()).to(torch.bfloat16)
    W = rand_bf16((N, K), seed=51 + N, scale=0.01)
    b = rand_bf16((N,), seed=52, scale=0.01) if bias else None
    ref = oracle.linear_blockwise(bits(X), bits(W), None if b is None else bits(b))
    Wq, sw = w8a8.quantize_weight(W.to(DEV), w8a8.BLOCK)
    Y, sx, Xq = w8a8.linear_blockwise(X.to(DEV), w8a8.pack_weight(Wq), sw, None if b is None else b.to(DEV),
                                      codes=True)
    assert np.array_equal(Xq.cpu().numpy(), ref["Xq"])
    assert np.array_equal(sx.cpu().numpy().view(np.uint32), ref["sx"].view(np.uint32))
    d = assert_bf16_close(bits(Y), ref["Y"], 1)
    assert d.max() == 0


def test_linear_fused_rejects_bad_arguments(w8a8):
    X = torch.zeros((4, 64), dtype=torch.bfloat16, device=DEV)
    Wimg = torch.zeros((8, 64), dtype=torch.bfloat16, device=DEV)
    sw = torch.ones(8, device=DEV)
    with pytest.raises(w8a8.W8A8Error, match="WORKSPACE"):
        w8a8.linear_postscale(X, Wimg, sw, workspace=torch.empty(16, dtype=torch.uint8, device=DEV))
    with pytest.raises(w8a8.W8A8Error, match="SHAPE"):
        w8a8.linear_blockwise(X, Wimg, torch.ones((1, 1), device=DEV))
    Y, sx, _ = w8a8.linear_postscale(torch.zeros((0, 64), dtype=torch.bfloat16, device=DEV), Wimg, sw)
    assert Y.shape == (0, 8)


# ----------------------------------------------------------------- Int8Linear module
@pytest.mark.parametrize("mode", ["postscale", "blockwise"])
def test_int8linear_module(w8a8, oracle, mode):
    from w8a8_int8_linear_gb300.module import Int8Linear
    torch.manual_seed(0)
    lin = torch.nn.Linear(384, 200, bias=True).to(DEV).to(torch.bfloat16)
    m = Int8Linear.from_linear(lin, mode)
    x = rand_bf16((3, 5, 384), seed=60).to(DEV)  # leading dims are flattened
    y = m(x)
    assert y.shape == (3, 5, 200) and y.dtype == torch.bfloat16
    X = bits(x.reshape(15, 384))
    W = bits(lin.weight)
    b = bits(lin.bias)
    ref = oracle.linear_postscale(X, W, b) if mode == "postscale" else oracle.linear_blockwise(X, W, b)
    d = assert_bf16_close(bits(y.reshape(15, 200)), ref["Y"], 1)
    assert d.max() == 0


@pytest.mark.parametrize("M", [1, 4, 8, 120, 250])
def test_int8linear_module_decode(w8a8, oracle, M):
    """With few tokens the post-scale module runs on the int8 codes: the GEMV
    up to 4 tokens, the int8-operand tensor-core kernels beyond (the wide
    one from 97 tokens; codes_preferred up to 256 at any N)."""
    from w8a8_int8_linear_gb300.module import Int8Linear
    torch.manual_seed(2)
    lin = torch.nn.Linear(1040, 300, bias=True).to(DEV).to(torch.bfloat16)
    m = Int8Linear.from_linear(lin)
    x = rand_bf16((M, 1, 1040), seed=62 + M, outliers=0.01, oscale=20.0).to(DEV)
    y = m(x)
    assert y.shape == (M, 1, 300)
    ref = oracle.linear_postscale(bits(x.reshape(M, 1040)), bits(lin.weight), bits(lin.bias))
    d = assert_bf16_close(bits(y.reshape(M, 300)), ref["Y"], 1)
    assert d.max() == 0


# ----------------------------------------------------------------- host-to-host pipeline
def test_host_pipeline_matches_direct_calls(w8a8):
    """HostPipeline overlaps each batch's copies with its neighbours' Linears;
    every result equals a direct call on the same batch, at every depth."""
    M, N, K = 300, 520, 1040
    W = rand_bf16((N, K), seed=90, scale=0.02).to(DEV)
    Wq, sw = w8a8.quantize_weight(W)
    Wimg = w8a8.pack_weight(Wq)
    b = rand_bf16((N,), seed=91, scale=0.01).to(DEV)
    xs = [rand_bf16((M, K), seed=100 + i, outliers=0.01, oscale=20.0).pin_memory() for i in range(7)]
    ys = [torch.empty((M, N), dtype=torch.bfloat16).pin_memory() for _ in range(7)]
    ws = torch.empty(w8a8.linear_workspace_size(M, N, K), dtype=torch.uint8, device=DEV)
    refs = [w8a8.linear_postscale(x.to(DEV), Wimg, sw, b)[0].cpu() for x in xs]
    for depth in (1, 2, 3):
        for y in ys:
            y.fill_(float("nan"))
        pipe = w8a8.HostPipeline(lambda X, Y: w8a8.linear_postscale(X, Wimg, sw, b, out=Y, workspace=ws),
                                 (M, K), (M, N), DEV, depth=depth)
        pipe.run(xs, ys)
        torch.cuda.synchronize()
        for y, r in zip(ys, refs):
            assert torch.equal(y, r)
    # one token per batch on the weight codes, the batch index picking a weight copy
    Wq2 = [Wq, Wq.flip(0).contiguous()]
    sw2 = [sw, sw.flip(0).contiguous()]
    xs1 = [x[:1].contiguous().pin_memory() for x in xs]
    ys1 = [torch.empty((1, N), dtype=torch.bfloat16).pin_memory() for _ in xs1]
    pipe = w8a8.HostPipeline(lambda X, Y, i: w8a8.linear_postscale_codes(X, Wq2[i % 2], sw2[i % 2], None, out=Y),
                             (1, K), (1, N), DEV, depth=2, pass_index=True)
    pipe.run(xs1, ys1)
    torch.cuda.synchronize()
    for i, (x, y) in enumerate(zip(xs1, ys1)):
        ref, _, _ = w8a8.linear_postscale_codes(x.to(DEV), Wq2[i % 2], sw2[i % 2], None)
        assert torch.equal(y, ref.cpu())
    assert w8a8.get_device_error() == (0, 0)


# ----------------------------------------------------------------- FFN up: GELU + 1x128 quantization epilogue
def _bf16_dev(u16):
    """uint16 bf16 bit patterns (numpy) -> bf16 CUDA tensor."""
    return torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).view(torch.bfloat16).to(DEV)


def test_gelu_export_matches_plain_definition_on_every_bf16(w8a8, oracle):
    """The epilogue's GELU (through its test export) on every bf16 bit
    pattern against the plain definition x * Phi(x) (fp64 erfc, rounded to
    fp32 and bf16): within 1 ulp on every finite input, and identical except
    on at most a handful of inputs whose exact value lies within the
    kernel's error of a bf16 rounding boundary."""
    allbits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = (allbits.astype(np.uint32) << 16).view(np.float32)
    fin = np.isfinite(vals)
    G = bits(w8a8.gelu_bf16(_bf16_dev(allbits)))
    Gp = oracle.gelu_bf16(allbits[fin])
    d = bf16_ulp_distance(G[fin], Gp)
    assert d.max() <= 1
    assert (d > 0).sum() <= 4, f"differing inputs: {vals[fin][d > 0]}"
    # tails: g = x from 4 up, -0 from -14 down, tiny negatives near -10
    x = vals[fin]
    assert np.array_equal(G[fin][x >= 4.0], allbits[fin][x >= 4.0])
    assert np.all(G[fin][x <= -14.0] == 0x8000)
    assert w8a8.get_device_error() == (0, 0)


@pytest.mark.parametrize("M,N,K,bias", [
    (64, 256, 256, True),      # one tile
    (5, 384, 512, True),       # few tokens (this epilogue never swaps operands)
    (300, 640, 1040, True),    # ragged M, K not a multiple of 64
    (1000, 1408, 2048, False),
    (2100, 2560, 512, True),   # several tiles in both directions
])
def test_ffn_up_gelu_quant(w8a8, oracle, M, N, K, bias):
    """Codes and 1x128 scales of bf16(gelu(y)) against the plain oracle (erf
    GELU in fp64): bit-exact wherever a block's GELU values agree, and always
    the plain quantization of the kernel's own GELU values (from the test
    export applied to the oracle's y, which the post-scale epilogue
    reproduces bit for bit)."""
    X = rand_bf16((M, K), seed=40 + M, outliers=0.01, oscale=20.0)
    W = rand_bf16((N, K), seed=41 + N, scale=0.05)
    b = rand_bf16((N,), seed=42, scale=0.5) if bias else None
    tail_blocks = bias and N >= 384
    if tail_blocks:
        # blocks whose GELU output is tiny (y ~ -6) or exactly zero (y ~ -1000)
        b[128:256] = -6.0
        b[-128:] = -1000.0
    ref = oracle.ffn_up_gelu_quant(bits(X), bits(W), None if b is None else bits(b))
    Wq, sw = w8a8.quantize_weight(W.to(DEV))
    G, sg, sx, Xq = w8a8.linear_postscale_gelu_quant(X.to(DEV), w8a8.pack_weight(Wq), sw,
                                                      None if b is None else b.to(DEV), codes=True)
    assert np.array_equal(Xq.cpu().numpy(), ref["Xq"])
    assert np.array_equal(sx.cpu().numpy().view(np.uint32), ref["sx"].view(np.uint32))
    Gf = G.float().cpu()
    assert torch.equal(Gf, Gf.round()) and Gf.abs().max() <= 127
    Gk = bits(w8a8.gelu_bf16(_bf16_dev(ref["Y"])))
    differing = assert_quant_follows_plain(oracle, Gk, ref["G"], Gf.to(torch.int8).numpy(), sg.cpu().numpy(),
                                           ref["Gq"], ref["sg"], 128)
    assert differing <= max(1, ref["sg"].size // 100)
    if tail_blocks:
        assert np.all(ref["sg"][:, -1] == 0) and np.all(ref["sg"][:, 1] > 0)
        assert np.array_equal(sg.cpu().numpy()[:, -1], ref["sg"][:, -1])
    assert w8a8.get_device_error() == (0, 0)
    # the blockwise down-projection consumes the image and the 1x128 scales
    N2 = 200
    W2 = rand_bf16((N2, N), seed=43, scale=0.02)
    Wq2, sw2 = w8a8.quantize_weight(W2.to(DEV), w8a8.BLOCK)
    Y2 = w8a8.gemm_blockwise_images(G, sg, w8a8.pack_weight(Wq2), sw2)
    oWq2, osw2 = oracle.quantize_weight(bits(W2), oracle.BLOCK)
    acc2 = oracle.gemm_blockwise_f32(Gf.to(torch.int8).numpy(), sg.cpu().numpy(), oWq2, osw2)
    d = assert_bf16_close(bits(Y2), oracle.epilogue_blockwise(acc2), 1)
    assert d.max() == 0


def test_ffn_up_gelu_quant_rejects_bad_arguments(w8a8):
    X = torch.zeros((4, 64), dtype=torch.bfloat16, device=DEV)
    Wimg = torch.zeros((200, 64), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(w8a8.W8A8Error, match="SHAPE"):  # N not a multiple of 128
        w8a8.linear_postscale_gelu_quant(X, Wimg, torch.ones(200, device=DEV))


# ----------------------------------------------------------------- normalization fused with quantization
@pytest.mark.parametrize("layer", [False, True])
@pytest.mark.parametrize("M,K", [(1, 8), (7, 128), (33, 264), (300, 4096), (64, 5120), (9, 8192), (11, 8200),
                                 (5, 13824), (3, 16384), (1000, 1040)])
def test_norm_quant(w8a8, oracle, layer, M, K):
    """Against the plain definition (fp64 statistics and normalization): the
    normalized bf16 row within 1 ulp, except where the exact value comes out
    of a cancellation (x close to the mean, or (x - mu) r gamma close to
    -beta), which no binary32 evaluation resolves to 1 ulp: there within the
    binary32 forward error bound (norm_error_bound), on at most 1e-5 of the
    values.  Codes and scales are the plain quantization of the kernel's row
    and equal to the plain oracle's wherever the values agree.  And bit for
    bit against the fixed-order binary32 statement the kernel evaluates."""
    X = rand_bf16((M, K), seed=60 + K, scale=2.0, outliers=0.01, oscale=30.0)
    if layer:
        X = (X.float() + 0.75).to(torch.bfloat16)  # a nonzero mean
    if M >= 7:
        X[3] = 0.0                                  # an all-zero row: y = beta (or 0), s = 0
        X[5] = 1.25                                 # a constant row
    g = rand_bf16((K,), seed=61, scale=0.2) + 1.0
    g = g.to(torch.bfloat16)
    b = rand_bf16((K,), seed=62, scale=0.2) if layer else None
    kind = oracle.LAYER_NORM if layer else oracle.RMS_NORM
    # also LayerNorm without beta, and RMSNorm given a beta (which it does not
    # use): the generic kernel for image-only calls
    other = (g, None) if layer else (g, rand_bf16((K,), seed=63, scale=0.2))
    for gg, bb in ((g, b), (None, None), other):
        args = (bits(X), None if gg is None else bits(gg), None if bb is None else bits(bb), 1e-5, kind)
        Yo, Xqo, sxo = oracle.norm_quant(*args)
        Yf, Xqf, sxf = oracle.norm_quant_fixed_order(*args)
        Ximg, sx, Xq, Y = w8a8.norm_quant(X.to(DEV), None if gg is None else gg.to(DEV),
                                          None if bb is None else bb.to(DEV), 1e-5, kind, codes=True, y=True)
        bound = norm_error_bound(bits(X), None if gg is None else bits(gg),
                                 None if (bb is None or not layer) else bits(bb), 1e-5, layer)
        assert_quant_follows_plain(oracle, bits(Y), Yo, Xq.cpu().numpy(), sx.cpu().numpy(), Xqo, sxo, K,
                                   err_bound=bound, max_frac_beyond_ulp=1e-5)
        assert np.array_equal(bits(Y), Yf)
        assert np.array_equal(Xq.cpu().numpy(), Xqf)
        assert np.array_equal(sx.cpu().numpy().view(np.uint32), sxf.view(np.uint32))
        assert torch.equal(Ximg.float().cpu(), Xq.float().cpu())
        # only the code image and the scales (the specialized kernels for
        # gamma with or without beta, rows up to 8192 elements)
        Ximg1, sx1, none_q, none_y = w8a8.norm_quant(X.to(DEV), None if gg is None else gg.to(DEV),
                                                     None if bb is None else bb.to(DEV), 1e-5, kind)
        assert none_q is None and none_y is None
        assert np.array_equal(Ximg1.float().cpu().numpy(), Xqf.astype(np.float32))
        assert np.array_equal(sx1.cpu().numpy().view(np.uint32), sxf.view(np.uint32))
    assert w8a8.get_device_error() == (0, 0)


@pytest.mark.parametrize("layer", [False, True])
@pytest.mark.parametrize("M,K", [(2000, 5120), (10000, 264), (5000, 1040)])
def test_norm_quant_many_rows(w8a8, oracle, layer, M, K):
    """Thousands of rows through the specialized kernels (gamma, beta for
    LayerNorm, code image only), rows of 33 and 130 chunks (padding chunk
    slots) and 640: codes and scales bit for bit against the fixed-order
    statement, an all-zero and a constant row included."""
    X = rand_bf16((M, K), seed=80 + K, scale=2.0, outliers=0.01, oscale=30.0)
    if layer:
        X = (X.float() - 0.5).to(torch.bfloat16)
    X[7] = 0.0
    X[M - 1] = -3.0
    g = (rand_bf16((K,), seed=81, scale=0.2) + 1.0).to(torch.bfloat16)
    b = rand_bf16((K,), seed=82, scale=0.2) if layer else None
    kind = oracle.LAYER_NORM if layer else oracle.RMS_NORM
    _, Xqf, sxf = oracle.norm_quant_fixed_order(bits(X), bits(g), None if b is None else bits(b), 1e-5, kind)
    Ximg, sx, _, _ = w8a8.norm_quant(X.to(DEV), g.to(DEV), None if b is None else b.to(DEV), 1e-5, kind)
    assert np.array_equal(Ximg.float().cpu().numpy(), Xqf.astype(np.float32))
    assert np.array_equal(sx.cpu().numpy().view(np.uint32), sxf.view(np.uint32))
    assert w8a8.get_device_error() == (0, 0)


def test_norm_then_postscale_gemm(w8a8, oracle):
    """RMSNorm -> codes image -> post-scale GEMM on images, against the oracle
    composition (few tokens, so the swapped split-K path, and a regular
    shape).  The norm's own accuracy is test_norm_quant's; here the
    fixed-order statement it matches bit for bit feeds the oracle GEMM."""
    for M, N, K in ((5, 1536, 2048), (520, 640, 1024)):
        X = rand_bf16((M, K), seed=70 + M, scale=1.5)
        g = (rand_bf16((K,), seed=71, scale=0.1) + 1.0).to(torch.bfloat16)
        W = rand_bf16((N, K), seed=72, scale=0.02)
        bias = rand_bf16((N,), seed=73, scale=0.1)
        _, Xqo, sxo = oracle.norm_quant_fixed_order(bits(X), bits(g), None, 1e-6, oracle.RMS_NORM)
        oWq, osw = oracle.quantize_weight(bits(W), oracle.PER_ROW)
        Yo = oracle.epilogue_postscale(oracle.gemm_s32(Xqo, oWq), sxo, osw, bits(bias))
        Ximg, sx, _, _ = w8a8.norm_quant(X.to(DEV), g.to(DEV), None, 1e-6, w8a8.RMS_NORM)
        Wq, sw = w8a8.quantize_weight(W.to(DEV))
        Y = w8a8.gemm_postscale_images(Ximg, sx, w8a8.pack_weight(Wq), sw, bias.to(DEV))
        d = assert_bf16_close(bits(Y), Yo, 1)
        assert d.max() == 0


def test_norm_quant_rejects_bad_arguments(w8a8):
    X = torch.zeros((4, 36), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(w8a8.W8A8Error, match="SHAPE"):       # K % 8 != 0
        w8a8.norm_quant(X)
    X = torch.zeros((2, 16392), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(w8a8.W8A8Error, match="SHAPE"):       # K > 16384
        w8a8.norm_quant(X)
    with pytest.raises(w8a8.W8A8Error, match="INVALID_ARG"):  # negative eps
        w8a8.norm_quant(torch.zeros((2, 64), dtype=torch.bfloat16, device=DEV), eps=-1.0)


def test_int8linear_with_fused_norm(w8a8, oracle):
    """Int8Linear(norm=...) = norm + per-token quant in one pass, then the
    post-scale GEMM on the code image (on the int8 codes where that is
    faster: every shape here), against the oracle composition (with the fixed-order norm
    statement that the kernel matches bit for bit; test_norm_quant checks it
    against the plain definition)."""
    torch.manual_seed(1)
    for norm, lead in (("rms", (2, 7)), ("layer", (2, 7)), ("rms", (1, 3)), ("layer", (8,))):  # 3: the GEMV; 8, 14: the int8-operand kernel
        T = int(np.prod(lead))
        W = rand_bf16((300, 512), seed=80, scale=0.03)
        b = rand_bf16((300,), seed=81, scale=0.1)
        g = (rand_bf16((512,), seed=82, scale=0.1) + 1.0).to(torch.bfloat16)
        be = rand_bf16((512,), seed=83, scale=0.1) if norm == "layer" else None
        m = w8a8.Int8Linear(W.to(DEV), b.to(DEV), norm=norm, norm_weight=g.to(DEV),
                            norm_bias=None if be is None else be.to(DEV), eps=1e-5)
        x = rand_bf16((*lead, 512), seed=84 + T, scale=2.0)
        y = m(x.to(DEV))
        assert y.shape == (*lead, 300)
        _, Xq, sx = oracle.norm_quant_fixed_order(bits(x.reshape(T, 512)), bits(g), None if be is None else bits(be), 1e-5,
                                      oracle.RMS_NORM if norm == "rms" else oracle.LAYER_NORM)
        Wq, sw = oracle.quantize_weight(bits(W), oracle.PER_ROW)
        Yo = oracle.epilogue_postscale(oracle.gemm_s32(Xq, Wq), sx, sw, bits(b))
        d = assert_bf16_close(bits(y.reshape(T, 300)), Yo, 1)
        assert d.max() == 0


def test_int8ffn_module(w8a8, oracle):
    """Int8FFN: up-projection with the GELU + 1x128 quant epilogue, then the
    blockwise down-projection on the code image, against the oracle."""
    D, H, O = 256, 384, 200
    Wu = rand_bf16((H, D), seed=90, scale=0.06)
    bu = rand_bf16((H,), seed=91, scale=0.3)
    Wd = rand_bf16((O, H), seed=92, scale=0.03)
    bd = rand_bf16((O,), seed=93, scale=0.05)
    m = w8a8.Int8FFN(Wu.to(DEV), Wd.to(DEV), bu.to(DEV), bd.to(DEV))
    x = rand_bf16((3, 11, D), seed=94)
    y = m(x.to(DEV))
    assert y.shape == (3, 11, O)
    r = oracle.ffn_up_gelu_quant(bits(x.reshape(33, D)), bits(Wu), bits(bu))
    # the kernel's GELU of the oracle's y (test_ffn_up_gelu_quant ties it to the plain definition)
    Gk = bits(w8a8.gelu_bf16(_bf16_dev(r["Y"])))
    assert bf16_ulp_distance(Gk, r["G"]).max() <= 1
    Gq, sg = oracle.quantize_act(Gk, oracle.BLOCK)
    Wq2, sw2 = oracle.quantize_weight(bits(Wd), oracle.BLOCK)
    Yo = oracle.epilogue_blockwise(oracle.gemm_blockwise_f32(Gq, sg, Wq2, sw2), bits(bd))
    d = assert_bf16_close(bits(y.reshape(33, O)), Yo, 1)
    assert d.max() == 0


# ----------------------------------------------------------------- failure detection
def test_bounded_wait_timeout_is_reported_and_the_context_survives(w8a8, oracle):
    """A kernel whose mbarrier wait nothing satisfies gives up after its
    bound, records the timeout (code 0x100 + site) and returns; the host
    reads W8A8_ERR_TIMEOUT, the word is cleared by the read, and the next
    GEMM on the same context is exact."""
    assert w8a8.get_device_error() == (0, 0)
    w8a8.probe_wait_timeout()
    st, code = w8a8.get_device_error()
    assert st == 6 and code == 0x100 + 30  # W8A8_ERR_TIMEOUT, probe site
    assert w8a8.get_device_error() == (0, 0)
    X = rand_bf16((40, 256), seed=95)
    W = rand_bf16((72, 256), seed=96, scale=0.03)
    ref = oracle.linear_postscale(bits(X), bits(W), None)
    Xq, sx = w8a8.quantize_act(X.to(DEV))
    Wq, sw = w8a8.quantize_weight(W.to(DEV))
    assert np.array_equal(bits(w8a8.gemm_postscale(Xq, sx, Wq, sw)), ref["Y"])
    assert w8a8.get_device_error() == (0, 0)
