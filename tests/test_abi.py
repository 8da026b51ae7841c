"""C-ABI checks that need no GPU: the library builds, loads, exports every
entry point include/w8a8.h declares, and rejects bad arguments before it
touches the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "w8a8.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"W8A8_API\s+[\w\s\*]+?\b(w8a8_\w+)\s*\(", src)))


@pytest.fixture(scope="module")
def cdll():
    from w8a8_int8_linear_gb300 import build as b
    path = b.build()
    import w8a8_int8_linear_gb300 as w
    return w.lib(), path


def test_header_declares_the_four_calls():
    names = declared_functions()
    for n in ("w8a8_quantize_weight", "w8a8_quantize_act", "w8a8_gemm_postscale", "w8a8_gemm_blockwise"):
        assert n in names
    assert len(names) >= 10


def test_library_exports_every_declared_symbol(cdll):
    L, path = cdll
    for name in declared_functions():
        assert hasattr(L, name), name
    from w8a8_int8_linear_gb300 import SIGNATURES
    assert sorted(n for n, _, _ in SIGNATURES) == declared_functions()


def test_status_strings(cdll):
    L, _ = cdll
    for code in range(8):
        s = L.w8a8_status_string(code).decode()
        assert s.startswith("W8A8_")
    assert L.w8a8_status_string(99).decode() == "unknown w8a8_status"


def test_argument_checks_before_device(cdll):
    """These return before any CUDA call, so they run without a GPU."""
    L, _ = cdll
    P = ctypes.c_void_p
    fake = P(0x1000)  # never dereferenced: every call below fails validation first
    odd = P(0x1001)
    null = None
    # bad mode / negative sizes
    assert L.w8a8_quantize_act(fake, 4, 16, 7, fake, fake, null) == 1
    assert L.w8a8_quantize_act(fake, -1, 16, 0, fake, fake, null) == 1
    # K rules
    assert L.w8a8_quantize_act(fake, 4, 24, 0, fake, fake, null) == 3
    assert L.w8a8_quantize_act(fake, 4, 0, 0, fake, fake, null) == 1
    assert L.w8a8_quantize_act(fake, 4, 144, 1, fake, fake, null) == 3
    assert L.w8a8_quantize_weight(fake, 4, 131072 + 16, 0, fake, fake, null) == 3
    # zero rows: nothing to do
    assert L.w8a8_quantize_act(null, 0, 16, 0, null, null, null) == 0
    assert L.w8a8_quantize_weight(null, 0, 128, 1, null, null, null) == 0
    # null / misaligned pointers
    assert L.w8a8_quantize_act(null, 4, 16, 0, fake, fake, null) == 1
    assert L.w8a8_quantize_act(odd, 4, 16, 0, fake, fake, null) == 2
    # GEMM: shapes, zero sizes, pointers, workspace
    g = L.w8a8_gemm_postscale
    assert g(fake, fake, fake, fake, null, fake, 4, 4, 20, fake, 1 << 20, null) == 3
    assert g(null, null, null, null, null, null, 0, 4, 16, null, 0, null) == 0
    assert g(null, null, null, null, null, null, 4, 0, 16, null, 0, null) == 0
    assert g(fake, null, fake, fake, null, fake, 4, 4, 16, fake, 1 << 20, null) == 1
    assert g(fake, fake, fake, fake, odd, fake, 4, 4, 16, fake, 1 << 20, null) == 2
    # (more than 288 tokens: the bf16-image path, which needs the workspace)
    assert g(fake, fake, fake, fake, null, fake, 300, 4, 16, null, 1 << 20, null) == 7
    assert g(fake, fake, fake, fake, null, fake, 300, 4, 16, fake, 10, null) == 7
    assert g(fake, fake, fake, fake, null, fake, 300, 4, 16, P(0x1010), 1 << 20, null) == 7
    # 5..288 tokens stream the int8 codes: the fp16 image of Xq, plus int32
    # sums [M][N] and counters (8 per 128 weight rows) where K may be split
    # (77 x 3072: 24 weight tiles; 77 x 13824 has 108, too many to split)
    s = s8_need(77, 3072, 5120)
    assert g(fake, fake, fake, fake, null, fake, 77, 3072, 5120, null, 0, null) == 7
    assert g(fake, fake, fake, fake, null, fake, 77, 3072, 5120, fake, s - 256, null) == 7
    assert g(fake, fake, fake, fake, null, fake, 77, 13824, 5120, fake, s8_need(77, 13824, 5120) - 256, null) == 7
    assert s8_need(77, 13824, 5120) == _a256(77 * 5120 * 2)
    s = s8_need(257, 3072, 5120)
    assert s == _a256(257 * 5120 * 2) + _a256(257 * 3072 * 4) + _a256(24 * 32)
    assert g(fake, fake, fake, fake, null, fake, 257, 3072, 5120, fake, s - 256, null) == 7
    assert g(fake, fake, fake, fake, null, fake, 200, 4, 16, null, 1 << 20, null) == 7
    # blockwise needs its workspace even for one token
    assert L.w8a8_gemm_blockwise(fake, fake, fake, fake, null, fake, 1, 4, 128, null, 0, null) == 7
    assert L.w8a8_gemm_blockwise(fake, fake, fake, fake, null, fake, 4, 4, 64, fake, 1 << 20, null) == 3
    assert L.w8a8_gemm_postscale_s32(fake, fake, null, 4, 4, 16, fake, 1 << 20, null) == 1
    assert L.w8a8_gemm_blockwise_f32(fake, null, fake, fake, fake, 4, 4, 128, fake, 1 << 20, null) == 1


def test_widened_entry_points_check_arguments_before_device(cdll):
    """The fused FFN up-projection, the image GEMMs and the norm + quant
    entry point validate shapes, pointers, alignment and workspace first."""
    L, _ = cdll
    P = ctypes.c_void_p
    fake = P(0x1000)
    odd = P(0x1001)
    null = None
    # norm + quant: kind, K % 8, K limit, eps, nothing to do, pointers, alignment
    n = L.w8a8_norm_quant
    assert n(fake, null, null, 1e-5, 5, 4, 64, null, null, fake, fake, null) == 1
    assert n(fake, null, null, 1e-5, 0, 4, 12, null, null, fake, fake, null) == 3
    assert n(fake, null, null, 1e-5, 0, 4, 16392, null, null, fake, fake, null) == 3
    assert n(fake, null, null, -1.0, 1, 4, 64, null, null, fake, fake, null) == 1
    assert n(fake, null, null, float("nan"), 1, 4, 64, null, null, fake, fake, null) == 1
    assert n(null, null, null, 1e-5, 0, 0, 64, null, null, null, null, null) == 0
    assert n(null, null, null, 1e-5, 0, 4, 64, null, null, fake, fake, null) == 1
    assert n(fake, null, null, 1e-5, 0, 4, 64, null, null, fake, null, null) == 1
    assert n(odd, null, null, 1e-5, 0, 4, 64, null, null, fake, fake, null) == 2
    assert n(fake, odd, null, 1e-5, 0, 4, 64, null, null, fake, fake, null) == 2
    # fused FFN up-projection: N % 128, pointers, workspace
    f = L.w8a8_linear_postscale_gelu_quant
    assert f(fake, fake, fake, null, fake, fake, 4, 200, 64, fake, null, fake, 1 << 20, null) == 3
    assert f(fake, fake, fake, null, null, fake, 4, 256, 64, fake, null, fake, 1 << 20, null) == 1
    assert f(fake, fake, fake, null, fake, fake, 4, 256, 64, fake, null, null, 1 << 20, null) == 7
    assert f(null, null, null, null, null, null, 0, 256, 64, null, null, null, 0, null) == 0
    # fused Linear on int8 weight codes: K rule, nothing to do, pointers, alignment, workspace
    c = L.w8a8_linear_postscale_codes
    assert c(fake, fake, fake, null, fake, 4, 4, 20, fake, null, fake, 1 << 20, null) == 3
    assert c(null, null, null, null, null, 0, 4, 16, null, null, null, 0, null) == 0
    assert c(fake, null, fake, null, fake, 4, 4, 16, fake, null, fake, 1 << 20, null) == 1
    assert c(fake, fake, fake, null, fake, 4, 4, 16, null, null, fake, 1 << 20, null) == 1
    assert c(odd, fake, fake, null, fake, 4, 4, 16, fake, null, fake, 1 << 20, null) == 2
    assert c(fake, fake, fake, null, fake, 4, 4, 16, fake, odd, fake, 1 << 20, null) == 2
    # (one or two tokens with M * K <= 131072: the one-kernel path needs no workspace)
    assert c(fake, fake, fake, null, fake, 16, 4, 16, fake, null, null, 1 << 20, null) == 7
    assert c(fake, fake, fake, null, fake, 16, 4, 16, fake, null, fake, 10, null) == 7
    assert c(fake, fake, fake, null, fake, 2, 4, 131072, fake, null, null, 1 << 20, null) == 7
    # image GEMMs
    assert L.w8a8_gemm_blockwise_images(fake, fake, fake, fake, null, fake, 4, 4, 100, null) == 3
    assert L.w8a8_gemm_blockwise_images(fake, null, fake, fake, null, fake, 4, 4, 128, null) == 1
    gi = L.w8a8_gemm_postscale_images
    assert gi(fake, fake, fake, fake, null, fake, 4, 4, 20, null, 0, null) == 3
    # a few-token shape that splits K needs the partial-sum workspace
    assert L.w8a8_splitk_workspace_size(1, 4096, 4096) > 0
    assert L.w8a8_splitk_workspace_size(4096, 4096, 4096) == 0
    assert gi(fake, fake, fake, fake, null, fake, 1, 4096, 4096, null, 0, null) == 7
    assert gi(fake, fake, fake, fake, odd, fake, 1, 4096, 4096, null, 0, null) == 2


def test_noalloc_and_gelu_export_check_arguments_before_device(cdll):
    L, _ = cdll
    P = ctypes.c_void_p
    fake = P(0x1000)
    odd = P(0x1001)
    null = None
    na = L.w8a8_gemm_postscale_noalloc
    assert na(fake, fake, fake, fake, null, fake, -1, 4, 16, null) == 1
    assert na(fake, fake, fake, fake, null, fake, 4, 4, 20, null) == 3
    assert na(fake, fake, fake, fake, null, fake, 1 << 31, 4, 16, null) == 3      # M > INT32_MAX: SHAPE
    assert na(null, null, null, null, null, null, 0, 4, 16, null) == 0
    assert na(fake, fake, fake, fake, null, fake, 4097, 4096, 4096, null) == 7   # beyond the 64 MiB scratch
    g = L.w8a8_gelu_bf16
    assert g(fake, -8, fake, null) == 1
    assert g(fake, 12, fake, null) == 3
    assert g(null, 0, null, null) == 0
    assert g(null, 8, fake, null) == 1
    assert g(odd, 8, fake, null) == 2


def _a256(v):
    return (v + 255) // 256 * 256


def s8_need(M, N, K):
    """Workspace of the GEMM on int8 operands (5..288 tokens): the fp16 image
    of Xq, and where K may be split (at most 76 tiles of 128 weight rows, K
    over 384) int32 sums [M][N] and 8 int32 counters per tile."""
    tiles = -(-N // 128)
    b = _a256(M * K * 2)
    if tiles <= 76 and -(-K // 128) >= 4:
        b += _a256(M * N * 4) + _a256(tiles * 32)
    return b


def test_workspace_size(cdll):
    L, _ = cdll
    assert L.w8a8_gemm_workspace_size(0, 5, 16) == 0
    # bf16 images of Xq [M,K] and Wq [N,K], each rounded up to 256 bytes
    assert L.w8a8_gemm_workspace_size(3, 5, 16) == 256 + 256
    assert L.w8a8_gemm_workspace_size(4096, 4096, 4096) == 2 * 4096 * 4096 * 2
    # few tokens with split K: images plus int32 partial sums (S splits x M x N)
    s = L.w8a8_splitk_workspace_size(1, 3072, 5120)
    assert s >= 6 * 1 * 3072 * 4 and s % 256 == 0
    assert L.w8a8_gemm_workspace_size(1, 3072, 5120) == 5120 * 2 + 3072 * 5120 * 2 + s
    assert L.w8a8_linear_workspace_size(1, 3072, 5120) == 256 * ((5120 * 2 + 255) // 256) + s
    assert L.w8a8_linear_workspace_size(4096, 4096, 4096) == 4096 * 4096 * 2
    # the fused Linear on codes: nothing for the one-kernel GEMV (M <= 2,
    # M * K <= 131072), the codes of X before the GEMV (M <= 4), else the codes
    # plus the GEMM's workspace
    assert L.w8a8_linear_codes_workspace_size(0, 3072, 5120) == 0
    assert L.w8a8_linear_codes_workspace_size(1, 3072, 5120) == 0
    assert L.w8a8_linear_codes_workspace_size(2, 64, 65536) == 0
    assert L.w8a8_linear_codes_workspace_size(1, 64, 131072) == 0
    assert L.w8a8_linear_codes_workspace_size(3, 5, 16) == 256
    assert L.w8a8_linear_codes_workspace_size(4, 13824, 32768) == 4 * 32768
    assert L.w8a8_linear_codes_workspace_size(8, 13824, 16384) == 8 * 16384 + s8_need(8, 13824, 16384)
    assert L.w8a8_linear_codes_workspace_size(8, 64, 16400) == _a256(8 * 16400) + s8_need(8, 64, 16400)
    assert L.w8a8_linear_codes_workspace_size(16, 4096, 4096) == 16 * 4096 + s8_need(16, 4096, 4096)
    assert L.w8a8_linear_codes_workspace_size(77, 13824, 5120) == _a256(77 * 5120) + s8_need(77, 13824, 5120)
    assert L.w8a8_linear_codes_workspace_size(200, 64, 256) == 200 * 256 + s8_need(200, 64, 256)
    assert L.w8a8_linear_codes_workspace_size(288, 3072, 5120) == 288 * 5120 + s8_need(288, 3072, 5120)
    assert L.w8a8_linear_codes_workspace_size(300, 64, 256) == 300 * 256 + L.w8a8_gemm_workspace_size(300, 64, 256)
    # the public size covers every path, the int8 path's need included
    for M, N, K in [(128, 4096, 16), (128, 4096, 512), (9, 9728, 512), (128, 128, 131072), (288, 64, 131072),
                    (257, 3072, 5120), (129, 9856, 400)]:
        assert L.w8a8_gemm_workspace_size(M, N, K) >= s8_need(M, N, K)


def test_few_token_routing():
    """The GEMV takes up to 4 tokens (their codes within 128 KB); the Linear
    on int8 codes is preferred up to 256 tokens, and up to 288 with at least
    2^25 weights."""
    import w8a8_int8_linear_gb300 as w
    assert w.gemv_takes(4, 5120) and not w.gemv_takes(5, 5120) and not w.gemv_takes(4, 32784)
    assert w.gemv_takes(1, 131072) and not w.gemv_takes(0, 16)
    assert w.codes_preferred(1, 3072, 5120) and w.codes_preferred(77, 3072, 5120)
    assert w.codes_preferred(128, 5120, 5120) and w.codes_preferred(256, 3072, 5120)
    assert not w.codes_preferred(257, 5120, 5120) and w.codes_preferred(257, 13824, 5120)
    assert w.codes_preferred(288, 15432, 5120) and not w.codes_preferred(289, 15432, 5120)
    assert not w.codes_preferred(0, 13824, 5120)


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    import w8a8_int8_linear_gb300 as w
    monkeypatch.setattr(w, "_lib", None)
    monkeypatch.setattr(w, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        w.lib()
