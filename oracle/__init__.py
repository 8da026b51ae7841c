"""CPU oracle for the W8A8 INT8 Linear path (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
may import this package.  The CUDA library never does, and this package never
imports the CUDA library.  It wraps the plain-C implementation in
``w8a8_oracle.c`` (ctypes); arrays are numpy, with bf16 values carried as their
uint16 bit patterns.

Every function follows "TurboDiffusion Integration Notes" (TurboT2AV
docs/acceleration.md), section "Reused Components" (W8A8 Linear: INT8 weights
quantized once, activations quantized dynamically before each Linear) and
section "Differences From TurboDiffusion" (post-scale kernel: continuous integer
accumulation over K, scales applied in the epilogue; original kernel:
blockwise-scaled).  The quantizer and epilogue formulas are the readings stated
at the top of ``w8a8_oracle.c``.
"""
import ctypes
import os

import numpy as np

from . import build as _build

PER_ROW = 0   # activations: per token; weights: per output channel
BLOCK = 1     # activations: per 1x128 block; weights: per 128x128 block
BLOCK_SIZE = 128

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        L.orc_quantize_act.argtypes = [P, I64, I64, ctypes.c_int, P, P]
        L.orc_quantize_act.restype = ctypes.c_int
        L.orc_quantize_weight.argtypes = [P, I64, I64, ctypes.c_int, P, P]
        L.orc_quantize_weight.restype = ctypes.c_int
        L.orc_gemm_s32.argtypes = [P, P, I64, I64, I64, P]
        L.orc_gemm_s32.restype = None
        L.orc_epilogue_postscale.argtypes = [P, P, P, P, I64, I64, P]
        L.orc_epilogue_postscale.restype = None
        L.orc_gemm_blockwise_f32.argtypes = [P, P, P, P, I64, I64, I64, P]
        L.orc_gemm_blockwise_f32.restype = None
        L.orc_epilogue_blockwise.argtypes = [P, P, I64, I64, P]
        L.orc_epilogue_blockwise.restype = None
        L.orc_bf16_from_f32.argtypes = [P, I64, P]
        L.orc_bf16_from_f32.restype = None
        L.orc_f32_from_bf16.argtypes = [P, I64, P]
        L.orc_f32_from_bf16.restype = None
        L.orc_gelu_f64.argtypes = [P, I64, P]
        L.orc_gelu_f64.restype = None
        L.orc_gelu_bf16.argtypes = [P, I64, P]
        L.orc_gelu_bf16.restype = None
        L.orc_norm_quant.argtypes = [P, P, P, ctypes.c_float, ctypes.c_int, I64, I64, P, P, P]
        L.orc_norm_quant.restype = ctypes.c_int
        L.orc_norm_quant_fixed_order.argtypes = [P, P, P, ctypes.c_float, ctypes.c_int, I64, I64, P, P, P]
        L.orc_norm_quant_fixed_order.restype = ctypes.c_int
        L.orc_num_threads.restype = ctypes.c_int
        L.orc_set_num_threads.argtypes = [ctypes.c_int]
        L.orc_set_num_threads.restype = None
        _lib = L
    return _lib


def _p(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    a = np.asarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {dtype}, got {a.dtype}")
    return np.ascontiguousarray(a)


def num_threads() -> int:
    return lib().orc_num_threads()


def set_num_threads(n: int) -> None:
    lib().orc_set_num_threads(int(n))


def bf16_from_f32(x) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); returns uint16 bits."""
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint16)
    lib().orc_bf16_from_f32(_p(x), x.size, _p(out))
    return out


def f32_from_bf16(h) -> np.ndarray:
    h = _c(h, np.uint16)
    out = np.empty(h.shape, np.float32)
    lib().orc_f32_from_bf16(_p(h), h.size, _p(out))
    return out


def quantize_act(X, mode=PER_ROW):
    """X: uint16 bf16 bits [M,K] -> (Xq int8 [M,K], sx fp32 [M] or [M,K/128])."""
    X = _c(X, np.uint16)
    M, K = X.shape
    Xq = np.empty((M, K), np.int8)
    sx = np.empty((M,) if mode == PER_ROW else (M, K // BLOCK_SIZE), np.float32)
    if lib().orc_quantize_act(_p(X), M, K, mode, _p(Xq), _p(sx)) != 0:
        raise ValueError("bad shape for activation quantization")
    return Xq, sx


def quantize_weight(W, mode=PER_ROW):
    """W: uint16 bf16 bits [N,K] -> (Wq int8 [N,K], sw fp32 [N] or [ceil(N/128),K/128])."""
    W = _c(W, np.uint16)
    N, K = W.shape
    Wq = np.empty((N, K), np.int8)
    if mode == PER_ROW:
        sw = np.empty((N,), np.float32)
    else:
        sw = np.empty(((N + BLOCK_SIZE - 1) // BLOCK_SIZE, K // BLOCK_SIZE), np.float32)
    if lib().orc_quantize_weight(_p(W), N, K, mode, _p(Wq), _p(sw)) != 0:
        raise ValueError("bad shape for weight quantization")
    return Wq, sw


def gemm_s32(Xq, Wq):
    Xq = _c(Xq, np.int8)
    Wq = _c(Wq, np.int8)
    M, K = Xq.shape
    N, K2 = Wq.shape
    assert K == K2
    acc = np.empty((M, N), np.int32)
    lib().orc_gemm_s32(_p(Xq), _p(Wq), M, N, K, _p(acc))
    return acc


def epilogue_postscale(acc, sx, sw, bias=None):
    acc = _c(acc, np.int32)
    sx = _c(sx, np.float32)
    sw = _c(sw, np.float32)
    M, N = acc.shape
    b = None if bias is None else _c(bias, np.uint16)
    Y = np.empty((M, N), np.uint16)
    lib().orc_epilogue_postscale(_p(acc), _p(sx), _p(sw), _p(b), M, N, _p(Y))
    return Y


def gemm_blockwise_f32(Xq, sx, Wq, sw):
    Xq = _c(Xq, np.int8)
    Wq = _c(Wq, np.int8)
    sx = _c(sx, np.float32)
    sw = _c(sw, np.float32)
    M, K = Xq.shape
    N = Wq.shape[0]
    acc = np.empty((M, N), np.float32)
    lib().orc_gemm_blockwise_f32(_p(Xq), _p(sx), _p(Wq), _p(sw), M, N, K, _p(acc))
    return acc


def epilogue_blockwise(acc, bias=None):
    acc = _c(acc, np.float32)
    M, N = acc.shape
    b = None if bias is None else _c(bias, np.uint16)
    Y = np.empty((M, N), np.uint16)
    lib().orc_epilogue_blockwise(_p(acc), _p(b), M, N, _p(Y))
    return Y


def linear_postscale(X, W, bias=None):
    """Whole post-scale W8A8 Linear from bf16 X [M,K], W [N,K] (uint16 bits).

    Returns dict with Xq, sx, Wq, sw, acc (int32) and Y (bf16 bits)."""
    Xq, sx = quantize_act(X, PER_ROW)
    Wq, sw = quantize_weight(W, PER_ROW)
    acc = gemm_s32(Xq, Wq)
    Y = epilogue_postscale(acc, sx, sw, bias)
    return dict(Xq=Xq, sx=sx, Wq=Wq, sw=sw, acc=acc, Y=Y)


def linear_blockwise(X, W, bias=None):
    """Whole blockwise-scaled W8A8 Linear (1x128 activation, 128x128 weight blocks)."""
    Xq, sx = quantize_act(X, BLOCK)
    Wq, sw = quantize_weight(W, BLOCK)
    acc = gemm_blockwise_f32(Xq, sx, Wq, sw)
    Y = epilogue_blockwise(acc, bias)
    return dict(Xq=Xq, sx=sx, Wq=Wq, sw=sw, acc=acc, Y=Y)


def gelu_f64(x):
    """GELU in its erf form, x * Phi(x), of fp64 values, evaluated in fp64 with
    the C library's erfc (Phi(x) = erfc(-x / sqrt 2) / 2)."""
    x = _c(x, np.float64)
    g = np.empty_like(x)
    lib().orc_gelu_f64(_p(x), x.size, _p(g))
    return g


def gelu_bf16(Y):
    """bf16(fp32(gelu(Y))) for bf16 Y given as uint16 bit patterns: the fp64
    value of the plain definition rounded to fp32, then to bf16."""
    Y = _c(Y, np.uint16)
    G = np.empty_like(Y)
    lib().orc_gelu_bf16(_p(Y), Y.size, _p(G))
    return G


def ffn_up_gelu_quant(X, W, bias=None):
    """FFN up-projection as the down-projection consumes it: the post-scale
    W8A8 Linear Y = linear_postscale(X, W, bias), G = bf16(gelu(Y)), then
    G quantized in 1x128 blocks.  N must be a multiple of 128.

    Returns linear_postscale's dict plus G (bf16 bits), Gq int8 [M,N] and
    sg fp32 [M, N/128]."""
    r = linear_postscale(X, W, bias)
    G = gelu_bf16(r["Y"])
    Gq, sg = quantize_act(G, BLOCK)
    r.update(G=G, Gq=Gq, sg=sg)
    return r


RMS_NORM = 0
LAYER_NORM = 1


def _norm_quant(fn, X, gamma, beta, eps, kind):
    X = _c(X, np.uint16)
    M, K = X.shape
    g = None if gamma is None else _c(gamma, np.uint16)
    b = None if beta is None else _c(beta, np.uint16)
    Y = np.empty((M, K), np.uint16)
    Xq = np.empty((M, K), np.int8)
    sx = np.empty(M, np.float32)
    if fn(_p(X), _p(g), _p(b), float(eps), int(kind), M, K, _p(Y), _p(Xq), _p(sx)) != 0:
        raise ValueError("norm_quant: bad shape")
    return Y, Xq, sx


def norm_quant(X, gamma=None, beta=None, eps=1e-6, kind=RMS_NORM):
    """RMSNorm (kind 0) or LayerNorm (kind 1) of bf16 X [M,K] (uint16 bits) by
    the plain definition: fp64 statistics (left-to-right sums) and fp64
    normalization, rounded to fp32 and then bf16; then per-token
    quantization of the bf16 result.

    Returns (Y bf16 bits [M,K], Xq int8 [M,K], sx fp32 [M])."""
    return _norm_quant(lib().orc_norm_quant, X, gamma, beta, eps, kind)


def norm_quant_fixed_order(X, gamma=None, beta=None, eps=1e-6, kind=RMS_NORM):
    """The same normalization stated in binary32 with one fixed summation
    order (chunks of 8, then a pairwise tree; see w8a8_oracle.c), then the
    per-token quantization.  K % 8 == 0, K <= 65536.

    Returns (Y bf16 bits [M,K], Xq int8 [M,K], sx fp32 [M])."""
    return _norm_quant(lib().orc_norm_quant_fixed_order, X, gamma, beta, eps, kind)


def linear_sampled(X, W, bias, rows, cols, mode=PER_ROW):
    """Outputs Y[rows[i], cols[j]] of the full Linear, computed only from the
    X rows and W rows (or 128-row W blocks) they depend on.

    Returns (Y_sub uint16 [len(rows), len(cols)], acc_sub) where acc_sub is int32
    (post-scale) or fp32 (blockwise, pre-bf16)."""
    X = np.asarray(X)
    W = np.asarray(W)
    rows = np.asarray(rows, np.int64)
    cols = np.asarray(cols, np.int64)
    Xs = np.ascontiguousarray(X[rows])
    Xq, sx = quantize_act(Xs, mode)
    bsub = None if bias is None else np.ascontiguousarray(np.asarray(bias)[cols])
    if mode == PER_ROW:
        Wq, sw = quantize_weight(np.ascontiguousarray(W[cols]), PER_ROW)
        acc = gemm_s32(Xq, Wq)
        return epilogue_postscale(acc, sx, sw, bsub), acc
    # blockwise: quantize each 128-row weight block the sampled columns fall in
    N, K = W.shape
    nbs = np.unique(cols // BLOCK_SIZE)
    Wq_cols = np.empty((len(cols), K), np.int8)
    sw_cols = np.empty((len(cols), K // BLOCK_SIZE), np.float32)
    for nb in nbs:
        n0 = int(nb) * BLOCK_SIZE
        n1 = min(n0 + BLOCK_SIZE, N)
        wq, swb = quantize_weight(np.ascontiguousarray(W[n0:n1]), BLOCK)
        sel = np.nonzero(cols // BLOCK_SIZE == nb)[0]
        Wq_cols[sel] = wq[cols[sel] - n0]
        sw_cols[sel] = swb[0]
    # columns are no longer grouped in 128-row blocks: evaluate one column at a
    # time with its own block scale row (a 1-row "block" carrying that scale)
    acc = np.empty((len(rows), len(cols)), np.float32)
    for j in range(len(cols)):
        acc[:, j] = gemm_blockwise_f32(Xq, sx, Wq_cols[j:j + 1], sw_cols[j:j + 1])[:, 0]
    return epilogue_blockwise(acc, bsub), acc


__all__ = [
    "PER_ROW", "BLOCK", "BLOCK_SIZE", "lib", "num_threads", "set_num_threads",
    "bf16_from_f32", "f32_from_bf16", "quantize_act", "quantize_weight", "gemm_s32",
    "epilogue_postscale", "gemm_blockwise_f32", "epilogue_blockwise", "linear_postscale",
    "linear_blockwise", "linear_sampled",
]
