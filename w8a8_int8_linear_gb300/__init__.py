"""GB300 (sm_103a) W8A8 INT8 Linear.

Thin Python binding of the C ABI declared in ``include/w8a8.h``: every
function here only checks tensor types, allocates outputs with PyTorch and
passes raw device pointers and the current CUDA stream to the library.  All
arithmetic runs in the library's CUDA kernels; there is no other code path.
If the library has not been built (``__graft_entry__.build()``), every call
raises.

The method is the W8A8 Linear of "TurboDiffusion Integration Notes"
(TurboT2AV docs/acceleration.md), sections "Reused Components" (INT8
weights quantized once, activations quantized dynamically before each
Linear) and "Differences From TurboDiffusion" (post-scale kernel with
continuous integer accumulation over K and scales in the epilogue; the
original blockwise-scaled kernel).
"""
import ctypes
import os

import torch

PER_ROW = 0  # activations: per token; weights: per output channel
BLOCK = 1    # activations: per 1x128 block; weights: per 128x128 block
BLOCK_SIZE = 128

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libw8a8_gb300.so")

_STATUS = {
    0: "W8A8_OK", 1: "W8A8_ERR_INVALID_ARG", 2: "W8A8_ERR_ALIGNMENT", 3: "W8A8_ERR_SHAPE",
    4: "W8A8_ERR_UNSUPPORTED_DEVICE", 5: "W8A8_ERR_CUDA", 6: "W8A8_ERR_TIMEOUT", 7: "W8A8_ERR_WORKSPACE",
}

# (name, restype, argtypes) of every entry point in include/w8a8.h
_P, _I64, _I32, _SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
SIGNATURES = [
    ("w8a8_status_string", ctypes.c_char_p, [_I32]),
    ("w8a8_last_error_detail", ctypes.c_char_p, []),
    ("w8a8_quantize_weight", _I32, [_P, _I64, _I64, _I32, _P, _P, _P]),
    ("w8a8_quantize_act", _I32, [_P, _I64, _I64, _I32, _P, _P, _P]),
    ("w8a8_gemm_workspace_size", _SZ, [_I64, _I64, _I64]),
    ("w8a8_gemm_postscale", _I32, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _P, _SZ, _P]),
    ("w8a8_gemm_blockwise", _I32, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _P, _SZ, _P]),
    ("w8a8_pack_weight", _I32, [_P, _I64, _I64, _P, _P]),
    ("w8a8_linear_workspace_size", _SZ, [_I64, _I64, _I64]),
    ("w8a8_linear_postscale", _I32, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _P, _P, _P, _SZ, _P]),
    ("w8a8_linear_blockwise", _I32, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _P, _P, _P, _SZ, _P]),
    ("w8a8_linear_codes_workspace_size", _SZ, [_I64, _I64, _I64]),
    ("w8a8_linear_postscale_codes", _I32, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _P, _P, _P, _SZ, _P]),
    ("w8a8_linear_postscale_gelu_quant", _I32, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _P, _P, _P, _SZ, _P]),
    ("w8a8_gemm_blockwise_images", _I32, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _P]),
    ("w8a8_norm_quant", _I32, [_P, _P, _P, ctypes.c_float, ctypes.c_int, _I64, _I64, _P, _P, _P, _P, _P]),
    ("w8a8_splitk_workspace_size", _SZ, [_I64, _I64, _I64]),
    ("w8a8_gemm_postscale_images", _I32, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _P, _SZ, _P]),
    ("w8a8_gemm_postscale_noalloc", _I32, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _P]),
    ("w8a8_gemm_postscale_s32", _I32, [_P, _P, _P, _I64, _I64, _I64, _P, _SZ, _P]),
    ("w8a8_gemm_blockwise_f32", _I32, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _P, _SZ, _P]),
    ("w8a8_gelu_bf16", _I32, [_P, _I64, _P, _P]),
    ("w8a8_get_device_error", _I32, [ctypes.POINTER(ctypes.c_int)]),
    ("w8a8_probe_wait_timeout", _I32, [_P]),
    ("w8a8_set_gemm_timing_events", _I32, [_P, _P]),
    ("w8a8_measure_imma_peak", _I32, [ctypes.POINTER(ctypes.c_double), _P]),
    ("w8a8_stream_floor", _I32, [_P, _I64, _P, _P]),
]

_lib = None


class W8A8Error(RuntimeError):
    def __init__(self, fn, status, detail=""):
        self.status = status
        msg = f"{fn} failed: {_STATUS.get(status, status)}"
        if detail:
            msg += f" ({detail})"
        super().__init__(msg)


def lib():
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"W8A8 CUDA library not built ({LIB_PATH} missing): run __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, res, args in SIGNATURES:
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check(fn, status):
    if status != 0:
        detail = lib().w8a8_last_error_detail().decode() if status == 5 else ""
        raise W8A8Error(fn, status, detail)


def _need(t, dtype, name, ndim=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims")


def quantize_weight(W, mode=PER_ROW):
    """W bf16 [N,K] -> (Wq int8 [N,K], sw fp32 [N] or [ceil(N/128), K/128])."""
    _need(W, torch.bfloat16, "W", 2)
    N, K = W.shape
    Wq = torch.empty((N, K), dtype=torch.int8, device=W.device)
    sw_shape = (N,) if mode == PER_ROW else ((N + BLOCK_SIZE - 1) // BLOCK_SIZE, K // BLOCK_SIZE)
    sw = torch.empty(sw_shape, dtype=torch.float32, device=W.device)
    _check("w8a8_quantize_weight",
           lib().w8a8_quantize_weight(_ptr(W), N, K, mode, _ptr(Wq), _ptr(sw), _stream()))
    return Wq, sw


def quantize_act(X, mode=PER_ROW, out=None):
    """X bf16 [M,K] -> (Xq int8 [M,K], sx fp32 [M] or [M, K/128])."""
    _need(X, torch.bfloat16, "X", 2)
    M, K = X.shape
    if out is None:
        Xq = torch.empty((M, K), dtype=torch.int8, device=X.device)
        sx = torch.empty((M,) if mode == PER_ROW else (M, K // BLOCK_SIZE), dtype=torch.float32, device=X.device)
    else:
        Xq, sx = out
    _check("w8a8_quantize_act", lib().w8a8_quantize_act(_ptr(X), M, K, mode, _ptr(Xq), _ptr(sx), _stream()))
    return Xq, sx


def workspace_size(M, N, K):
    return int(lib().w8a8_gemm_workspace_size(M, N, K))


class Workspace:
    """Caller-owned GEMM workspace, grown on demand (PyTorch allocation)."""

    def __init__(self, device=None):
        self.device = device
        self.buf = None

    def get(self, M, N, K, device):
        need = workspace_size(M, N, K)
        if self.buf is None or self.buf.numel() < need or self.buf.device != device:
            self.buf = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
        return self.buf


_default_ws = {}


def _workspace(ws, M, N, K, device):
    if isinstance(ws, torch.Tensor):
        return ws
    if ws is None:
        ws = _default_ws.setdefault(str(device), Workspace())
    return ws.get(M, N, K, device)


# Up to this many tokens, with M * K up to GEMV_MAX_CODE_BYTES, the post-scale
# GEMM is a CUDA-core GEMV on the int8 codes, which needs no workspace.
GEMV_MAX_TOKENS = 4
GEMV_MAX_CODE_BYTES = 131072
# Up to this many tokens the post-scale GEMM on int8 codes streams the codes
# itself (the int8-operand tensor-core kernels) instead of bf16 images.
INT8_OPERAND_MAX_TOKENS = 288


def gemv_takes(M, K):
    return 1 <= M <= GEMV_MAX_TOKENS and M * K <= GEMV_MAX_CODE_BYTES


def codes_preferred(M, N, K):
    """Whether a post-scale Linear of M tokens is faster on the int8 weight
    codes (linear_postscale_codes: the GEMV, or the int8-operand kernels that
    read each weight byte once) than on the packed bf16 image.  Measured in
    steady state on GB300 (K = 5120, N = 3072 / 5120 / 13824 / 15432): the
    codes are at least as fast up to 256 tokens at every N, and up to 288
    once the weights hold 2^25 values; beyond that the image path runs."""
    if M < 1 or M > INT8_OPERAND_MAX_TOKENS:
        return False
    return M <= 256 or N * K >= 1 << 25


def _postscale_workspace(ws, M, N, K, device):
    if ws is None and gemv_takes(M, K):
        return None
    return _workspace(ws, M, N, K, device)


def gemm_postscale(Xq, sx, Wq, sw, bias=None, out=None, workspace=None):
    """Y bf16 [M,N] = bf16(((acc * sx[m]) * sw[n]) + bias[n]), acc = Xq . Wq^T exact in int32."""
    _need(Xq, torch.int8, "Xq", 2)
    _need(Wq, torch.int8, "Wq", 2)
    _need(sx, torch.float32, "sx")
    _need(sw, torch.float32, "sw")
    if bias is not None:
        _need(bias, torch.bfloat16, "bias", 1)
    M, K = Xq.shape
    N = Wq.shape[0]
    Y = out if out is not None else torch.empty((M, N), dtype=torch.bfloat16, device=Xq.device)
    ws = _postscale_workspace(workspace, M, N, K, Xq.device)
    _check("w8a8_gemm_postscale",
           lib().w8a8_gemm_postscale(_ptr(Xq), _ptr(sx), _ptr(Wq), _ptr(sw), _ptr(bias), _ptr(Y), M, N, K,
                                     _ptr(ws), 0 if ws is None else ws.numel(), _stream()))
    return Y


def gemm_blockwise(Xq, sx, Wq, sw, bias=None, out=None, workspace=None):
    """Blockwise-scaled GEMM: 1x128 activation scales, 128x128 weight scales, bf16 out."""
    _need(Xq, torch.int8, "Xq", 2)
    _need(Wq, torch.int8, "Wq", 2)
    _need(sx, torch.float32, "sx", 2)
    _need(sw, torch.float32, "sw", 2)
    if bias is not None:
        _need(bias, torch.bfloat16, "bias", 1)
    M, K = Xq.shape
    N = Wq.shape[0]
    Y = out if out is not None else torch.empty((M, N), dtype=torch.bfloat16, device=Xq.device)
    ws = _workspace(workspace, M, N, K, Xq.device)
    _check("w8a8_gemm_blockwise",
           lib().w8a8_gemm_blockwise(_ptr(Xq), _ptr(sx), _ptr(Wq), _ptr(sw), _ptr(bias), _ptr(Y), M, N, K,
                                     _ptr(ws), ws.numel(), _stream()))
    return Y


NOALLOC_SCRATCH_BYTES = 64 << 20


def gemm_postscale_noalloc(Xq, sx, Wq, sw, bias=None, out=None):
    """Post-scale GEMM using the library's fixed 64 MiB device scratch instead
    of a caller workspace (for callers that cannot allocate device memory at
    the call site).  Calls overlapping on the GPU race on the shared scratch."""
    _need(Xq, torch.int8, "Xq", 2)
    _need(Wq, torch.int8, "Wq", 2)
    _need(sx, torch.float32, "sx")
    _need(sw, torch.float32, "sw")
    if bias is not None:
        _need(bias, torch.bfloat16, "bias", 1)
    M, K = Xq.shape
    N = Wq.shape[0]
    Y = out if out is not None else torch.empty((M, N), dtype=torch.bfloat16, device=Xq.device)
    _check("w8a8_gemm_postscale_noalloc",
           lib().w8a8_gemm_postscale_noalloc(_ptr(Xq), _ptr(sx), _ptr(Wq), _ptr(sw), _ptr(bias), _ptr(Y), M, N, K,
                                             _stream()))
    return Y


def gemm_postscale_s32(Xq, Wq, workspace=None):
    """Debug export: int32 accumulator [M,N] of the post-scale mainloop."""
    _need(Xq, torch.int8, "Xq", 2)
    _need(Wq, torch.int8, "Wq", 2)
    M, K = Xq.shape
    N = Wq.shape[0]
    acc = torch.empty((M, N), dtype=torch.int32, device=Xq.device)
    ws = _postscale_workspace(workspace, M, N, K, Xq.device)
    _check("w8a8_gemm_postscale_s32",
           lib().w8a8_gemm_postscale_s32(_ptr(Xq), _ptr(Wq), _ptr(acc), M, N, K, _ptr(ws),
                                         0 if ws is None else ws.numel(), _stream()))
    return acc


def gemm_blockwise_f32(Xq, sx, Wq, sw, workspace=None):
    """Debug export: fp32 blockwise accumulator [M,N] before bias and bf16 rounding."""
    _need(Xq, torch.int8, "Xq", 2)
    _need(Wq, torch.int8, "Wq", 2)
    _need(sx, torch.float32, "sx", 2)
    _need(sw, torch.float32, "sw", 2)
    M, K = Xq.shape
    N = Wq.shape[0]
    acc = torch.empty((M, N), dtype=torch.float32, device=Xq.device)
    ws = _workspace(workspace, M, N, K, Xq.device)
    _check("w8a8_gemm_blockwise_f32",
           lib().w8a8_gemm_blockwise_f32(_ptr(Xq), _ptr(sx), _ptr(Wq), _ptr(sw), _ptr(acc), M, N, K, _ptr(ws),
                                         ws.numel(), _stream()))
    return acc


def pack_weight(Wq):
    """Exact bf16 image [N,K] of INT8 weight codes, made once at init; the
    fused Linear entry points take it in place of Wq."""
    _need(Wq, torch.int8, "Wq", 2)
    N, K = Wq.shape
    Wimg = torch.empty((N, K), dtype=torch.bfloat16, device=Wq.device)
    _check("w8a8_pack_weight", lib().w8a8_pack_weight(_ptr(Wq), N, K, _ptr(Wimg), _stream()))
    return Wimg


def linear_workspace_size(M, N, K):
    return int(lib().w8a8_linear_workspace_size(M, N, K))


def _linear(fn, mode, X, Wimg, sw, bias, out, workspace, sx_out, codes):
    _need(X, torch.bfloat16, "X", 2)
    _need(Wimg, torch.bfloat16, "Wimg", 2)
    _need(sw, torch.float32, "sw")
    if bias is not None:
        _need(bias, torch.bfloat16, "bias", 1)
    M, K = X.shape
    N = Wimg.shape[0]
    Y = out if out is not None else torch.empty((M, N), dtype=torch.bfloat16, device=X.device)
    if sx_out is None:
        sx_out = torch.empty((M,) if mode == PER_ROW else (M, K // BLOCK_SIZE), dtype=torch.float32, device=X.device)
    Xq = None
    if codes is True:
        Xq = torch.empty((M, K), dtype=torch.int8, device=X.device)
    elif isinstance(codes, torch.Tensor):
        Xq = codes
    ws = workspace
    if ws is None:
        ws = torch.empty(max(linear_workspace_size(M, N, K), 256), dtype=torch.uint8, device=X.device)
    _check(fn, getattr(lib(), fn)(_ptr(X), _ptr(Wimg), _ptr(sw), _ptr(bias), _ptr(Y), M, N, K, _ptr(sx_out), _ptr(Xq),
                                  _ptr(ws), ws.numel(), _stream()))
    return Y, sx_out, Xq


def linear_postscale(X, Wimg, sw, bias=None, out=None, workspace=None, sx_out=None, codes=False):
    """Fused W8A8 Linear, post-scale: per-token quantization of X, then the
    exact INT8 GEMM against the packed weight image, scales and bias in the
    epilogue.  Returns (Y, sx, Xq or None); codes=True also returns Xq."""
    return _linear("w8a8_linear_postscale", PER_ROW, X, Wimg, sw, bias, out, workspace, sx_out, codes)


def linear_blockwise(X, Wimg, sw, bias=None, out=None, workspace=None, sx_out=None, codes=False):
    """Fused W8A8 Linear, blockwise (1x128 activation, 128x128 weight scales)."""
    return _linear("w8a8_linear_blockwise", BLOCK, X, Wimg, sw, bias, out, workspace, sx_out, codes)


def linear_codes_workspace_size(M, N, K):
    return int(lib().w8a8_linear_codes_workspace_size(M, N, K))


def linear_postscale_codes(X, Wq, sw, bias=None, out=None, workspace=None, sx_out=None, codes=False):
    """Fused W8A8 Linear, post-scale, against the int8 weight codes (no
    image): per-token quantization of X, then the post-scale GEMM on the
    codes, which reads each weight code once (one or two tokens: one GEMV
    kernel that quantizes X itself; up to 4: the GEMV; up to 288: the
    int8-operand tensor-core kernels).  Returns (Y, sx, Xq or None);
    codes=True also returns Xq."""
    _need(X, torch.bfloat16, "X", 2)
    _need(Wq, torch.int8, "Wq", 2)
    _need(sw, torch.float32, "sw")
    if bias is not None:
        _need(bias, torch.bfloat16, "bias", 1)
    M, K = X.shape
    N = Wq.shape[0]
    Y = out if out is not None else torch.empty((M, N), dtype=torch.bfloat16, device=X.device)
    sx = sx_out if sx_out is not None else torch.empty((M,), dtype=torch.float32, device=X.device)
    Xq = None
    if codes is True:
        Xq = torch.empty((M, K), dtype=torch.int8, device=X.device)
    elif isinstance(codes, torch.Tensor):
        Xq = codes
    ws = workspace
    need = linear_codes_workspace_size(M, N, K)
    if ws is None and need:
        ws = torch.empty(need, dtype=torch.uint8, device=X.device)
    _check("w8a8_linear_postscale_codes",
           lib().w8a8_linear_postscale_codes(_ptr(X), _ptr(Wq), _ptr(sw), _ptr(bias), _ptr(Y), M, N, K, _ptr(sx),
                                             _ptr(Xq), _ptr(ws), 0 if ws is None else ws.numel(), _stream()))
    return Y, sx, Xq


def linear_postscale_gelu_quant(X, Wimg, sw, bias=None, out=None, sg_out=None, workspace=None, sx_out=None,
                                codes=False):
    """Fused FFN up-projection: post-scale W8A8 Linear, GELU, then 1x128
    quantization of the GELU output, which is returned as the exact bf16 image
    of its codes.  N % 128 == 0.  Returns (Gimg [M,N] bf16, sg [M,N/128],
    sx [M], Xq or None)."""
    _need(X, torch.bfloat16, "X", 2)
    _need(Wimg, torch.bfloat16, "Wimg", 2)
    _need(sw, torch.float32, "sw")
    if bias is not None:
        _need(bias, torch.bfloat16, "bias", 1)
    M, K = X.shape
    N = Wimg.shape[0]
    G = out if out is not None else torch.empty((M, N), dtype=torch.bfloat16, device=X.device)
    sg = sg_out if sg_out is not None else torch.empty((M, N // BLOCK_SIZE), dtype=torch.float32, device=X.device)
    sx = sx_out if sx_out is not None else torch.empty((M,), dtype=torch.float32, device=X.device)
    Xq = None
    if codes is True:
        Xq = torch.empty((M, K), dtype=torch.int8, device=X.device)
    elif isinstance(codes, torch.Tensor):
        Xq = codes
    ws = workspace
    if ws is None:
        ws = torch.empty(max(linear_workspace_size(M, N, K), 256), dtype=torch.uint8, device=X.device)
    _check("w8a8_linear_postscale_gelu_quant",
           lib().w8a8_linear_postscale_gelu_quant(_ptr(X), _ptr(Wimg), _ptr(sw), _ptr(bias), _ptr(G), _ptr(sg), M, N,
                                                  K, _ptr(sx), _ptr(Xq), _ptr(ws), ws.numel(), _stream()))
    return G, sg, sx, Xq


def gemm_blockwise_images(Ximg, sx, Wimg, sw, bias=None, out=None):
    """Blockwise GEMM on exact bf16 images of int8 codes (for example the
    output of linear_postscale_gelu_quant and a packed weight)."""
    _need(Ximg, torch.bfloat16, "Ximg", 2)
    _need(Wimg, torch.bfloat16, "Wimg", 2)
    _need(sx, torch.float32, "sx")
    _need(sw, torch.float32, "sw")
    if bias is not None:
        _need(bias, torch.bfloat16, "bias", 1)
    M, K = Ximg.shape
    N = Wimg.shape[0]
    Y = out if out is not None else torch.empty((M, N), dtype=torch.bfloat16, device=Ximg.device)
    _check("w8a8_gemm_blockwise_images",
           lib().w8a8_gemm_blockwise_images(_ptr(Ximg), _ptr(sx), _ptr(Wimg), _ptr(sw), _ptr(bias), _ptr(Y), M, N, K,
                                            _stream()))
    return Y


RMS_NORM = 0
LAYER_NORM = 1


def norm_quant(X, gamma=None, beta=None, eps=1e-6, kind=RMS_NORM, image=True, codes=False, y=False):
    """RMSNorm (kind RMS_NORM) or LayerNorm (LAYER_NORM) of bf16 X [M,K]
    fused with per-token quantization.  Returns (Ximg or None, sx, Xq or None,
    Y or None): the bf16 image of the codes (image=True), the per-token
    scales, the int8 codes (codes=True) and the normalized bf16 rows (y=True)."""
    _need(X, torch.bfloat16, "X", 2)
    M, K = X.shape
    for t, name in ((gamma, "gamma"), (beta, "beta")):
        if t is not None:
            _need(t, torch.bfloat16, name, 1)
    dev = X.device
    Ximg = torch.empty((M, K), dtype=torch.bfloat16, device=dev) if image else None
    Xq = torch.empty((M, K), dtype=torch.int8, device=dev) if codes else None
    Y = torch.empty((M, K), dtype=torch.bfloat16, device=dev) if y else None
    sx = torch.empty((M,), dtype=torch.float32, device=dev)
    _check("w8a8_norm_quant", lib().w8a8_norm_quant(_ptr(X), _ptr(gamma), _ptr(beta), float(eps), int(kind), M, K,
                                                    _ptr(Y), _ptr(Xq), _ptr(Ximg), _ptr(sx), _stream()))
    return Ximg, sx, Xq, Y


def gemm_postscale_images(Ximg, sx, Wimg, sw, bias=None, out=None, workspace=None):
    """Post-scale GEMM on exact bf16 images of int8 codes (for example the
    output of norm_quant and a packed weight)."""
    _need(Ximg, torch.bfloat16, "Ximg", 2)
    _need(Wimg, torch.bfloat16, "Wimg", 2)
    _need(sx, torch.float32, "sx")
    _need(sw, torch.float32, "sw")
    if bias is not None:
        _need(bias, torch.bfloat16, "bias", 1)
    M, K = Ximg.shape
    N = Wimg.shape[0]
    Y = out if out is not None else torch.empty((M, N), dtype=torch.bfloat16, device=Ximg.device)
    need = int(lib().w8a8_splitk_workspace_size(M, N, K))
    ws = workspace
    if ws is None and need:
        ws = torch.empty(need, dtype=torch.uint8, device=Ximg.device)
    _check("w8a8_gemm_postscale_images",
           lib().w8a8_gemm_postscale_images(_ptr(Ximg), _ptr(sx), _ptr(Wimg), _ptr(sw), _ptr(bias), _ptr(Y), M, N, K,
                                            _ptr(ws), 0 if ws is None else ws.numel(), _stream()))
    return Y


def gelu_bf16(Y, out=None):
    """Test export: bf16(gelu(Y)) elementwise with the FFN up-projection
    epilogue's device function (Y bf16 on the device, numel % 8 == 0)."""
    _need(Y, torch.bfloat16, "Y")
    G = torch.empty_like(Y) if out is None else out
    _need(G, torch.bfloat16, "out")
    _check("w8a8_gelu_bf16", lib().w8a8_gelu_bf16(_ptr(Y), Y.numel(), _ptr(G), _stream()))
    return G


def get_device_error():
    """Synchronizes, then reads and clears the device error word: (status, code)."""
    code = ctypes.c_int(0)
    st = lib().w8a8_get_device_error(ctypes.byref(code))
    return st, code.value


def probe_wait_timeout():
    """Launch the failure-detection probe: a kernel whose bounded wait runs
    out (nothing arrives) and records a timeout; read it with get_device_error."""
    _check("w8a8_probe_wait_timeout", lib().w8a8_probe_wait_timeout(_stream()))


def set_gemm_timing_events(start=None, end=None):
    """Record torch.cuda.Event `start`/`end` around the tensor-core kernel of
    every following GEMM call on this thread (None, None stops)."""
    def handle(ev):
        if ev is None:
            return None
        if ev.cuda_event == 0:
            ev.record()  # materialize the underlying cudaEvent_t
        return ctypes.c_void_p(ev.cuda_event)
    _check("w8a8_set_gemm_timing_events", lib().w8a8_set_gemm_timing_events(handle(start), handle(end)))


def stream_floor(src, dst):
    """Move the bytes of an activation quantization of `src` (bf16) into
    `dst` (int8, same element count) as a plain stream: the memory floor of
    that quantization."""
    _need(src, torch.bfloat16, "src")
    _need(dst, torch.int8, "dst")
    if dst.numel() != src.numel():
        raise ValueError("dst must have as many elements as src")
    _check("w8a8_stream_floor", lib().w8a8_stream_floor(_ptr(src), src.numel(), _ptr(dst), _stream()))


def measure_imma_peak():
    """Measured warp-level INT8 MMA throughput of this GPU, TOPS."""
    v = ctypes.c_double(0.0)
    _check("w8a8_measure_imma_peak", lib().w8a8_measure_imma_peak(ctypes.byref(v), _stream()))
    return v.value


from .module import Int8FFN, Int8Linear
from .pipeline import HostPipeline  # noqa: E402  (the modules use the functions above)
