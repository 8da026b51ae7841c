"""Int8Linear: a torch module over the W8A8 C ABI.

"Acceleration Backends" names an `Int8Linear` module and a `quant_linear`
switch; "TurboDiffusion Integration Notes", section "Reused Components",
describes what it does: weights quantized to INT8 once at model
initialization, activations quantized dynamically before every Linear.  This
module does exactly that through the library: the weight is quantized and its
exact bf16 image packed once (`from_linear` / `__init__`), and every forward
is one fused call (per-token or 1x128 quantization plus the INT8 GEMM).  With
few tokens (decoding, and up to 288 tokens where that is faster:
`codes_preferred`) a post-scale forward runs against the int8 codes instead of
the image, reading each weight byte once.  It keeps no
bf16 copy of the original weight and has no fallback path: every shape runs
the INT8 kernels.
"""
import torch

from . import BLOCK, LAYER_NORM, PER_ROW, RMS_NORM, codes_preferred, gemm_blockwise_images, gemm_postscale, \
    gemm_postscale_images, linear_blockwise, linear_codes_workspace_size, linear_postscale, \
    linear_postscale_codes, linear_postscale_gelu_quant, linear_workspace_size, norm_quant, pack_weight, \
    quantize_weight


class Int8Linear(torch.nn.Module):
    """y = W8A8(x) for x [..., in_features] bf16 on a sm_103 device.

    With `norm` ("rms" or "layer", post-scale mode only) the module first
    applies that normalization (optional `norm_weight` / `norm_bias`, `eps`)
    and the normalized rows go straight to int8 codes in the same pass
    ("Reused Components": FastNorm with W8A8)."""

    def __init__(self, weight, bias=None, mode="postscale", norm=None, norm_weight=None, norm_bias=None, eps=1e-6):
        super().__init__()
        if mode not in ("postscale", "blockwise"):
            raise ValueError("mode must be 'postscale' or 'blockwise'")
        if norm not in (None, "rms", "layer"):
            raise ValueError("norm must be None, 'rms' or 'layer'")
        if norm is not None and mode != "postscale":
            raise ValueError("a fused norm needs per-token (post-scale) activation scales")
        self.norm = norm
        self.eps = float(eps)
        for name, t in (("norm_weight", norm_weight), ("norm_bias", norm_bias)):
            self.register_buffer(name, None if t is None else t.detach().to(torch.bfloat16).contiguous())
        if weight.dtype != torch.bfloat16 or not weight.is_cuda or weight.dim() != 2:
            raise ValueError("weight must be a 2-D bf16 CUDA tensor [out_features, in_features]")
        self.mode = mode
        self.out_features, self.in_features = weight.shape
        qmode = PER_ROW if mode == "postscale" else BLOCK
        wq, sw = quantize_weight(weight.contiguous(), qmode)
        self.register_buffer("weight_q", wq)
        self.register_buffer("weight_scale", sw)
        self.register_buffer("weight_image", pack_weight(wq))
        self.register_buffer("bias", None if bias is None else bias.detach().to(torch.bfloat16).contiguous())
        self._ws = None

    @classmethod
    def from_linear(cls, linear, mode="postscale"):
        """Quantize an nn.Linear (bf16 weights on the GPU) once."""
        w = linear.weight.detach().to(torch.bfloat16).contiguous()
        b = None if linear.bias is None else linear.bias.detach()
        return cls(w, b, mode)

    def _workspace(self, M, device, codes=False):
        size = linear_codes_workspace_size if codes else linear_workspace_size
        need = max(size(M, self.out_features, self.in_features), 256)
        if self._ws is None or self._ws.numel() < need or self._ws.device != device:
            self._ws = torch.empty(need, dtype=torch.uint8, device=device)
        return self._ws

    def forward(self, x):
        if x.dtype != torch.bfloat16:
            raise TypeError("Int8Linear takes bf16 activations")
        lead = x.shape[:-1]
        x2 = x.reshape(-1, self.in_features).contiguous()
        M = x2.shape[0]
        decode = self.mode == "postscale" and codes_preferred(M, self.out_features, self.in_features)
        if self.norm is not None:
            kind = RMS_NORM if self.norm == "rms" else LAYER_NORM
            if decode:
                _, sx, xq, _ = norm_quant(x2, self.norm_weight, self.norm_bias, self.eps, kind, image=False,
                                          codes=True)
                y = gemm_postscale(xq, sx, self.weight_q, self.weight_scale, self.bias)
            else:
                ximg, sx, _, _ = norm_quant(x2, self.norm_weight, self.norm_bias, self.eps, kind)
                y = gemm_postscale_images(ximg, sx, self.weight_image, self.weight_scale, self.bias,
                                          workspace=self._workspace(M, x2.device))
        elif decode:
            ws = self._workspace(M, x2.device, codes=True) if linear_codes_workspace_size(
                M, self.out_features, self.in_features) else None
            y, _, _ = linear_postscale_codes(x2, self.weight_q, self.weight_scale, self.bias, workspace=ws)
        else:
            ws = self._workspace(M, x2.device)
            fn = linear_postscale if self.mode == "postscale" else linear_blockwise
            y, _, _ = fn(x2, self.weight_image, self.weight_scale, self.bias, workspace=ws)
        return y.reshape(*lead, self.out_features)

    def extra_repr(self):
        s = f"in_features={self.in_features}, out_features={self.out_features}, mode={self.mode}"
        return s + (f", norm={self.norm}" if self.norm else "")


class Int8FFN(torch.nn.Module):
    """FFN y = down(GELU(up(x))) on the W8A8 path: the up-projection is a
    post-scale Linear whose epilogue applies GELU and the 1x128 quantization
    the blockwise down-projection consumes, so the hidden activation never
    exists in bf16 ("Differences From TurboDiffusion": the post-scale kernel
    for LTX FFN shapes; the original blockwise kernel).  up_weight [H, D],
    down_weight [D_out, H], H % 128 == 0."""

    def __init__(self, up_weight, down_weight, up_bias=None, down_bias=None):
        super().__init__()
        for name, t in (("up_weight", up_weight), ("down_weight", down_weight)):
            if t.dtype != torch.bfloat16 or not t.is_cuda or t.dim() != 2:
                raise ValueError(f"{name} must be a 2-D bf16 CUDA tensor")
        self.hidden, self.in_features = up_weight.shape
        self.out_features = down_weight.shape[0]
        if down_weight.shape[1] != self.hidden or self.hidden % 128 != 0:
            raise ValueError("down_weight must be [out, hidden] with hidden % 128 == 0")
        wq, sw = quantize_weight(up_weight.contiguous(), PER_ROW)
        self.register_buffer("up_image", pack_weight(wq))
        self.register_buffer("up_scale", sw)
        wq2, sw2 = quantize_weight(down_weight.contiguous(), BLOCK)
        self.register_buffer("down_image", pack_weight(wq2))
        self.register_buffer("down_scale", sw2)
        self.register_buffer("up_bias", None if up_bias is None else up_bias.detach().to(torch.bfloat16).contiguous())
        self.register_buffer("down_bias",
                             None if down_bias is None else down_bias.detach().to(torch.bfloat16).contiguous())
        self._ws = None

    def forward(self, x):
        if x.dtype != torch.bfloat16:
            raise TypeError("Int8FFN takes bf16 activations")
        lead = x.shape[:-1]
        x2 = x.reshape(-1, self.in_features).contiguous()
        M = x2.shape[0]
        need = max(linear_workspace_size(M, self.hidden, self.in_features), 256)
        if self._ws is None or self._ws.numel() < need or self._ws.device != x2.device:
            self._ws = torch.empty(need, dtype=torch.uint8, device=x2.device)
        gimg, sg, _, _ = linear_postscale_gelu_quant(x2, self.up_image, self.up_scale, self.up_bias, workspace=self._ws)
        y = gemm_blockwise_images(gimg, sg, self.down_image, self.down_scale, self.down_bias)
        return y.reshape(*lead, self.out_features)

    def extra_repr(self):
        return f"in_features={self.in_features}, hidden={self.hidden}, out_features={self.out_features}"
