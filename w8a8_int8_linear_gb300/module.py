"""Int8Linear: a torch module over the W8A8 C ABI.

"Acceleration Backends" names an `Int8Linear` module and a `quant_linear`
switch; "TurboDiffusion Integration Notes", section "Reused Components",
describes what it does: weights quantized to INT8 once at model
initialization, activations quantized dynamically before every Linear.  This
module does exactly that through the library: the weight is quantized and its
exact bf16 image packed once (`from_linear` / `__init__`), and every forward
is one fused call (per-token or 1x128 quantization plus the INT8 GEMM).  It
keeps no bf16 copy of the original weight and has no fallback path: every
shape runs the INT8 kernels.
"""
import torch

from . import BLOCK, PER_ROW, linear_blockwise, linear_postscale, linear_workspace_size, pack_weight, \
    quantize_weight


class Int8Linear(torch.nn.Module):
    """y = W8A8(x) for x [..., in_features] bf16 on a sm_103 device."""

    def __init__(self, weight, bias=None, mode="postscale"):
        super().__init__()
        if mode not in ("postscale", "blockwise"):
            raise ValueError("mode must be 'postscale' or 'blockwise'")
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

    def _workspace(self, M, device):
        need = max(linear_workspace_size(M, self.out_features, self.in_features), 256)
        if self._ws is None or self._ws.numel() < need or self._ws.device != device:
            self._ws = torch.empty(need, dtype=torch.uint8, device=device)
        return self._ws

    def forward(self, x):
        if x.dtype != torch.bfloat16:
            raise TypeError("Int8Linear takes bf16 activations")
        lead = x.shape[:-1]
        x2 = x.reshape(-1, self.in_features).contiguous()
        fn = linear_postscale if self.mode == "postscale" else linear_blockwise
        y, _, _ = fn(x2, self.weight_image, self.weight_scale, self.bias,
                     workspace=self._workspace(x2.shape[0], x2.device))
        return y.reshape(*lead, self.out_features)

    def extra_repr(self):
        return f"in_features={self.in_features}, out_features={self.out_features}, mode={self.mode}"
