"""Seeded synthetic inputs for the W8A8 Linear workloads.

This module holds no arithmetic of the method: it only draws bf16 inputs
with the shapes and value distributions of the workloads, so that the CUDA
path and the CPU oracle can be fed the same bytes.  The workloads stand in
for the LTX-2 FFN Linears the pages measure ("TurboDiffusion Integration
Notes", section "Differences From TurboDiffusion": TileLang post-scale kernel
tuned for LTX FFN shapes); no model weights or datasets are involved.

Recipe (every tensor drawn in fp32, then rounded to bf16):
  X      ~ N(0, 1), generator seeded with `seed`; a fixed random set of
         round(frac * K) input channels (columns), chosen by randperm(K)
         from a generator seeded with seed + 1, is multiplied by `scale`
         (activation outliers);
  X_gelu = GELU(N(0, 1)) (erf form) for the FFN down-projection;
  W      ~ N(0, std), generator seeded with seed + 1000;
  bias   ~ N(0, std), generator seeded with seed + 2000.
The separate seed offsets keep X, W and bias from sharing a random stream.
"""
import dataclasses

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    mode: str                 # "postscale" | "blockwise"
    x_kind: str = "gauss"     # "gauss" | "gelu"
    outlier_frac: float = 0.0
    outlier_scale: float = 1.0
    w_std: float = 0.02
    bias_std: float = 0.0     # 0: no bias
    seed: int = 0

    @property
    def ops(self) -> float:
        return 2.0 * self.M * self.N * self.K


def _gen(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def outlier_channels(K, frac, seed, device="cpu"):
    n = int(round(frac * K))
    if n == 0:
        return torch.empty(0, dtype=torch.long, device=device)
    return torch.randperm(K, generator=_gen(seed + 1, device), device=device)[:n]


def make_x(wl: Workload, device="cpu", M=None):
    M = wl.M if M is None else M
    x = torch.randn((M, wl.K), generator=_gen(wl.seed, device), device=device, dtype=torch.float32)
    if wl.x_kind == "gelu":
        x = torch.nn.functional.gelu(x)
    elif wl.outlier_frac > 0:
        idx = outlier_channels(wl.K, wl.outlier_frac, wl.seed, device)
        x[:, idx] *= wl.outlier_scale
    return x.to(torch.bfloat16)


def make_w(wl: Workload, device="cpu"):
    w = torch.randn((wl.N, wl.K), generator=_gen(wl.seed + 1000, device), device=device, dtype=torch.float32)
    return (w * wl.w_std).to(torch.bfloat16)


def make_bias(wl: Workload, device="cpu"):
    if wl.bias_std <= 0:
        return None
    b = torch.randn((wl.N,), generator=_gen(wl.seed + 2000, device), device=device, dtype=torch.float32)
    return (b * wl.bias_std).to(torch.bfloat16)


# The five workload families.
TINY = Workload("tiny_postscale_64x128x256", 64, 128, 256, "postscale", w_std=0.02, bias_std=0.01)
SQUARE = Workload("square_postscale_4096", 4096, 4096, 4096, "postscale", outlier_frac=0.01, outlier_scale=20.0,
                  w_std=0.02)
FFN_UP = Workload("ffn_up_postscale_32768x13824x5120", 32768, 13824, 5120, "postscale", outlier_frac=0.005,
                  outlier_scale=30.0, w_std=0.015, bias_std=0.01)
FFN_DOWN = Workload("ffn_down_blockwise_32768x5120x13824", 32768, 5120, 13824, "blockwise", x_kind="gelu",
                    w_std=0.01)
RAGGED_M = (1, 77, 257, 1000, 28672, 32769)
RAGGED_N = (3072, 5120, 13824, 15432)


def ragged(M, N):
    return Workload(f"ragged_postscale_{M}x{N}x5120", M, N, 5120, "postscale", outlier_frac=0.01,
                    outlier_scale=20.0, w_std=0.02)


ALL = {w.name: w for w in (TINY, SQUARE, FFN_UP, FFN_DOWN)}


def bf16_bits(t):
    """bf16 tensor -> numpy uint16 bit patterns (host copy)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")
