"""The allocation-free post-scale GEMM entry point, through the C ABI.

w8a8_gemm_postscale_noalloc serves callers that cannot allocate device memory
where they call (a host callback or real-time loop that must not trigger
cudaMalloc's synchronization, or a plugin whose framework owns the
allocator): its scratch is a fixed 64 MiB device array inside the library.
This file is collected last so that a failure here leaves every other test
already run; it also passes when run alone in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

from gpu_helpers import assert_bf16_close, bits, edge_indices

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _inputs(M, N, K, seed, bias):
    g = torch.Generator().manual_seed(seed)
    X = (torch.randn((M, K), generator=g)).to(torch.bfloat16).to(DEV)
    W = (torch.randn((N, K), generator=g) * 0.02).to(torch.bfloat16).to(DEV)
    b = (torch.randn((N,), generator=g) * 0.01).to(torch.bfloat16).to(DEV) if bias else None
    return X, W, b


def _call_noalloc(L, Xq, sx, Wq, sw, b, Y):
    M, K = Xq.shape
    N = Wq.shape[0]
    P = ctypes.c_void_p
    return L.w8a8_gemm_postscale_noalloc(P(Xq.data_ptr()), P(sx.data_ptr()), P(Wq.data_ptr()), P(sw.data_ptr()),
                                         None if b is None else P(b.data_ptr()), P(Y.data_ptr()), M, N, K,
                                         P(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_workspace_entry_point_twice(w8a8):
    L = w8a8.lib()
    # two calls in a row, different shapes (the second at the 64 MiB limit),
    # each against the workspace entry point on the same inputs
    for (M, N, K, bias, seed) in [(300, 520, 1040, True, 1), (4096, 4096, 4096, False, 2)]:
        X, W, b = _inputs(M, N, K, seed, bias)
        Xq, sx = w8a8.quantize_act(X)
        Wq, sw = w8a8.quantize_weight(W)
        Y_ref = w8a8.gemm_postscale(Xq, sx, Wq, sw, b)
        Y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=DEV)
        assert _call_noalloc(L, Xq, sx, Wq, sw, b, Y) == 0
        torch.cuda.synchronize()
        assert_bf16_close(bits(Y), bits(Y_ref), 1)
    assert w8a8.get_device_error() == (0, 0)


def test_noalloc_repeat_same_shape_and_limit(w8a8):
    L = w8a8.lib()
    X, W, b = _inputs(129, 264, 4112, 3, True)
    Xq, sx = w8a8.quantize_act(X)
    Wq, sw = w8a8.quantize_weight(W)
    Y_ref = w8a8.gemm_postscale(Xq, sx, Wq, sw, b)
    for _ in range(2):
        Y = torch.zeros((129, 264), dtype=torch.bfloat16, device=DEV)
        assert _call_noalloc(L, Xq, sx, Wq, sw, b, Y) == 0
        torch.cuda.synchronize()
        assert_bf16_close(bits(Y), bits(Y_ref), 1)
    # one row past the limit is rejected with W8A8_ERR_WORKSPACE, nothing launched
    M, N, K = 4097, 4096, 4096
    Xq = torch.zeros((M, K), dtype=torch.int8, device=DEV)
    Wq = torch.zeros((N, K), dtype=torch.int8, device=DEV)
    Y = torch.zeros((M, N), dtype=torch.bfloat16, device=DEV)
    st = _call_noalloc(L, Xq, torch.ones(M, device=DEV), Wq, torch.ones(N, device=DEV), None, Y)
    assert st == 7
    assert "no-alloc scratch holds" in L.w8a8_last_error_detail().decode()
    assert torch.all(Y == 0)


def test_noalloc_few_token_paths(w8a8):
    """The two few-token routes use the scratch differently: the GEMV (M <= 4)
    needs none, the int8-operand GEMM (5..288 tokens) the fp16 image of the
    tokens and, where K is split (77 x 3072), int32 sums and counters that
    its first kernel zeroes.  77 x 13824 x 5120 would need ~142 MB as bf16
    images but fits through the int8 route; two calls in a row each, against
    the workspace entry point."""
    L = w8a8.lib()
    for (M, N, K, seed) in [(4, 3072, 5120, 4), (77, 13824, 5120, 5), (77, 13824, 5120, 6), (77, 3072, 5120, 7),
                            (77, 3072, 5120, 8), (257, 13824, 5120, 9), (200, 3072, 5120, 10),
                            (200, 3072, 5120, 11)]:
        X, W, b = _inputs(M, N, K, seed, True)
        Xq, sx = w8a8.quantize_act(X)
        Wq, sw = w8a8.quantize_weight(W)
        Y_ref = w8a8.gemm_postscale(Xq, sx, Wq, sw, b)
        Y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=DEV)
        assert _call_noalloc(L, Xq, sx, Wq, sw, b, Y) == 0
        torch.cuda.synchronize()
        if not torch.equal(Y, Y_ref):
            # which side moved: each path once more
            Y_ref2 = w8a8.gemm_postscale(Xq, sx, Wq, sw, b)
            Y2 = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=DEV)
            _call_noalloc(L, Xq, sx, Wq, sw, b, Y2)
            torch.cuda.synchronize()
            bad = Y != Y_ref
            rows = bad.any(dim=1).nonzero().flatten().tolist()
            cols = bad.any(dim=0).nonzero().flatten().tolist()
            pytest.fail(f"{M}x{N}x{K}: {int(bad.sum())} outputs differ, NaN in Y {int(torch.isnan(Y).sum())}, "
                        f"rows {rows[:3]}..{rows[-3:]} ({len(rows)}), cols {cols[:3]}..{cols[-3:]} ({len(cols)}), "
                        f"workspace repeat equal {torch.equal(Y_ref, Y_ref2)}, no-alloc repeat equal "
                        f"{torch.equal(Y, Y2)}, no-alloc repeat vs workspace {torch.equal(Y2, Y_ref)}, "
                        f"device error {w8a8.get_device_error()}")
    assert w8a8.get_device_error() == (0, 0)


def test_noalloc_against_oracle_and_allocates_nothing(w8a8, oracle):
    """At the 64 MiB limit (4096 x 4096 x 4096): sampled outputs (every tile
    edge and random points) against the CPU oracle, and a second call that
    changes neither the device's free memory nor torch's allocation count."""
    L = w8a8.lib()
    M = N = K = 4096
    X, W, b = _inputs(M, N, K, 7, True)
    Xq, sx = w8a8.quantize_act(X)
    Wq, sw = w8a8.quantize_weight(W)
    Y = torch.zeros((M, N), dtype=torch.bfloat16, device=DEV)
    assert _call_noalloc(L, Xq, sx, Wq, sw, b, Y) == 0  # warm-up: kernels loaded
    torch.cuda.synchronize()
    free0, alloc0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
    Y.zero_()
    assert _call_noalloc(L, Xq, sx, Wq, sw, b, Y) == 0
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0 and torch.cuda.memory_allocated() == alloc0
    rng = np.random.default_rng(0)
    rows = edge_indices(M, 128, 16, rng)
    cols = edge_indices(N, 224, 16, rng)
    Xs = bits(X[torch.from_numpy(rows).to(DEV)])
    Yo, _ = oracle.linear_sampled(Xs, bits(W), bits(b), np.arange(len(rows)), cols, oracle.PER_ROW)
    Yg = bits(Y[torch.from_numpy(rows).to(DEV)][:, torch.from_numpy(cols).to(DEV)])
    d = assert_bf16_close(Yg, Yo, 1)
    assert d.max() == 0
    assert w8a8.get_device_error() == (0, 0)
