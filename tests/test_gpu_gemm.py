"""GPU: the weight-streaming GEMM kernels through the fs_gemm_bf16 test hook.

Reference: the same bf16 operands multiplied in f64 on the host. The bound
is the f32 accumulation error of a K-term dot product, relative to the sum
of |terms|. Batch invariance: a lane's outputs are bit-identical whatever
the number of lanes in the call.
"""
import numpy as np
import pytest

from continuous_transformer_decode_gb300 import fs

pytestmark = pytest.mark.gpu


def _case(N, K, B, seed):
    import torch
    g = torch.Generator().manual_seed(seed)
    W = (torch.randn(N, K, generator=g) * 0.02).to(torch.bfloat16)
    X = torch.randn(B, K, generator=g).to(torch.bfloat16)
    return W, X


def _ref(W, X):
    return X.double() @ W.double().T, X.double().abs() @ W.double().abs().T


@pytest.mark.parametrize("N,K,B,splits", [
    (128, 64, 1, 1), (960, 576, 1, 4), (960, 576, 17, 4), (576, 1536, 64, 4),
    (3072, 576, 256, 1), (200, 128, 33, 2), (1000, 576, 600, 3),
    (576, 576, 5, 8)])
def test_tcgen05_gemm_matches_f64(N, K, B, splits):
    import torch
    W, X = _case(N, K, B, N * 7 + K + B)
    Y = torch.empty(B, N, dtype=torch.float32, device="cuda")
    fs.fs_gemm_bf16(W.cuda(), X.cuda(), Y, splits=splits, path=1)
    ref, mag = _ref(W, X)
    err = (Y.cpu().double() - ref).abs()
    bound = 1e-5 * mag + 1e-6
    assert bool((err <= bound).all()), float((err / mag.clamp_min(1e-9)).max())


def test_gemv_matches_f64():
    import torch
    W, X = _case(960, 576, 9, 5)
    Y = torch.empty(9, 960, dtype=torch.float32, device="cuda")
    fs.fs_gemm_bf16(W.cuda(), X.cuda(), Y, path=0)
    ref, mag = _ref(W, X)
    assert bool(((Y.cpu().double() - ref).abs() <= 1e-5 * mag + 1e-6).all())


@pytest.mark.parametrize("splits", [1, 4])
def test_tcgen05_gemm_batch_invariance_bitwise(splits):
    import torch
    W, X = _case(960, 576, 300, 11)
    Wd, Xd = W.cuda(), X.cuda()
    full = torch.empty(300, 960, dtype=torch.float32, device="cuda")
    fs.fs_gemm_bf16(Wd, Xd, full, splits=splits, path=1)
    for B in (1, 2, 16, 17, 100, 256):
        Y = torch.empty(B, 960, dtype=torch.float32, device="cuda")
        fs.fs_gemm_bf16(Wd, Xd[:B].contiguous(), Y, splits=splits, path=1)
        assert torch.equal(Y.view(torch.int32), full[:B].view(torch.int32)), B


@pytest.mark.parametrize("N,K,B,width", [
    (960, 576, 1, 5), (960, 576, 17, 13), (960, 576, 130, 72), (1000, 576, 33, 50),
    (3072, 576, 256, 7), (576, 1536, 64, 113), (4096, 1024, 9, 152), (200, 128, 300, 3)])
def test_tcgen05_stream_k_widths_match_f64(N, K, B, width):
    """Widths whose ranges end inside row tiles: partial pieces, two slots
    per block and multi-piece reductions."""
    import torch
    W, X = _case(N, K, B, N + 3 * K + B + width)
    Y = torch.empty(B, N, dtype=torch.float32, device="cuda")
    fs.fs_gemm_bf16_width(W.cuda(), X.cuda(), Y, width)
    ref, mag = _ref(W, X)
    err = (Y.cpu().double() - ref).abs()
    assert bool((err <= 1e-5 * mag + 1e-6).all()), float((err / mag.clamp_min(1e-9)).max())


def test_tcgen05_stream_k_batch_invariance_bitwise():
    import torch
    W, X = _case(1000, 576, 300, 12)
    Wd, Xd = W.cuda(), X.cuda()
    full = torch.empty(300, 1000, dtype=torch.float32, device="cuda")
    fs.fs_gemm_bf16_width(Wd, Xd, full, 23)
    for B in (1, 16, 33, 257):
        Y = torch.empty(B, 1000, dtype=torch.float32, device="cuda")
        fs.fs_gemm_bf16_width(Wd, Xd[:B].contiguous(), Y, 23)
        assert torch.equal(Y.view(torch.int32), full[:B].view(torch.int32)), B


@pytest.mark.parametrize("N,K,B,splits", [
    (960, 576, 1, 3), (960, 576, 256, 3), (576, 1536, 64, 8), (3072, 576, 200, 3),
    (576, 576, 17, 2), (6144, 4096, 128, 2), (4096, 14336, 3, 4)])
def test_cluster_and_workspace_reductions_give_the_same_bits(N, K, B, splits):
    """The K splits of a row tile summed inside a thread-block cluster
    (distributed shared memory) and through the global workspace: the same
    partial tiles added in the same split order, so the same bits."""
    import torch
    W, X = _case(N, K, B, N + K + B + splits)
    Wd, Xd = W.cuda(), X.cuda()
    a = torch.empty(B, N, dtype=torch.float32, device="cuda")
    b = torch.full((B, N), float("nan"), dtype=torch.float32, device="cuda")
    fs.fs_gemm_bf16(Wd, Xd, a, splits=splits, path=1)
    fs.fs_gemm_bf16(Wd, Xd, b, splits=splits, path=2)
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    ref, mag = _ref(W, X)
    assert bool(((a.cpu().double() - ref).abs() <= 1e-5 * mag + 1e-6).all())
