"""GPU: fs_gemm_bf16_noalloc, the GEMM entry point that allocates nothing.

It serves callers that cannot call cudaMalloc or cudaFree (device memory
owned by another framework's allocator, latency-critical loops, fixed
memory budgets). Its K-split workspace lives in a static device array of the
library. This file is collected last so that a run stopping at the first
failure has already run every other test; it also passes on its own.
"""
import numpy as np
import pytest

from continuous_transformer_decode_gb300 import build, fs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


@pytest.mark.parametrize("N,K,B,splits", [(960, 576, 17, 4), (576, 1536, 64, 8),
                                          (3072, 576, 5, 2), (1000, 256, 40, 1)])
def test_noalloc_matches_allocating_entry_point_twice(N, K, B, splits):
    import torch
    g = torch.Generator().manual_seed(N + K + B)
    W = (torch.randn(N, K, generator=g) * 0.02).to(torch.bfloat16).cuda()
    X = torch.randn(B, K, generator=g).to(torch.bfloat16).cuda()
    ref = torch.empty(B, N, dtype=torch.float32, device="cuda")
    fs.fs_gemm_bf16(W, X, ref, splits=splits, path=1)
    ref_h = ref.cpu().numpy()
    for _ in range(2):  # two calls in a row share the static scratch
        Y = torch.full((B, N), float("nan"), dtype=torch.float32, device="cuda")
        fs.fs_gemm_bf16_noalloc(W, X, Y, splits=splits)
        got = Y.cpu().numpy()
        # same kernel and decomposition: within the GEMM tests' f64 bound, and
        # in fact bit-identical
        assert np.allclose(got, ref_h, rtol=1e-5, atol=1e-6)
        assert np.array_equal(got.view(np.uint32), ref_h.view(np.uint32))


def test_noalloc_rejects_requests_beyond_its_scratch():
    import torch
    N, K, B = 4096, 1024, 256  # 8 splits x 256 lanes x 4096 rows of f32 > 8 MiB
    W = torch.zeros(N, K, dtype=torch.bfloat16, device="cuda")
    X = torch.zeros(B, K, dtype=torch.bfloat16, device="cuda")
    Y = torch.zeros(B, N, dtype=torch.float32, device="cuda")
    with pytest.raises(fs.FsError) as e:
        fs.fs_gemm_bf16_noalloc(W, X, Y, splits=8)
    assert e.value.name == "FS_ERR_SCRATCH"


def test_noalloc_scratch_limit_boundary():
    """N = 4096 with 4 K splits needs 64 KiB of partials per lane: 127 lanes
    fit the 8 MiB - 64 KiB partial area, 128 do not."""
    import torch
    N, K = 4096, 256
    W = torch.zeros(N, K, dtype=torch.bfloat16, device="cuda")
    for B, ok in ((127, True), (128, False)):
        X = torch.zeros(B, K, dtype=torch.bfloat16, device="cuda")
        Y = torch.full((B, N), 1.0, dtype=torch.float32, device="cuda")
        if ok:
            fs.fs_gemm_bf16_noalloc(W, X, Y, splits=4)
            assert float(Y.abs().max()) == 0.0
        else:
            with pytest.raises(fs.FsError) as e:
                fs.fs_gemm_bf16_noalloc(W, X, Y, splits=4)
            assert e.value.name == "FS_ERR_SCRATCH"
