"""GPU: greedy decode without materialising logits (fs_decode_step_greedy).

The tokens must equal, step after step, those of fs_decode_step_batch
followed by fs_sample with temperature 0 (argmax, lowest index on ties), for
bf16 and Q8_0 heads (argmax epilogue of the tensor-core GEMM) and the f32
model (logits + sampler kernel); a greedy step leaves no logits to sample.
"""
import numpy as np
import pytest

from continuous_transformer_decode_gb300 import fs, synth
from tests import _gpu_util as U

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from continuous_transformer_decode_gb300 import build
    build.build()


def _run(cfg, W, wdt, kvdt, B, steps=6, device_out=False):
    import torch
    V = cfg["V"]
    h1 = U.make_gpu(cfg, W, wdt, kvdt, max_lanes=64, max_pos=32)
    h2 = U.make_gpu(cfg, W, wdt, kvdt, max_lanes=64, max_pos=32)
    try:
        rng = np.random.default_rng(B)
        lanes = list(range(B))
        toks = [int(t) for t in rng.integers(0, V, B)]
        p1 = np.zeros(B, np.int32)
        p2 = np.zeros(B, np.int32)
        for _ in range(steps):
            fs.fs_decode_step_batch(h1, lanes, p1, toks)
            want = fs.fs_sample(h1, np.zeros(B), np.zeros(B), np.zeros(B))
            if device_out:
                out = torch.empty(B, dtype=torch.int32, device="cuda")
                fs.fs_decode_step_greedy(h2, lanes, p2, toks, out)
                torch.cuda.synchronize()
                got = out.cpu().numpy()
            else:
                got = fs.fs_decode_step_greedy(h2, lanes, p2, toks)
            assert got.tolist() == want.tolist()
            toks = [int(t) for t in got]
        assert p1.tolist() == p2.tolist()
        with pytest.raises(fs.FsError):
            fs.fs_sample(h2, np.zeros(B), np.zeros(B), np.zeros(B))
    finally:
        fs.fs_destroy(h1)
        fs.fs_destroy(h2)


@pytest.fixture(scope="module")
def smol_l2():
    cfg = synth.with_layers(synth.MODEL_S, 2)
    return cfg, synth.make_weights(cfg, seed=1, fmt="bf16")


@pytest.mark.parametrize("B", [1, 7, 64])
def test_greedy_bf16_equals_sampler(smol_l2, B):
    cfg, W = smol_l2
    _run(cfg, W, fs.FS_DTYPE_BF16, fs.FS_DTYPE_BF16, B, device_out=(B == 7))


def test_greedy_q8_equals_sampler(smol_l2):
    cfg, W = smol_l2
    _run(cfg, U.quantize_weights(W), fs.FS_DTYPE_Q8_0, fs.FS_DTYPE_BF16, 13)


def test_greedy_f32_equals_sampler():
    cfg = synth.MODEL_T
    W = synth.make_weights(cfg, seed=1, fmt="f32")
    _run(cfg, W, fs.FS_DTYPE_F32, fs.FS_DTYPE_F32, 4)
