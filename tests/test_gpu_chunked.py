"""GPU: chunked prefill (fs_step_batch_chunked).

A lane's prompt consumed in chunks, next to other lanes decoding in the same
steps, must give bit for bit the logits and KV of feeding the same tokens one
per call (every row's K/V are appended before attention, with the same
rounding as the one-token path). Covered: the TMA attention (long-context
handle), the cp.async attention (short-context handle) and the tiled
attention of f32-KV handles; rows of a lane in any order; atomic refusals.
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


@pytest.fixture(scope="module")
def smol_l2():
    cfg = synth.with_layers(synth.MODEL_S, 2)
    return cfg, synth.make_weights(cfg, seed=1, fmt="bf16")


def _logits(h, fn, lanes, pos, toks, V):
    import torch
    buf = torch.empty((len(lanes), V), dtype=torch.float32, device="cuda")
    p = np.array(pos, np.int32)
    fn(h, lanes, p, toks, logits_out=buf)
    torch.cuda.synchronize()
    return buf.cpu().numpy(), p


def _compare(cfg, W, wdt, kvdt, max_pos, expect_path):
    V = cfg["V"]
    rng = np.random.default_rng(7)
    prompt = [int(t) for t in rng.integers(0, V, 45)]
    other = [int(t) for t in rng.integers(0, V, 60)]
    chunks = [13, 17, 15]
    # reference: one token per call; lane 0 ingests the prompt, lane 1 decodes
    # its own tokens in the same calls
    h1 = U.make_gpu(cfg, W, wdt, kvdt, max_lanes=32, max_pos=max_pos)
    h2 = U.make_gpu(cfg, W, wdt, kvdt, max_lanes=32, max_pos=max_pos)
    try:
        if expect_path:
            assert fs.fs_attention_path(h1) == expect_path
        ref = {}
        for t in range(45):
            lg, _ = _logits(h1, fs.fs_decode_step_batch, [0, 1], [t, t], [prompt[t], other[t]], V)
            ref[(0, t)] = lg[0]
            ref[(1, t)] = lg[1]
        # chunked: each step carries one chunk of lane 0, rows in reverse
        # position order
        pos0 = 0
        for c in chunks:
            rows_l = [0] * c
            p0 = list(range(pos0 + c - 1, pos0 - 1, -1))
            toks = [prompt[p] for p in p0]
            lg, pnew = _logits(h2, fs.fs_step_batch_chunked, rows_l, p0, toks, V)
            assert pnew.tolist() == [p + 1 for p in p0]
            for r, p in enumerate(p0):
                assert np.array_equal(lg[r].view(np.int32), ref[(0, p)].view(np.int32)), (c, p)
            pos0 += c
        for t in range(45):  # lane 1 one token per call, as in the reference
            lg, _ = _logits(h2, fs.fs_decode_step_batch, [1], [t], [other[t]], V)
            assert np.array_equal(lg[0].view(np.int32), ref[(1, t)].view(np.int32)), t
        # a mixed step: lane 0's decode row next to a 5-token chunk of lane 2
        lg2, _ = _logits(h2, fs.fs_step_batch_chunked, [2, 0, 2, 2, 2, 2],
                         [0, 45, 1, 2, 3, 4], [3, 9, 4, 5, 6, 7], V)
        lg1, _ = _logits(h1, fs.fs_decode_step_batch, [0], [45], [9], V)
        assert np.array_equal(lg2[1].view(np.int32), lg1[0].view(np.int32))
        assert fs.fs_lane_length(h2, 2) == 5 and fs.fs_lane_length(h2, 0) == 46
        hd, Hkv = cfg["hd"], cfg["Hkv"]
        for l in range(cfg["L"]):
            k1, v1 = fs.fs_lane_export_kv(h1, 0, l, Hkv, hd)
            k2, v2 = fs.fs_lane_export_kv(h2, 0, l, Hkv, hd)
            assert np.array_equal(k1.view(np.int32), k2.view(np.int32))
            assert np.array_equal(v1.view(np.int32), v2.view(np.int32))
        # pages hold the same tokens (their indices differ: lane 0 took its
        # pages in another order relative to lane 1)
        assert len(fs.fs_lane_pages(h1, 0)) == len(fs.fs_lane_pages(h2, 0)) == 3
    finally:
        fs.fs_destroy(h1)
        fs.fs_destroy(h2)


def test_chunked_equals_one_token_steps_tma(smol_l2):
    cfg, W = smol_l2
    _compare(cfg, W, fs.FS_DTYPE_BF16, fs.FS_DTYPE_BF16, 600, "tma-mma")


def test_chunked_equals_one_token_steps_cp_async(smol_l2):
    cfg, W = smol_l2
    _compare(cfg, W, fs.FS_DTYPE_BF16, fs.FS_DTYPE_BF16, 200, "cp.async-mma")


def test_chunked_equals_one_token_steps_f32_tiled():
    cfg = synth.MODEL_T
    W = synth.make_weights(cfg, seed=1, fmt="f32")
    _compare(cfg, W, fs.FS_DTYPE_F32, fs.FS_DTYPE_F32, 128, None)


def test_chunked_refusals_are_atomic(smol_l2):
    cfg, W = smol_l2
    h = U.make_gpu(cfg, W, fs.FS_DTYPE_BF16, max_lanes=8, max_pos=64)
    try:
        fs.fs_step_batch_chunked(h, [0, 0, 0], [0, 1, 2], [1, 2, 3])
        before = (fs.fs_lane_pages(h, 0), fs.fs_lane_length(h, 0))
        bad = [([0, 0], [3, 5], [1, 1]),          # gap in the positions
               ([0, 0], [3, 3], [1, 1]),          # a position twice
               ([0, 1], [2, 0], [1, 1]),          # not the lane's next position
               ([0] * 9, list(range(3, 12)), [1] * 9)]  # more rows than lanes
        for la, po, to in bad:
            with pytest.raises(fs.FsError):
                fs.fs_step_batch_chunked(h, la, po, to)
        assert (fs.fs_lane_pages(h, 0), fs.fs_lane_length(h, 0)) == before
    finally:
        fs.fs_destroy(h)
