"""GPU failure detection and memory-safety checks, without faulting a GPU.

- A bounded device wait that nothing satisfies gives up after its limit and
  reports an error status the host reads; the handle then keeps computing
  exactly as before (the context stays usable).
- Canary pages: a spare lane holds seeded K/V that no other lane may touch;
  after decode, chunked, clone and evict work on the other lanes, its K/V
  are bit for bit unchanged (no write strays out of a lane's own pages).
"""
import numpy as np
import pytest

from continuous_transformer_decode_gb300 import build, fs, synth
from tests import _gpu_util as U

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


def _bits(a):
    return np.ascontiguousarray(a).view(np.uint32)


def _logits(h, lanes, toks, V):
    import torch
    pos = np.array([fs.fs_lane_length(h, k) for k in lanes], np.int32)
    buf = torch.empty((len(lanes), V), dtype=torch.float32, device="cuda")
    fs.fs_decode_step_batch(h, list(lanes), pos, list(toks), logits_out=buf)
    torch.cuda.synchronize()
    return buf.cpu().numpy()


def test_bounded_wait_gives_up_and_the_handle_stays_usable():
    cfg = synth.with_layers(synth.MODEL_S, 2)
    W = synth.make_weights(cfg, seed=1, fmt="bf16")
    h = U.make_gpu(cfg, W, fs.FS_DTYPE_BF16, max_lanes=4, max_pos=64)
    try:
        before = _logits(h, [0, 1], [5, 6], cfg["V"])
        assert fs.fs_device_error(h) == 0
        assert fs.fs_selftest_bounded_wait(h, 2000) == 99
        assert fs.fs_device_error(h) == 0  # read and cleared
        fs.fs_lane_reset(h, 0)
        fs.fs_lane_reset(h, 1)
        after = _logits(h, [0, 1], [5, 6], cfg["V"])
        assert np.array_equal(_bits(before), _bits(after))
        with pytest.raises(fs.FsError):
            fs.fs_selftest_bounded_wait(h, 0)
    finally:
        fs.fs_destroy(h)


def test_canary_lane_is_untouched_by_other_lanes_work():
    cfg = synth.with_layers(synth.MODEL_S, 2)
    W = synth.make_weights(cfg, seed=1, fmt="bf16")
    h = U.make_gpu(cfg, W, fs.FS_DTYPE_BF16, max_lanes=6, max_pos=96)
    try:
        spare = 5
        fs.fs_lane_fill_random_kv(h, spare, 80, 1234)
        snap = [fs.fs_lane_export_kv(h, spare, l, cfg["Hkv"], cfg["hd"]) for l in range(cfg["L"])]
        toks = [int(t) for t in synth.make_prompts(1, 40, cfg["V"], seed=3)[0]]
        for t in toks[:20]:  # one-token steps on four lanes, ragged
            ls = [k for k in range(4) if fs.fs_lane_length(h, k) < 10 + 5 * k]
            if ls:
                _logits(h, ls, [t] * len(ls), cfg["V"])
        # chunked prefill rows
        import torch
        n0 = fs.fs_lane_length(h, 0)
        pos = np.array([n0 + i for i in range(6)], np.int32)
        fs.fs_step_batch_chunked(h, [0] * 6, pos, toks[20:26])
        torch.cuda.synchronize()
        fs.fs_lane_clone(h, 1, 4)
        fs.fs_lane_evict(h, 1, 3, 9)
        fs.fs_lane_evict(h, 4, 10, fs.fs_lane_length(h, 4))
        _logits(h, [0, 1, 2, 3, 4], [7] * 5, cfg["V"])
        for l in range(cfg["L"]):
            k, v = fs.fs_lane_export_kv(h, spare, l, cfg["Hkv"], cfg["hd"])
            assert np.array_equal(_bits(k), _bits(snap[l][0])), l
            assert np.array_equal(_bits(v), _bits(snap[l][1])), l
        assert fs.fs_device_error(h) == 0
    finally:
        fs.fs_destroy(h)
