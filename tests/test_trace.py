"""Kernel timeline tracing: the analysis of records (CPU, hand-built
records), and on the GPU that a traced step yields one launch per kernel
the step enqueued, with ordered stamps."""
import numpy as np
import pytest

from continuous_transformer_decode_gb300 import trace as tr


def _rec(tag, waited, sm, block, t0, t1, t2):
    w0 = (tag << 40) | (int(waited) << 39) | (sm << 24) | block
    return [w0, t0, t1, t2]


def test_launch_grouping_and_summary_by_hand():
    R = np.array([
        _rec(2, 1, 0, 0, 0, 1000, 3000),      # rmsnorm, one block
        _rec(16, 1, 1, 0, 500, 4000, 9000),   # gemm: two blocks
        _rec(16, 1, 2, 1, 600, 4500, 10000),
        _rec(6, 0, 3, 5, 700, 700, 800),      # attention block that left early: ignored
        _rec(6, 1, 3, 0, 2000, 11000, 15000),  # attention
    ], dtype=np.uint64)
    ls = tr.launches(R)
    assert [l["name"] for l in ls] == ["rmsnorm", "gemm_store", "attn_tma"]
    assert ls[1]["blocks"] == 2 and ls[1]["first_ready"] == 4000 and ls[1]["last_exit"] == 10000
    s = tr.summarize(R, steps=1)
    g = s["kernels"]["gemm_store"]
    assert g["mean_gap_us"] == pytest.approx(1.0)      # 4000 - 3000
    assert g["mean_body_us"] == pytest.approx(6.0)     # 10000 - 4000
    assert g["mean_ahead_us"] == pytest.approx(3.5)    # 4000 - 500
    a = s["kernels"]["attn_tma"]
    assert a["mean_gap_us"] == pytest.approx(1.0) and a["mean_body_us"] == pytest.approx(4.0)
    assert s["us_per_step"] == pytest.approx(12.0)     # 15000 - 3000
    assert g["share"] + a["share"] == pytest.approx(1.0)


@pytest.mark.gpu
def test_traced_steps_give_one_launch_per_kernel():
    import torch
    import oracle.core as O
    from continuous_transformer_decode_gb300 import build, fs, synth
    from tests import _gpu_util as U
    build.build()
    T = synth.MODEL_T
    W = synth.make_weights(T, seed=1, fmt="bf16")
    h = U.make_gpu(T, W, fs.FS_DTYPE_BF16, max_lanes=4, max_pos=64)
    try:
        lanes = [0, 1, 2, 3]
        pos = np.zeros(4, np.int32)
        out = torch.empty(4, dtype=torch.int32, device="cuda")
        for t in range(3):
            fs.fs_decode_step_greedy(h, lanes, pos, [1, 2, 3, 4], out)
        torch.cuda.synchronize()
        fs.fs_trace_enable(h, 1 << 16)
        l0 = fs.fs_kernel_launches(h)
        for t in range(4):
            fs.fs_decode_step_greedy(h, lanes, pos, [1, 2, 3, 4], out)
        recs, n = fs.fs_trace_read(h)
        launched = fs.fs_kernel_launches(h) - l0
        assert n == len(recs) > 0
        d = tr.decode(recs)
        assert np.all(d["t_entry"] <= d["t_ready"]) and np.all(d["t_ready"] <= d["t_exit"])
        assert len(tr.launches(recs)) == launched
        # off: nothing more is recorded
        fs.fs_trace_enable(h, 0)
        fs.fs_decode_step_greedy(h, lanes, pos, [1, 2, 3, 4], out)
        torch.cuda.synchronize()
        with pytest.raises(fs.FsError):
            fs.fs_trace_read(h)
    finally:
        fs.fs_destroy(h)
