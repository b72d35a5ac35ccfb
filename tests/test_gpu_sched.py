"""GPU: continuous batching through fs_sched over the CUDA decode step.

Per-job tokens must equal the same job run alone (the parity gate of "Fat-
station continuous batching", "Parity"): against the oracle's serial runs on
the f32 tiny model, and bit for bit against GPU serial runs on the bf16
SmolLM2 shape (the GPU step is batch-invariant).
"""
import numpy as np
import pytest

import oracle.core as O
from oracle import sched as S
from continuous_transformer_decode_gb300 import build, fs, synth
from tests import _gpu_util as U

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


def _jobs(n, vocab, seed, max_prompt=12, max_new=10, shared=0):
    """Random jobs; with shared > 0 their prompts start with one of two common
    prefixes of up to `shared` tokens (prefix reuse)."""
    g = np.random.default_rng(seed)
    heads = [[int(t) for t in g.integers(0, vocab, shared)] for _ in range(2)] if shared else []
    jobs = []
    for j in range(n):
        head = heads[j % 2][:int(g.integers(1, shared + 1))] if shared else []
        jobs.append(dict(id=j, arrive=int(g.integers(0, 2 * n)),
                         prompt=head + [int(t) for t in
                                        g.integers(0, vocab, int(g.integers(1, max_prompt)))],
                         max_new=int(g.integers(1, max_new)),
                         temperature=0.0 if j % 2 else 0.8, seed=1000 + 7 * j))
    return jobs


def _run_sched(h, jobs, lanes, budget, chunk=1, reuse=0):
    s = fs.fs_sched_create(h, lanes, budget, prefill_chunk=chunk, prefix_reuse_min=reuse)
    try:
        order = sorted(jobs, key=lambda j: (j["arrive"], j["id"]))
        ids, i, tick = {}, 0, 0
        while i < len(order) or fs.fs_sched_get_stats(s)["active"] or \
                fs.fs_sched_get_stats(s)["queued"]:
            while i < len(order) and order[i]["arrive"] <= tick:
                j = order[i]
                ids[j["id"]] = fs.fs_sched_submit(s, j["prompt"], j["max_new"],
                                                  j["temperature"], j["seed"])
                i += 1
            fs.fs_sched_step(s)
            tick += 1
        st = fs.fs_sched_get_stats(s)
        return {j["id"]: fs.fs_sched_take(s, ids[j["id"]]) for j in jobs}, st
    finally:
        fs.fs_sched_destroy(s)


def test_scheduler_tiny_f32_per_job_equals_oracle_serial():
    cfg = synth.MODEL_T
    W = synth.make_weights(cfg, seed=1, fmt="f32")
    m = O.Model(cfg, W, O.F32)
    jobs = _jobs(14, cfg["V"], 3)
    h = U.make_gpu(cfg, W, fs.FS_DTYPE_F32, fs.FS_DTYPE_F32, max_lanes=4, max_pos=32)
    try:
        got, st = _run_sched(h, jobs, 4, 2)
    finally:
        fs.fs_destroy(h)
    assert st["occupancy_max"] >= 3
    ln = m.lane(32)

    def step_fn(ks, poss, toks):
        return m.step_batch([ln], toks)

    def reset_fn(k):
        ln.reset()

    def sample_fn(row, temp, seed, counter):
        return O.sample(row, temp, seed, counter)
    for j in jobs:
        assert got[j["id"]] == S.serial_job(j, step_fn, sample_fn, reset_fn), j["id"]


@pytest.mark.parametrize("budget,chunk,max_prompt,reuse", [
    (3, 1, 12, 0), (10, 6, 40, 0),
    # prefix reuse: admitted jobs clone a running lane's shared prefix
    (3, 1, 12, 1), (10, 6, 20, 4)])
def test_scheduler_smollm2_bf16_per_job_equals_gpu_serial_bitwise(budget, chunk, max_prompt,
                                                                 reuse):
    """One token per lane per step, chunked prefill (several prompt tokens of
    a lane per step through fs_step_batch_chunked), and prefix reuse (Clone of
    a running lane, Evict of the clone's suffix)."""
    cfg = synth.with_layers(synth.MODEL_S, 2)
    Wb = synth.make_weights(cfg, seed=1, fmt="bf16")
    jobs = _jobs(12, cfg["V"], 5, max_prompt=max_prompt, shared=16 if reuse else 0)
    h = U.make_gpu(cfg, Wb, fs.FS_DTYPE_BF16, max_lanes=6, max_pos=64)
    try:
        got, st = _run_sched(h, jobs, 6, budget, chunk, reuse)
        if chunk > 1:
            assert st["occupancy_max"] > 1
        if reuse:
            assert st["prefix_hits"] > 0
        for k in range(6):
            fs.fs_lane_reset(h, k)
        for j in jobs:  # each job alone on lane 0, one token per step
            fs.fs_lane_reset(h, 0)
            pos = np.zeros(1, np.int32)
            out = []
            for t in j["prompt"]:
                fs.fs_decode_step_batch(h, [0], pos, [t])
            while True:
                tok = int(fs.fs_sample(h, [j["temperature"]], [j["seed"]], [len(out)])[0])
                out.append(tok)
                if len(out) >= j["max_new"]:
                    break
                fs.fs_decode_step_batch(h, [0], pos, [tok])
            assert got[j["id"]] == out, j["id"]
    finally:
        fs.fs_destroy(h)


def test_scheduler_refuses_a_job_longer_than_a_lane():
    """The GPU engine's lane holds max_pos tokens: a job needing more is
    refused at submit (FS_ERR_KV_BUDGET) and counted in the telemetry."""
    cfg = synth.MODEL_T
    W = synth.make_weights(cfg, seed=1, fmt="f32")
    h = U.make_gpu(cfg, W, fs.FS_DTYPE_F32, fs.FS_DTYPE_F32, max_lanes=2, max_pos=32)
    s = fs.fs_sched_create(h, 2, 4, prefill_chunk=4)
    try:
        with pytest.raises(fs.FsError) as e:
            fs.fs_sched_submit(s, list(range(30)), 5)
        assert e.value.name == "FS_ERR_KV_BUDGET"
        jid = fs.fs_sched_submit(s, list(range(20)), 5)
        fs.fs_sched_run(s)
        assert len(fs.fs_sched_take(s, jid)) == 5
        st = fs.fs_sched_get_stats(s)
        assert st["rejected_kv_budget"] == 1 and st["rejected"] == 1
        assert st["kv_reserved_tokens"] == 0 and st["kv_reserved_max"] == 25
        assert st["decode_tok_s"] > 0 and st["seconds"] > 0
    finally:
        fs.fs_sched_destroy(s)
        fs.fs_destroy(h)
