"""Pins of the scheduler and page-allocator references."""
import json
import os

import numpy as np
import pytest

import oracle.core as O
from oracle import pages as P
from oracle import sched as S
from continuous_transformer_decode_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_dgr012_concurrency_sweep_replay():
    g = json.load(open(os.path.join(GOLDEN, "dgr012_concurrency_sweep.json")))
    for row in g["rows"]:
        r = S.tick_sweep(row["concurrency"], g["sessions"], g["prompt_len"],
                         g["new_tokens"])
        assert r["ticks"] == row["ticks"]
        assert round(r["avg_occupancy"], 3) == row["avg_occupancy"]
        assert r["max_occupancy"] == row["max_occupancy"]
        assert round(r["tokens_per_tick"], 3) == row["tokens_per_tick"]
    tot = g["total_tokens"]
    assert g["sessions"] * (g["new_tokens"] - 1) == tot["decode"]
    assert g["sessions"] * g["prompt_len"] == tot["prefill"]


def test_page_model_lowest_free_and_counts():
    pm = P.PageModel(n_pages=8, page_size=4, max_lanes=3, max_pages_per_lane=4)
    assert pm.step([0, 1], [0, 0], [1, 1], 10) == P.OK
    assert pm.table(0) == [0] and pm.table(1) == [1]
    for p in range(1, 9):
        assert pm.step([1], [p], [1], 10) == P.OK
    assert pm.table(1) == [1, 2, 3]  # lengths 9 -> ceil(9/4) = 3 pages
    assert pm.reset(0) == P.OK
    assert pm.step([2], [0], [1], 10) == P.OK
    assert pm.table(2) == [0]  # lowest free index reused
    for k in range(3):
        assert len(pm.table(k)) == -(-pm.length[k] // 4)


def test_page_model_errors_are_atomic():
    pm = P.PageModel(n_pages=2, page_size=2, max_lanes=4, max_pages_per_lane=8)
    assert pm.step([0, 1], [0, 0], [0, 0], 5) == P.OK
    snap = ([list(t) for t in pm.tables], list(pm.length), sorted(pm.free))
    assert pm.step([0, 0], [1, 1], [0, 0], 5) == P.ERR_DUP_LANE
    assert pm.step([0], [0], [0], 5) == P.ERR_POSITION
    assert pm.step([0], [1], [5], 5) == P.ERR_TOKEN
    assert pm.step([4], [0], [0], 5) == P.ERR_LANE
    assert pm.step([2], [0], [0], 5) == P.ERR_KV_FULL  # pool exhausted
    assert ([list(t) for t in pm.tables], list(pm.length), sorted(pm.free)) == snap


@pytest.fixture(scope="module")
def tiny_engine():
    cfg = synth.MODEL_T
    m = O.Model(cfg, synth.make_weights(cfg, seed=1, fmt="f32"), O.F32)
    return cfg, m


def _engine(m, n_lanes, max_pos=96):
    lanes = [m.lane(max_pos) for _ in range(n_lanes)]

    def step_fn(ks, poss, toks):
        for k, p in zip(ks, poss):
            assert lanes[k].pos == p
        return m.step_batch([lanes[k] for k in ks], toks)

    def reset_fn(k):
        lanes[k].reset()

    def sample_fn(row, temp, seed, counter):
        return O.sample(row, temp, seed, counter)
    return step_fn, reset_fn, sample_fn


def _engine_rows(m, n_lanes, max_pos=96):
    """Rows in order through serial Step: a lane on several rows (chunked
    prefill) consumes them one after another."""
    lanes = [m.lane(max_pos) for _ in range(n_lanes)]

    def step_fn(ks, poss, toks):
        out = []
        for k, p, t in zip(ks, poss, toks):
            assert lanes[k].pos == p
            out.append(m.step(lanes[k], t))
        return out

    def reset_fn(k):
        lanes[k].reset()

    def sample_fn(row, temp, seed, counter):
        return O.sample(row, temp, seed, counter)
    return step_fn, reset_fn, sample_fn


def test_scheduler_reference_chunked_prefill_per_job_equals_serial(tiny_engine):
    cfg, m = tiny_engine
    g = np.random.default_rng(5)
    jobs = [dict(id=j, arrive=int(g.integers(0, 12)),
                 prompt=synth.make_prompts(1, int(g.integers(1, 25)), cfg["V"],
                                           seed=200 + j)[0],
                 max_new=int(g.integers(1, 8)),
                 temperature=0.0 if j % 2 else 0.8, seed=2000 + j) for j in range(8)]
    step_fn, reset_fn, sample_fn = _engine_rows(m, 3)
    ref = S.Reference(3, 7, step_fn, sample_fn, reset_fn, prefill_chunk=5)
    done = ref.run(jobs)
    s_step, s_reset, s_sample = _engine(m, 1)
    for job in jobs:
        assert done[job["id"]] == S.serial_job(job, s_step, s_sample, s_reset), job["id"]
    assert max(ref.prefill_per_step) <= 7 and max(ref.occupancy) <= 3
    assert ref.prefill_tokens == sum(len(j["prompt"]) for j in jobs)


def test_scheduler_reference_per_job_equals_serial(tiny_engine):
    cfg, m = tiny_engine
    g = np.random.default_rng(4)
    jobs = []
    for j in range(10):
        jobs.append(dict(id=j, arrive=int(g.integers(0, 12)),
                         prompt=synth.make_prompts(1, int(g.integers(1, 9)),
                                                   cfg["V"], seed=100 + j)[0],
                         max_new=int(g.integers(1, 10)),
                         temperature=0.0 if j % 2 else 0.8, seed=1000 + j))
    step_fn, reset_fn, sample_fn = _engine(m, 3)
    ref = S.Reference(3, 2, step_fn, sample_fn, reset_fn)
    done = ref.run(jobs)
    assert sorted(done) == list(range(10))
    s_step, s_reset, s_sample = _engine(m, 1)
    for job in jobs:
        solo = S.serial_job(job, s_step, s_sample, s_reset)
        assert done[job["id"]] == solo, job["id"]
        assert len(solo) == job["max_new"]
    assert max(ref.occupancy) <= 3
    assert ref.prefill_tokens == sum(len(j["prompt"]) for j in jobs)
    assert ref.decode_tokens == sum(j["max_new"] - 1 for j in jobs)


def test_scheduler_reference_decode_first_bounded_prefill(tiny_engine):
    cfg, m = tiny_engine
    seen = []
    step_fn, reset_fn, sample_fn = _engine(m, 4)

    def spy(ks, poss, toks):
        seen.append(list(ks))
        return step_fn(ks, poss, toks)
    ref = S.Reference(4, 1, spy, sample_fn, reset_fn)
    ref.submit(dict(id=0, prompt=[1], max_new=12, temperature=0.0, seed=0))
    ref.step()  # lane 0 consumes its one prompt token -> decoding from now on
    for j in range(1, 4):
        ref.submit(dict(id=j, prompt=[2, 3, 4, 5], max_new=2,
                        temperature=0.0, seed=0))
    for _ in range(6):
        ref.step()
    for ks in seen[1:]:
        assert 0 in ks            # the in-flight decode runs every step
    assert max(ref.prefill_per_step) == 1  # at most one prompt token per step
    assert sum(ref.prefill_per_step) == 1 + 6  # budget used on every step


def test_scheduler_reference_stop_id_and_lane_reuse(tiny_engine):
    cfg, m = tiny_engine
    step_fn, reset_fn, sample_fn = _engine(m, 1)
    job = dict(id=0, prompt=[7, 8], max_new=20, temperature=0.0, seed=0)
    full = S.serial_job(job, step_fn, sample_fn, reset_fn)
    stop = full[3]
    first = full.index(stop)
    ref = S.Reference(1, 1, step_fn, sample_fn, reset_fn)
    done = ref.run([dict(job, stop=stop), dict(job, id=1, arrive=0)])
    assert done[0] == full[:first + 1]  # retired on the stop id
    assert done[1] == full              # the freed lane serves the next job


def test_scheduler_reference_kv_budget_admission(tiny_engine):
    """Bounded admission ("DGR-012", "Summary"): a job whose prompt + new
    tokens exceed the budget is rejected up front; the others wait until the
    running jobs' reservations leave room, never exceed the budget, release
    it as they retire, and still get their serial tokens."""
    cfg, m = tiny_engine
    g = np.random.default_rng(6)
    jobs = [dict(id=j, arrive=int(g.integers(0, 6)),
                 prompt=synth.make_prompts(1, int(g.integers(1, 20)), cfg["V"],
                                           seed=300 + j)[0],
                 max_new=int(g.integers(1, 10)),
                 temperature=0.0 if j % 2 else 0.8, seed=3000 + j) for j in range(10)]
    budget = 22
    step_fn, reset_fn, sample_fn = _engine_rows(m, 4)
    ref = S.Reference(4, 8, step_fn, sample_fn, reset_fn, prefill_chunk=4,
                      kv_budget_tokens=budget)
    done = ref.run(jobs)
    too_big = [j["id"] for j in jobs if len(j["prompt"]) + j["max_new"] > budget]
    assert ref.rejected == too_big and too_big
    assert sorted(done) == sorted(j["id"] for j in jobs if j["id"] not in too_big)
    assert ref.reserved == 0 and ref.reserved_max <= budget and ref.kv_wait_steps > 0
    s_step, s_reset, s_sample = _engine(m, 1)
    for job in jobs:
        if job["id"] in done:
            assert done[job["id"]] == S.serial_job(job, s_step, s_sample, s_reset), job["id"]


def test_scheduler_reference_prefix_reuse_per_job_equals_serial(tiny_engine):
    """Prefix reuse (Clone of a running lane, then Evict of the clone's
    suffix): every job's tokens equal its serial run bit for bit, because a
    position's K/V depend only on the tokens up to it; jobs share prompt
    prefixes so that clones happen, and the reused tokens are not fed."""
    cfg, m = tiny_engine
    g = np.random.default_rng(9)
    heads = [synth.make_prompts(1, 10, cfg["V"], seed=300 + i)[0] for i in range(2)]
    jobs = []
    for j in range(10):
        head = [int(t) for t in heads[j % 2][:int(g.integers(3, 11))]]
        tail = [int(t) for t in synth.make_prompts(1, int(g.integers(1, 6)), cfg["V"],
                                                   seed=400 + j)[0]]
        jobs.append(dict(id=j, arrive=int(g.integers(0, 10)), prompt=head + tail,
                         max_new=int(g.integers(1, 8)),
                         temperature=0.0 if j % 2 else 0.8, seed=3000 + j))
    lanes = [m.lane(96) for _ in range(3)]

    def step_fn(ks, poss, toks):
        out = []
        for k, p, t in zip(ks, poss, toks):
            assert lanes[k].pos == p
            out.append(m.step(lanes[k], t))
        return out

    def clone_fn(src, dst):
        assert lanes[dst].pos == 0
        lanes[dst].clone_from(lanes[src])

    ref = S.Reference(3, 4, step_fn, lambda r, t, s, c: O.sample(r, t, s, c),
                      lambda k: lanes[k].reset(), prefill_chunk=3, prefix_reuse_min=2,
                      clone_fn=clone_fn, evict_fn=lambda k, a, b: lanes[k].evict(a, b))
    done = ref.run(jobs)
    assert ref.prefix_hits > 0
    assert ref.prefill_tokens + ref.prefix_tokens == sum(len(j["prompt"]) for j in jobs)
    s_step, s_reset, s_sample = _engine(m, 1)
    for job in jobs:
        assert done[job["id"]] == S.serial_job(job, s_step, s_sample, s_reset), job["id"]



def test_scheduler_reference_cancellation_keeps_the_others_serial(tiny_engine):
    """Cancelling queued and running jobs between steps frees their lanes for
    others; every job not cancelled still gives its serial tokens, and a
    cancelled running job keeps the tokens it had (a prefix of its serial
    run)."""
    cfg, m = tiny_engine
    g = np.random.default_rng(12)
    jobs = [dict(id=j, arrive=int(g.integers(0, 8)),
                 prompt=synth.make_prompts(1, int(g.integers(1, 7)), cfg["V"],
                                           seed=500 + j)[0],
                 max_new=int(g.integers(2, 9)),
                 temperature=0.0 if j % 2 else 0.8, seed=4000 + j) for j in range(10)]
    step_fn, reset_fn, sample_fn = _engine(m, 3)
    ref = S.Reference(3, 2, step_fn, sample_fn, reset_fn)
    order = sorted(jobs, key=lambda j: (j["arrive"], j["id"]))
    i, tick, cancelled = 0, 0, set()
    while i < len(order) or not ref.idle():
        while i < len(order) and order[i]["arrive"] <= tick:
            ref.submit(order[i])
            i += 1
        if tick in (3, 6, 9):  # a running job, then whatever is oldest queued
            running = [l["job"]["id"] for l in ref.lanes if l is not None]
            target = running[0] if tick != 6 or not ref.pending else ref.pending[0]["id"]
            if running or ref.pending:
                assert ref.cancel(target)
                cancelled.add(target)
        ref.step()
        tick += 1
    assert ref.cancelled == len(cancelled) > 0 and ref.reserved == 0
    s_step, s_reset, s_sample = _engine(m, 1)
    for job in jobs:
        solo = S.serial_job(job, s_step, s_sample, s_reset)
        if job["id"] in cancelled:
            assert ref.status(job["id"]) == "cancelled"
            assert ref.done[job["id"]] == solo[:len(ref.done[job["id"]])]
        else:
            assert ref.done[job["id"]] == solo, job["id"]
