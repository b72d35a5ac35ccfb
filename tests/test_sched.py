"""The product scheduler (C++, fs_sched_*) against the scheduler reference.

CPU: both drive the same model-free stand-in for a model (a per-lane running
hash of consumed tokens, as fs_sched.h defines it, restated here in Python),
so every step's batch, every job's tokens and the counters must match.
"""
import numpy as np
import pytest

from oracle import sched as S
from continuous_transformer_decode_gb300 import build, fs, synth

M64 = (1 << 64) - 1


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


def _mix64(z):
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M64
    return z ^ (z >> 31)


class HashModel:
    """Python restatement of the model-free engine, for the reference (the
    running hash after every consumed token, so that a clone copies a lane
    and an evict of a suffix returns to an earlier hash)."""

    INIT = 0xCBF29CE484222325

    def __init__(self, n_lanes, vocab):
        self.hist = [[] for _ in range(n_lanes)]
        self.vocab = vocab
        self.batches = []

    def h(self, k):
        return self.hist[k][-1] if self.hist[k] else self.INIT

    def reset(self, k):
        self.hist[k] = []

    def clone(self, src, dst):
        assert not self.hist[dst]
        self.hist[dst] = list(self.hist[src])

    def evict(self, k, start, end):
        assert end == len(self.hist[k])  # suffixes only
        del self.hist[k][start:]

    def step(self, ks, poss, toks):
        self.batches.append(list(ks))
        out = []
        for k, p, t in zip(ks, poss, toks):
            assert p == len(self.hist[k])
            self.hist[k].append(((self.h(k) ^ (t & 0xFFFFFFFF)) * 0x100000001B3) & M64)
            out.append(self.hist[k][-1])
        return out  # "logits": each row's state

    def sample(self, state, temp, seed, counter):
        v = state
        if temp != 0.0:
            v = state ^ _mix64((seed + 0x9E3779B97F4A7C15 * (counter + 1)) & M64)
        return int(v % self.vocab)


def _jobs(n, vocab, seed, max_prompt=9, max_new=9, shared=0):
    """Random jobs; with shared > 0, prompts start with one of three common
    prefixes of up to `shared` tokens (prefix reuse)."""
    g = np.random.default_rng(seed)
    heads = [[int(t) for t in g.integers(0, vocab, int(g.integers(2, shared + 1)))]
             for _ in range(3)] if shared else []
    jobs = []
    for j in range(n):
        tail = [int(t) for t in g.integers(0, vocab, int(g.integers(1, max_prompt)))]
        head = heads[int(g.integers(0, 3))][:int(g.integers(1, shared + 1))] if shared else []
        jobs.append(dict(id=j, arrive=int(g.integers(0, 3 * n)),
                         prompt=head + tail,
                         max_new=int(g.integers(1, max_new)),
                         temperature=0.0 if g.uniform() < 0.5 else 0.8,
                         seed=int(g.integers(0, 2**63)),
                         stop=int(g.integers(0, vocab)) if g.uniform() < 0.3 else None))
    return jobs


@pytest.mark.parametrize("lanes,budget,chunk,kv,seed,reuse", [
    (1, 1, 1, 0, 0, 0), (3, 1, 1, 0, 1, 0), (4, 2, 1, 0, 2, 0), (8, 3, 1, 0, 3, 0),
    (5, 100, 1, 0, 4, 0),
    # chunked prefill: several prompt tokens of a lane in one step
    (4, 6, 3, 0, 5, 0), (3, 20, 8, 0, 6, 0), (8, 5, 2, 0, 7, 0), (2, 1, 4, 0, 8, 0),
    (6, 100, 100, 0, 9, 0),
    # bounded admission: a KV budget (tokens) smaller than the lanes could hold
    (4, 2, 1, 14, 10, 0), (6, 8, 4, 35, 11, 0), (3, 100, 100, 25, 12, 0),
    # prefix reuse: jobs sharing prompt prefixes clone a running lane
    (4, 2, 1, 0, 13, 1), (6, 8, 4, 0, 14, 2), (8, 100, 100, 0, 15, 3), (3, 3, 2, 60, 16, 1)])
def test_product_scheduler_matches_reference(lanes, budget, chunk, kv, seed, reuse):
    vocab = 97
    jobs = _jobs(24, vocab, seed, max_prompt=9 if chunk == 1 else 30,
                 shared=12 if reuse else 0)
    model = HashModel(lanes, vocab)
    ref = S.Reference(lanes, budget, model.step, model.sample, model.reset,
                      prefill_chunk=chunk, kv_budget_tokens=kv, prefix_reuse_min=reuse,
                      clone_fn=model.clone, evict_fn=model.evict)
    want = ref.run(jobs)

    s = fs.fs_sched_create_model_free(lanes, vocab, budget, prefill_chunk=chunk,
                                      kv_budget_tokens=kv, prefix_reuse_min=reuse)
    try:
        order = sorted(jobs, key=lambda j: (j["arrive"], j["id"]))
        ids, i, tick, batches, rejected = {}, 0, 0, [], []
        while i < len(order) or fs.fs_sched_get_stats(s)["active"] or \
                fs.fs_sched_get_stats(s)["queued"]:
            while i < len(order) and order[i]["arrive"] <= tick:
                j = order[i]
                try:
                    ids[j["id"]] = fs.fs_sched_submit(
                        s, j["prompt"], j["max_new"], j["temperature"], j["seed"],
                        -1 if j["stop"] is None else j["stop"])
                except fs.FsError as e:
                    assert e.code == -13, e  # FS_ERR_KV_BUDGET
                    rejected.append(j["id"])
                i += 1
            before = fs.fs_sched_get_stats(s)["steps"]
            fs.fs_sched_step(s)
            st = fs.fs_sched_get_stats(s)
            if kv:
                assert st["kv_reserved_tokens"] <= kv
            if st["steps"] > before:
                batches.append(fs.fs_sched_last_batch(s))
            tick += 1
        assert batches == model.batches
        assert rejected == ref.rejected
        for j in jobs:
            if j["id"] not in rejected:
                assert fs.fs_sched_take(s, ids[j["id"]]) == want[j["id"]]
        st = fs.fs_sched_get_stats(s)
        assert st["rejected_kv_budget"] == len(ref.rejected) == st["rejected"]
        assert st["kv_reserved_tokens"] == 0 and st["kv_budget_tokens"] == kv
        assert st["kv_reserved_max"] == ref.reserved_max
        assert st["kv_wait_steps"] == ref.kv_wait_steps
        if kv:
            assert ref.kv_wait_steps > 0 or len(ref.rejected) > 0
        assert st["steps"] == ref.steps
        assert st["prefill_tokens"] == ref.prefill_tokens
        assert st["decode_tokens"] == ref.decode_tokens
        assert st["occupancy_max"] == max(ref.occupancy)
        assert abs(st["occupancy_avg"] - np.mean(ref.occupancy)) < 1e-12
        assert st["jobs_done"] == len(jobs) - len(rejected)
        assert st["prefix_hits"] == ref.prefix_hits
        assert st["prefix_tokens"] == ref.prefix_tokens
        if reuse:
            assert ref.prefix_hits > 0
            assert st["prefill_tokens"] + st["prefix_tokens"] == sum(
                len(j["prompt"]) for j in jobs if j["id"] not in rejected)
    finally:
        fs.fs_sched_destroy(s)


def test_decode_first_and_prefill_budget():
    s = fs.fs_sched_create_model_free(4, 50, max_prefill_tokens_per_tick=1)
    try:
        a = fs.fs_sched_submit(s, [1], 20)
        fs.fs_sched_step(s)  # lane 0 consumes its only prompt token
        for _ in range(3):
            fs.fs_sched_submit(s, [2, 3, 4, 5], 2)
        for _ in range(8):
            fs.fs_sched_step(s)
            lanes = fs.fs_sched_last_batch(s)
            assert 0 in lanes  # the in-flight decode runs every step
        st = fs.fs_sched_get_stats(s)
        assert st["prefill_tokens"] == 1 + 8  # one prompt token per step
    finally:
        fs.fs_sched_destroy(s)


def test_backpressure_and_argument_errors():
    s = fs.fs_sched_create_model_free(1, 50, 1, max_queue=2)
    try:
        fs.fs_sched_submit(s, [1], 3)
        fs.fs_sched_submit(s, [1], 3)
        with pytest.raises(fs.FsError) as e:
            fs.fs_sched_submit(s, [1], 3)
        assert e.value.name == "FS_ERR_QUEUE_FULL"
        with pytest.raises(fs.FsError):
            fs.fs_sched_submit(s, [], 3)
        with pytest.raises(fs.FsError):
            fs.fs_sched_submit(s, [1], 0)
        assert fs.fs_sched_get_stats(s)["rejected"] == 1
        fs.fs_sched_run(s)
        st = fs.fs_sched_get_stats(s)
        assert st["jobs_done"] == 2 and st["active"] == 0 and st["queued"] == 0
        with pytest.raises(fs.FsError):
            fs.fs_sched_take(s, 99)
    finally:
        fs.fs_sched_destroy(s)


def test_failed_lane_reset_takes_no_kv_reservation():
    """Host-side fault injection: a lane reset that fails during fill leaves
    the job pending and the KV reservation untaken; once resets succeed the
    job runs and every reservation is released at the end."""
    s = fs.fs_sched_create_model_free(2, 50, 1, kv_budget_tokens=40)
    try:
        fs.fs_sched_submit(s, [1, 2, 3], 5)       # needs 8 tokens of KV
        fs.fs_sched_model_free_fail_resets(s, 1)
        with pytest.raises(fs.FsError) as e:
            fs.fs_sched_step(s)
        assert e.value.name == "FS_ERR_CUDA"
        st = fs.fs_sched_get_stats(s)
        assert st["kv_reserved_tokens"] == 0
        assert st["queued"] == 1 and st["active"] == 0
        fs.fs_sched_run(s)
        st = fs.fs_sched_get_stats(s)
        assert st["jobs_done"] == 1 and st["kv_reserved_tokens"] == 0
        assert st["kv_reserved_max"] == 8
        with pytest.raises(fs.FsError):
            fs.fs_sched_model_free_fail_resets(s, -1)
    finally:
        fs.fs_sched_destroy(s)


def test_dgr_sweep_shape_with_the_product_scheduler():
    """DGR-012 sweep workload (8 sessions, prompt 4, 8 new tokens) through the
    product scheduler with one prompt token per step: per-session tokens are
    identical at every concurrency level and occupancy rises with it."""
    outs, occ = [], []
    for c in (1, 2, 4, 8):
        s = fs.fs_sched_create_model_free(c, 1000, max_prefill_tokens_per_tick=1)
        try:
            ids = [fs.fs_sched_submit(s, [10 + k, 20, 30, 40], 8) for k in range(8)]
            fs.fs_sched_run(s)
            outs.append([fs.fs_sched_take(s, i) for i in ids])
            occ.append(fs.fs_sched_get_stats(s)["occupancy_avg"])
        finally:
            fs.fs_sched_destroy(s)
    assert all(o == outs[0] for o in outs)
    assert occ == sorted(occ) and occ[0] == 1.0


_STATE = {fs.JOB_UNKNOWN: "unknown", fs.JOB_QUEUED: "queued", fs.JOB_RUNNING: "running",
          fs.JOB_DONE_LENGTH: "done_length", fs.JOB_DONE_STOP: "done_stop",
          fs.JOB_CANCELLED: "cancelled"}


@pytest.mark.parametrize("lanes,budget,chunk,kv,seed", [
    (3, 2, 1, 0, 20), (5, 6, 3, 0, 21), (4, 3, 2, 40, 22)])
def test_cancellation_matches_reference(lanes, budget, chunk, kv, seed):
    """Cancellations between steps (queued and running jobs, and refused ones
    for finished jobs): the same batches, tokens, states and counters as the
    reference; a cancelled running job's lane and KV reservation are freed."""
    vocab = 97
    jobs = _jobs(20, vocab, seed, max_prompt=12, max_new=14)
    g = np.random.default_rng(seed + 100)
    model = HashModel(lanes, vocab)
    ref = S.Reference(lanes, budget, model.step, model.sample, model.reset,
                      prefill_chunk=chunk, kv_budget_tokens=kv)
    s = fs.fs_sched_create_model_free(lanes, vocab, budget, prefill_chunk=chunk,
                                      kv_budget_tokens=kv)
    try:
        order = sorted(jobs, key=lambda j: (j["arrive"], j["id"]))
        ids, i, tick, batches, n_refused = {}, 0, 0, [], 0
        while i < len(order) or not ref.idle():
            while i < len(order) and order[i]["arrive"] <= tick:
                j = order[i]
                assert ref.submit(j)
                ids[j["id"]] = fs.fs_sched_submit(
                    s, j["prompt"], j["max_new"], j["temperature"], j["seed"],
                    -1 if j["stop"] is None else j["stop"])
                i += 1
            if ids and g.uniform() < 0.25:  # cancel a submitted job, maybe finished
                jid = int(g.choice(sorted(ids)))
                assert _STATE[fs.fs_sched_status(s, ids[jid])] == ref.status(jid)
                ok = ref.cancel(jid)
                if ok:
                    fs.fs_sched_cancel(s, ids[jid])
                else:
                    n_refused += 1
                    with pytest.raises(fs.FsError) as e:
                        fs.fs_sched_cancel(s, ids[jid])
                    assert e.value.name == "FS_ERR_STATE"
            before = len(model.batches)
            ref.step()
            fs.fs_sched_step(s)
            if len(model.batches) > before:
                batches.append(fs.fs_sched_last_batch(s))
            tick += 1
        assert batches == model.batches
        st = fs.fs_sched_get_stats(s)
        assert st["jobs_cancelled"] == ref.cancelled > 0
        assert st["jobs_done"] == len(jobs) - ref.cancelled
        assert st["kv_reserved_tokens"] == 0 and ref.reserved == 0
        for j in jobs:
            assert _STATE[fs.fs_sched_status(s, ids[j["id"]])] == ref.status(j["id"])
            assert fs.fs_sched_take(s, ids[j["id"]]) == ref.done[j["id"]]
            assert fs.fs_sched_status(s, ids[j["id"]]) == fs.JOB_UNKNOWN
        assert st["steps"] == ref.steps
    finally:
        fs.fs_sched_destroy(s)
