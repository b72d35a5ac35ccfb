"""Scheduler references — test infrastructure only.

1. ``Reference`` — the fill / gather / fold loop of "Fat-station continuous
   batching" ("Components", item 3) with the decode-first, bounded-prefill
   policy of "DGR-012 — Continuous batching and bounded admission"
   ("Summary": in-flight decodes run first, prefill per tick is capped but at
   least one). Readings (the pages leave them open):
     * fill: at the start of a step each free lane, in lane-index order, takes
       the next pending job (FIFO by arrival); a lane freed in step t is
       refilled at the start of step t+1;
     * gather: a prompt is fed one token per step through the batched step;
       every lane past its prompt is included; prompt-phase lanes are added
       oldest-admitted first until max_prefill_tokens_per_tick tokens
       (at least one);
     * fold: the step that consumes the last prompt token yields the first
       generated token; a job retires at max_new_tokens or on its stop id;
     * sampling of a job's t-th generated token uses (seed, counter = t),
       so a job's tokens do not depend on its lane, step or neighbours;
     * prefix reuse ("MODEL-BATCHING-RESULTS", "Why in-kernel batching,
       not vLLM": Clone for prefix reuse), when prefix_reuse_min > 0: a job
       admitted into lane k takes the history of the busy lane whose fed
       tokens (prompt, then generated tokens fed back) share the longest
       prefix with its prompt (ties: lowest lane), capped at its prompt
       length - 1, by a clone and an evict of the clone's suffix, if that
       prefix has at least prefix_reuse_min tokens; it then feeds only the
       rest of its prompt;
     * cancellation ("DGR-012", "Summary": KV released when a session ends),
       between steps: a queued job leaves the queue, a running job's lane is
       reset and freed with its KV reservation; the tokens generated so far
       are kept. States: queued, running, done by length, done by stop id,
       cancelled.
   ``step_fn(lanes, positions, tokens) -> logits[n, V]`` is the engine
   (the oracle model, or anything with the decode_step_batch contract);
   ``sample_fn(logits_row, temp, seed, counter) -> token``.

2. ``tick_sweep`` — the model-free tick model of the DGR-012 concurrency sweep
   ("Concurrency 1/2/4/8 sweep"): a whole-prompt prefill takes one tick and
   yields the first token, at most one prefill per tick, the active cap is
   the concurrency level, decode runs before prefill, and a slot retired in
   tick t is reusable in tick t+1.
"""
from __future__ import annotations

from collections import deque


class Reference:
    def __init__(self, n_lanes: int, max_prefill_tokens_per_tick: int,
                 step_fn, sample_fn, reset_fn=None, prefill_chunk: int = 1,
                 kv_budget_tokens: int = 0, lane_tokens: int = 0,
                 prefix_reuse_min: int = 0, clone_fn=None, evict_fn=None):
        self.n_lanes = n_lanes
        self.budget = max(1, int(max_prefill_tokens_per_tick))
        # prompt tokens one lane may consume in one step (chunked prefill,
        # "Fat-station continuous batching", "What /generate does today")
        self.chunk = max(1, int(prefill_chunk))
        # bounded admission ("DGR-012", "Summary"): a job reserves its whole
        # generation (prompt + new tokens) of KV; one that can never fit is
        # rejected at submit, one that fits waits until the reservations of
        # the running jobs leave room (oldest first)
        self.kv_budget = int(kv_budget_tokens)
        self.lane_tokens = int(lane_tokens)
        self.reserved = 0
        self.reserved_max = 0
        self.rejected = []
        self.kv_wait_steps = 0
        self.step_fn = step_fn
        self.sample_fn = sample_fn
        self.reset_fn = reset_fn
        self.prefix_min = int(prefix_reuse_min)
        self.clone_fn = clone_fn
        self.evict_fn = evict_fn
        self.prefix_hits = 0
        self.prefix_tokens = 0
        self.state = {}  # job id -> "done_length" | "done_stop" | "cancelled"
        self.cancelled = 0
        self.pending = deque()
        self.lanes = [None] * n_lanes
        self.positions = [0] * n_lanes
        self.done = {}
        self.admit_seq = 0
        self.steps = 0
        self.occupancy = []
        self.prefill_tokens = 0
        self.decode_tokens = 0
        self.prefill_per_step = []

    def submit(self, job: dict) -> bool:
        """job: id, prompt (len >= 1), max_new (>= 1), temperature, seed,
        optional stop. False: rejected (its prompt + new tokens exceed the
        KV budget or the tokens one lane holds)."""
        need = len(job["prompt"]) + job["max_new"]
        if (self.kv_budget and need > self.kv_budget) or \
                (self.lane_tokens and need > self.lane_tokens):
            self.rejected.append(job["id"])
            return False
        self.pending.append(job)
        return True

    def idle(self) -> bool:
        return not self.pending and all(l is None for l in self.lanes)

    def _fill(self) -> None:
        for k in range(self.n_lanes):
            if self.lanes[k] is None and self.pending:
                need = len(self.pending[0]["prompt"]) + self.pending[0]["max_new"]
                if self.kv_budget and self.reserved + need > self.kv_budget:
                    self.kv_wait_steps += 1
                    break
                self.reserved += need
                self.reserved_max = max(self.reserved_max, self.reserved)
                job = self.pending.popleft()
                if self.reset_fn:
                    self.reset_fn(k)
                self.positions[k] = 0
                self.lanes[k] = dict(job=job, feed=0, gen=[], last=None,
                                     seq=self.admit_seq)
                self.admit_seq += 1
                if self.prefix_min > 0:
                    self._reuse_prefix(k)

    def _fed(self, j: int) -> list:
        """Tokens lane j fed so far: its prompt, then its generated tokens."""
        ln = self.lanes[j]
        return (list(ln["job"]["prompt"]) + ln["gen"])[:self.positions[j]]

    def _reuse_prefix(self, k: int) -> None:
        prompt = [int(t) for t in self.lanes[k]["job"]["prompt"]]
        best, src = 0, None
        for j in range(self.n_lanes):
            if j == k or self.lanes[j] is None:
                continue
            fed = self._fed(j)
            c = 0
            while c < min(len(prompt) - 1, len(fed)) and int(fed[c]) == prompt[c]:
                c += 1
            if c > best:
                best, src = c, j
        if src is None or best < self.prefix_min:
            return
        self.clone_fn(src, k)
        self.evict_fn(k, best, self.positions[src])
        self.positions[k] = best
        self.lanes[k]["feed"] = best
        self.prefix_hits += 1
        self.prefix_tokens += best

    def step(self):
        """One scheduler step; returns the list of job ids retired."""
        self._fill()
        decode = [k for k in range(self.n_lanes) if self.lanes[k] is not None
                  and self.lanes[k]["feed"] >= len(self.lanes[k]["job"]["prompt"])]
        prompt = [k for k in range(self.n_lanes) if self.lanes[k] is not None
                  and self.lanes[k]["feed"] < len(self.lanes[k]["job"]["prompt"])]
        prompt.sort(key=lambda k: self.lanes[k]["seq"])
        # decode first; then prompt lanes oldest first, each up to `chunk`
        # tokens, within the step's prompt-token budget and within n_lanes
        # rows in all ("DGR-012", "Prefill does not starve decode")
        take = {k: 1 for k in decode}
        left, rows_left = self.budget, self.n_lanes - len(decode)
        for k in prompt:
            ln = self.lanes[k]
            t = min(len(ln["job"]["prompt"]) - ln["feed"], self.chunk, left, rows_left)
            if t <= 0:
                break
            take[k] = t
            left -= t
            rows_left -= t
        if not take:
            return []
        # rows: lanes ascending, a lane's positions ascending
        rows, toks, poss = [], [], []
        for k in sorted(take):
            ln = self.lanes[k]
            p = ln["job"]["prompt"]
            for r in range(take[k]):
                f = ln["feed"] + r
                rows.append(k)
                toks.append(int(p[f]) if f < len(p) else ln["last"])
                poss.append(self.positions[k] + r)
        logits = self.step_fn(rows, poss, toks)
        self.steps += 1
        self.occupancy.append(len(rows))
        retired = []
        self.prefill_per_step.append(
            sum(1 for k, f in zip(rows, poss)
                if f < len(self.lanes[k]["job"]["prompt"])))
        i = 0
        for k in sorted(take):
            ln = self.lanes[k]
            job = ln["job"]
            for r in range(take[k]):
                if ln["feed"] < len(job["prompt"]):
                    self.prefill_tokens += 1
                else:
                    self.decode_tokens += 1
                ln["feed"] += 1
                self.positions[k] += 1
            last = i + take[k] - 1  # the lane's last row of this step
            i += take[k]
            if ln["feed"] < len(job["prompt"]):
                continue
            t = self.sample_fn(logits[last], job["temperature"], job["seed"],
                               len(ln["gen"]))
            ln["gen"].append(int(t))
            ln["last"] = int(t)
            stop = job.get("stop")
            if len(ln["gen"]) >= job["max_new"] or (stop is not None
                                                    and t == stop):
                self.done[job["id"]] = list(ln["gen"])
                self.state[job["id"]] = ("done_stop" if stop is not None and t == stop
                                         else "done_length")
                self.reserved -= len(job["prompt"]) + job["max_new"]
                self.lanes[k] = None
                retired.append(job["id"])
        return retired

    def status(self, job_id) -> str:
        if any(j["id"] == job_id for j in self.pending):
            return "queued"
        if any(l is not None and l["job"]["id"] == job_id for l in self.lanes):
            return "running"
        return self.state.get(job_id, "unknown")

    def cancel(self, job_id) -> bool:
        """Between steps; False when the job is unknown or already finished."""
        for j in list(self.pending):
            if j["id"] == job_id:
                self.pending.remove(j)
                self.done[job_id] = []
                self.state[job_id] = "cancelled"
                self.cancelled += 1
                return True
        for k, ln in enumerate(self.lanes):
            if ln is not None and ln["job"]["id"] == job_id:
                if self.reset_fn:
                    self.reset_fn(k)
                self.positions[k] = 0
                self.done[job_id] = list(ln["gen"])
                self.state[job_id] = "cancelled"
                self.reserved -= len(ln["job"]["prompt"]) + ln["job"]["max_new"]
                self.lanes[k] = None
                self.cancelled += 1
                return True
        return False

    def run(self, jobs, max_steps: int = 10**7) -> dict:
        """Run jobs with ``arrive`` ticks (0 if absent) to completion."""
        order = sorted(jobs, key=lambda j: (j.get("arrive", 0), j["id"]))
        i = 0
        tick = 0
        while (i < len(order) or not self.idle()) and tick < max_steps:
            while i < len(order) and order[i].get("arrive", 0) <= tick:
                self.submit(order[i])
                i += 1
            self.step()
            tick += 1
        return self.done


def serial_job(job: dict, step_fn, sample_fn, reset_fn=None, lane: int = 0):
    """One job alone on one lane: the per-job reference of the parity gate."""
    if reset_fn:
        reset_fn(lane)
    pos = 0
    out = []
    logits = None
    for t in job["prompt"]:
        logits = step_fn([lane], [pos], [int(t)])
        pos += 1
    while True:
        tok = int(sample_fn(logits[0], job["temperature"], job["seed"],
                            len(out)))
        out.append(tok)
        stop = job.get("stop")
        if len(out) >= job["max_new"] or (stop is not None and tok == stop):
            return out
        logits = step_fn([lane], [pos], [tok])
        pos += 1


def tick_sweep(concurrency: int, n_sessions: int = 8, prompt_len: int = 4,
               new_tokens: int = 8, max_prefill_per_tick: int = 1) -> dict:
    """Model-free tick simulation of the DGR-012 sweep."""
    pending = deque(range(n_sessions))
    active = {}  # session -> generated tokens so far
    ticks = 0
    occ = []
    while pending or active:
        ticks += 1
        retired = []
        decoders = sorted(active)
        if decoders:
            occ.append(len(decoders))
        for s in decoders:
            active[s] += 1
            if active[s] >= new_tokens:
                retired.append(s)
        started = []
        n_pref = 0
        while (pending and len(active) + len(started) < concurrency
               and n_pref < max_prefill_per_tick):
            s = pending.popleft()
            started.append(s)
            n_pref += 1
        for s in retired:
            del active[s]  # slot reusable from the next tick on
        for s in started:
            active[s] = 1  # the prefill tick yields the first token
            if new_tokens <= 1:
                del active[s]
    total = n_sessions * prompt_len + n_sessions * (new_tokens - 1)
    return dict(ticks=ticks,
                avg_occupancy=(sum(occ) / len(occ)) if occ else 0.0,
                max_occupancy=max(occ) if occ else 0,
                tokens_per_tick=total / ticks)
