"""Pins of Clone and Evict ("MODEL-BATCHING-RESULTS", "Why in-kernel batching,
not vLLM": per-user prefix reuse and quarantine of a span, kept under
batching) in the oracle: the model's lane operations and the page model's
sharing.

What fixes them independently of the oracle's own code:
- a clone is the same history, so both lanes continue bit for bit alike;
- evicting a suffix leaves exactly the lane that was fed only the prefix;
- layer 0's K/V of a token depend only on the token and its position, so
  after a middle span is evicted, layer 0 equals that of a lane fed the
  sequence without the span (a wrong shift, a missing re-rope or a re-rope
  at the old position fails this);
- page counts: every page's holder count is the number of tables holding
  it, the free list is the pages held by none, a lane's partly filled last
  page is held by that lane alone; and small hand-worked tables.
"""
import random

import numpy as np
import pytest

import oracle.core as O
from oracle import pages as P
from continuous_transformer_decode_gb300 import synth

T = synth.MODEL_T


@pytest.fixture(scope="module")
def tiny():
    W = synth.make_weights(T, seed=1, fmt="f32")
    return O.Model(T, W, O.F32)


def _bits(a):
    return a.view(np.uint32)


def _fed(m, toks, max_pos=64):
    ln = m.lane(max_pos)
    for t in toks:
        m.step(ln, int(t))
    return ln


def test_clone_continues_bitwise_like_its_source(tiny):
    m = tiny
    toks = synth.make_prompts(1, 11, T["V"], seed=5)[0]
    a = _fed(m, toks)
    b = m.lane(64)
    b.clone_from(a)
    assert b.pos == a.pos == 11
    for l in range(T["L"]):
        for w in ("K", "Kraw", "V"):
            assert np.array_equal(_bits(a.export(l, w)), _bits(b.export(l, w)))
    nxt = synth.make_prompts(1, 4, T["V"], seed=6)[0]
    for t in nxt:
        la, lb = m.step(a, int(t)), m.step(b, int(t))
        assert np.array_equal(_bits(la), _bits(lb))
    # the two histories are independent afterwards
    m.step(a, 1)
    assert a.pos == b.pos + 1


def test_evict_suffix_is_the_prefix_lane(tiny):
    m = tiny
    toks = synth.make_prompts(1, 14, T["V"], seed=7)[0]
    full = _fed(m, toks)
    full.evict(9, 14)
    pre = _fed(m, toks[:9])
    assert full.pos == pre.pos == 9
    for l in range(T["L"]):
        for w in ("K", "Kraw", "V"):
            assert np.array_equal(_bits(full.export(l, w)), _bits(pre.export(l, w)))
    for t in (3, 17, 40):
        assert np.array_equal(_bits(m.step(full, t)), _bits(m.step(pre, t)))


@pytest.mark.parametrize("span", [(2, 5), (0, 3), (6, 7), (4, 12)])
def test_evict_middle_span_layer0_is_the_lane_without_the_span(tiny, span):
    m = tiny
    a, b = span
    toks = [int(t) for t in synth.make_prompts(1, 13, T["V"], seed=8)[0]]
    ln = _fed(m, toks)
    ln.evict(a, b)
    kept = toks[:a] + toks[b:]
    ref = _fed(m, kept)
    assert ln.pos == len(kept)
    for w in ("K", "Kraw", "V"):
        assert np.array_equal(_bits(ln.export(0, w)), _bits(ref.export(0, w))), w
    # deeper layers were computed with the span present: V and un-roped K
    # of the kept entries are the lane's own rows, moved
    whole = _fed(m, toks)
    for l in range(1, T["L"]):
        for w in ("Kraw", "V"):
            e, o = ln.export(l, w), whole.export(l, w)
            assert np.array_equal(_bits(e[:a]), _bits(o[:a]))
            assert np.array_equal(_bits(e[a:]), _bits(o[b:]))
    # and the lane goes on at its new length
    m.step(ln, 5)
    assert ln.pos == len(kept) + 1


def test_evict_edge_cases(tiny):
    m = tiny
    toks = synth.make_prompts(1, 6, T["V"], seed=9)[0]
    ln = _fed(m, toks)
    before = [ln.export(l, "K").copy() for l in range(T["L"])]
    ln.evict(3, 3)  # empty span: nothing changes
    assert ln.pos == 6
    for l in range(T["L"]):
        assert np.array_equal(_bits(ln.export(l, "K")), _bits(before[l]))
    for bad in ((-1, 2), (4, 3), (2, 7)):
        with pytest.raises(ValueError):
            ln.evict(*bad)
    assert ln.pos == 6
    ln.evict(0, 6)  # everything: an empty lane that starts again at 0
    assert ln.pos == 0
    fresh = m.lane(64)
    assert np.array_equal(_bits(m.step(ln, 7)), _bits(m.step(fresh, 7)))


# ---- page model

def _check_pages(pm: P.PageModel, n_pages: int):
    held = [0] * n_pages
    for k in range(pm.max_lanes):
        t = pm.table(k)
        assert len(t) == -(-pm.length[k] // pm.page_size)
        assert len(set(t)) == len(t)
        for p in t:
            held[p] += 1
        if pm.length[k] % pm.page_size:
            assert pm.ref[t[-1]] == 1  # the page the lane writes next is its own
    assert held == pm.ref
    assert sorted(pm.free) == [p for p in range(n_pages) if held[p] == 0]


def test_page_model_clone_and_evict_hand_worked():
    pm = P.PageModel(n_pages=8, page_size=4, max_lanes=3, max_pages_per_lane=4)
    for t in range(6):
        assert pm.step([0], [t], [1], 10) == P.OK
    assert pm.table(0) == [0, 1]
    # clone: full page 0 shared, partial page 1 copied into page 2
    assert pm.clone(0, 1) == P.OK
    assert pm.table(1) == [0, 2] and pm.length[1] == 6
    assert pm.ref[:3] == [2, 1, 1]
    # lane 1 evicts [1, 3): new length 4, one page kept, page 0 is written
    # and shared, so it is replaced by the lowest free page (3); page 2 goes
    assert pm.evict(1, 1, 3) == P.OK
    assert pm.table(1) == [3] and pm.length[1] == 4
    assert pm.ref[:4] == [1, 1, 0, 1]
    # a suffix evict inside the unshared last page moves nothing
    assert pm.evict(0, 5, 6) == P.OK
    assert pm.table(0) == [0, 1] and pm.length[0] == 5
    # clone at a page boundary shares everything and takes no page
    assert pm.evict(0, 4, 5) == P.OK
    assert pm.clone(0, 2) == P.OK
    assert pm.table(2) == [0] and pm.ref[0] == 2
    # resetting the source keeps the shared page held by the clone
    assert pm.reset(0) == P.OK
    assert pm.ref[0] == 1 and 0 not in pm.free
    _check_pages(pm, 8)


def test_page_model_errors_are_atomic():
    pm = P.PageModel(n_pages=3, page_size=4, max_lanes=3, max_pages_per_lane=3)
    for t in range(6):
        assert pm.step([0], [t], [1], 10) == P.OK
    assert pm.clone(0, 1) == P.OK  # takes the last free page
    snap = ([pm.table(k) for k in range(3)], list(pm.ref), sorted(pm.free))
    assert pm.clone(0, 2) == P.ERR_KV_FULL
    assert pm.clone(0, 0) == P.ERR_ARG
    assert pm.clone(0, 1) == P.ERR_STATE
    assert pm.clone(0, 3) == P.ERR_LANE
    assert pm.evict(1, 2, 1) == P.ERR_ARG
    assert pm.evict(1, 0, 7) == P.ERR_ARG
    # lane 1 writes its shared page 0 after this evict: no page to copy to
    assert pm.evict(1, 1, 2) == P.ERR_KV_FULL
    assert ([pm.table(k) for k in range(3)], list(pm.ref), sorted(pm.free)) == snap


def test_page_model_random_operations_keep_counts():
    rng = random.Random(3)
    n_pages, ps, lanes = 24, 4, 5
    pm = P.PageModel(n_pages, ps, lanes, 8)
    for _ in range(3000):
        op = rng.random()
        k = rng.randrange(lanes)
        if op < 0.55:
            pm.step([k], [pm.length[k]], [0], 10)
        elif op < 0.7:
            pm.clone(rng.randrange(lanes), k)
        elif op < 0.85:
            n = pm.length[k]
            a = rng.randint(0, n)
            pm.evict(k, a, rng.randint(a, n))
        elif op < 0.9:
            pm.reset(k)
        _check_pages(pm, n_pages)
