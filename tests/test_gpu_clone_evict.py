"""GPU: Clone and Evict of a lane's KV through the C ABI ("MODEL-BATCHING-
RESULTS", "Why in-kernel batching, not vLLM": per-user prefix reuse and
quarantine of a span, kept under batching).

Bit-exact: a clone continues exactly like its source and like a lane fed
the same tokens; a suffix evict leaves exactly the lane fed the prefix;
moved V rows; page tables (against the oracle's page model); a clone's
history when another lane holding its pages evicts (copy on write).
Within tolerance: a middle-span evict against the oracle (f32 path: K/V
max-abs 1e-4 and logits 2e-3, the f32 parity bounds; bf16: logits max-abs
5e-2 and cosine >= 0.9995), and re-rotated keys against the rotation by
-delta positions computed here in f64 (bf16 storage: one bf16 unit in the
last place).
"""
import numpy as np
import pytest

import oracle.core as O
from oracle import pages as P
from continuous_transformer_decode_gb300 import fs, synth
from tests import _gpu_util as U

pytestmark = pytest.mark.gpu

T = synth.MODEL_T
BF16_MAX_ABS, BF16_MIN_COS = 5e-2, 0.9995


@pytest.fixture(scope="module", autouse=True)
def _built():
    from continuous_transformer_decode_gb300 import build
    build.build()
    O.set_threads(8)


@pytest.fixture(scope="module")
def tiny():
    W = synth.make_weights(T, seed=1, fmt="f32")
    return W, O.Model(T, W, O.F32)


@pytest.fixture(scope="module")
def smol_l2():
    cfg = synth.with_layers(synth.MODEL_S, 2)
    Wb = synth.make_weights(cfg, seed=1, fmt="bf16")
    return cfg, Wb, O.Model(cfg, Wb, O.BF16)


def _bits(a):
    return np.ascontiguousarray(a).view(np.uint32)


def _feed(h, lane, toks, V):
    """Feeds a lane its tokens one step at a time."""
    import torch
    buf = torch.empty((1, V), dtype=torch.float32, device="cuda")
    for t in toks:
        pos = np.array([fs.fs_lane_length(h, lane)], np.int32)
        fs.fs_decode_step_batch(h, [lane], pos, [int(t)], logits_out=buf)
    torch.cuda.synchronize()


def _step(h, lanes, toks, V):
    """One step of several lanes; returns their logits rows."""
    import torch
    pos = np.array([fs.fs_lane_length(h, k) for k in lanes], np.int32)
    buf = torch.empty((len(lanes), V), dtype=torch.float32, device="cuda")
    fs.fs_decode_step_batch(h, list(lanes), pos, [int(t) for t in toks], logits_out=buf)
    torch.cuda.synchronize()
    return buf.cpu().numpy()


def _kv(h, cfg, lane):
    return [fs.fs_lane_export_kv(h, lane, l, cfg["Hkv"], cfg["hd"]) for l in range(cfg["L"])]


def _model(max_lanes, max_pos, page_size, n_pages):
    return P.PageModel(n_pages, page_size, max_lanes, -(-max_pos // page_size))


def _pm_feed(pm, lane, n):
    for _ in range(n):
        assert pm.step([lane], [pm.length[lane]], [0], 1 << 30) == P.OK


@pytest.mark.parametrize("kvdtype", [fs.FS_DTYPE_F32, fs.FS_DTYPE_BF16])
def test_clone_continues_bitwise_like_source_and_like_a_fed_lane(tiny, kvdtype):
    W, m = tiny
    ps, max_pos, lanes, n_pages = 16, 64, 6, 24
    h = U.make_gpu(T, W, fs.FS_DTYPE_F32, kvdtype, max_lanes=lanes, max_pos=max_pos,
                   n_pages=n_pages, page_size=ps)
    pm = _model(lanes, max_pos, ps, n_pages)
    try:
        toks = [int(t) for t in synth.make_prompts(1, 21, T["V"], seed=11)[0]]
        _feed(h, 0, toks, T["V"])
        _pm_feed(pm, 0, 21)
        fs.fs_lane_clone(h, 0, 2)
        assert pm.clone(0, 2) == P.OK
        for k in range(lanes):
            assert fs.fs_lane_pages(h, k) == pm.table(k), k
        assert fs.fs_lane_length(h, 2) == 21
        for a, b in zip(_kv(h, T, 0), _kv(h, T, 2)):
            assert np.array_equal(_bits(a[0]), _bits(b[0]))
            assert np.array_equal(_bits(a[1]), _bits(b[1]))
        # same tokens: the same rows, bit for bit; past the page boundary too
        nxt = [int(t) for t in synth.make_prompts(1, 14, T["V"], seed=12)[0]]
        for t in nxt[:6]:
            r = _step(h, [0, 2], [t, t], T["V"])
            assert np.array_equal(_bits(r[0]), _bits(r[1]))
            _pm_feed(pm, 0, 1)
            _pm_feed(pm, 2, 1)
        # different tokens: each lane is the lane fed its sequence from scratch
        _feed(h, 3, toks + nxt[:6] + nxt[6:10], T["V"])
        _feed(h, 4, toks + nxt[:6] + nxt[10:14], T["V"])
        for i in range(4):
            r = _step(h, [0, 2], [nxt[6 + i], nxt[10 + i]], T["V"])
            _pm_feed(pm, 0, 1)
            _pm_feed(pm, 2, 1)
        r3 = _step(h, [3, 4, 0, 2], [7, 7, 7, 7], T["V"])
        assert np.array_equal(_bits(r3[2]), _bits(r3[0]))
        assert np.array_equal(_bits(r3[3]), _bits(r3[1]))
        # against the oracle: a cloned oracle lane
        src = m.lane(max_pos)
        for t in toks:
            m.step(src, t)
        cl = m.lane(max_pos)
        cl.clone_from(src)
        for t in nxt[:6] + nxt[10:14]:
            m.step(cl, t)
        ref = m.step(cl, 7)
        tol = 2e-3 if kvdtype == fs.FS_DTYPE_F32 else BF16_MAX_ABS
        assert np.abs(r3[3] - ref).max() <= tol
    finally:
        fs.fs_destroy(h)


def test_evict_suffix_is_the_prefix_lane_bitwise(smol_l2):
    cfg, Wb, m = smol_l2
    h = U.make_gpu(cfg, Wb, fs.FS_DTYPE_BF16, max_lanes=4, max_pos=64)
    try:
        toks = [int(t) for t in synth.make_prompts(1, 37, cfg["V"], seed=13)[0]]
        _feed(h, 0, toks, cfg["V"])
        _feed(h, 1, toks[:19], cfg["V"])
        pages_before = fs.fs_lane_pages(h, 0)
        fs.fs_lane_evict(h, 0, 19, 37)
        assert fs.fs_lane_length(h, 0) == 19
        assert fs.fs_lane_pages(h, 0) == pages_before[:2]
        for a, b in zip(_kv(h, cfg, 0), _kv(h, cfg, 1)):
            assert np.array_equal(_bits(a[0]), _bits(b[0]))
            assert np.array_equal(_bits(a[1]), _bits(b[1]))
        for t in (5, 99, 1234):
            r = _step(h, [0, 1], [t, t], cfg["V"])
            assert np.array_equal(_bits(r[0]), _bits(r[1]))
    finally:
        fs.fs_destroy(h)


@pytest.mark.parametrize("span", [(3, 9), (0, 17), (20, 21), (5, 33)])
def test_evict_middle_span_f32_against_oracle(tiny, span):
    W, m = tiny
    a, b = span
    h = U.make_gpu(T, W, fs.FS_DTYPE_F32, fs.FS_DTYPE_F32, max_lanes=3, max_pos=64,
                   page_size=16)
    try:
        toks = [int(t) for t in synth.make_prompts(1, 40, T["V"], seed=14)[0]]
        _feed(h, 0, toks, T["V"])
        fs.fs_lane_evict(h, 0, a, b)
        ln = m.lane(64)
        for t in toks:
            m.step(ln, t)
        ln.evict(a, b)
        assert fs.fs_lane_length(h, 0) == ln.pos == 40 - (b - a)
        for l, (k, v) in enumerate(_kv(h, T, 0)):
            assert np.abs(k - ln.export(l, "K")).max() < 1e-4
            assert np.abs(v - ln.export(l, "V")).max() < 1e-4
        nxt = [int(t) for t in synth.make_prompts(1, 5, T["V"], seed=15)[0]]
        for t in nxt:
            got = _step(h, [0], [t], T["V"])[0]
            ref = m.step(ln, t)
            assert np.abs(got - ref).max() <= 2e-3
        # layer 0 is the lane fed the sequence without the span: V bit for
        # bit (it depends on the token alone), K up to the rotation's rounding
        kept = toks[:a] + toks[b:]
        _feed(h, 1, kept + nxt, T["V"])
        k0, v0 = fs.fs_lane_export_kv(h, 0, 0, T["Hkv"], T["hd"])
        k1, v1 = fs.fs_lane_export_kv(h, 1, 0, T["Hkv"], T["hd"])
        assert np.array_equal(_bits(v0), _bits(v1))
        assert np.abs(k0 - k1).max() <= 1e-5 * max(1.0, np.abs(k1).max())
    finally:
        fs.fs_destroy(h)


def test_evict_middle_span_bf16_logits_against_oracle(smol_l2):
    cfg, Wb, m = smol_l2
    h = U.make_gpu(cfg, Wb, fs.FS_DTYPE_BF16, max_lanes=4, max_pos=64)
    try:
        toks = [int(t) for t in synth.make_prompts(1, 45, cfg["V"], seed=16)[0]]
        _feed(h, 0, toks, cfg["V"])
        fs.fs_lane_evict(h, 0, 7, 26)
        ln = m.lane(64)
        for t in toks:
            m.step(ln, t)
        ln.evict(7, 26)
        nxt = [int(t) for t in synth.make_prompts(1, 6, cfg["V"], seed=17)[0]]
        got = np.stack([_step(h, [0], [t], cfg["V"])[0] for t in nxt])
        ref = np.stack([m.step(ln, t) for t in nxt])
        U.compare_logits(got, ref, BF16_MAX_ABS, BF16_MIN_COS)
    finally:
        fs.fs_destroy(h)


def _rotate_back(k, delta, hd, theta):
    """Rotate-half RoPE pairs of k [n, Hkv, hd] turned back by delta
    positions, in f64."""
    half = hd // 2
    inv = theta ** (-2.0 * np.arange(half) / hd)
    c, s = np.cos(delta * inv), np.sin(delta * inv)
    x0, x1 = k[..., :half].astype(np.float64), k[..., half:].astype(np.float64)
    return np.concatenate([x0 * c + x1 * s, x1 * c - x0 * s], axis=-1)


@pytest.mark.parametrize("span", [(100, 103), (0, 1), (16, 500), (250, 333)])
def test_evict_long_random_context_rows_moved_and_rotated(smol_l2, span):
    """600 seeded random rows (several relocation batches, spans that
    overlap their destinations) on the long-context attention path."""
    cfg, Wb, m = smol_l2
    a, b = span
    n, d = 600, b - a
    h = U.make_gpu(cfg, Wb, fs.FS_DTYPE_BF16, max_lanes=4, max_pos=1024)
    try:
        fs.fs_lane_fill_random_kv(h, 0, n, 77)
        fs.fs_lane_clone(h, 0, 1)  # lane 1 keeps the original history
        before = _kv(h, cfg, 1)
        fs.fs_lane_evict(h, 0, a, b)
        assert fs.fs_lane_length(h, 0) == n - d
        after = _kv(h, cfg, 0)
        for l in range(cfg["L"]):
            k_old, v_old = before[l]
            k_new, v_new = after[l]
            assert np.array_equal(_bits(k_new[:a]), _bits(k_old[:a]))
            assert np.array_equal(_bits(v_new[:a]), _bits(v_old[:a]))
            assert np.array_equal(_bits(v_new[a:]), _bits(v_old[b:]))
            exp = _rotate_back(k_old[b:], d, cfg["hd"], cfg["rope_theta"])
            bound = 2.0 ** -7 * np.abs(exp) + 1e-5 * np.abs(k_old).max()
            assert np.all(np.abs(k_new[a:] - exp) <= bound), l
        # the clone's history is untouched (its shared pages were copied
        # before lane 0 wrote them)
        for l, (k, v) in enumerate(_kv(h, cfg, 1)):
            assert np.array_equal(_bits(k), _bits(before[l][0]))
            assert np.array_equal(_bits(v), _bits(before[l][1]))
        # lane 1 now holds its pages from a // page_size on alone, so the same
        # evict compacts them in place: bit for bit lane 0's result
        fs.fs_lane_evict(h, 1, a, b)
        for l, (k, v) in enumerate(_kv(h, cfg, 1)):
            assert np.array_equal(_bits(k), _bits(after[l][0]))
            assert np.array_equal(_bits(v), _bits(after[l][1]))
        r = _step(h, [0, 1], [3, 3], cfg["V"])
        assert np.all(np.isfinite(r)) and np.array_equal(_bits(r[0]), _bits(r[1]))
    finally:
        fs.fs_destroy(h)


def test_copy_on_write_keeps_the_other_holder_and_pages_match_model(tiny):
    W, m = tiny
    ps, max_pos, lanes, n_pages = 16, 64, 4, 14
    h = U.make_gpu(T, W, fs.FS_DTYPE_F32, fs.FS_DTYPE_F32, max_lanes=lanes,
                   max_pos=max_pos, n_pages=n_pages, page_size=ps)
    pm = _model(lanes, max_pos, ps, n_pages)
    try:
        toks = [int(t) for t in synth.make_prompts(1, 37, T["V"], seed=18)[0]]
        _feed(h, 0, toks, T["V"])
        _pm_feed(pm, 0, 37)
        fs.fs_lane_clone(h, 0, 1)
        assert pm.clone(0, 1) == P.OK
        snap = _kv(h, T, 1)
        fs.fs_lane_evict(h, 0, 5, 9)  # writes pages 0.. of lane 0, shared with lane 1
        assert pm.evict(0, 5, 9) == P.OK
        for k in range(lanes):
            assert fs.fs_lane_pages(h, k) == pm.table(k), k
        for l, (k, v) in enumerate(_kv(h, T, 1)):
            assert np.array_equal(_bits(k), _bits(snap[l][0]))
            assert np.array_equal(_bits(v), _bits(snap[l][1]))
        # lane 1 still decodes as the lane fed the whole sequence
        _feed(h, 2, toks, T["V"])
        r = _step(h, [1, 2], [11, 11], T["V"])
        assert np.array_equal(_bits(r[0]), _bits(r[1]))
        _pm_feed(pm, 1, 1)
        _pm_feed(pm, 2, 38)
        # errors change nothing
        snap_t = [fs.fs_lane_pages(h, k) for k in range(lanes)]
        snap_n = [fs.fs_lane_length(h, k) for k in range(lanes)]
        cases = [(lambda: fs.fs_lane_clone(h, 0, 1), "FS_ERR_STATE"),
                 (lambda: fs.fs_lane_clone(h, 0, 0), "FS_ERR_ARG"),
                 (lambda: fs.fs_lane_clone(h, 0, 4), "FS_ERR_LANE"),
                 (lambda: fs.fs_lane_evict(h, 0, 4, 2), "FS_ERR_ARG"),
                 (lambda: fs.fs_lane_evict(h, 0, 0, 34), "FS_ERR_ARG")]
        for f, name in cases:
            with pytest.raises(fs.FsError) as e:
                f()
            assert e.value.name == name
        assert [fs.fs_lane_pages(h, k) for k in range(lanes)] == snap_t
        assert [fs.fs_lane_length(h, k) for k in range(lanes)] == snap_n
        # resets return every page once no lane holds it
        for k in range(lanes):
            fs.fs_lane_reset(h, k)
            assert pm.reset(k) == P.OK
        _feed(h, 3, list(range(n_pages * ps // 4)), T["V"])  # one lane can again take pages
        _pm_feed(pm, 3, n_pages * ps // 4)
        assert fs.fs_lane_pages(h, 3) == pm.table(3)
    finally:
        fs.fs_destroy(h)
