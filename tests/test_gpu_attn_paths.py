"""GPU: the TMA-fed decode attention (k_attn_tma) against the cp.async one
(k_attn_mma) and against the oracle.

The two kernels do the same arithmetic in the same order, so their logits
must agree bit for bit; the oracle comparison uses the bf16 tolerances of
the parity tests (max-abs 5e-2, cosine >= 0.9995). Covered: page sizes 8 to
128 (one page per copy, or 64 rows of one page), head dims 64 / 128 / 256,
ragged contexts spanning several attention splits with a partial last page.
"""
import os

import numpy as np
import pytest

import oracle.core as O
from continuous_transformer_decode_gb300 import fs, synth
from tests import _gpu_util as U

pytestmark = pytest.mark.gpu

BF16_MAX_ABS, BF16_MIN_COS = 5e-2, 0.9995
HD256 = dict(name="hd256-llama", L=2, d=512, H=2, Hkv=1, hd=256, F=1024, V=512,
             rms_eps=1e-5, rope_theta=1e4, tied=True)


@pytest.fixture(scope="module", autouse=True)
def _built():
    from continuous_transformer_decode_gb300 import build
    build.build()
    O.set_threads(8)


def _handle(cfg, Wb, page_size, max_pos, force=None, max_lanes=4):
    old = os.environ.get("FS_ATTN")
    try:
        if force:
            os.environ["FS_ATTN"] = force
        else:
            os.environ.pop("FS_ATTN", None)
        return U.make_gpu(cfg, Wb, fs.FS_DTYPE_BF16, max_lanes=max_lanes, max_pos=max_pos,
                          page_size=page_size)
    finally:
        if old is None:
            os.environ.pop("FS_ATTN", None)
        else:
            os.environ["FS_ATTN"] = old


def _kv(cfg, ctx, seed):
    out = []
    for b, n in enumerate(ctx):
        Ks, Vs = [], []
        for l in range(cfg["L"]):
            K, V = synth.make_kv(n, cfg["Hkv"], cfg["hd"], seed=seed, path=(b, l))
            Ks.append(synth.bf16_to_f32(synth.bf16_bits(K)))
            Vs.append(synth.bf16_to_f32(synth.bf16_bits(V)))
        out.append((np.stack(Ks), np.stack(Vs)))
    return out


def _run_gpu(h, cfg, ctx, kv, toks):
    import torch
    for b, (K, V) in enumerate(kv):
        fs.fs_lane_import_kv(h, b, K, V)
    pos = np.array(ctx, np.int32)
    lanes = list(range(len(ctx)))
    out = []
    for t in toks:
        buf = torch.empty((len(ctx), cfg["V"]), dtype=torch.float32, device="cuda")
        fs.fs_decode_step_batch(h, lanes, pos, t, logits_out=buf)
        torch.cuda.synchronize()
        out.append(buf.cpu().numpy())
    return np.stack(out)


def _run_oracle(cfg, Wb, ctx, kv, toks, max_pos):
    m = O.Model(cfg, Wb, O.BF16)
    lanes = []
    for K, V in kv:
        ln = m.lane(max_pos)
        for l in range(cfg["L"]):
            ln.import_kv(l, K[l], V[l])
        lanes.append(ln)
    return np.stack([m.step_batch(lanes, t) for t in toks])


def _check(cfg, Wb, page_size, ctx, with_oracle, max_lanes=4, max_pos=None):
    max_pos = max_pos or max(ctx) + 8
    kv = _kv(cfg, ctx, seed=41)
    rng = np.random.default_rng(page_size)
    toks = [[int(x) for x in rng.integers(0, cfg["V"], len(ctx))] for _ in range(3)]
    h_t = _handle(cfg, Wb, page_size, max_pos, max_lanes=max_lanes)
    h_m = _handle(cfg, Wb, page_size, max_pos, force="mma", max_lanes=max_lanes)
    try:
        assert fs.fs_attention_path(h_t) == "tma-mma"
        assert fs.fs_attention_path(h_m) == "cp.async-mma"
        got_t = _run_gpu(h_t, cfg, ctx, kv, toks)
        got_m = _run_gpu(h_m, cfg, ctx, kv, toks)
    finally:
        fs.fs_destroy(h_t)
        fs.fs_destroy(h_m)
    assert np.array_equal(got_t.view(np.int32), got_m.view(np.int32))
    if with_oracle:
        ref = _run_oracle(cfg, Wb, ctx, kv, toks, max_pos)
        U.compare_logits(got_t.reshape(-1, cfg["V"]), ref.reshape(-1, cfg["V"]),
                         BF16_MAX_ABS, BF16_MIN_COS)


@pytest.fixture(scope="module")
def smol_l2():
    cfg = synth.with_layers(synth.MODEL_S, 2)
    return cfg, synth.make_weights(cfg, seed=1, fmt="bf16")


@pytest.mark.parametrize("page_size", [8, 16, 32, 64, 128])
def test_tma_attention_page_sizes_hd64(smol_l2, page_size):
    cfg, Wb = smol_l2
    _check(cfg, Wb, page_size, [37, 200, 650], with_oracle=page_size in (8, 128))


def test_tma_attention_hd128_mistral_shape():
    cfg = synth.with_layers(synth.MODEL_M, 2)
    Wb = synth.make_weights(cfg, seed=1, fmt="bf16")
    _check(cfg, Wb, 16, [300, 1100], with_oracle=True)


@pytest.mark.parametrize("page_size", [16, 64])
def test_tma_attention_hd256(page_size):
    Wb = synth.make_weights(HD256, seed=3, fmt="bf16")
    _check(HD256, Wb, page_size, [5, 130, 700], with_oracle=True)


def test_tma_attention_long_splits(smol_l2):
    """A handle large enough (128 lanes x 3 KV heads x 4 chunks of 1024) to
    take 1024-position attention splits: contexts of 300 / 1100 / 2100 tokens
    are 1, 2 and 3 splits."""
    cfg, Wb = smol_l2
    _check(cfg, Wb, 16, [300, 1100, 2100], with_oracle=True, max_lanes=128, max_pos=3100)


def _check_warp(cfg, Wb, page_size, ctx, max_pos=64):
    """The one-warp kernel (handles of at most 64 positions; FS_ATTN=warp
    takes it for calls of any size) against the cp.async kernel, bit for
    bit, and against the oracle."""
    kv = _kv(cfg, ctx, seed=43)
    rng = np.random.default_rng(7)
    steps = min(3, max_pos - max(ctx))
    toks = [[int(x) for x in rng.integers(0, cfg["V"], len(ctx))] for _ in range(steps)]
    h_w = _handle(cfg, Wb, page_size, max_pos, force="warp", max_lanes=8)
    h_m = _handle(cfg, Wb, page_size, max_pos, force="mma", max_lanes=8)
    try:
        assert fs.fs_attention_path(h_w) == "warp-mma"
        assert fs.fs_attention_path(h_m) == "cp.async-mma"
        got_w = _run_gpu(h_w, cfg, ctx, kv, toks)
        got_m = _run_gpu(h_m, cfg, ctx, kv, toks)
    finally:
        fs.fs_destroy(h_w)
        fs.fs_destroy(h_m)
    assert np.array_equal(got_w.view(np.int32), got_m.view(np.int32))
    ref = _run_oracle(cfg, Wb, ctx, kv, toks, max_pos)
    U.compare_logits(got_w.reshape(-1, cfg["V"]), ref.reshape(-1, cfg["V"]),
                     BF16_MAX_ABS, BF16_MIN_COS)


@pytest.mark.parametrize("page_size", [8, 16, 64])
def test_warp_attention_hd64(smol_l2, page_size):
    """Contexts of 0 to 60 tokens: empty and partial 16-position chunks, a
    lane whose position is the tile's last row."""
    cfg, Wb = smol_l2
    _check_warp(cfg, Wb, page_size, [0, 1, 15, 16, 37, 60])


def test_warp_attention_hd128_mistral_shape():
    cfg = synth.with_layers(synth.MODEL_M, 2)
    Wb = synth.make_weights(cfg, seed=1, fmt="bf16")
    _check_warp(cfg, Wb, 16, [3, 33, 61])


def test_warp_attention_chunked_prefill(smol_l2):
    """Chunked steps (every row's k, v appended before attention reads them)
    on the one-warp and the cp.async kernels give the same bits."""
    import torch
    cfg, Wb = smol_l2
    outs = []
    for force in ("warp", "mma"):
        h = _handle(cfg, Wb, 16, 64, force=force, max_lanes=8)
        try:
            pos = np.zeros(3, np.int32)
            rows, lg = [], []
            prompts = synth.make_prompts(3, [20, 9, 33], cfg["V"], seed=5)
            # lane 0 takes 4 rows a step, lane 1 one, lane 2 three
            p = np.zeros(3, np.int64)
            while any(p[k] < len(prompts[k]) for k in range(3)):
                lanes, poss, toks = [], [], []
                for k, take in enumerate((4, 1, 3)):
                    for _ in range(take):
                        if p[k] < len(prompts[k]):
                            lanes.append(k)
                            poss.append(int(p[k]))
                            toks.append(int(prompts[k][p[k]]))
                            p[k] += 1
                po = np.array([poss[i] for i in range(len(lanes))], np.int32)
                buf = torch.empty((len(lanes), cfg["V"]), dtype=torch.float32, device="cuda")
                fs.fs_step_batch_chunked(h, lanes, po, toks, logits_out=buf)
                torch.cuda.synchronize()
                lg.append(buf.cpu().numpy())
            outs.append(np.concatenate(lg))
        finally:
            fs.fs_destroy(h)
    assert np.array_equal(outs[0].view(np.int32), outs[1].view(np.int32))
