"""Pins of the oracle model: the pages' batched == serial gates, an f64 brute
force of the whole tiny model, structural invariants (GQA grouping, tied head,
thread count) and the Q8_0 faithfulness gate."""
import json
import os

import numpy as np
import pytest

import oracle.core as O
from continuous_transformer_decode_gb300 import synth
from tests._f64_model import forward_logits

T = synth.MODEL_T
PROMPT_LENS = [3, 5, 7, 9]  # the tiny workload's ragged prompts


@pytest.fixture(scope="module")
def tiny():
    W = synth.make_weights(T, seed=1, fmt="f32")
    return W, O.Model(T, W, O.F32)


def test_f64_brute_force_whole_model(tiny):
    W, m = tiny
    toks = synth.make_prompts(1, 12, T["V"], seed=2)[0]
    ref = forward_logits(T, W, toks)
    ln = m.lane(64)
    for t, tok in enumerate(toks):
        lg = m.step(ln, tok)
        err = np.abs(lg - ref[t]).max()
        assert err < 2e-5 * max(1.0, np.abs(ref[t]).max()), (t, err)
    assert ln.pos == len(toks)


def test_f64_brute_force_with_bf16_kv_storage(tiny):
    """kv_bf16: keys and values enter the cache rounded to bf16. Pinned by
    the f64 brute force with the same storage rounding, which the f32-KV
    oracle misses by far more than the tolerance (so the rounding is really
    applied, to both keys and values); every stored value is bf16-exact."""
    W, m = tiny
    mb = O.Model(T, W, O.F32, kv_bf16=True)
    toks = synth.make_prompts(1, 12, T["V"], seed=2)[0]
    ref_b = forward_logits(T, W, toks, kv_bf16=True)
    ref_f = forward_logits(T, W, toks)
    lb, lf = mb.lane(64), m.lane(64)
    worst_f = 0.0
    for t, tok in enumerate(toks):
        gb, gf = mb.step(lb, tok), m.step(lf, tok)
        scale = max(1.0, np.abs(ref_b[t]).max())
        assert np.abs(gb - ref_b[t]).max() < 2e-5 * scale, t
        worst_f = max(worst_f, np.abs(gf - ref_b[t]).max() / scale)
    assert worst_f > 1e-4  # the f32-KV oracle is not the bf16-storage model
    for l in range(T["L"]):
        for which in ("K", "V"):
            a = lb.export(l, which)
            assert np.array_equal(synth.bf16_to_f32(synth.bf16_bits(a)), a)
    # batched == serial holds in this storage too
    prompts = synth.make_prompts(3, [4, 6, 5], T["V"], seed=8)
    ser = [mb.lane(64) for _ in range(3)]
    bat = [mb.lane(64) for _ in range(3)]
    for b in range(3):
        mb.prefill(ser[b], prompts[b])
        mb.prefill(bat[b], prompts[b])
    tk = [int(p[-1]) for p in prompts]
    for _ in range(4):
        out = mb.step_batch(bat, tk)
        for b in range(3):
            assert np.array_equal(mb.step(ser[b], tk[b]).view(np.uint32), out[b].view(np.uint32))
        tk = [int(np.argmax(r)) for r in out]


def test_batched_equals_serial_bitwise_logits_and_kv(tiny):
    """StepBatch == serial Step per lane: logits and the full K/Kraw/V/pos."""
    W, m = tiny
    prompts = synth.make_prompts(4, PROMPT_LENS, T["V"], seed=2)
    ser = [m.lane(64) for _ in range(4)]
    bat = [m.lane(64) for _ in range(4)]
    # ragged prefill, serial on both sides
    for b in range(4):
        m.prefill(ser[b], prompts[b])
        m.prefill(bat[b], prompts[b])
    toks = [int(p[-1]) for p in prompts]
    for step in range(8):
        lb = m.step_batch(bat, toks)
        for b in range(4):
            ls = m.step(ser[b], toks[b])
            assert np.array_equal(ls.view(np.uint32), lb[b].view(np.uint32))
        toks = [int(np.argmax(lb[b])) for b in range(4)]
    for b in range(4):
        assert ser[b].pos == bat[b].pos == PROMPT_LENS[b] + 8
        for l in range(T["L"]):
            for which in ("K", "Kraw", "V"):
                a, c = ser[b].export(l, which), bat[b].export(l, which)
                assert np.array_equal(a.view(np.uint32), c.view(np.uint32))


def test_lockstep_greedy_equals_serial_generate(tiny):
    W, m = tiny
    prompts = synth.make_prompts(4, PROMPT_LENS, T["V"], seed=2)
    lanes = [m.lane(64) for _ in range(4)]
    got = m.generate_batch(lanes, prompts, 8)
    for b in range(4):
        ref = m.generate(m.lane(64), prompts[b], 8)
        assert np.array_equal(got[b], ref)


def test_batch_composition_does_not_change_a_lane(tiny):
    W, m = tiny
    prompts = synth.make_prompts(6, 4, T["V"], seed=9)
    lanes = [m.lane(32) for _ in range(6)]
    for b in range(6):
        m.prefill(lanes[b], prompts[b])
    solo = m.lane(32)
    m.prefill(solo, prompts[2])
    a = m.step_batch([lanes[5], lanes[2], lanes[0]], [1, 2, 3])[1]
    b = m.step(solo, 2)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_thread_count_does_not_change_bits(tiny):
    W, m = tiny
    toks = synth.make_prompts(1, 6, T["V"], seed=4)[0]
    outs = []
    for nt in (1, 4):
        O.set_threads(nt)
        ln = m.lane(16)
        outs.append(m.prefill(ln, toks))
    O.set_threads(1)
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))


def test_gqa_equals_mha_with_repeated_kv_heads(tiny):
    """Head h reads KV head h // (H/Hkv): a GQA model equals the MHA model
    whose K/V projections repeat each KV head's rows for its query heads."""
    W, m = tiny
    hd, H, Hkv = T["hd"], T["H"], T["Hkv"]
    rep = H // Hkv
    mha_cfg = dict(T, Hkv=H)
    W2 = dict(W, layers=[])
    for ly in W["layers"]:
        l2 = dict(ly)
        for k in ("wk", "wv"):
            blocks = ly[k].reshape(Hkv, hd, -1)
            l2[k] = np.repeat(blocks, rep, axis=0).reshape(H * hd, -1).copy()
        W2["layers"].append(l2)
    m2 = O.Model(mha_cfg, W2, O.F32)
    toks = synth.make_prompts(1, 7, T["V"], seed=6)[0]
    a = m.prefill(m.lane(16), toks)
    b = m2.prefill(m2.lane(16), toks)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_tied_head_equals_untied_copy(tiny):
    W, m = tiny
    tied = O.Model(dict(T, tied=True), dict(W, lm_head=None), O.F32)
    untied = O.Model(T, dict(W, lm_head=W["embed"].copy()), O.F32)
    toks = [5, 9, 200]
    a = tied.prefill(tied.lane(8), toks)
    b = untied.prefill(untied.lane(8), toks)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_bf16_weights_equal_their_f32_upcast():
    Wb = synth.make_weights(T, seed=1, fmt="bf16")
    up = lambda a: synth.bf16_to_f32(a) if a is not None and a.dtype == np.uint16 else a
    Wf = {"embed": up(Wb["embed"]), "lm_head": up(Wb["lm_head"]),
          "final_norm": Wb["final_norm"],
          "layers": [{k: up(v) for k, v in ly.items()} for ly in Wb["layers"]]}
    a = O.Model(T, Wb, O.BF16)
    b = O.Model(T, Wf, O.F32)
    toks = [1, 2, 3, 4]
    x = a.prefill(a.lane(8), toks)
    y = b.prefill(b.lane(8), toks)
    assert np.array_equal(x.view(np.uint32), y.view(np.uint32))


def quantize_weights(W):
    q = lambda a: O.quantize_q8_0(synth.bf16_to_f32(a) if a.dtype == np.uint16 else a)
    return {"embed": q(W["embed"]),
            "lm_head": None if W["lm_head"] is None else q(W["lm_head"]),
            "final_norm": W["final_norm"],
            "layers": [{k: (q(v) if k not in ("attn_norm", "ffn_norm") else v)
                        for k, v in ly.items()} for ly in W["layers"]]}


def test_q8_gate_against_f32_on_reduced_smollm2():
    """Q8_0 oracle vs the f32 oracle on the unquantised bf16 weights: the
    pages' gate (decisive first-token argmax exact, teacher-forced top-1 at
    least 80%, mean cosine at least 0.99) on the SmolLM2 shape with 2 layers."""
    gate = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                       "q8_gate.json")))
    cfg = synth.with_layers(synth.MODEL_S, 2)
    Wb = synth.make_weights(cfg, seed=1, fmt="bf16")
    O.set_threads(os.cpu_count() or 1)
    try:
        f32 = O.Model(cfg, Wb, O.BF16)
        q8 = O.Model(cfg, quantize_weights(Wb), O.Q8_0)
        prompts = synth.make_prompts(3, 16, cfg["V"], seed=2)
        agree, cos, n = 0, [], 0
        for b in range(3):
            lf, lq = f32.lane(32), q8.lane(32)
            a = f32.prefill(lf, prompts[b])
            c = q8.prefill(lq, prompts[b])
            srt = np.sort(a)
            if srt[-1] - srt[-2] > 0.05:  # decisive first token
                assert np.argmax(a) == np.argmax(c)
            for t in range(12):  # teacher-forced on the f32 tokens
                agree += int(np.argmax(a) == np.argmax(c))
                cos.append(np.dot(a, c) / np.linalg.norm(a) / np.linalg.norm(c))
                n += 1
                tok = int(np.argmax(a))
                a = f32.step(lf, tok)
                c = q8.step(lq, tok)
        assert agree / n >= gate["top1_min"]
        assert np.mean(cos) >= gate["mean_cos_min"]
    finally:
        O.set_threads(1)
