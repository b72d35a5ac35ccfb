"""Helpers for the GPU parity tests: drive the C ABI and the oracle on the same
seeded inputs and collect per-(lane, step) logits."""
from __future__ import annotations

import os

import numpy as np

import oracle.core as O
from continuous_transformer_decode_gb300 import fs, synth

ORACLE_DTYPE = {fs.FS_DTYPE_F32: O.F32, fs.FS_DTYPE_BF16: O.BF16,
                fs.FS_DTYPE_Q8_0: O.Q8_0}


def quantize_weights(W: dict) -> dict:
    """Q8_0 blocks of every matrix (the oracle's quantiser: input prep)."""
    q = lambda a: O.quantize_q8_0(synth.bf16_to_f32(a) if a.dtype == np.uint16 else a)
    return {"embed": q(W["embed"]),
            "lm_head": None if W["lm_head"] is None else q(W["lm_head"]),
            "final_norm": W["final_norm"],
            "layers": [{k: (v if k in ("attn_norm", "ffn_norm") else q(v))
                        for k, v in ly.items()} for ly in W["layers"]]}


def make_gpu(cfg, W, wdtype, kvdtype=fs.FS_DTYPE_BF16, max_lanes=8,
             max_pos=64, n_pages=None, page_size=16, act_split=0, env=None):
    """env: environment variables set while fs_create reads its knobs."""
    if n_pages is None:
        n_pages = max_lanes * (-(-max_pos // page_size))
    desc = fs.make_desc(cfg, wdtype, kvdtype, max_lanes, n_pages, max_pos,
                        page_size, act_split)
    old = {k: os.environ.get(k) for k in (env or {})}
    try:
        os.environ.update(env or {})
        return fs.fs_create(desc, W)
    finally:
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


def oracle_runs(model, prompts, n_steps, max_pos=64):
    """Serial oracle per lane: prompt then n_steps greedy tokens. Returns the
    fed token sequences and the logits after each fed token."""
    seqs, logits = [], []
    for p in prompts:
        ln = model.lane(max_pos)
        toks = [int(t) for t in p]
        rows = []
        i = 0
        while i < len(toks):
            lg = model.step(ln, toks[i])
            rows.append(lg)
            if i == len(toks) - 1 and len(toks) < len(p) + n_steps:
                toks.append(int(np.argmax(lg)))
            i += 1
        seqs.append(toks)
        logits.append(np.stack(rows))
    return seqs, logits


def gpu_teacher_forced(h, cfg, lanes, seqs, V):
    """Feeds each lane its token sequence in lockstep steps (ragged: a lane
    drops out when its sequence ends). Returns per-lane logits [T_b, V]."""
    import torch
    T = max(len(s) for s in seqs)
    out = [np.zeros((len(s), V), dtype=np.float32) for s in seqs]
    pos = {k: fs.fs_lane_length(h, k) for k in lanes}
    for t in range(T):
        idx = [i for i, s in enumerate(seqs) if t < len(s)]
        ls = [lanes[i] for i in idx]
        toks = [seqs[i][t] for i in idx]
        ps = np.array([pos[k] for k in ls], dtype=np.int32)
        buf = torch.empty((len(idx), V), dtype=torch.float32, device="cuda")
        fs.fs_decode_step_batch(h, ls, ps, toks, logits_out=buf)
        torch.cuda.synchronize()
        lg = buf.cpu().numpy()
        for j, i in enumerate(idx):
            out[i][t] = lg[j]
            pos[lanes[i]] += 1
    return out


def compare_logits(got, ref, max_abs, min_cos):
    """Per-row max-abs and cosine; returns (worst max-abs, mean cosine)."""
    err = np.abs(got - ref).max(axis=-1)
    cos = (got * ref).sum(-1) / (np.linalg.norm(got, axis=-1) *
                                 np.linalg.norm(ref, axis=-1))
    assert err.max() <= max_abs, f"max-abs {err.max()} > {max_abs}"
    assert cos.min() >= min_cos, f"cosine {cos.min()} < {min_cos}"
    return float(err.max()), float(cos.mean())


def decisive_token_agreement(got, ref, err_bound):
    """Greedy token equality wherever the oracle's top-1/top-2 margin exceeds
    2 x the measured logit error (elsewhere several tokens are correct)."""
    srt = np.sort(ref, axis=-1)
    margin = srt[..., -1] - srt[..., -2]
    decisive = margin > 2 * err_bound
    same = np.argmax(got, -1) == np.argmax(ref, -1)
    assert np.all(same[decisive]), np.nonzero(~same & decisive)
    return int(decisive.sum()), int(same.size)
