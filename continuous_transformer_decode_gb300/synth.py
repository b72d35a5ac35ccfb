"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This module holds no arithmetic of the decode method: it draws random weights,
prompts and context lengths with fixed seeds and encodes them in the storage
formats the library accepts (f32, or bf16 bits by round-to-nearest-even).

Shapes follow the workloads measured on the pages: a tiny dense Llama for
exact checks, a SmolLM2-135M-shaped model (MODEL-BATCHING-RESULTS, "Measured":
16-token prompts, 12 decode steps) and a Mistral-7B-shaped model (the
fat-station deployment of "Fat-station continuous batching", whose live model
is a Mistral). No real weights or datasets are used anywhere.
"""
from __future__ import annotations

import os

import numpy as np

# name: L layers, d width, H/Hkv heads, hd head dim, F ffn, V vocab
MODEL_T = dict(name="tiny-llama", L=2, d=64, H=4, Hkv=2, hd=16, F=172, V=256,
               rms_eps=1e-5, rope_theta=1e4, tied=False)
MODEL_S = dict(name="smollm2-135m", L=30, d=576, H=9, Hkv=3, hd=64, F=1536,
               V=49152, rms_eps=1e-5, rope_theta=1e4, tied=True)
MODEL_M = dict(name="mistral-7b", L=32, d=4096, H=32, Hkv=8, hd=128, F=14336,
               V=32000, rms_eps=1e-5, rope_theta=1e6, tied=False)

LAYER_KEYS = ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down",
              "attn_norm", "ffn_norm")

WEIGHT_STD = 0.02


def with_layers(cfg: dict, L: int) -> dict:
    """Same shape with fewer layers (the first L layers draw identical weights)."""
    c = dict(cfg)
    c["L"] = L
    return c


def _rng(seed: int, *path: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([seed, *path]))


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """f32 -> bf16 bit patterns (uint16), round to nearest even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32)
            << np.uint32(16)).view(np.float32)


def matrix_shapes(cfg: dict) -> dict:
    d, qd, kvd, F = cfg["d"], cfg["H"] * cfg["hd"], cfg["Hkv"] * cfg["hd"], cfg["F"]
    return {"wq": (qd, d), "wk": (kvd, d), "wv": (kvd, d), "wo": (d, qd),
            "w_gate": (F, d), "w_up": (F, d), "w_down": (d, F)}


def _normal(seed: int, path, shape) -> np.ndarray:
    g = _rng(seed, *path)
    return (g.standard_normal(size=shape, dtype=np.float32)
            * np.float32(WEIGHT_STD)).astype(np.float32)


def make_weights(cfg: dict, seed: int = 1, fmt: str = "bf16",
                 workers: int = 0) -> dict:
    """Random-init weights N(0, 0.02), norm gains 1.

    fmt "f32": float32 matrices; "bf16": uint16 bf16 bits of the same draws.
    Returns the dict layout of the library's and the oracle's weight inputs.
    Every matrix draws from its own seeded stream, so `workers` threads
    (0: one per core) give the same values as one.
    """
    assert fmt in ("f32", "bf16")
    enc = (lambda a: a) if fmt == "f32" else bf16_bits
    d, V = cfg["d"], cfg["V"]
    shapes = matrix_shapes(cfg)
    jobs = [("embed", (0, 0), (V, d))]
    if not cfg["tied"]:
        jobs.append(("lm_head", (0, 1), (V, d)))
    for l in range(cfg["L"]):
        for j, k in enumerate(LAYER_KEYS[:7]):
            jobs.append(((l, k), (1, l, j), shapes[k]))
    n_workers = workers or os.cpu_count() or 1
    draw = lambda job: enc(_normal(seed, job[1], job[2]))
    if n_workers > 1 and len(jobs) > 1:
        from concurrent.futures import ThreadPoolExecutor
        with ThreadPoolExecutor(min(n_workers, len(jobs))) as ex:
            mats = list(ex.map(draw, jobs))
    else:
        mats = [draw(j) for j in jobs]
    got = {job[0]: m for job, m in zip(jobs, mats)}
    w = {"embed": got["embed"], "lm_head": got.get("lm_head"),
         "final_norm": np.ones(d, dtype=np.float32), "layers": []}
    for l in range(cfg["L"]):
        ly = {k: got[(l, k)] for k in LAYER_KEYS[:7]}
        ly["attn_norm"] = np.ones(d, dtype=np.float32)
        ly["ffn_norm"] = np.ones(d, dtype=np.float32)
        w["layers"].append(ly)
    return w


def make_prompts(n_lanes: int, lengths, vocab: int, seed: int = 2):
    """Uniform-random token prompts; lane i draws from its own stream."""
    if np.isscalar(lengths):
        lengths = [int(lengths)] * n_lanes
    return [_rng(seed, i).integers(0, vocab, size=int(lengths[i]),
                                   dtype=np.int64).astype(np.int32)
            for i in range(n_lanes)]


def make_context_lengths(n_lanes: int, lo: int = 128, hi: int = 4096,
                         seed: int = 3) -> np.ndarray:
    """Per-lane context lengths drawn uniformly from [lo, hi]."""
    return _rng(seed).integers(lo, hi + 1, size=n_lanes).astype(np.int32)


def make_kv(n_tokens: int, Hkv: int, hd: int, seed: int, path=()) -> tuple:
    """Random N(0, 1) K and V for a synthetic long context, f32 [n, Hkv, hd]."""
    g = _rng(seed, 7, *path)
    K = g.standard_normal(size=(n_tokens, Hkv, hd), dtype=np.float32)
    V = g.standard_normal(size=(n_tokens, Hkv, hd), dtype=np.float32)
    return K, V


def make_trace(n_jobs: int, vocab: int, seed: int = 5, lanes: int = 8,
               prompt_lo: int = 8, prompt_hi: int = 2048, new_lo: int = 16,
               new_hi: int = 512, p_temp: float = 0.5, temp: float = 0.8):
    """Continuous-batching job trace: Poisson arrivals on a tick clock,
    log-uniform prompt lengths, uniform max_new_tokens, temperature 0 or
    `temp` with per-job seeds. Arrival rate = 1.5 * lanes / mean job ticks."""
    g = _rng(seed, 11)
    plen = np.floor(np.exp(g.uniform(np.log(prompt_lo), np.log(prompt_hi),
                                     size=n_jobs))).astype(np.int64)
    new = g.integers(new_lo, new_hi + 1, size=n_jobs)
    mean_ticks = float(np.mean(plen + new))
    rate = 1.5 * lanes / mean_ticks
    gaps = g.exponential(1.0 / rate, size=n_jobs)
    arrive = np.floor(np.cumsum(gaps)).astype(np.int64)
    temps = np.where(g.uniform(size=n_jobs) < p_temp, np.float32(temp),
                     np.float32(0.0)).astype(np.float32)
    seeds = g.integers(1, 2**63 - 1, size=n_jobs, dtype=np.int64)
    jobs = []
    for j in range(n_jobs):
        toks = _rng(seed, 12, j).integers(0, vocab, size=int(plen[j]))
        jobs.append(dict(id=j, arrive=int(arrive[j]),
                         prompt=toks.astype(np.int32),
                         max_new=int(new[j]), temperature=float(temps[j]),
                         seed=int(seeds[j])))
    return jobs
