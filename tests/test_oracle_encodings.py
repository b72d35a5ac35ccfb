"""Pins of the oracle's encodings against libraries and published vectors.

fp16 / bf16 conversions are checked against numpy's float16 and torch's
bfloat16 casts (both round to nearest even); Q8_0 against the properties its
definition fixes; Philox4x32-10 against the Random123 known-answer vectors.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle.core as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_f16_to_f32_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float32)
    got = np.array([O.f16_to_f32(int(b)) for b in bits], dtype=np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def _f32_samples(n=40000, seed=0):
    g = np.random.default_rng(seed)
    x = np.concatenate([
        g.standard_normal(n).astype(np.float32) * np.float32(0.02),
        g.standard_normal(n).astype(np.float32) * np.float32(1000.0),
        (g.uniform(-1, 1, n) * 2.0 ** g.integers(-30, 20, n)).astype(np.float32),
        np.array([0.0, -0.0, 65504.0, 65520.0, 65519.99, 1e9, -1e9, 2.0**-24,
                  2.0**-25, 2.0**-25 * 1.5, 2.0**-26, 6.1e-5, 5.96e-8,
                  np.inf, -np.inf], dtype=np.float32)])
    # values exactly halfway between fp16 neighbours (ties)
    h = g.integers(0, 0x7bff, 2000).astype(np.uint16)
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).view(np.float16).astype(np.float64)
    mid = ((lo + hi) / 2).astype(np.float32)
    return np.concatenate([x, mid])


def test_f32_to_f16_matches_numpy_rne():
    x = _f32_samples()
    with np.errstate(over="ignore"):  # the samples include values beyond fp16's range
        ref = x.astype(np.float16).view(np.uint16)
    got = np.array([O.f32_to_f16(float(v)) for v in x], dtype=np.uint16)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(x[i], hex(got[i]), hex(ref[i])) for i in bad[:5]]


def test_f32_to_bf16_matches_torch_rne():
    x = _f32_samples(seed=3)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy()
    ref = ref.view(np.uint16)
    got = np.array([O.f32_to_bf16(float(v)) for v in x], dtype=np.uint16)
    assert np.array_equal(got, ref)


def test_q8_0_block_properties():
    g = np.random.default_rng(5)
    x = (g.standard_normal(32 * 500) * 0.02).astype(np.float32)
    x[:32] = 0.0                       # all-zero block
    x[32:64] = np.linspace(-1, 1, 32)  # exact extremes
    blocks = O.quantize_q8_0(x)
    assert blocks.shape == (500, 34)
    d16 = blocks[:, 0].astype(np.uint16) | (blocks[:, 1].astype(np.uint16) << 8)
    d = d16.view(np.float16).astype(np.float32)
    q = blocks[:, 2:].view(np.int8).astype(np.int32)
    xb = x.reshape(-1, 32)
    amax = np.abs(xb).max(axis=1)
    # zero block: d = 0 and every code 0
    assert d[0] == 0.0 and np.all(q[0] == 0)
    # codes within [-127, 127]; the largest magnitude maps to +-127
    assert np.all(np.abs(q) <= 127)
    nz = amax > 0
    assert np.all(np.abs(q[nz]).max(axis=1) == 127)
    # d is the fp16 rounding of amax / 127 (relative error <= 2^-11)
    want = amax / np.float32(127.0)
    assert np.all(np.abs(d - want) <= want * 2.0**-11 + 1e-30)
    # round trip: |x - q*d| <= d_f32/2 (rounding) + 127*|d - d_f32| (scale)
    deq = O.dequantize_q8_0(blocks).reshape(-1, 32)
    assert np.array_equal(deq, q.astype(np.float32) * d[:, None])
    bound = want[:, None] / 2 + 127 * np.abs(d - want)[:, None] + 1e-12
    assert np.all(np.abs(xb - deq) <= bound * (1 + 1e-6))
    # sign symmetry: quantising -x negates every code
    qn = O.quantize_q8_0(-x)[:, 2:].view(np.int8).astype(np.int32)
    assert np.array_equal(qn, -q)


def test_philox_known_answer_vectors():
    rows = []
    with open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            v = [int(t, 16) for t in line.split()]
            rows.append(v)
    assert len(rows) == 3
    for v in rows:
        assert O.philox4x32_10(v[0:4], v[4:6]) == tuple(v[6:10])


def test_uniform_range_and_spread():
    u = np.array([O.uniform(1234, c) for c in range(20000)])
    assert np.all((u >= 0) & (u < 1))
    # mean and variance of U[0,1) within ~6 sigma
    assert abs(u.mean() - 0.5) < 6 * np.sqrt(1 / 12 / u.size)
    assert abs(u.var() - 1 / 12) < 0.01
    # distinct seeds give distinct streams
    assert O.uniform(1, 0) != O.uniform(2, 0)


def test_q8_gate_golden_is_the_pages_gate():
    g = json.load(open(os.path.join(GOLDEN, "q8_gate.json")))
    assert g["top1_min"] == 0.80 and g["mean_cos_min"] == 0.99
