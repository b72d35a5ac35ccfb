"""The roofline arithmetic of bench.py (host logic, no GPU), pinned to
numbers from outside the code: the published parameter counts of the two
model shapes, the weight bytes per token that MODEL-BATCHING-RESULTS ("The
lever") gives for SmolLM2-135M at Q8_0, and sums written out by hand."""
import hashlib
import json

import pytest

import bench
from continuous_transformer_decode_gb300 import synth

PEAKS = dict(hbm=6689.1, bf16=1946.7, bf16_sus=1751.0, src="measured")


def _n_params(cfg):
    # step_roofline with 1 byte per weight, no lanes: the streamed parameters
    return bench.step_roofline(cfg, 1.0, 0, 0, PEAKS)["bytes_per_step"]


@pytest.mark.parametrize("cfg,published", [
    (synth.MODEL_S, 134_515_008),     # SmolLM2-135M (tied embeddings)
    (synth.MODEL_M, 7_241_732_096),   # Mistral-7B (separate LM head)
])
def test_streamed_parameters_plus_norm_gains_are_the_published_model_size(cfg, published):
    # every parameter but the 2L + 1 RMSNorm gain vectors is a streamed weight
    norms = (2 * cfg["L"] + 1) * cfg["d"]
    assert _n_params(cfg) + norms == published


def test_smollm2_q8_0_bytes_per_token_match_the_pages():
    # "~150 MB at Q8_0" per generated token, batch 1 (34 bytes per 32 weights)
    b = bench.step_roofline(synth.MODEL_S, 34 / 32, 1, 0, PEAKS)["bytes_per_step"]
    assert 140e6 < b < 150e6
    # the weights dominate: one lane's KV at position 0 is a few KB
    assert b - _n_params(synth.MODEL_S) * 34 / 32 == 2 * 30 * 3 * 64 * 2


def test_step_roofline_bounds_by_hand():
    cfg = synth.MODEL_S
    n = _n_params(cfg)
    kv_tok = 2 * 30 * 3 * 64 * 2                  # K and V, bf16, every layer
    r = bench.step_roofline(cfg, 2.0, 256, 17.0, PEAKS)
    assert r["bytes_per_step"] == 2 * n + 256 * 18 * kv_tok
    assert r["flops_per_token"] == 2 * n + 4 * 9 * 64 * 18 * 30
    hbm = 256 * 6689.1e9 / r["bytes_per_step"]
    tc = 1751.0e12 / r["flops_per_token"]
    assert r["bound"] == "hbm" and r["tok_s_ceiling"] == pytest.approx(min(hbm, tc))
    # 960 Q8_0 lanes: compute binds (the pages' large-B regime)
    assert bench.step_roofline(cfg, 34 / 32, 960, 20.0, PEAKS)["bound"] == "tensor"
    assert bench.step_roofline(cfg, 34 / 32, 1, 20.0, PEAKS)["bound"] == "hbm"


def test_gemm_bytes_per_step_by_hand():
    cfg = synth.MODEL_S
    d, F, V, B = 576, 1536, 49152, 4
    q, kv = 9 * 64, 3 * 64
    layer = (
        (q + 2 * kv) * d * 2 + B * d * 2 + B * (q + 2 * kv) * 4   # QKV: f32 rows out
        + d * q * 2 + B * q * 2 + B * d * 4                       # O
        + 2 * F * d * 2 + B * d * 2 + B * F * 2                   # gate/up: bf16 SwiGLU out
        + d * F * 2 + B * F * 2 + B * d * 4)                      # down
    head_greedy = V * d * 2 + B * d * 2 + B * (V // 128) * 8      # per-tile (max, index)
    head_logits = V * d * 2 + B * d * 2 + B * V * 4
    assert bench.gemm_bytes_per_step(cfg, 2.0, B, greedy=True) == (30 * layer + head_greedy, 121)
    assert bench.gemm_bytes_per_step(cfg, 2.0, B, greedy=False) == (30 * layer + head_logits, 121)


def test_traffic_record_follows_the_kernel_source(tmp_path, monkeypatch):
    csrc = tmp_path / "continuous_transformer_decode_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    src = csrc / "k.cu"
    src.write_bytes(b"kernel v1")
    rec = {"w@8": {"source_sha256": hashlib.sha256(b"kernel v1").hexdigest(),
                   "dram_bytes_per_launch": 1234}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_for("k.cu", "w", 8) == 1234
    assert bench.traffic_for("k.cu", "w", 16) is None        # no record for that size
    src.write_bytes(b"kernel v2")                            # counters now stale
    assert bench.traffic_for("k.cu", "w", 8) is None

