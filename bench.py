#!/usr/bin/env python
"""Benchmark of decode_step_batch: aggregate decode tokens/s and roofline.

One step = one fs_decode_step_batch over B lanes (embed, all layers, final
norm, LM head) plus the per-lane sampler. Default workload: the
SmolLM2-135M-shaped model with bf16 random weights N(0, 0.02), B = 256
lanes, 16-token uniform random prompts ingested before timing, then decode
steps (the workload of MODEL-BATCHING-RESULTS, "Measured": 16-token
prompts, 12 decode steps; the B sweep there tops out at 256 for this shape).

  value      device time (CUDA events on the handle's stream) of K steps,
             inputs resident on the device; tokens/s = B * K / time.
  e2e        the same K steps through the host API: host arrays in
             (fs_decode_step_batch), host tokens out (fs_sample), timed with
             the host clock including every copy.
  roofline   the weight-streaming GEMM (dominant kernel class): its
             algorithmic bytes per step / its time per step, where its time
             per step = the CUDA-event step time x the GEMM launches' share
             of a traced step (the library's per-block %globaltimer tracer
             over graph replays identical to the timed ones; a launch's share
             is its dependency gap plus its body, so the shares partition the
             step), against the measured HBM copy bandwidth.
  workloads  the other measured configurations, each on its own handle
             (SmolLM2-135M Q8_0 at 960 lanes, Mistral-7B bf16 at 1 and 128
             lanes with contexts U[128, 4096]): device ms per step, tokens/s,
             the step roofline fraction and the clocks of its timed region.
  cpu_baseline  the C++ f32 oracle (StepBatch) on this host's cores over a
             bounded sample of the same workload.

Multi-GPU (torchrun): replicas, one per GPU, no collective on the data path;
value = all ranks' tokens / max over ranks of the time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOADS = {
    "smollm2-135m-bf16": dict(model="S", wdtype="bf16", B=256, prompt=16),
    "smollm2-135m-q8_0": dict(model="S", wdtype="q8_0", B=960, prompt=16),
    # split activations: the configuration whose full-depth logits meet the
    # 5e-2 bound against the oracle (bf16 panels alone drift by ~0.15)
    "mistral-7b-bf16": dict(model="M", wdtype="bf16", B=128, ctx=(128, 4096), act_split=1),
    # continuous batching through the native scheduler (fill / gather / fold,
    # decode-first, bounded prefill) over a synthetic Poisson job trace
    "mistral-7b-trace": dict(model="M", wdtype="bf16", B=128, trace=True, act_split=1),
}
METRIC = "aggregate decode tokens/s"


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        j = json.load(open(p))
        return dict(hbm=j["hbm_gbs"], bf16=j["bf16_tflops"],
                    bf16_sus=j.get("bf16_tflops_sustained"), src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


class Clocks:
    """nvidia-smi sampling of SM clock and throttle reasons during timing."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.p = None
        self.out = os.path.join("/tmp", f"fs_clocks_{os.getpid()}.csv")
        try:
            self.p = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", gpu_id],
                stdout=open(self.out, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.p = None

    def stop(self):
        if self.p is None:
            return None
        time.sleep(0.25)
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except Exception:
            self.p.kill()
        rows = []
        for line in open(self.out):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append((float(f[1]), float(f[2]), f[5], f[6], f[7], f[8]))
            except ValueError:
                continue
        os.unlink(self.out)
        if not rows:
            return None
        sm = [r[0] for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if r[2 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(vals, world_size: int, device: str = "cpu"):
    """Element-wise max of per-rank timings over the process group (the
    slowest replica bounds the job); identity for a single process."""
    if world_size <= 1:
        return [float(v) for v in vals]
    import torch
    t = torch.tensor(vals, dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def aggregate_throughput(tokens_per_rank: int, ms_per_rank: float, world_size: int,
                         device: str = "cpu") -> float:
    """Whole-job tokens/s of replicas: all ranks' tokens over the slowest
    rank's time."""
    (ms,) = max_over_ranks([ms_per_rank], world_size, device)
    return tokens_per_rank * world_size / (ms / 1e3)


def model_cfg(name):
    from continuous_transformer_decode_gb300 import synth
    return {"S": synth.MODEL_S, "M": synth.MODEL_M, "T": synth.MODEL_T}[name]


def device_weights(cfg, seed=1):
    """Random-init bf16 weights N(0, 0.02) drawn on the device (seeded torch
    generator): for the 7B shape, where host draws would dominate the run.
    The timing does not depend on the values."""
    import torch
    from continuous_transformer_decode_gb300 import synth
    g = torch.Generator(device="cuda").manual_seed(seed)

    def mat(rows, cols):
        return (torch.randn(rows, cols, generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    d, V = cfg["d"], cfg["V"]
    shapes = synth.matrix_shapes(cfg)
    ones = torch.ones(d, dtype=torch.float32, device="cuda")
    W = {"embed": mat(V, d), "lm_head": None if cfg["tied"] else mat(V, d),
         "final_norm": ones, "layers": []}
    for _ in range(cfg["L"]):
        ly = {k: mat(*shapes[k]) for k in synth.LAYER_KEYS[:7]}
        ly["attn_norm"] = ones
        ly["ffn_norm"] = ones
        W["layers"].append(ly)
    return W


def gpu_weights(cfg, wdtype, seed=1):
    """Random-init weights. bf16: N(0, 0.02) drawn on the host (seeded), or
    on the device for the 7B shape; q8_0: the same bf16 values quantised on
    the device by the library."""
    import torch
    from continuous_transformer_decode_gb300 import fs, synth
    if cfg["d"] >= 4096 and wdtype == "bf16":
        return device_weights(cfg, seed), fs.FS_DTYPE_BF16
    W = synth.make_weights(cfg, seed=seed, fmt="bf16")
    if wdtype == "bf16":
        return W, fs.FS_DTYPE_BF16

    def q(a):
        x = torch.from_numpy(synth.bf16_to_f32(a).reshape(-1)).cuda()
        out = torch.empty((x.numel() // 32, 34), dtype=torch.uint8, device="cuda")
        fs.fs_quantize_q8_0(x, out)
        return out
    Q = {"embed": q(W["embed"]), "lm_head": None if W["lm_head"] is None else q(W["lm_head"]),
         "final_norm": W["final_norm"],
         "layers": [{k: (v if k in ("attn_norm", "ffn_norm") else q(v))
                     for k, v in ly.items()} for ly in W["layers"]]}
    return Q, fs.FS_DTYPE_Q8_0


def make_handle(cfg, wl, B, extra, W=None):
    """A handle for B lanes of workload `wl`, its lanes filled the way the
    pages' runs start: 16-token prompts ingested one token per lane per step,
    or (long contexts) per-lane random KV of U[lo, hi] tokens. Returns the
    handle and the step inputs (lanes, positions, next tokens, prompts,
    contexts, weight dtype)."""
    from continuous_transformer_decode_gb300 import fs, synth
    prompt = wl.get("prompt", 0)
    if "ctx" in wl:
        ctx = synth.make_context_lengths(B, *wl["ctx"], seed=3)
    else:
        ctx = np.full(B, prompt, dtype=np.int32)
    max_pos = int(ctx.max()) + extra
    ps = 16
    n_pages = int(sum(-(-(int(c) + extra) // ps) for c in ctx)) + B
    if W is None:
        W, wdt = gpu_weights(cfg, wl["wdtype"])
    else:
        W, wdt = W
    desc = fs.make_desc(cfg, wdt, fs.FS_DTYPE_BF16, B, n_pages, max_pos, ps,
                        wl.get("act_split", 0))
    h = fs.fs_create(desc, W)
    del W
    return h, ctx, wdt


def fill_lanes(h, cfg, wl, B, ctx):
    from continuous_transformer_decode_gb300 import fs, synth
    lanes = np.arange(B, dtype=np.int32)
    prompts = None
    if "ctx" in wl:  # long synthetic contexts: random KV (content irrelevant)
        for b in range(B):
            fs.fs_lane_fill_random_kv(h, b, int(ctx[b]), 1000 + b)
        pos = ctx.astype(np.int32).copy()
        toks = np.array([p[0] for p in synth.make_prompts(B, 1, cfg["V"], seed=2)], np.int32)
    else:  # prompt ingestion, one token per lane per step, outside timing
        prompts = np.stack(synth.make_prompts(B, wl["prompt"], cfg["V"], seed=2))
        pos = np.zeros(B, dtype=np.int32)
        for t in range(wl["prompt"]):
            fs.fs_decode_step_batch(h, lanes, pos, prompts[:, t])
        toks = prompts[:, -1].astype(np.int32).copy()
    return lanes, pos, toks, prompts


def gpu_id_of(local):
    import torch
    props = torch.cuda.get_device_properties(local)
    gpu_id = "GPU-" + str(props.uuid) if hasattr(props, "uuid") else str(local)
    return gpu_id[4:] if gpu_id.startswith("GPU-GPU-") else gpu_id


def run_ours(args, wl, ws, rank, local):
    import torch
    from continuous_transformer_decode_gb300 import build, fs, synth
    build.build()
    torch.cuda.set_device(local)
    cfg = model_cfg(wl["model"])
    if args.layers:
        cfg = synth.with_layers(cfg, args.layers)
    B = args.batch or wl["B"]
    K, Wm = args.steps, args.warmup
    extra = Wm + 2 * K + 8 + args.trace  # warm-up, timed, end-to-end, traced steps
    h, ctx, wdt = make_handle(cfg, wl, B, extra)
    gemm_path = fs.fs_gemm_path(h)
    stream = torch.cuda.Stream()
    torch.cuda.set_stream(stream)
    fs.fs_set_stream(h, stream)
    lanes, pos, toks, prompts = fill_lanes(h, cfg, wl, B, ctx)
    prompt = wl.get("prompt", 0)
    dtok = torch.empty(B, dtype=torch.int32, device="cuda")

    def device_step():  # greedy decode: tokens straight from the LM head's epilogue
        fs.fs_decode_step_greedy(h, lanes, pos, toks, dtok)

    for _ in range(Wm):
        device_step()
    torch.cuda.synchronize()
    clocks = Clocks(gpu_id_of(local))
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    l0 = fs.fs_kernel_launches(h)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(K):
        device_step()
    e1.record(stream)
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    ms = e0.elapsed_time(e1)
    launches = fs.fs_kernel_launches(h) - l0
    clk = clocks.stop()

    # end to end through the host API
    tk = torch.cuda.current_stream()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    htoks = toks.copy()
    for i in range(K):
        htoks = fs.fs_decode_step_greedy(h, lanes, pos, htoks)
    tk.synchronize()
    e2e_s = time.perf_counter() - t0

    # kernel timeline of a few more identical steps (outside every timed
    # region): per-launch gap + body, whose GEMM share times the timed step
    # gives the GEMMs' time per step
    timeline = None
    if args.trace:
        from continuous_transformer_decode_gb300 import trace as tr
        fs.fs_trace_enable(h, 400000 * args.trace)
        for _ in range(args.trace):
            device_step()
        recs, appended = fs.fs_trace_read(h)
        fs.fs_trace_enable(h, 0)
        timeline = tr.summarize(recs, args.trace)
        timeline["records"] = int(appended)
        print(tr.table(timeline), file=sys.stderr)

    fs.fs_destroy(h)

    # ---- B sweep, device-timed like `value`: each B on the workload's handle
    # (its lane capacity) and, below it, on a handle sized to B (the lane
    # capacity sets the GEMMs' K splits: a small handle splits short K)
    sweep = []
    if not args.no_sweep and "ctx" not in wl:
        Wsw = gpu_weights(cfg, wl["wdtype"])
        for Bs in [b for b in (1, 4, 16, 64, 256, 512, 960) if b <= B]:
            for cap in sorted({B, Bs}, reverse=True):
                hs, _, _ = make_handle(cfg, wl, cap, prompt + 12, W=Wsw)
                try:
                    fs.fs_set_stream(hs, stream)
                    ls = np.arange(Bs, dtype=np.int32)
                    ps_ = np.zeros(Bs, dtype=np.int32)
                    for t in range(prompt):
                        fs.fs_decode_step_batch(hs, ls, ps_, prompts[:Bs, t])
                    tk_ = prompts[:Bs, -1].astype(np.int32).copy()
                    for _ in range(2):
                        fs.fs_decode_step_greedy(hs, ls, ps_, tk_, dtok[:Bs])
                    torch.cuda.synchronize()
                    k_sw = 6
                    a0 = torch.cuda.Event(enable_timing=True)
                    a1 = torch.cuda.Event(enable_timing=True)
                    a0.record(stream)
                    for _ in range(k_sw):
                        fs.fs_decode_step_greedy(hs, ls, ps_, tk_, dtok[:Bs])
                    a1.record(stream)
                    torch.cuda.synchronize()
                finally:
                    fs.fs_destroy(hs)
                ms_sw = a0.elapsed_time(a1) / k_sw
                sweep.append({"lanes": Bs, "handle_lanes": cap, "ms_per_step": ms_sw,
                              "tok_s": Bs / (ms_sw / 1e3),
                              "positions": f"{prompt + 2}..{prompt + 2 + k_sw}"})
        del Wsw

    # ---- aggregate over ranks (max time)
    ms, e2e_s = max_over_ranks([ms, e2e_s], ws, "cuda")
    total_tokens = B * K * ws
    value = total_tokens / (ms / 1e3)
    peaks = _peaks()
    wb = {0: 4.0, 1: 2.0, 2: 34 / 32}[wdt]
    g_bytes, g_launches = gemm_bytes_per_step(cfg, wb, B, greedy=True)
    ms_step = ms / K
    roof = {"kernel": "weight-streaming GEMM (" + fs_path_name(cfg, wdt) + ")",
            "bound": "hbm", "achieved": None, "peak": peaks["hbm"], "unit": "GB/s",
            "frac": None, "traffic": None, "peak_source": peaks["src"],
            "launches_per_step": g_launches,
            "algorithmic_bytes_per_launch": g_bytes / g_launches,
            # tcgen05-q8_0+bf16: calls of many lane groups multiply bf16
            # copies of the Q8_0 matrices (more bytes than the algorithmic ones)
            "gemm_path": gemm_path}
    if timeline:
        share = sum(k["share"] or 0.0 for n, k in timeline["kernels"].items()
                    if n.startswith("gemm"))
        g_ms = share * ms_step
        # the GEMMs' time cannot exceed the step: the shares partition it
        assert 0.0 < g_ms <= ms_step, (g_ms, ms_step)
        achieved = g_bytes / (g_ms / 1e3) / 1e9
        roof.update(achieved=achieved, frac=achieved / peaks["hbm"],
                    ms_per_step_of_kernel=g_ms, share_of_step=share,
                    mean_launch_us=g_ms / g_launches * 1e3,
                    method="CUDA-event step time x GEMM share of the traced step "
                           "(gap + body per launch, %globaltimer per block)")
    arg_bytes = (7 * B + 1) * 4
    e2e = {"value": total_tokens / e2e_s, "unit": "tok/s",
           "h2d_bytes_per_step": arg_bytes,
           "d2h_bytes_per_step": B * 4}
    return dict(value=value, ms=ms, B=B, launches=launches, clocks=clk, roofline=roof,
                e2e=e2e, ctx=ctx, cfg=cfg, wdt=wdt, sweep=sweep, timeline=timeline)


def time_steps(h, lanes, pos, toks, dtok, steps, warmup, local):
    """Device time per greedy step (CUDA events on the handle's stream) and
    the clocks sampled meanwhile."""
    import torch
    from continuous_transformer_decode_gb300 import fs
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        fs.fs_decode_step_greedy(h, lanes, pos, toks, dtok)
    torch.cuda.synchronize()
    clocks = Clocks(gpu_id_of(local))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fs.fs_decode_step_greedy(h, lanes, pos, toks, dtok)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps, clocks.stop()


def run_workloads(args, local):
    """The other configurations of the pages' measurements, each briefly on
    its own handle: SmolLM2-135M Q8_0 at 960 lanes (MODEL-BATCHING-RESULTS,
    "Measured": B = 512 -> 960) and Mistral-7B bf16 at 1 and 128 lanes with
    contexts U[128, 4096]."""
    import torch
    from continuous_transformer_decode_gb300 import fs
    peaks = _peaks()
    out = []
    steps, warm = 10, 3
    plan = [("smollm2-135m-q8_0", [960]), ("mistral-7b-bf16", [1, 128])]
    for name, Bs in plan:
        wl = WORKLOADS[name]
        cfg = model_cfg(wl["model"])
        Wshared = gpu_weights(cfg, wl["wdtype"]) if len(Bs) > 1 else None
        for B in Bs:
            t0 = time.perf_counter()
            h, ctx, wdt = make_handle(cfg, wl, B, warm + steps + 4, W=Wshared)
            gemm_path = fs.fs_gemm_path(h)
            try:
                fs.fs_set_stream(h, torch.cuda.current_stream())
                lanes, pos, toks, _ = fill_lanes(h, cfg, wl, B, ctx)
                dtok = torch.empty(B, dtype=torch.int32, device="cuda")
                ms, clk = time_steps(h, lanes, pos, toks, dtok, steps, warm, local)
            finally:
                fs.fs_destroy(h)
            wb = {0: 4.0, 1: 2.0, 2: 34 / 32}[wdt]
            ctx_mean = float(np.mean(ctx)) + warm + steps / 2.0
            sr = step_roofline(cfg, wb, B, ctx_mean, peaks)
            tok_s = B / (ms / 1e3)
            out.append({"workload": name, "lanes": B, "ms_per_step": ms, "tok_s": tok_s,
                        "gemm_path": gemm_path,
                        "activations": ("bf16 + bf16 remainder (act_split)"
                                        if wl.get("act_split") else "bf16"),
                        "context": (f"16-token prompts" if "ctx" not in wl else
                                    f"U[{wl['ctx'][0]},{wl['ctx'][1]}] mean {np.mean(ctx):.0f}"),
                        "step_roofline": dict(sr, frac=tok_s / sr["tok_s_ceiling"]),
                        "clocks": clk, "wall_s": time.perf_counter() - t0})
        del Wshared
        torch.cuda.empty_cache()
    return out


def step_roofline(cfg, wbytes_per_param, lanes, ctx_mean, peaks):
    """Whole-step ceiling min(B*BW/bytes_step, P_tc/flops_token): weights
    once per step, each lane's KV read plus its append (logits stay on the
    device and are not counted); flops = 2 * streamed params + attention."""
    L, Hkv, hd, H = cfg["L"], cfg["Hkv"], cfg["hd"], cfg["H"]
    n_par = cfg["V"] * cfg["d"] * (1 if cfg["tied"] else 2) + L * (
        (H * hd * 2 + Hkv * hd * 2) * cfg["d"] + 3 * cfg["F"] * cfg["d"])
    w_bytes = n_par * wbytes_per_param
    kv_tok = 2 * L * Hkv * hd * 2
    bytes_step = w_bytes + lanes * (ctx_mean + 1) * kv_tok
    flops_tok = 2 * n_par + 4 * H * hd * (ctx_mean + 1) * L
    hbm = lanes * peaks["hbm"] * 1e9 / bytes_step
    tc = (peaks["bf16_sus"] or peaks["bf16"]) * 1e12 / flops_tok
    return {"tok_s_ceiling": min(hbm, tc), "bound": "hbm" if hbm < tc else "tensor",
            "bytes_per_step": bytes_step, "flops_per_token": flops_tok}


def gemm_bytes_per_step(cfg, wbytes_per_param, lanes, greedy=True):
    """Algorithmic bytes of every weight GEMM of one step: each weight once,
    the bf16 input panel, the output (f32 rows; bf16 for the SwiGLU product;
    per-tile (max, index) pairs for the greedy LM head)."""
    d, F, V = cfg["d"], cfg["F"], cfg["V"]
    nq, nkv = cfg["H"] * cfg["hd"], cfg["Hkv"] * cfg["hd"]
    B = lanes
    per_layer = ((nq + 2 * nkv) * d * wbytes_per_param + B * d * 2 + B * (nq + 2 * nkv) * 4
                 + d * nq * wbytes_per_param + B * nq * 2 + B * d * 4
                 + 2 * F * d * wbytes_per_param + B * d * 2 + B * F * 2
                 + d * F * wbytes_per_param + B * F * 2 + B * d * 4)
    head = V * d * wbytes_per_param + B * d * 2 + (B * -(-V // 128) * 8 if greedy else B * V * 4)
    return cfg["L"] * per_layer + head, cfg["L"] * 4 + 1


def traffic_for(kernel_src: str, workload: str, lanes: int):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary, or None when the kernel source changed since the capture."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    rec = json.load(open(p)).get(f"{workload}@{lanes}")
    if not rec:
        return None
    src = os.path.join(ROOT, "continuous_transformer_decode_gb300", "csrc", kernel_src)
    digest = hashlib.sha256(open(src, "rb").read()).hexdigest()
    return rec["dram_bytes_per_launch"] if rec.get("source_sha256") == digest else None


def fs_path_name(cfg, wdt):
    return {0: "f32", 1: "bf16", 2: "q8_0"}[wdt] + " weights"


def workload_config(args, wl, B, ws):
    """The workload's `config` record, the same dict for both arms: the model
    shape, lanes, context and what the step streams."""
    from continuous_transformer_decode_gb300 import synth
    cfg = model_cfg(wl["model"])
    if args.layers:
        cfg = synth.with_layers(cfg, args.layers)
    wbytes = {"bf16": 2, "q8_0": 34 / 32}[wl["wdtype"]]
    weight_mb = step_roofline(cfg, wbytes, 0, 0, _peaks())["bytes_per_step"] / 1e6
    if "ctx" in wl:  # the lanes' context lengths: the draw make_handle makes
        ctx = synth.make_context_lengths(B, *wl["ctx"], seed=3)
        context = f"ctx U[{wl['ctx'][0]},{wl['ctx'][1]}] mean {float(np.mean(ctx)):.0f}"
    else:
        context = f"16-token prompts, positions 16..{16 + args.warmup + args.steps}"
    return {"workload": args.workload, "model_shape": cfg["name"], "lanes": B,
            "layers": cfg["L"], "d": cfg["d"], "vocab": cfg["V"], "context": context,
            "l2": f"no flush: inputs larger than L2 ({weight_mb:.0f} MB of weights "
                  "streamed per step vs 129 MB L2)",
            "parallelism": f"replicas x{ws}"}


class OracleArm:
    """The oracle as it stands, on this host's cores: StepBatch over a bounded
    number of the workload's lanes (up to 32), after seeding each lane with
    the workload's context as random KV (content does not change the work)."""

    def __init__(self, wl, B, max_steps=64):
        import oracle.core as O
        from continuous_transformer_decode_gb300 import synth
        cfg = model_cfg(wl["model"])
        self.scale = 1.0
        if wl["model"] == "M":  # bounded: 2 of 32 layers, scaled by work share
            full = cfg
            cfg = synth.with_layers(cfg, 2)
            per_layer = (cfg["H"] * cfg["hd"] * 2 + cfg["Hkv"] * cfg["hd"] * 2) * cfg["d"] \
                + 3 * cfg["F"] * cfg["d"]
            head = cfg["V"] * cfg["d"]
            self.scale = (2 * per_layer + head) / (full["L"] * per_layer + head)
        self.cores = os.cpu_count() or 1
        O.set_threads(self.cores)
        W = synth.make_weights(cfg, seed=1, fmt="bf16")
        if wl["wdtype"] == "q8_0":
            q = lambda a: O.quantize_q8_0(synth.bf16_to_f32(a))
            W = {"embed": q(W["embed"]),
                 "lm_head": None if W["lm_head"] is None else q(W["lm_head"]),
                 "final_norm": W["final_norm"],
                 "layers": [{k: (v if k in ("attn_norm", "ffn_norm") else q(v))
                             for k, v in ly.items()} for ly in W["layers"]]}
            self.m = O.Model(cfg, W, O.Q8_0)
        else:
            self.m = O.Model(cfg, W, O.BF16)
        del W
        self.nb = min(B, 32)
        self.B = B
        self.ctx = wl.get("prompt", 16) if "ctx" not in wl else 1024
        self.lanes = [self.m.lane(self.ctx + max_steps + 2) for _ in range(self.nb)]
        for b, ln in enumerate(self.lanes):
            for l in range(cfg["L"]):
                K, V = synth.make_kv(self.ctx, cfg["Hkv"], cfg["hd"], seed=9, path=(b, l))
                ln.import_kv(l, K, V)
        self.L = cfg["L"]
        self.steps = 0
        self.seconds = 0.0

    def step(self) -> float:
        t0 = time.perf_counter()
        self.m.step_batch(self.lanes, [1] * self.nb)
        dt = time.perf_counter() - t0
        self.steps += 1
        self.seconds += dt
        return self.nb / dt * self.scale

    def describe(self, value):
        return {"value": value, "unit": "tok/s", "cores": self.cores, "kind": "oracle",
                "sample": f"oracle StepBatch over {self.nb} of {self.B} lanes, "
                          f"{self.steps} steps after {self.ctx} tokens of context, "
                          f"{self.L} layers" + (" (scaled to the full depth by weight share)"
                                                if self.scale != 1.0 else "")}


def cpu_baseline(wl, B, seconds=15.0):
    arm = OracleArm(wl, B)
    vals = []
    while not vals or (arm.seconds < seconds and arm.steps < 48):
        vals.append(arm.step())
    return arm.describe(arm.nb * arm.steps / arm.seconds * arm.scale)


def run_trace(args, wl, ws, rank):
    """The continuous-batching trace: jobs with Poisson arrivals on the
    scheduler's step clock, log-uniform prompts of 8..2048 tokens (consumed in
    chunks, decode first), U[16, 512] new tokens, temperature 0 or 0.8 with per-job seeds,
    through fs_sched over the decode step. Returns the JSON line's fields.
    Gate: a few jobs re-run alone on the same handle give the same tokens."""
    import torch
    from continuous_transformer_decode_gb300 import fs, synth
    cfg = model_cfg(wl["model"])
    if args.layers:
        cfg = synth.with_layers(cfg, args.layers)
    lanes = args.batch or wl["B"]
    n_jobs = args.jobs or min(512, 4 * lanes)
    jobs = synth.make_trace(n_jobs, cfg["V"], seed=5 + rank, lanes=lanes)
    if args.shared_prefix:  # one system prompt ahead of every job's own prompt
        head = [int(t) for t in synth.make_prompts(1, args.shared_prefix, cfg["V"], seed=77)[0]]
        jobs = [dict(j, prompt=head + [int(t) for t in j["prompt"]]) for j in jobs]
    max_pos = max(len(j["prompt"]) + j["max_new"] for j in jobs) + 1
    ps = 16
    n_pages = lanes * ((max_pos + ps - 1) // ps)
    W, wdt = gpu_weights(cfg, wl["wdtype"])
    h = fs.fs_create(fs.make_desc(cfg, wdt, fs.FS_DTYPE_BF16, lanes, n_pages, max_pos, ps,
                                  wl.get("act_split", 0)), W)
    budget = args.prefill_budget or max(1, lanes // 2)
    chunk = args.prefill_chunk or budget

    def run(sched_lanes, js):
        s = fs.fs_sched_create(h, sched_lanes, budget, prefill_chunk=chunk,
                               prefix_reuse_min=args.prefix_reuse)
        try:
            order = sorted(js, key=lambda j: (j["arrive"], j["id"]))
            ids, i, tick = {}, 0, 0
            st = fs.fs_sched_get_stats(s)
            while i < len(order) or st["active"] or st["queued"]:
                if not st["active"] and not st["queued"]:
                    tick = max(tick, order[i]["arrive"])  # idle: jump to the next arrival
                while i < len(order) and order[i]["arrive"] <= tick:
                    j = order[i]
                    ids[j["id"]] = fs.fs_sched_submit(s, j["prompt"], j["max_new"],
                                                      j["temperature"], j["seed"])
                    i += 1
                fs.fs_sched_step(s)
                tick += 1
                st = fs.fs_sched_get_stats(s)
            return {j["id"]: fs.fs_sched_take(s, ids[j["id"]]) for j in js}, st
        finally:
            fs.fs_sched_destroy(s)

    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    tokens, st = run(lanes, jobs)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    if ws > 1:
        t = torch.tensor([dt], device="cuda")
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        dt = float(t.item())
    # gate: the three shortest jobs, each alone (one lane, arrival at 0)
    short = sorted(jobs, key=lambda j: len(j["prompt"]) + j["max_new"])[:3]
    alone_ok = []
    for j in short:
        got, _ = run(1, [dict(j, arrive=0)])
        alone_ok.append(got[j["id"]] == tokens[j["id"]])
    fs.fs_destroy(h)
    total = st["prefill_tokens"] + st["decode_tokens"]
    # served: every job's prompt and generated tokens, whether fed or taken
    # from a clone (prefix reuse)
    served = sum(len(j["prompt"]) for j in jobs) + sum(len(t) for t in tokens.values())
    return dict(cfg=cfg, lanes=lanes, jobs=n_jobs, seconds=dt, steps=st["steps"],
                tok_s=total * ws / dt, decode_tok_s=st["decode_tokens"] * ws / dt,
                served_tok_s=served * ws / dt, prefix_hits=st["prefix_hits"],
                prefix_tokens=st["prefix_tokens"],
                prefill_tokens=st["prefill_tokens"], decode_tokens=st["decode_tokens"],
                occupancy_avg=st["occupancy_avg"], occupancy_max=st["occupancy_max"],
                budget=budget, chunk=chunk, alone_ok=alone_ok, max_pos=max_pos)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=12)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="smollm2-135m-bf16", choices=sorted(WORKLOADS))
    ap.add_argument("--batch", type=int, default=0)
    ap.add_argument("--layers", type=int, default=0,
                    help="use only the first L layers (same per-layer shapes; for "
                         "small profiling captures, never for a reported number)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--shared-prefix", type=int, default=0,
                    help="trace workload: a common system prompt of N tokens ahead of "
                         "every job's prompt")
    ap.add_argument("--prefix-reuse", type=int, default=0,
                    help="trace workload: the scheduler's prefix_reuse_min (0: off)")
    ap.add_argument("--trace", type=int, default=2,
                    help="after the timed steps, trace N more steps' kernel timeline "
                         "(%%globaltimer per block): the GEMM roofline's time share "
                         "and the line's kernel_timeline (0: off, no roofline)")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the other configurations' record (Q8_0 at 960 lanes, "
                         "Mistral-7B at 1 and 128 lanes)")
    ap.add_argument("--jobs", type=int, default=0,
                    help="trace workload: number of jobs (default min(512, 4 x lanes))")
    ap.add_argument("--prefill-budget", type=int, default=0,
                    help="trace workload: prompt tokens per step (default lanes / 2)")
    ap.add_argument("--prefill-chunk", type=int, default=0,
                    help="trace workload: prompt tokens per lane per step (default the "
                         "budget; 1 = no chunking)")
    args = ap.parse_args()
    wl = WORKLOADS[args.workload]
    ws, rank, local = _dist()

    if wl.get("trace"):
        if args.impl == "reference":
            if rank == 0:
                print(json.dumps({"impl": "reference", "unavailable":
                                  "the trace workload has no oracle arm: a 7B f32 oracle "
                                  "runs at seconds per token"}))
            return
        if ws > 1:
            import torch
            torch.cuda.set_device(local)
            torch.distributed.init_process_group("nccl")
        r = run_trace(args, wl, ws, rank)
        if rank == 0:
            cfg = r["cfg"]
            print(json.dumps({
                "metric": "aggregate tokens/s (continuous-batching trace)", "value": r["tok_s"],
                "unit": "tok/s", "n_gpus": ws, "steps": r["steps"], "warmup": 0,
                "ms_per_step": r["seconds"] * 1e3 / max(1, r["steps"]),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": wl["wdtype"], "data": "synthetic job trace (random N(0,0.02) weights)",
                "config": {"workload": args.workload, "model_shape": cfg["name"],
                           "layers": cfg["L"], "lanes": r["lanes"], "jobs": r["jobs"],
                           "max_prefill_tokens_per_tick": r["budget"],
                           "prefill_chunk": r["chunk"], "max_pos": r["max_pos"],
                           "shared_prefix": args.shared_prefix,
                           "prefix_reuse_min": args.prefix_reuse,
                           "parallelism": f"replicas x{ws}"},
                "served_tok_s": r["served_tok_s"], "prefix_hits": r["prefix_hits"],
                "prefix_tokens": r["prefix_tokens"],
                "decode_tok_s": r["decode_tok_s"], "prefill_tokens": r["prefill_tokens"],
                "decode_tokens": r["decode_tokens"], "occupancy_avg": r["occupancy_avg"],
                "occupancy_max": r["occupancy_max"],
                "per_job_equals_alone": {"jobs_checked": len(r["alone_ok"]),
                                         "equal": all(r["alone_ok"])},
                "e2e": {"value": r["tok_s"], "unit": "tok/s",
                        "note": "host-driven scheduler loop; host tokens each step"}}))
        if ws > 1:
            import torch
            torch.distributed.destroy_process_group()
        return

    if args.impl == "reference":
        if rank != 0:
            return
        B = args.batch or wl["B"]
        arm = OracleArm(wl, B, max_steps=args.warmup + args.steps + 2)
        for _ in range(args.warmup):
            arm.step()
        arm.steps, arm.seconds = 0, 0.0
        for _ in range(args.steps):
            arm.step()
        v = arm.nb * arm.steps / arm.seconds * arm.scale
        cb = arm.describe(v)
        print(json.dumps({"metric": METRIC, "value": v, "unit": "tok/s", "impl": "reference",
                          "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
                          "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                          "dtype": "f32", "data": "synthetic",
                          "config": workload_config(args, wl, B, ws),
                          "cpu_baseline": cb,
                          "e2e": {"value": v, "unit": "tok/s", "h2d_bytes_per_step": 0,
                                  "d2h_bytes_per_step": 0}}))
        return

    if ws > 1:
        import torch
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl")
    r = run_ours(args, wl, ws, rank, local)
    if rank != 0:
        if ws > 1:
            import torch
            torch.distributed.destroy_process_group()
        return
    workloads = None
    if (ws == 1 and not args.no_workloads and not args.layers and not args.batch
            and args.workload == "smollm2-135m-bf16"):
        workloads = run_workloads(args, local)
    cb = None if args.no_cpu_baseline else cpu_baseline(wl, r["B"])
    cfg = r["cfg"]
    wbytes = {"bf16": 2, "q8_0": 34 / 32}[wl["wdtype"]]
    peaks = _peaks()
    ctx_mean = float(np.mean(r["ctx"])) + args.warmup + args.steps / 2.0
    sr = step_roofline(cfg, wbytes, r["B"], ctx_mean, peaks)
    line = {
        "metric": METRIC, "value": r["value"], "unit": "tok/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["ms"] / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": wl["wdtype"], "data": "synthetic (random N(0,0.02) weights, uniform prompts)",
        "config": workload_config(args, wl, r["B"], ws),
        "roofline": dict(r["roofline"], traffic=traffic_for("k_gemm_tc.cu", args.workload, r["B"])),
        "step_roofline": dict(sr, frac=r["value"] / ws / sr["tok_s_ceiling"], peak_source=peaks["src"]),
        "sweep": [dict(p, frac_of_step_roofline=p["tok_s"] / step_roofline(
            cfg, wbytes, p["lanes"], 17 + 3, peaks)["tok_s_ceiling"]) for p in r["sweep"]],
        "cpu_baseline": cb, "e2e": r["e2e"],
        **({"reduced_layers_for_profiling": args.layers} if args.layers else {}),
        "clocks": r["clocks"], "gpu_launches": r["launches"],
        **({"kernel_timeline": r["timeline"]} if r["timeline"] else {}),
        **({"workloads": workloads} if workloads else {}),
    }
    print(json.dumps(line))
    if ws > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
