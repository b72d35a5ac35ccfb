"""Thin Python binding of the C ABI in include/fs.h (argument marshalling only).

Every step of the decode path runs inside ``_build/libfs.so``; this module
only converts Python/numpy/torch arguments to pointers and sizes. If the
library is missing the import of any entry point raises: there is no
fallback implementation.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from . import build as _build

FS_OK = 0
ERRORS = {-1: "FS_ERR_ARG", -2: "FS_ERR_LANE", -3: "FS_ERR_DUP_LANE",
          -4: "FS_ERR_POSITION", -5: "FS_ERR_TOKEN", -6: "FS_ERR_KV_FULL",
          -7: "FS_ERR_OOM", -8: "FS_ERR_CUDA", -9: "FS_ERR_STATE",
          -10: "FS_ERR_DEVICE", -11: "FS_ERR_SCRATCH", -12: "FS_ERR_QUEUE_FULL",
          -13: "FS_ERR_KV_BUDGET"}
CODES = {v: k for k, v in ERRORS.items()}
FS_DTYPE_F32, FS_DTYPE_BF16, FS_DTYPE_Q8_0 = 0, 1, 2


class FsError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{ERRORS.get(code, code)}: {msg}")
        self.code = code
        self.name = ERRORS.get(code, str(code))


class fs_model_desc(C.Structure):
    _fields_ = [("n_layers", C.c_int32), ("d_model", C.c_int32),
                ("n_heads", C.c_int32), ("n_kv_heads", C.c_int32),
                ("head_dim", C.c_int32), ("d_ffn", C.c_int32),
                ("vocab", C.c_int32), ("rms_eps", C.c_float),
                ("rope_theta", C.c_double), ("tied_embeddings", C.c_int32),
                ("weight_dtype", C.c_int32), ("kv_dtype", C.c_int32),
                ("max_lanes", C.c_int32), ("page_size", C.c_int32),
                ("n_pages", C.c_int32), ("max_pos", C.c_int32),
                ("act_split", C.c_int32)]


class fs_layer_weights(C.Structure):
    _fields_ = [(k, C.c_void_p) for k in ("wq", "wk", "wv", "wo", "w_gate",
                                          "w_up", "w_down", "attn_norm",
                                          "ffn_norm")]


class fs_weights(C.Structure):
    _fields_ = [("embed", C.c_void_p), ("lm_head", C.c_void_p),
                ("final_norm", C.c_void_p),
                ("layers", C.POINTER(fs_layer_weights))]


class fs_sched_config(C.Structure):
    _fields_ = [("lanes", C.c_int32), ("max_prefill_tokens_per_tick", C.c_int32),
                ("max_queue", C.c_int32), ("prefill_chunk", C.c_int32),
                ("kv_budget_tokens", C.c_int64), ("prefix_reuse_min", C.c_int32)]


class fs_job(C.Structure):
    _fields_ = [("prompt", C.c_void_p), ("prompt_len", C.c_int32),
                ("max_new_tokens", C.c_int32), ("temperature", C.c_float),
                ("seed", C.c_uint64), ("stop_token", C.c_int32)]


class fs_sched_stats(C.Structure):
    _fields_ = [("steps", C.c_int64), ("prefill_tokens", C.c_int64),
                ("decode_tokens", C.c_int64), ("jobs_submitted", C.c_int64),
                ("jobs_done", C.c_int64), ("rejected", C.c_int64),
                ("active", C.c_int32), ("queued", C.c_int32),
                ("occupancy_last", C.c_int32), ("occupancy_max", C.c_int32),
                ("occupancy_avg", C.c_double),
                ("rejected_queue_full", C.c_int64), ("rejected_kv_budget", C.c_int64),
                ("kv_reserved_tokens", C.c_int64), ("kv_reserved_max", C.c_int64),
                ("kv_budget_tokens", C.c_int64), ("kv_wait_steps", C.c_int64),
                ("seconds", C.c_double), ("prefill_tok_s", C.c_double),
                ("decode_tok_s", C.c_double),
                ("prefix_hits", C.c_int64), ("prefix_tokens", C.c_int64),
                ("jobs_cancelled", C.c_int64)]


LIB_PATH = _build.LIB
_lib = None


def lib():
    """Loads libfs.so (built by ``build.build()``); raises if it is absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"CUDA library not built: {LIB_PATH} is missing "
                          "(run __graft_entry__.build())")
    L = C.CDLL(LIB_PATH)
    p, i32, i64, u64 = C.c_void_p, C.c_int32, C.c_int64, C.c_uint64
    sig = {
        "fs_create": (C.c_int, [C.POINTER(fs_model_desc),
                                C.POINTER(fs_weights), C.POINTER(p)]),
        "fs_destroy": (C.c_int, [p]),
        "fs_last_error": (C.c_char_p, [p]),
        "fs_set_stream": (C.c_int, [p, p]),
        "fs_lane_reset": (C.c_int, [p, i32]),
        "fs_lane_clone": (C.c_int, [p, i32, i32]),
        "fs_trace_enable": (C.c_int, [p, i64]),
        "fs_selftest_bounded_wait": (C.c_int, [p, i32, p]),
        "fs_trace_read": (C.c_int, [p, p, i64, p, C.c_int]),
        "fs_lane_evict": (C.c_int, [p, i32, i32, i32]),
        "fs_decode_step_batch": (C.c_int, [p, p, p, p, i32, p]),
        "fs_step_batch_chunked": (C.c_int, [p, p, p, p, i32, p]),
        "fs_decode_step_greedy": (C.c_int, [p, p, p, p, i32, p]),
        "fs_sample": (C.c_int, [p, i32, p, p, p, p]),
        "fs_lane_length": (C.c_int, [p, i32, p]),
        "fs_lane_pages": (C.c_int, [p, i32, p, i32, p]),
        "fs_lane_export_kv": (C.c_int, [p, i32, i32, p, p]),
        "fs_lane_import_kv": (C.c_int, [p, i32, p, p, i32]),
        "fs_lane_fill_random_kv": (C.c_int, [p, i32, i32, u64]),
        "fs_quantize_q8_0": (C.c_int, [p, i64, p, p]),
        "fs_sample_device": (C.c_int, [p, i32, p, p, p, p]),
        "fs_profile_enable": (C.c_int, [p, i32]),
        "fs_profile_read": (C.c_int, [p, i32, p, p, p]),
        "fs_kernel_launches": (C.c_int, [p, p]),
        "fs_gemm_path": (C.c_char_p, [p]),
        "fs_gemm_plan": (C.c_int, [i64, i64, i32, i32, i32, i32, p]),
        "fs_lane_capacity": (C.c_int, [p, p]),
        "fs_attention_path": (C.c_char_p, [p]),
        "fs_device_error": (C.c_int, [p, p]),
        "fs_copy_logits": (C.c_int, [p, p]),
        "fs_gemm_bf16_noalloc": (C.c_int, [p, i32, i32, p, i32, p, i32, p]),
        "fs_sched_create": (C.c_int, [p, C.POINTER(fs_sched_config), C.POINTER(p)]),
        "fs_sched_create_model_free": (C.c_int, [C.POINTER(fs_sched_config), i32,
                                                 C.POINTER(p)]),
        "fs_sched_destroy": (C.c_int, [p]),
        "fs_sched_submit": (C.c_int, [p, C.POINTER(fs_job), p]),
        "fs_sched_step": (C.c_int, [p, p]),
        "fs_sched_run": (C.c_int, [p, i64, p]),
        "fs_sched_take": (C.c_int, [p, i64, p, i32, p]),
        "fs_sched_get_stats": (C.c_int, [p, C.POINTER(fs_sched_stats)]),
        "fs_sched_status": (C.c_int, [p, i64, p]),
        "fs_sched_cancel": (C.c_int, [p, i64]),
        "fs_sched_last_batch": (C.c_int, [p, p, i32, p]),
        "fs_sched_last_error": (C.c_char_p, [p]),
        "fs_sched_model_free_fail_resets": (C.c_int, [p, i32]),
        "fs_gemm_bf16": (C.c_int, [p, i32, i32, p, i32, p, i32, i32, p]),
        "fs_gemm_bf16_width": (C.c_int, [p, i32, i32, p, i32, p, i32, p]),
        "fs_gemm_bf16_time": (C.c_int, [p, i32, i32, p, i32, p, i32, i32, p, p]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


def exported_symbols() -> list:
    """Names of the entry points declared in include/fs.h."""
    return ["fs_create", "fs_destroy", "fs_last_error", "fs_set_stream",
            "fs_lane_reset", "fs_lane_clone", "fs_lane_evict", "fs_trace_enable", "fs_trace_read", "fs_selftest_bounded_wait", "fs_decode_step_batch", "fs_step_batch_chunked", "fs_decode_step_greedy", "fs_sample",
            "fs_lane_length", "fs_lane_pages", "fs_lane_export_kv",
            "fs_lane_import_kv", "fs_lane_fill_random_kv", "fs_quantize_q8_0",
            "fs_kernel_launches", "fs_gemm_path", "fs_gemm_plan", "fs_lane_capacity", "fs_attention_path", "fs_sample_device",
            "fs_profile_enable", "fs_profile_read", "fs_device_error",
            "fs_gemm_bf16", "fs_gemm_bf16_width", "fs_gemm_bf16_time", "fs_copy_logits", "fs_gemm_bf16_noalloc",
            "fs_sched_create", "fs_sched_create_model_free", "fs_sched_destroy",
            "fs_sched_submit", "fs_sched_step", "fs_sched_run", "fs_sched_take",
            "fs_sched_get_stats", "fs_sched_status", "fs_sched_cancel", "fs_sched_last_batch",
            "fs_sched_last_error", "fs_sched_model_free_fail_resets"]


def _check(h, rc: int) -> None:
    if rc != FS_OK:
        msg = lib().fs_last_error(h)
        raise FsError(rc, msg.decode() if msg else "")


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(C.c_void_p)


def _dptr(x):
    """Address of a host numpy array, a torch tensor (host or device) or None."""
    if x is None:
        return None
    if isinstance(x, np.ndarray):
        assert x.flags["C_CONTIGUOUS"]
        return x.ctypes.data
    if hasattr(x, "data_ptr"):
        assert x.is_contiguous()
        return x.data_ptr()
    return int(x)


def make_desc(cfg: dict, weight_dtype: int, kv_dtype: int, max_lanes: int,
              n_pages: int, max_pos: int, page_size: int = 16,
              act_split: int = 0) -> fs_model_desc:
    return fs_model_desc(cfg["L"], cfg["d"], cfg["H"], cfg["Hkv"], cfg["hd"],
                         cfg["F"], cfg["V"], cfg["rms_eps"], cfg["rope_theta"],
                         1 if cfg["tied"] else 0, weight_dtype, kv_dtype,
                         max_lanes, page_size, n_pages, max_pos, act_split)


LAYER_KEYS = ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down",
              "attn_norm", "ffn_norm")


def fs_create(desc: fs_model_desc, weights: dict):
    """weights: dict of host numpy arrays or torch tensors (host or device):
    embed, lm_head (or None), final_norm, layers[list of LAYER_KEYS dicts]."""
    layers = (fs_layer_weights * len(weights["layers"]))()
    for i, ly in enumerate(weights["layers"]):
        for k in LAYER_KEYS:
            setattr(layers[i], k, _dptr(ly[k]))
    w = fs_weights(_dptr(weights["embed"]), _dptr(weights.get("lm_head")),
                   _dptr(weights["final_norm"]), layers)
    h = C.c_void_p()
    _check(None, lib().fs_create(C.byref(desc), C.byref(w), C.byref(h)))
    return h


def fs_destroy(h) -> None:
    lib().fs_destroy(h)


def fs_last_error(h) -> str:
    m = lib().fs_last_error(h)
    return m.decode() if m else ""


def fs_set_stream(h, stream) -> None:
    """stream: a torch.cuda.Stream, a raw cudaStream_t int, or None."""
    raw = getattr(stream, "cuda_stream", stream)
    _check(h, lib().fs_set_stream(h, raw))


def fs_lane_reset(h, lane: int) -> None:
    _check(h, lib().fs_lane_reset(h, int(lane)))


TRACE_TAGS = {1: "embed", 2: "rmsnorm", 3: "sample", 4: "argmax_tiles",
              5: "attn_mma", 6: "attn_tma", 7: "attn_tiled", 8: "attn_warp",
              9: "rope_append", 10: "gemv", 11: "attn_partial", 12: "attn_combine",
              13: "gemv_swiglu",
              16: "gemm_store", 17: "gemm_resid",
              18: "gemm_swiglu", 19: "gemm_argmax"}


def fs_trace_enable(h, capacity: int) -> None:
    """Kernel timeline tracing into a device buffer of ``capacity`` records
    (0 turns it off)."""
    _check(h, lib().fs_trace_enable(h, int(capacity)))


def fs_trace_read(h, reset: bool = True):
    """Returns (records [n, 4] uint64, appended count)."""
    n = C.c_int64()
    _check(h, lib().fs_trace_read(h, None, 0, C.byref(n), 0))
    out = np.zeros((max(1, n.value), 4), dtype=np.uint64)
    _check(h, lib().fs_trace_read(h, _ptr(out), n.value, C.byref(n), int(bool(reset))))
    return out[:min(n.value, out.shape[0])], n.value


def fs_lane_clone(h, src: int, dst: int) -> None:
    """Empty lane ``dst`` takes lane ``src``'s history (full pages shared,
    the partial last page copied)."""
    _check(h, lib().fs_lane_clone(h, int(src), int(dst)))


def fs_lane_evict(h, lane: int, start: int, end: int) -> None:
    """Positions [start, end) leave the lane; later entries move down, their
    keys rotated back by end - start positions."""
    _check(h, lib().fs_lane_evict(h, int(lane), int(start), int(end)))


def fs_decode_step_batch(h, lanes, positions, tokens, logits_out=None):
    """Advances lanes by one token. ``positions`` (np.int32) is incremented
    in place on success and returned. logits_out: torch CUDA f32 [n, V]."""
    la = _i32(lanes)
    to = _i32(tokens)
    if (isinstance(positions, np.ndarray) and positions.dtype == np.int32
            and positions.flags["C_CONTIGUOUS"]):
        po = positions
    else:
        po = _i32(positions)
    n = la.size
    assert po.size == n and to.size == n
    _check(h, lib().fs_decode_step_batch(h, _ptr(la), _ptr(po), _ptr(to), n,
                                         _dptr(logits_out)))
    return po


def fs_decode_step_greedy(h, lanes, positions, tokens, tokens_out=None):
    """Decode step + greedy token per lane without materialising logits.
    tokens_out: torch CUDA int32 [n] (no synchronisation) or None for a host
    numpy array. ``positions`` (np.int32) is incremented in place."""
    la = _i32(lanes)
    to = _i32(tokens)
    if (isinstance(positions, np.ndarray) and positions.dtype == np.int32
            and positions.flags["C_CONTIGUOUS"]):
        po = positions
    else:
        po = _i32(positions)
    n = la.size
    assert po.size == n and to.size == n
    host = tokens_out is None
    out = np.empty(n, dtype=np.int32) if host else tokens_out
    _check(h, lib().fs_decode_step_greedy(h, _ptr(la), _ptr(po), _ptr(to), n,
                                          _ptr(out) if host else _dptr(out)))
    return out


def fs_step_batch_chunked(h, lanes, positions, tokens, logits_out=None):
    """Chunked prefill step: a lane may appear on several rows at its next
    consecutive positions. ``positions`` (np.int32) is incremented in place
    on success and returned. logits_out: torch CUDA f32 [n, V]."""
    la = _i32(lanes)
    to = _i32(tokens)
    if (isinstance(positions, np.ndarray) and positions.dtype == np.int32
            and positions.flags["C_CONTIGUOUS"]):
        po = positions
    else:
        po = _i32(positions)
    n = la.size
    assert po.size == n and to.size == n
    _check(h, lib().fs_step_batch_chunked(h, _ptr(la), _ptr(po), _ptr(to), n,
                                          _dptr(logits_out)))
    return po


def fs_sample(h, temps, seeds, counters) -> np.ndarray:
    t = np.ascontiguousarray(np.asarray(temps, dtype=np.float32))
    s = np.ascontiguousarray(np.asarray(seeds, dtype=np.uint64))
    c = np.ascontiguousarray(np.asarray(counters, dtype=np.uint64))
    out = np.empty(t.size, dtype=np.int32)
    _check(h, lib().fs_sample(h, t.size, _ptr(t), _ptr(s), _ptr(c), _ptr(out)))
    return out


def fs_sample_device(h, temps, seeds, counters, tokens_out) -> None:
    """All four are torch CUDA tensors (f32, int64/uint64, int64/uint64,
    int32) of n entries; no synchronisation."""
    _check(h, lib().fs_sample_device(h, tokens_out.numel(), _dptr(temps),
                                     _dptr(seeds), _dptr(counters),
                                     _dptr(tokens_out)))


FS_PROF_GEMM, FS_PROF_ATTN, FS_PROF_OTHER = 0, 1, 2


def fs_profile_enable(h, enable: bool) -> None:
    _check(h, lib().fs_profile_enable(h, 1 if enable else 0))


def fs_profile_read(h, cls: int):
    """(ms, launches, algorithmic bytes) of kernel class `cls` since the
    last read."""
    ms, n, b = C.c_double(), C.c_int64(), C.c_double()
    _check(h, lib().fs_profile_read(h, int(cls), C.byref(ms), C.byref(n),
                                    C.byref(b)))
    return ms.value, n.value, b.value


def fs_lane_length(h, lane: int) -> int:
    v = C.c_int32()
    _check(h, lib().fs_lane_length(h, int(lane), C.byref(v)))
    return v.value


def fs_lane_pages(h, lane: int) -> list:
    n = C.c_int32()
    _check(h, lib().fs_lane_pages(h, int(lane), None, 0, C.byref(n)))
    out = np.empty(max(1, n.value), dtype=np.int32)
    _check(h, lib().fs_lane_pages(h, int(lane), _ptr(out), n.value, C.byref(n)))
    return out[:n.value].tolist()


def fs_lane_export_kv(h, lane: int, layer: int, Hkv: int, hd: int):
    n = fs_lane_length(h, lane)
    k = np.empty((n, Hkv, hd), dtype=np.float32)
    v = np.empty((n, Hkv, hd), dtype=np.float32)
    _check(h, lib().fs_lane_export_kv(h, int(lane), int(layer), _ptr(k), _ptr(v)))
    return k, v


def fs_lane_import_kv(h, lane: int, k: np.ndarray, v: np.ndarray) -> None:
    """k, v: f32 [n_layers, n, Hkv, hd] (K already rotated)."""
    k = np.ascontiguousarray(k, dtype=np.float32)
    v = np.ascontiguousarray(v, dtype=np.float32)
    _check(h, lib().fs_lane_import_kv(h, int(lane), _ptr(k), _ptr(v),
                                      k.shape[1]))


def fs_lane_fill_random_kv(h, lane: int, n: int, seed: int) -> None:
    _check(h, lib().fs_lane_fill_random_kv(h, int(lane), int(n), int(seed)))


def fs_quantize_q8_0(src, blocks_out, stream=None) -> None:
    """src: torch CUDA f32 tensor; blocks_out: torch CUDA uint8 [n/32, 34]."""
    raw = getattr(stream, "cuda_stream", stream)
    rc = lib().fs_quantize_q8_0(_dptr(src), src.numel(), _dptr(blocks_out), raw)
    if rc != FS_OK:
        raise FsError(rc, "fs_quantize_q8_0 failed")


def fs_kernel_launches(h) -> int:
    v = C.c_int64()
    _check(h, lib().fs_kernel_launches(h, C.byref(v)))
    return v.value


def fs_gemm_path(h) -> str:
    return lib().fs_gemm_path(h).decode()


PLAN_KEYS = ("P", "lanes_per_group", "groups", "tmem_cols", "q8_copy_kept",
             "q8_copy_used", "m_tiles", "k_blocks")


def fs_gemm_plan(n_rows: int, k_inputs: int, max_lanes: int, n: int, sms: int,
                 weight_dtype: int) -> dict:
    """The tcgen05 GEMM's work split for one matrix and call (host only)."""
    out = (C.c_int32 * 8)()
    _check(None, lib().fs_gemm_plan(n_rows, k_inputs, max_lanes, n, sms, weight_dtype, out))
    return dict(zip(PLAN_KEYS, [int(v) for v in out]))


def fs_attention_path(h) -> str:
    return lib().fs_attention_path(h).decode()


def fs_device_error(h) -> int:
    v = C.c_int32()
    _check(h, lib().fs_device_error(h, C.byref(v)))
    return v.value


def fs_selftest_bounded_wait(h, timeout_us: int = 2000) -> int:
    """Failure-detection check: a kernel's bounded wait on a barrier nothing
    arrives on gives up after timeout_us; returns the device error code it
    set (99), which is then cleared."""
    v = C.c_int32()
    _check(h, lib().fs_selftest_bounded_wait(h, int(timeout_us), C.byref(v)))
    return v.value


def fs_gemm_bf16(W, X, Y, splits: int = 1, path: int = 1, stream=None) -> None:
    """Test hook: Y = X @ W^T on the device (torch bf16 W [N, K], X [B, K],
    f32 Y [B, N])."""
    raw = getattr(stream, "cuda_stream", stream)
    N, K = W.shape
    B = X.shape[0]
    rc = lib().fs_gemm_bf16(_dptr(W), N, K, _dptr(X), B, _dptr(Y), splits,
                            path, raw)
    if rc != FS_OK:
        raise FsError(rc, "fs_gemm_bf16 failed")


def fs_gemm_bf16_width(W, X, Y, width: int, stream=None) -> None:
    """Test hook: the tcgen05 GEMM with the stream-K width given directly."""
    raw = getattr(stream, "cuda_stream", stream)
    N, K = W.shape
    B = X.shape[0]
    rc = lib().fs_gemm_bf16_width(_dptr(W), N, K, _dptr(X), B, _dptr(Y), width, raw)
    if rc != FS_OK:
        raise FsError(rc, "fs_gemm_bf16_width failed")


def fs_gemm_bf16_time(W, X, Y, width: int, reps: int = 10, stream=None) -> float:
    """Tuning hook: mean device ms of one tcgen05 GEMM launch with the given
    stream-K width, over `reps` launches each after an L2-evicting memset."""
    raw = getattr(stream, "cuda_stream", stream)
    N, K = W.shape
    B = X.shape[0]
    ms = C.c_double()
    rc = lib().fs_gemm_bf16_time(_dptr(W), N, K, _dptr(X), B, _dptr(Y), width, reps,
                                 C.byref(ms), raw)
    if rc != FS_OK:
        raise FsError(rc, "fs_gemm_bf16_time failed")
    return ms.value


def fs_copy_logits(h, dst) -> None:
    """Copies the last step's logits [n, V] f32 into dst (numpy or torch)."""
    _check(h, lib().fs_copy_logits(h, _dptr(dst)))


def fs_gemm_bf16_noalloc(W, X, Y, splits: int = 1, stream=None) -> None:
    """fs_gemm_bf16 (tcgen05 path) with its workspace in the library's static
    device scratch instead of allocations (see include/fs.h)."""
    raw = getattr(stream, "cuda_stream", stream)
    N, K = W.shape
    B = X.shape[0]
    rc = lib().fs_gemm_bf16_noalloc(_dptr(W), N, K, _dptr(X), B, _dptr(Y),
                                    splits, raw)
    if rc != FS_OK:
        raise FsError(rc, "fs_gemm_bf16_noalloc failed")


# ------------------------------------------------------------------ scheduler
def _sched_check(s, rc: int) -> None:
    if rc != FS_OK:
        msg = lib().fs_sched_last_error(s)
        raise FsError(rc, msg.decode() if msg else "")


def fs_sched_create(h, lanes: int, max_prefill_tokens_per_tick: int = 1,
                    max_queue: int = 0, prefill_chunk: int = 1, kv_budget_tokens: int = 0,
                    prefix_reuse_min: int = 0):
    s = C.c_void_p()
    cfg = fs_sched_config(lanes, max_prefill_tokens_per_tick, max_queue, prefill_chunk,
                          kv_budget_tokens, prefix_reuse_min)
    rc = lib().fs_sched_create(h, C.byref(cfg), C.byref(s))
    if rc != FS_OK:
        raise FsError(rc, "fs_sched_create failed")
    return s


def fs_sched_create_model_free(lanes: int, vocab: int,
                               max_prefill_tokens_per_tick: int = 1,
                               max_queue: int = 0, prefill_chunk: int = 1,
                               kv_budget_tokens: int = 0, prefix_reuse_min: int = 0):
    s = C.c_void_p()
    cfg = fs_sched_config(lanes, max_prefill_tokens_per_tick, max_queue, prefill_chunk,
                          kv_budget_tokens, prefix_reuse_min)
    rc = lib().fs_sched_create_model_free(C.byref(cfg), vocab, C.byref(s))
    if rc != FS_OK:
        raise FsError(rc, "fs_sched_create_model_free failed")
    return s


def fs_sched_destroy(s) -> None:
    lib().fs_sched_destroy(s)


def fs_sched_submit(s, prompt, max_new_tokens: int, temperature: float = 0.0,
                    seed: int = 0, stop_token: int = -1) -> int:
    p = _i32(prompt)
    job = fs_job(p.ctypes.data, p.size, max_new_tokens, temperature,
                 int(seed) & (2**64 - 1), stop_token)
    jid = C.c_int64()
    _sched_check(s, lib().fs_sched_submit(s, C.byref(job), C.byref(jid)))
    return jid.value


def fs_sched_step(s) -> int:
    n = C.c_int32()
    _sched_check(s, lib().fs_sched_step(s, C.byref(n)))
    return n.value


def fs_sched_run(s, max_steps: int = 10**9) -> int:
    n = C.c_int64()
    _sched_check(s, lib().fs_sched_run(s, max_steps, C.byref(n)))
    return n.value


def fs_sched_take(s, job_id: int) -> list:
    n = C.c_int32()
    buf = np.empty(1 << 16, dtype=np.int32)
    _sched_check(s, lib().fs_sched_take(s, job_id, _ptr(buf), buf.size, C.byref(n)))
    return buf[:n.value].tolist()


def fs_sched_get_stats(s) -> dict:
    st = fs_sched_stats()
    _sched_check(s, lib().fs_sched_get_stats(s, C.byref(st)))
    return {k: getattr(st, k) for k, _ in st._fields_}


JOB_UNKNOWN, JOB_QUEUED, JOB_RUNNING, JOB_DONE_LENGTH, JOB_DONE_STOP, JOB_CANCELLED = (
    -1, 0, 1, 2, 3, 4)


def fs_sched_status(s, job_id: int) -> int:
    """One of the JOB_* states."""
    v = C.c_int32()
    _sched_check(s, lib().fs_sched_status(s, int(job_id), C.byref(v)))
    return v.value


def fs_sched_cancel(s, job_id: int) -> None:
    _sched_check(s, lib().fs_sched_cancel(s, int(job_id)))


def fs_sched_last_batch(s) -> list:
    n = C.c_int32()
    buf = np.empty(4096, dtype=np.int32)
    _sched_check(s, lib().fs_sched_last_batch(s, _ptr(buf), buf.size, C.byref(n)))
    return buf[:n.value].tolist()


def fs_sched_model_free_fail_resets(s, n: int) -> None:
    """Test hook: the model-free engine fails its next n lane resets."""
    _sched_check(s, lib().fs_sched_model_free_fail_resets(s, int(n)))


def fs_sched_last_error(s) -> str:
    m = lib().fs_sched_last_error(s)
    return m.decode() if m else ""
