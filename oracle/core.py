"""ctypes binding of the C++ f32 oracle (oracle.cpp) — test infrastructure only.

Every function here is a thin marshaller; the arithmetic lives in oracle.cpp.
Build: ``build()`` compiles oracle.cpp with g++ -O2 -ffp-contract=off into
``oracle/_build/liboracle.so`` (no -ffast-math, no -march flags, so x86_64
and aarch64 builds compute the same IEEE f32 operations).
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")

F32, BF16, Q8_0 = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile the oracle shared library (idempotent)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class or_desc(C.Structure):
    _fields_ = [("L", C.c_int), ("d", C.c_int), ("H", C.c_int),
                ("Hkv", C.c_int), ("hd", C.c_int), ("F", C.c_int),
                ("V", C.c_int), ("rms_eps", C.c_float),
                ("rope_theta", C.c_double), ("tied", C.c_int)]


_lib = None


def lib():
    global _lib
    if _lib is None:
        path = build()
        L = C.CDLL(path)
        p, i, f, u64 = C.c_void_p, C.c_int, C.c_float, C.c_uint64
        sig = {
            "or_bf16_to_f32": (C.c_float, [C.c_uint16]),
            "or_f16_to_f32": (C.c_float, [C.c_uint16]),
            "or_f32_to_f16": (C.c_uint16, [C.c_float]),
            "or_f32_to_bf16": (C.c_uint16, [C.c_float]),
            "or_quantize_q8_0": (None, [p, C.c_int64, p]),
            "or_dequantize_q8_0": (None, [p, C.c_int64, p]),
            "or_philox4x32_10": (None, [p, p, p]),
            "or_uniform": (C.c_double, [u64, u64]),
            "or_sample": (i, [p, i, f, u64, u64]),
            "or_set_threads": (None, [i]),
            "or_get_threads": (i, []),
            "or_matvec": (None, [p, i, i, p, p]),
            "or_matmul_panel": (None, [p, i, i, p, i, p]),
            "or_rmsnorm": (None, [p, p, i, f, p]),
            "or_rope_table": (None, [i, i, C.c_double, p, p]),
            "or_rope": (None, [p, i, i, i, C.c_double]),
            "or_softmax": (None, [p, i]),
            "or_attend_head": (None, [p, p, p, i, i, C.c_int64, p]),
            "or_silu": (C.c_float, [C.c_float]),
            "or_model_create": (p, [C.POINTER(or_desc), i, p, p, p, p]),
            "or_model_free": (None, [p]),
            "or_model_set_kv_bf16": (None, [p, i]),
            "or_lane_create": (p, [p, i]),
            "or_lane_free": (None, [p]),
            "or_lane_reset": (None, [p]),
            "or_lane_pos": (i, [p]),
            "or_lane_export": (None, [p, p, i, i, p]),
            "or_lane_import": (None, [p, p, i, p, p, i]),
            "or_lane_clone": (C.c_int, [p, p]),
            "or_lane_evict": (C.c_int, [p, p, i, i]),
            "or_step": (i, [p, p, i, p]),
            "or_step_batch": (i, [p, p, p, i, p]),
            "or_prefill": (i, [p, p, p, i, p]),
            "or_generate": (i, [p, p, p, i, i, p]),
            "or_generate_batch": (i, [p, p, p, p, i, i, p]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(C.c_void_p)


# ---------------------------------------------------------------- encodings
def f16_to_f32(h: int) -> float:
    return lib().or_f16_to_f32(h)


def f32_to_f16(x: float) -> int:
    return lib().or_f32_to_f16(x)


def f32_to_bf16(x: float) -> int:
    return lib().or_f32_to_bf16(x)


def quantize_q8_0(x: np.ndarray) -> np.ndarray:
    """f32 array (size multiple of 32) -> uint8 blocks [n/32, 34]."""
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    assert x.size % 32 == 0
    out = np.empty((x.size // 32, 34), dtype=np.uint8)
    lib().or_quantize_q8_0(_ptr(x), x.size, _ptr(out))
    return out


def dequantize_q8_0(blocks: np.ndarray) -> np.ndarray:
    blocks = np.ascontiguousarray(blocks, dtype=np.uint8)
    n = blocks.size // 34 * 32
    out = np.empty(n, dtype=np.float32)
    lib().or_dequantize_q8_0(_ptr(blocks), n, _ptr(out))
    return out


def philox4x32_10(ctr, key) -> tuple:
    c = np.asarray(ctr, dtype=np.uint32)
    k = np.asarray(key, dtype=np.uint32)
    o = np.zeros(4, dtype=np.uint32)
    lib().or_philox4x32_10(_ptr(c), _ptr(k), _ptr(o))
    return tuple(int(v) for v in o)


def uniform(seed: int, counter: int) -> float:
    return lib().or_uniform(seed, counter)


def sample(logits: np.ndarray, temp: float = 0.0, seed: int = 0,
           counter: int = 0) -> int:
    lg = np.ascontiguousarray(logits, dtype=np.float32)
    return lib().or_sample(_ptr(lg), lg.size, temp, seed, counter)


def set_threads(n: int) -> None:
    lib().or_set_threads(n)


# ---------------------------------------------------------- building blocks
def matvec(W: np.ndarray, x: np.ndarray) -> np.ndarray:
    W = np.ascontiguousarray(W, dtype=np.float32)
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty(W.shape[0], dtype=np.float32)
    lib().or_matvec(_ptr(W), W.shape[0], W.shape[1], _ptr(x), _ptr(y))
    return y


def matmul_panel(W: np.ndarray, X: np.ndarray) -> np.ndarray:
    W = np.ascontiguousarray(W, dtype=np.float32)
    X = np.ascontiguousarray(X, dtype=np.float32)
    Y = np.empty((X.shape[0], W.shape[0]), dtype=np.float32)
    lib().or_matmul_panel(_ptr(W), W.shape[0], W.shape[1], _ptr(X),
                          X.shape[0], _ptr(Y))
    return Y


def rmsnorm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    g = np.ascontiguousarray(g, dtype=np.float32)
    y = np.empty_like(x)
    lib().or_rmsnorm(_ptr(x), _ptr(g), x.size, eps, _ptr(y))
    return y


def rope_table(pos: int, hd: int, theta: float):
    c = np.empty(hd // 2, dtype=np.float32)
    s = np.empty(hd // 2, dtype=np.float32)
    lib().or_rope_table(pos, hd, theta, _ptr(c), _ptr(s))
    return c, s


def rope(v: np.ndarray, nheads: int, hd: int, pos: int,
         theta: float) -> np.ndarray:
    v = np.array(v, dtype=np.float32, copy=True).reshape(-1)
    lib().or_rope(_ptr(v), nheads, hd, pos, theta)
    return v


def softmax(s: np.ndarray) -> np.ndarray:
    s = np.array(s, dtype=np.float32, copy=True).reshape(-1)
    lib().or_softmax(_ptr(s), s.size)
    return s


def attend_head(q: np.ndarray, K: np.ndarray, V: np.ndarray) -> np.ndarray:
    """q [hd], K/V [n, hd] -> o [hd]."""
    q = np.ascontiguousarray(q, dtype=np.float32)
    K = np.ascontiguousarray(K, dtype=np.float32)
    V = np.ascontiguousarray(V, dtype=np.float32)
    o = np.empty(q.size, dtype=np.float32)
    lib().or_attend_head(_ptr(q), _ptr(K), _ptr(V), K.shape[0], q.size,
                         K.shape[1], _ptr(o))
    return o


def silu(z: float) -> float:
    return lib().or_silu(z)


# -------------------------------------------------------------------- model
LAYER_KEYS = ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down",
              "attn_norm", "ffn_norm")


class Model:
    """Oracle model over host weights.

    ``weights`` is a dict: ``embed`` [V, d], ``lm_head`` [V, d] or None when
    tied, ``final_norm`` [d] f32, ``layers``: list of dicts with LAYER_KEYS.
    Matrices are np.float32, np.uint16 (bf16 bits) or np.uint8 Q8_0 blocks
    [rows*cols/32, 34], matching ``dtype`` (F32, BF16 or Q8_0).
    """

    def __init__(self, cfg: dict, weights: dict, dtype: int, kv_bf16: bool = False):
        self.cfg = dict(cfg)
        d = or_desc(cfg["L"], cfg["d"], cfg["H"], cfg["Hkv"], cfg["hd"],
                    cfg["F"], cfg["V"], cfg["rms_eps"], cfg["rope_theta"],
                    1 if cfg["tied"] else 0)
        self._keep = []

        def p(a):
            if a is None:
                return None
            a = np.ascontiguousarray(a)
            self._keep.append(a)
            return a.ctypes.data_as(C.c_void_p)

        L = cfg["L"]
        arr = (C.c_void_p * (L * 9))()
        for l, ly in enumerate(weights["layers"]):
            for j, k in enumerate(LAYER_KEYS):
                arr[l * 9 + j] = p(ly[k])
        self._h = lib().or_model_create(
            C.byref(d), dtype, p(weights["embed"]),
            p(weights.get("lm_head")), p(weights["final_norm"]), arr)
        self._keep = []  # the oracle keeps its own f32 copies
        self.V = cfg["V"]
        # KV storage of a bf16 arena: keys (roped) and values enter the
        # cache rounded to bf16
        lib().or_model_set_kv_bf16(self._h, 1 if kv_bf16 else 0)

    def __del__(self):
        if getattr(self, "_h", None):
            lib().or_model_free(self._h)
            self._h = None

    def lane(self, max_pos: int) -> "Lane":
        return Lane(self, max_pos)

    def step(self, lane: "Lane", token: int) -> np.ndarray:
        out = np.empty(self.V, dtype=np.float32)
        rc = lib().or_step(self._h, lane._h, int(token), _ptr(out))
        if rc:
            raise RuntimeError("oracle lane full")
        return out

    def step_batch(self, lanes, tokens) -> np.ndarray:
        n = len(lanes)
        arr = (C.c_void_p * n)(*[l._h for l in lanes])
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        out = np.empty((n, self.V), dtype=np.float32)
        rc = lib().or_step_batch(self._h, arr, _ptr(t), n, _ptr(out))
        if rc:
            raise RuntimeError("oracle lane full")
        return out

    def prefill(self, lane: "Lane", tokens) -> np.ndarray:
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        out = np.empty(self.V, dtype=np.float32)
        rc = lib().or_prefill(self._h, lane._h, _ptr(t), t.size, _ptr(out))
        if rc:
            raise RuntimeError("oracle lane full")
        return out

    def generate(self, lane: "Lane", prompt, n_new: int) -> np.ndarray:
        t = np.ascontiguousarray(prompt, dtype=np.int32)
        out = np.empty(n_new, dtype=np.int32)
        rc = lib().or_generate(self._h, lane._h, _ptr(t), t.size, n_new,
                               _ptr(out))
        if rc:
            raise RuntimeError("oracle lane full")
        return out

    def generate_batch(self, lanes, prompts, n_new: int) -> np.ndarray:
        n = len(lanes)
        arr = (C.c_void_p * n)(*[l._h for l in lanes])
        flat = np.ascontiguousarray(np.concatenate(prompts), dtype=np.int32)
        lens = np.array([len(p) for p in prompts], dtype=np.int32)
        out = np.empty((n, n_new), dtype=np.int32)
        rc = lib().or_generate_batch(self._h, arr, _ptr(flat), _ptr(lens), n,
                                     n_new, _ptr(out))
        if rc:
            raise RuntimeError("oracle lane full")
        return out


class Lane:
    """Per-lane oracle KV cache: K (roped), Kraw (un-roped), V, pos."""

    def __init__(self, model: Model, max_pos: int):
        self.model = model
        self._h = lib().or_lane_create(model._h, max_pos)

    def __del__(self):
        if getattr(self, "_h", None):
            lib().or_lane_free(self._h)
            self._h = None

    @property
    def pos(self) -> int:
        return lib().or_lane_pos(self._h)

    def reset(self) -> None:
        lib().or_lane_reset(self._h)

    def export(self, layer: int, which: str) -> np.ndarray:
        c = self.model.cfg
        w = {"K": 0, "Kraw": 1, "V": 2}[which]
        out = np.empty((self.pos, c["Hkv"], c["hd"]), dtype=np.float32)
        lib().or_lane_export(self.model._h, self._h, layer, w, _ptr(out))
        return out

    def clone_from(self, src: "Lane") -> None:
        """This lane becomes a copy of ``src``'s history (Clone)."""
        if lib().or_lane_clone(src._h, self._h):
            raise ValueError("lanes of different max_pos")

    def evict(self, start: int, end: int) -> None:
        """Positions [start, end) leave the cache; later entries move down,
        keys re-roped at their new positions (Evict)."""
        if lib().or_lane_evict(self.model._h, self._h, int(start), int(end)):
            raise ValueError("span outside [0, length]")

    def import_kv(self, layer: int, K: np.ndarray, V: np.ndarray) -> None:
        K = np.ascontiguousarray(K, dtype=np.float32)
        V = np.ascontiguousarray(V, dtype=np.float32)
        lib().or_lane_import(self.model._h, self._h, layer, _ptr(K), _ptr(V),
                             K.shape[0])
