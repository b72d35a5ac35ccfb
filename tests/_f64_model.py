"""An independent f64 numpy formulation of the dense Llama decode, used only to
pin the f32 oracle end to end on tiny shapes (brute force).

It is written as whole-sequence causal attention with complex-number RoPE and
an explicit KV-head repeat for GQA, so it shares neither structure nor
ordering with the oracle's per-token scalar loops.
"""
import numpy as np


def _norm(x, g, eps):
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * g


def _rope(x, pos, theta):
    # x: [T, nh, hd]; pos: [T]
    hd = x.shape[-1]
    half = hd // 2
    z = x[..., :half] + 1j * x[..., half:]
    ang = pos[:, None] * theta ** (-2.0 * np.arange(half) / hd)
    z = z * np.exp(1j * ang)[:, None, :]
    return np.concatenate([z.real, z.imag], axis=-1)


def _bf16_round(a):
    """Nearest-even bf16 rounding of the values' float32 images (a bf16 KV
    arena's storage), written with integer bit arithmetic."""
    u = np.asarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return r.astype(np.uint32).view(np.float32).astype(np.float64)


def forward_logits(cfg, W, tokens, kv_bf16=False):
    """Logits [T, V] for every position of one sequence (causal). kv_bf16:
    the roped keys and the values are stored rounded to bf16 before any
    query reads them (the storage of a bf16 KV arena)."""
    f = lambda a: np.asarray(a, dtype=np.float64)
    d, H, Hkv, hd = cfg["d"], cfg["H"], cfg["Hkv"], cfg["hd"]
    T = len(tokens)
    pos = np.arange(T, dtype=np.float64)
    x = f(W["embed"])[np.asarray(tokens)]
    mask = np.triu(np.full((T, T), -np.inf), k=1)
    for ly in W["layers"]:
        h = _norm(x, f(ly["attn_norm"]), cfg["rms_eps"])
        q = (h @ f(ly["wq"]).T).reshape(T, H, hd)
        k = (h @ f(ly["wk"]).T).reshape(T, Hkv, hd)
        v = (h @ f(ly["wv"]).T).reshape(T, Hkv, hd)
        q = _rope(q, pos, cfg["rope_theta"])
        k = _rope(k, pos, cfg["rope_theta"])
        if kv_bf16:
            k, v = _bf16_round(k), _bf16_round(v)
        rep = H // Hkv
        k = np.repeat(k, rep, axis=1)  # head h uses kv head h // rep
        v = np.repeat(v, rep, axis=1)
        s = np.einsum("thd,shd->hts", q, k) / np.sqrt(hd) + mask
        p = np.exp(s - s.max(-1, keepdims=True))
        p /= p.sum(-1, keepdims=True)
        o = np.einsum("hts,shd->thd", p, v).reshape(T, H * hd)
        x = x + o @ f(ly["wo"]).T
        h = _norm(x, f(ly["ffn_norm"]), cfg["rms_eps"])
        a = h @ f(ly["w_gate"]).T
        a = a / (1 + np.exp(-a)) * (h @ f(ly["w_up"]).T)
        x = x + a @ f(ly["w_down"]).T
    h = _norm(x, f(W["final_norm"]), cfg["rms_eps"])
    head = W["embed"] if cfg["tied"] else W["lm_head"]
    return h @ f(head).T
