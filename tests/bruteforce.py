"""Brute-force reference used only to pin the oracle.

A separate statement of the same model as the oracle, written the other way
round: the whole token sequence is run at once with full causal attention
over contiguous (unpaged) keys and values, in numpy float64.  It shares no
code with ``oracle/`` and reads no KV cache: keys and values of every position
are recomputed from the token prefix.  The only thing it shares with the
oracle is the list of readings (NeoX RoPE with fp64 angles and fp32 cos/sin,
bf16 rounding of cached k and v, top-k by logit with ties to the lower index,
renormalised router weights).

``mlp`` selects the expert block:
  * ``"moe"``   -- routed top-k SwiGLU experts (the model);
  * ``"dense"`` -- one plain SwiGLU MLP with expert 0's weights (the E=1, k=1
    special case must reduce to this);
  * ``"soft"``  -- every expert weighted by its full softmax probability (the
    k=E special case must reduce to this dense soft mixture).
"""
from __future__ import annotations

import numpy as np


def bf16_to_f64(u16):
    return (np.asarray(u16, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def round_bf16(x):
    """float -> float32 -> bf16 (round to nearest even) -> float64."""
    f = np.asarray(x, dtype=np.float32)
    bits = f.view(np.uint32).astype(np.uint64)
    bits = (bits + 0x7FFF + ((bits >> 16) & 1)) >> 16
    return bf16_to_f64(bits.astype(np.uint16))


def round_q8(x):
    """float -> float32 -> q8_0 blocks of 32 along the last axis -> float64.  The cache reading of
    the Kinetic pages' quantized cache: per block d = max|x| / 127 in float32, kept as IEEE half
    (numpy's conversion); codes x * (1/d) in float32, rounded to the nearest integer with ties away
    from zero; a value reads back as code * d."""
    f = np.asarray(x, dtype=np.float32)
    shp = f.shape
    b = f.reshape(shp[:-1] + (shp[-1] // 32, 32))
    amax = np.abs(b).max(axis=-1, keepdims=True)
    d = (amax / np.float32(127)).astype(np.float32)
    safe = np.where(d != 0, d, np.float32(1)).astype(np.float32)
    inv = np.where(d != 0, np.float32(1) / safe, np.float32(0)).astype(np.float32)
    v = (b * inv).astype(np.float32).astype(np.float64)
    t = np.trunc(v)
    q = np.where(np.abs(v - t) >= 0.5, t + np.sign(v), t)
    return (q * d.astype(np.float16).astype(np.float64)).reshape(shp)


def _rms(x, g, eps):
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * g


def _rope_table(T, D, theta):
    half = D // 2
    inv = theta ** (-2.0 * np.arange(half) / D)
    ang = np.arange(T)[:, None] * inv[None, :]
    return np.cos(ang).astype(np.float32).astype(np.float64), np.sin(ang).astype(np.float32).astype(np.float64)


def _rotate(v, cos, sin):
    # v: [T, heads, D]; pairs (i, i+D/2)
    half = v.shape[-1] // 2
    a, b = v[..., :half], v[..., half:]
    c, s = cos[:, None, :], sin[:, None, :]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def _silu(a):
    return a / (1.0 + np.exp(-a))


def forward_sequence(model: dict, w: dict, tokens, mlp: str = "moe", router_bias=None, kv_round: str = "bf16"):
    """Logits [T, V] for every position of ``tokens`` (causal).  ``kv_round`` is how cached keys
    and values are stored: "bf16" or "q8" (q8_0 blocks along head_dim)."""
    rnd = round_bf16 if kv_round == "bf16" else round_q8
    H, D, Hq, Hkv = model["hidden"], model["head_dim"], model["n_q"], model["n_kv"]
    E, K, F = model["n_exp"], model["top_k"], model["ffn"]
    eps, theta = model["rms_eps"], model["rope_theta"]
    G = Hq // Hkv
    tokens = np.asarray(tokens)
    T = tokens.size
    x = bf16_to_f64(w["embed"])[tokens]                     # [T, H]
    cos, sin = _rope_table(T, D, theta)
    mask = np.triu(np.ones((T, T), dtype=bool), k=1)
    routes = []
    for l, lw in enumerate(w["layers"]):
        y = _rms(x, bf16_to_f64(lw["attn_norm"]), eps)
        qkv = y @ bf16_to_f64(lw["w_qkv"]).T
        q = qkv[:, :Hq * D].reshape(T, Hq, D)
        k = qkv[:, Hq * D:(Hq + Hkv) * D].reshape(T, Hkv, D)
        v = qkv[:, (Hq + Hkv) * D:].reshape(T, Hkv, D)
        q = _rotate(q, cos, sin)
        k = rnd(_rotate(k, cos, sin))
        v = rnd(v)
        o = np.empty((T, Hq, D))
        for h in range(Hq):
            s = (q[:, h, :] @ k[:, h // G, :].T) / np.sqrt(D)
            s = np.where(mask, -np.inf, s)
            p = np.exp(s - s.max(axis=1, keepdims=True))
            p /= p.sum(axis=1, keepdims=True)
            o[:, h, :] = p @ v[:, h // G, :]
        x = x + o.reshape(T, Hq * D) @ bf16_to_f64(lw["w_o"]).T
        y2 = _rms(x, bf16_to_f64(lw["ffn_norm"]), eps)
        gu = bf16_to_f64(lw["w_gate_up"])        # [E, 2F, H]
        dn = bf16_to_f64(lw["w_down"])           # [E, H, F]
        if mlp == "dense":
            h = _silu(y2 @ gu[0, :F].T) * (y2 @ gu[0, F:].T)
            x = x + h @ dn[0].T
            continue
        r = y2 @ bf16_to_f64(lw["w_router"]).T
        if router_bias is not None:
            r = r + np.asarray(router_bias[l], dtype=np.float64)
        p = np.exp(r - r.max(axis=1, keepdims=True))
        p /= p.sum(axis=1, keepdims=True)
        out = np.zeros_like(x)
        if mlp == "soft":
            for e in range(E):
                h = _silu(y2 @ gu[e, :F].T) * (y2 @ gu[e, F:].T)
                out += p[:, e:e + 1] * (h @ dn[e].T)
            x = x + out
            continue
        ids = np.argsort(-r, axis=1, kind="stable")[:, :K]
        routes.append(ids)
        for t in range(T):
            sel = p[t, ids[t]]
            wts = sel / sel.sum() if model.get("norm_topk", 1) else sel
            for j, e in enumerate(ids[t]):
                h = _silu(gu[e, :F] @ y2[t]) * (gu[e, F:] @ y2[t])
                out[t] += wts[j] * (dn[e] @ h)
        x = x + out
    yf = _rms(x, bf16_to_f64(w["final_norm"]), eps)
    return yf @ bf16_to_f64(w["lm_head"]).T, routes
