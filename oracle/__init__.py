"""Python side of the CPU oracle (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It loads ``liboracle.so`` (built from
``oracle.cpp`` by :func:`build`) through ctypes and offers:

* the oracle's primitives (GEMV, RMSNorm, RoPE, softmax, top-k, bf16 rounding)
  so that the self-checks in ``tests/`` can pin them;
* :meth:`Oracle.decode_step` -- one whole decode step with every weight in
  host memory (the small configurations);
* :meth:`Oracle.decode_step_lazy` -- the same step driven layer by layer from
  Python, fetching each layer's weights, KV slice and only the routed experts
  through callbacks, for configurations whose weights do not fit in host
  memory.  It calls the same C functions in the same order as
  ``decode_step``; Python only moves buffers.

The forward pass follows "Inside the megakernel serving engine for North Mini
Code" (section "What is a Megakernel?": ordinary GEMMs and ordinary paged
attention), with the readings listed at the top of ``oracle.cpp``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.cpp`` into ``_build/liboracle.so`` (plain g++, OpenMP)."""
    src = os.path.join(_HERE, "oracle.cpp")
    os.makedirs(_BUILD, exist_ok=True)
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(src):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-std=c++17", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
           "-shared", "-fPIC", src, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class Dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "layers", "hidden", "n_q", "n_kv", "head_dim", "n_exp", "top_k", "ffn", "vocab",
        "page_size", "num_pages", "max_pages_per_seq", "norm_topk", "kv_q8")] + [
        ("rope_theta", ctypes.c_double), ("rms_eps", ctypes.c_double)]


class Layer(ctypes.Structure):
    _fields_ = [("attn_norm", ctypes.c_void_p), ("w_qkv", ctypes.c_void_p), ("w_o", ctypes.c_void_p),
                ("ffn_norm", ctypes.c_void_p), ("w_router", ctypes.c_void_p), ("router_bias", ctypes.c_void_p),
                ("w_gate_up", ctypes.c_void_p), ("w_down", ctypes.c_void_p)]


def _bind(lib):
    vp, i32 = ctypes.c_void_p, ctypes.c_int
    for suf in ("f32", "f64"):
        getattr(lib, f"orc_gemv_{suf}").argtypes = [i32, i32, vp, vp, vp]
        getattr(lib, f"orc_rmsnorm_{suf}").argtypes = [i32, vp, vp, ctypes.c_double, vp]
        getattr(lib, f"orc_rope_{suf}").argtypes = [i32, i32, ctypes.c_double, vp]
        getattr(lib, f"orc_softmax_{suf}").argtypes = [i32, vp, vp]
        getattr(lib, f"orc_topk_{suf}").argtypes = [i32, i32, vp, vp]
        getattr(lib, f"orc_embed_{suf}").argtypes = [vp, vp, i32, vp, vp]
        getattr(lib, f"orc_attn_block_{suf}").argtypes = [vp, vp, i32, vp, vp, vp, vp, vp, vp, i32]
        getattr(lib, f"orc_attn_block_{suf}").restype = i32
        getattr(lib, f"orc_route_{suf}").argtypes = [vp, vp, i32, vp, vp, vp, vp, vp]
        getattr(lib, f"orc_moe_{suf}").argtypes = [vp, i32, vp, vp, vp, vp, vp, vp, vp, vp]
        getattr(lib, f"orc_final_{suf}").argtypes = [vp, vp, vp, i32, vp, vp]
        getattr(lib, f"orc_decode_step_{suf}").argtypes = [vp, vp, vp, vp, vp, i32, vp, vp, vp, vp, vp]
        getattr(lib, f"orc_decode_step_{suf}").restype = i32
    lib.orc_f32_to_bf16.argtypes = [ctypes.c_float]
    lib.orc_f32_to_bf16.restype = ctypes.c_uint16
    lib.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
    lib.orc_bf16_to_f32.restype = ctypes.c_float
    lib.orc_f32_to_f16.argtypes = [ctypes.c_float]
    lib.orc_f32_to_f16.restype = ctypes.c_uint16
    lib.orc_f16_to_f32.argtypes = [ctypes.c_uint16]
    lib.orc_f16_to_f32.restype = ctypes.c_float
    lib.orc_q8_quantize.argtypes = [i32, vp, vp, vp]
    return lib


def _load(path: str | None = None):
    """Load (once per path) the oracle library; ``path=None`` builds and loads the default one."""
    global _lib
    with _lock:
        if path is None:
            if _lib is None:
                build()
                _lib = _bind(ctypes.CDLL(_LIB_PATH))
            return _lib
        return _bind(ctypes.CDLL(path))


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _u16(a):
    """View a bf16 payload (numpy uint16/int16 array) as contiguous uint16."""
    a = np.ascontiguousarray(a)
    return a.view(np.uint16) if a.dtype != np.uint16 else a


def make_dims(model: dict, page_size: int, num_pages: int, max_pages_per_seq: int, kv_q8: bool = False) -> Dims:
    """Shape of a step; ``kv_q8`` selects the q8_0 cache (per layer: int8 code plane
    [pages][2][Hkv][page_size][D], then f16 scale plane [pages][2][Hkv][page_size][D/32])."""
    d = Dims()
    for k in ("layers", "hidden", "n_q", "n_kv", "head_dim", "n_exp", "top_k", "ffn", "vocab"):
        setattr(d, k, int(model[k]))
    d.page_size, d.num_pages, d.max_pages_per_seq = int(page_size), int(num_pages), int(max_pages_per_seq)
    d.norm_topk = int(model.get("norm_topk", 1))
    d.kv_q8 = 1 if kv_q8 else 0
    d.rope_theta = float(model["rope_theta"])
    d.rms_eps = float(model["rms_eps"])
    return d


class Oracle:
    """CPU forward step; ``precision`` is ``"f32"`` (parity reference) or ``"f64"`` (self-checks)."""

    def __init__(self, precision: str = "f32", lib_path: str | None = None):
        assert precision in ("f32", "f64")
        self.suf = precision
        self.dt = np.float32 if precision == "f32" else np.float64
        self.lib = _load(lib_path)

    def _fn(self, name):
        return getattr(self.lib, f"orc_{name}_{self.suf}")

    # ---- primitives ----------------------------------------------------
    def gemv(self, W, x):
        W = _u16(W)
        x = np.ascontiguousarray(x, dtype=self.dt)
        y = np.empty(W.shape[0], dtype=self.dt)
        self._fn("gemv")(W.shape[0], W.shape[1], _p(W), _p(x), _p(y))
        return y

    def rmsnorm(self, x, g, eps):
        x = np.ascontiguousarray(x, dtype=self.dt)
        g = _u16(g)
        y = np.empty_like(x)
        self._fn("rmsnorm")(x.size, _p(x), _p(g), float(eps), _p(y))
        return y

    def rope(self, v, pos, theta):
        v = np.array(v, dtype=self.dt, copy=True)
        self._fn("rope")(v.size, int(pos), float(theta), _p(v))
        return v

    def softmax(self, r):
        r = np.ascontiguousarray(r, dtype=self.dt)
        p = np.empty_like(r)
        self._fn("softmax")(r.size, _p(r), _p(p))
        return p

    def topk(self, r, k):
        r = np.ascontiguousarray(r, dtype=self.dt)
        ids = np.empty(k, dtype=np.int32)
        self._fn("topk")(r.size, int(k), _p(r), _p(ids))
        return ids

    def f32_to_bf16(self, f):
        return int(self.lib.orc_f32_to_bf16(float(f)))

    def f32_to_f16(self, f):
        return int(self.lib.orc_f32_to_f16(float(f)))

    def f16_to_f32(self, h):
        return float(self.lib.orc_f16_to_f32(int(h)))

    def q8_quantize(self, x):
        """q8_0 blocks of ``x`` (fp32, length a multiple of 32): (int8 codes, f16 scale bits)."""
        x = np.ascontiguousarray(x, dtype=np.float32).ravel()
        n = x.size // 32
        q = np.empty(n * 32, dtype=np.int8)
        d = np.empty(n, dtype=np.uint16)
        self.lib.orc_q8_quantize(n, _p(x), _p(q), _p(d))
        return q, d

    # ---- whole step, all weights on the host -------------------------------
    @staticmethod
    def _layer_struct(lw: dict, keep: list) -> Layer:
        L = Layer()
        for name in ("attn_norm", "w_qkv", "w_o", "ffn_norm", "w_router", "w_gate_up", "w_down"):
            a = lw.get(name)
            if a is not None:
                a = _u16(a)
                keep.append(a)
                setattr(L, name, a.ctypes.data)
        rb = lw.get("router_bias")
        if rb is not None:
            rb = np.ascontiguousarray(rb, dtype=np.float32)
            keep.append(rb)
            L.router_bias = rb.ctypes.data
        return L

    def decode_step(self, dims: Dims, weights: dict, tokens, seq_lens, block_tables, kv):
        """One decode step.  ``kv`` is updated in place: uint16 bf16 bits [L][P][2][Hkv][ps][D], or
        with ``dims.kv_q8`` a uint8 array holding each layer's q8_0 planes one after the other."""
        keep = []
        layers = (Layer * dims.layers)(*[self._layer_struct(lw, keep) for lw in weights["layers"]])
        tok = np.ascontiguousarray(tokens, dtype=np.int32)
        sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
        bt = np.ascontiguousarray(block_tables, dtype=np.int32)
        assert kv.dtype == (np.uint8 if dims.kv_q8 else np.uint16) and kv.flags.c_contiguous
        emb, fn, head = _u16(weights["embed"]), _u16(weights["final_norm"]), _u16(weights["lm_head"])
        B = tok.size
        logits = np.empty((B, dims.vocab), dtype=self.dt)
        rc = self._fn("decode_step")(ctypes.byref(dims), _p(emb), layers, _p(fn), _p(head), B, _p(tok), _p(sl),
                                     _p(bt), _p(kv), _p(logits))
        if rc != 0:
            raise ValueError(f"oracle decode_step rejected its inputs (code {rc})")
        return logits

    def final(self, dims: Dims, final_norm, lm_head, x):
        """Final RMSNorm and LM head of the residual rows ``x`` ([B, H]); returns [B, vocab]."""
        x = np.ascontiguousarray(x, dtype=self.dt)
        fn, head = _u16(final_norm), _u16(lm_head)
        B = x.shape[0]
        logits = np.empty((B, dims.vocab), dtype=self.dt)
        self._fn("final")(ctypes.byref(dims), _p(fn), _p(head), B, _p(x), _p(logits))
        return logits

    @staticmethod
    def _expert_ptrs(ids, expert):
        """Per (row, slot) of ``ids`` ([B, K], row-major), the addresses of the routed expert's
        gate/up and down matrices; ``expert(e)`` returns that expert's (gate_up, down) arrays,
        which must stay alive while the addresses are used."""
        flat = [int(e) for e in np.asarray(ids).ravel()]
        gu_p = (ctypes.c_void_p * len(flat))(*[expert(e)[0].ctypes.data for e in flat])
        dn_p = (ctypes.c_void_p * len(flat))(*[expert(e)[1].ctypes.data for e in flat])
        return gu_p, dn_p

    # ---- the same step, layer by layer, fetching weights on demand ------------
    def decode_step_lazy(self, dims: Dims, fetch, tokens, seq_lens, block_tables, trace: dict | None = None):
        """Decode step with weights fetched per layer.

        ``fetch`` provides host arrays (bf16 as uint16):
          ``fetch.embed_rows(tokens) -> [B, H]``; ``fetch.layer(l) -> dict`` of the
          non-expert tensors; ``fetch.expert(l, e) -> (gate_up [2F,H], down [H,F])``;
          ``fetch.kv_layer(l) -> [P][2][Hkv][ps][D]`` (a writable copy);
          ``fetch.final() -> (final_norm, lm_head)``.
        ``trace`` (optional dict) receives per-layer router ids/weights/logits.
        """
        tok = np.ascontiguousarray(tokens, dtype=np.int32)
        sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
        bt = np.ascontiguousarray(block_tables, dtype=np.int32)
        B, H, E, K = tok.size, dims.hidden, dims.n_exp, dims.top_k
        rows = _u16(fetch.embed_rows(tok)).reshape(B, H)
        x = np.empty((B, H), dtype=self.dt)
        local_tok = np.arange(B, dtype=np.int32)
        self._fn("embed")(ctypes.byref(dims), _p(rows), B, _p(local_tok), _p(x))
        y = np.empty((B, H), dtype=self.dt)
        r = np.empty((B, E), dtype=self.dt)
        ids = np.empty((B, K), dtype=np.int32)
        wts = np.empty((B, K), dtype=self.dt)
        for l in range(dims.layers):
            keep = []
            L = self._layer_struct(fetch.layer(l), keep)
            kv = fetch.kv_layer(l)
            assert kv.dtype == (np.uint8 if dims.kv_q8 else np.uint16) and kv.flags.c_contiguous
            rc = self._fn("attn_block")(ctypes.byref(dims), ctypes.byref(L), B, _p(x), _p(sl), _p(bt), _p(kv),
                                        None, None, 1)
            if rc != 0:
                raise ValueError(f"oracle attention rejected its inputs (code {rc})")
            self._fn("route")(ctypes.byref(dims), ctypes.byref(L), B, _p(x), _p(y), _p(r), _p(ids), _p(wts))
            if trace is not None:
                trace.setdefault("ids", []).append(ids.copy())
                trace.setdefault("w", []).append(wts.copy())
                trace.setdefault("logits", []).append(r.copy())
            experts = {}
            for e in sorted(set(int(v) for v in ids.ravel())):
                gu, dn = fetch.expert(l, e)
                experts[e] = (_u16(gu), _u16(dn))
            gu_p, dn_p = self._expert_ptrs(ids, lambda e: experts[e])
            self._fn("moe")(ctypes.byref(dims), B, _p(y), _p(ids), _p(wts), gu_p, dn_p, _p(x), None, None)
            del experts, keep, kv
        fn, head = fetch.final()
        return self.final(dims, fn, head, x)

    # ---- one layer's pieces (for per-op traces in the tests) ----------------
    def layer_trace(self, dims: Dims, lw: dict, x, seq_lens, block_tables, kv_layer, append: bool = True):
        """Run one layer on ``x`` ([B,H]); return a dict of every intermediate.  With
        ``append=False`` the cache already holds the current token's k and v (codes written by
        the implementation under test) and attention reads them instead of writing its own."""
        keep = []
        L = self._layer_struct(lw, keep)
        x = np.array(x, dtype=self.dt, copy=True, order="C")
        B, H, E, K, F = x.shape[0], dims.hidden, dims.n_exp, dims.top_k, dims.ffn
        nqkv = (dims.n_q + 2 * dims.n_kv) * dims.head_dim
        sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
        bt = np.ascontiguousarray(block_tables, dtype=np.int32)
        qkv = np.empty((B, nqkv), dtype=self.dt)
        attn = np.empty((B, dims.n_q * dims.head_dim), dtype=self.dt)
        rc = self._fn("attn_block")(ctypes.byref(dims), ctypes.byref(L), B, _p(x), _p(sl), _p(bt), _p(kv_layer),
                                    _p(qkv), _p(attn), 1 if append else 0)
        if rc != 0:
            raise ValueError(f"oracle attention rejected its inputs (code {rc})")
        x_mid = x.copy()
        y = np.empty((B, H), dtype=self.dt)
        r = np.empty((B, E), dtype=self.dt)
        ids = np.empty((B, K), dtype=np.int32)
        wts = np.empty((B, K), dtype=self.dt)
        self._fn("route")(ctypes.byref(dims), ctypes.byref(L), B, _p(x), _p(y), _p(r), _p(ids), _p(wts))
        gu_all, dn_all = _u16(lw["w_gate_up"]), _u16(lw["w_down"])
        gu_p, dn_p = self._expert_ptrs(ids, lambda e: (gu_all[e], dn_all[e]))
        h = np.empty((B, K, F), dtype=self.dt)
        moe_out = np.empty((B, H), dtype=self.dt)
        self._fn("moe")(ctypes.byref(dims), B, _p(y), _p(ids), _p(wts), gu_p, dn_p, _p(x), _p(h), _p(moe_out))
        return dict(qkv=qkv, attn=attn, x_mid=x_mid, y_ffn=y, router_logits=r, ids=ids, w=wts, h=h,
                    moe_out=moe_out, x_out=x)
