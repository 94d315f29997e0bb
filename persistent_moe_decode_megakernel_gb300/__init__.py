"""Python binding of the persistent MoE decode megakernel (``libmk.so``).

Argument marshalling only: every step of the decode path runs in the CUDA
library.  The library is built in-tree by :func:`build` (nvcc, sm_103a) and
loaded with ctypes; if it is missing, every entry point raises -- there is no
CPU fallback.  PyTorch is used for device memory and the current stream.

The C ABI is declared in ``include/mk.h`` (step) and ``include/mk_debug.h``
(host-side planning, simulation and inspection).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_HERE)
_CSRC = os.path.join(_HERE, "csrc")
_INC = os.path.join(_ROOT, "include")
# MK_TRACE=1 in the environment selects a separate build that records the per-tile timeline
# (mk_debug_trace); the default build compiles that instrumentation out of the step kernel.
TRACE = os.environ.get("MK_TRACE", "0") == "1"
_BUILD = os.path.join(_HERE, "_build_trace" if TRACE else "_build")
LIB_PATH = os.path.join(_BUILD, "libmk.so")
ARCH = "-gencode=arch=compute_103a,code=sm_103a"

MK_OK, MK_ERR_INVALID_ARG, MK_ERR_CUDA, MK_ERR_OOM = 0, -1, -2, -3
MK_ERR_UNSUPPORTED, MK_ERR_TIMEOUT, MK_ERR_DEVICE_BOUNDS = -4, -5, -6
OPS = {1: "embed", 2: "qkv", 3: "attn", 4: "oproj", 5: "router", 6: "moe", 7: "head", 8: "end"}
WAITS = {0: None, 1: "data", 2: "ring", 3: "route"}   # mk_status.wait
DBG = dict(x=1, qkv=2, attn=3, router=4, route_ids=5, route_w=6, h=7)


class MkError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"mk error {code}: {msg}")
        self.code = code


def _sources():
    return [os.path.join(_CSRC, f) for f in sorted(os.listdir(_CSRC)) if f.endswith((".cu", ".cuh", ".cpp", ".h"))] + [
        os.path.join(_INC, f) for f in sorted(os.listdir(_INC)) if f.endswith(".h")]


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile ``csrc/*.cu`` and ``csrc/*.cpp`` for sm_103a into ``_build/libmk.so``."""
    os.makedirs(_BUILD, exist_ok=True)
    srcs = _sources()
    if not force and os.path.exists(LIB_PATH) and os.path.getmtime(LIB_PATH) >= max(os.path.getmtime(s) for s in srcs):
        return LIB_PATH
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    nvcc = os.path.join(cuda, "bin", "nvcc")
    units = [f for f in sorted(os.listdir(_CSRC)) if f.endswith((".cu", ".cpp"))]
    cmds = []
    objs = []
    for f in units:
        obj = os.path.join(_BUILD, f.rsplit(".", 1)[0] + ".o")
        objs.append(obj)
        src = os.path.join(_CSRC, f)
        if f.endswith(".cu"):
            cmds.append([nvcc, ARCH, "-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", _INC, "-I", _CSRC,
                         "-DMK_TRACE=%d" % TRACE, "-c", src, "-o", obj] + (["-Xptxas", "-v"] if verbose else []))
        else:
            cmds.append(["g++", "-O2", "-std=c++17", "-fPIC", "-Wall", "-I", _INC, "-I", _CSRC, "-I",
                         os.path.join(cuda, "include"), "-DMK_TRACE=%d" % TRACE, "-c", src, "-o", obj])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"build failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        return r.stdout + r.stderr

    with ThreadPoolExecutor(max_workers=len(cmds)) as ex:
        logs = list(ex.map(run, cmds))
    if verbose:
        print("\n".join(logs))
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    run([nvcc, ARCH, "-shared", "-o", tmp] + objs)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


# ---------------------------------------------------------------- ctypes mirror of include/mk.h
class Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("num_layers", "hidden", "num_q_heads", "num_kv_heads", "head_dim",
                                               "num_experts", "top_k", "expert_ffn", "vocab")] + [
        ("rope_theta", ctypes.c_float), ("rms_eps", ctypes.c_float)] + [
        (n, ctypes.c_int32) for n in ("page_size", "num_pages", "max_batch", "max_pages_per_seq", "norm_topk",
                                      "flags")] + [("watchdog_ms", ctypes.c_uint32)]


class LayerWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("attn_norm", "w_qkv", "w_o", "ffn_norm", "w_router", "router_bias",
                                                "w_gate_up", "w_down")]


class Weights(ctypes.Structure):
    _fields_ = [("embed", ctypes.c_void_p), ("final_norm", ctypes.c_void_p), ("lm_head", ctypes.c_void_p),
                ("layers", ctypes.POINTER(LayerWeights))]


class Status(ctypes.Structure):
    _fields_ = [("code", ctypes.c_int32), ("op", ctypes.c_int32), ("layer", ctypes.c_int32), ("cta", ctypes.c_int32),
                ("wait", ctypes.c_uint32), ("observed", ctypes.c_uint32), ("tag", ctypes.c_uint32),
                ("detail", ctypes.c_int32)]


class Task(ctypes.Structure):
    _fields_ = [("op", ctypes.c_uint16), ("layer", ctypes.c_uint16), ("lo", ctypes.c_uint32), ("hi", ctypes.c_uint32),
                ("reserved", ctypes.c_uint32)]


class AttnItem(ctypes.Structure):
    _fields_ = [("b", ctypes.c_uint16), ("kvh", ctypes.c_uint16), ("split", ctypes.c_uint16),
                ("nsplit", ctypes.c_uint16), ("page_lo", ctypes.c_uint32), ("page_hi", ctypes.c_uint32)]


class PlanInfo(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("n_ctas", "n_tasks", "n_qkv_tiles", "n_o_tiles", "n_router_tiles",
                                               "n_head_tiles", "n_embed_tiles", "n_down_ranges", "reserved0",
                                               "reserved1", "reserved2", "n_flags", "max_items")]


class SimResult(ctypes.Structure):
    _fields_ = [("finished", ctypes.c_int32), ("deadlocked", ctypes.c_int32), ("events", ctypes.c_int64),
                ("tiles_run", ctypes.c_int32 * 9), ("writes_ok", ctypes.c_int32),
                ("moe_units_ok", ctypes.c_int32)]


EXPORTS = ("mk_create", "mk_decode_step", "mk_decode_step_greedy", "mk_get_status", "mk_last_error", "mk_destroy", "mk_plan_static",
           "mk_plan_attention", "mk_simulate", "mk_debug_read", "mk_debug_inject_stall", "mk_num_ctas",
           "mk_debug_trace", "mk_debug_trace_read", "mk_paged_attention_noalloc", "mk_kv_pool_create",
           "mk_kv_pool_destroy", "mk_kv_admit", "mk_kv_reserve", "mk_kv_evict", "mk_kv_fill", "mk_kv_free_pages",
           "mk_kv_len", "mk_graph_create", "mk_graph_launch", "mk_graph_destroy")

_lib = None
_lock = threading.Lock()


def lib():
    """The loaded CUDA library.  Raises if it has not been built: there is no fallback."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"CUDA library not built ({LIB_PATH} missing); call build() first")
            L = ctypes.CDLL(LIB_PATH)
            vp, i32, u32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint32
            L.mk_create.argtypes = [ctypes.POINTER(Config), ctypes.POINTER(Weights), ctypes.POINTER(vp)]
            L.mk_decode_step.argtypes = [vp, i32, vp, vp, vp, vp, vp, vp]
            L.mk_decode_step_greedy.argtypes = [vp, i32, vp, vp, vp, vp, vp, vp, vp, vp]
            L.mk_kv_pool_create.argtypes = [i32, i32, i32, i32, vp, ctypes.POINTER(vp)]
            L.mk_kv_pool_destroy.argtypes = [vp]
            L.mk_kv_pool_destroy.restype = None
            L.mk_kv_admit.argtypes = [vp, i32, ctypes.POINTER(i32)]
            L.mk_kv_reserve.argtypes = [vp, i32, i32]
            L.mk_kv_evict.argtypes = [vp, i32]
            L.mk_kv_fill.argtypes = [vp, vp, i32, vp, vp]
            L.mk_kv_free_pages.argtypes = [vp]
            L.mk_kv_len.argtypes = [vp, i32]
            L.mk_get_status.argtypes = [vp, ctypes.POINTER(Status)]
            L.mk_last_error.restype = ctypes.c_char_p
            L.mk_destroy.argtypes = [vp]
            L.mk_destroy.restype = None
            L.mk_plan_static.argtypes = [ctypes.POINTER(Config), i32, ctypes.POINTER(PlanInfo), vp, vp]
            L.mk_plan_attention.argtypes = [ctypes.POINTER(Config), i32, i32, vp, vp, i32, vp, ctypes.POINTER(i32)]
            L.mk_simulate.argtypes = [ctypes.POINTER(Config), i32, i32, vp, vp, ctypes.c_uint64, i32,
                                      ctypes.POINTER(SimResult)]
            L.mk_debug_read.argtypes = [vp, i32, i32, vp, ctypes.c_size_t]
            L.mk_debug_inject_stall.argtypes = [vp, i32, u32]
            L.mk_num_ctas.argtypes = [vp]
            L.mk_graph_create.argtypes = [vp, i32, vp, vp, vp, vp, ctypes.POINTER(vp)]
            L.mk_graph_launch.argtypes = [vp, vp, vp]
            L.mk_graph_destroy.argtypes = [vp]
            L.mk_graph_destroy.restype = None
            L.mk_debug_trace.argtypes = [vp, i32, i32]
            L.mk_debug_trace_read.argtypes = [vp, vp, ctypes.c_size_t]
            _lib = L
    return _lib


def _check(rc):
    if rc != MK_OK:
        raise MkError(rc, lib().mk_last_error().decode())
    return rc


# mk_config.flags: skip the transposed down-projection copy (every batch takes the general MoE path)
FLAG_NO_DOWN_COPY = 1
# mk_config.flags: the KV pool holds q8_0 blocks (uint8 [L][layer_bytes]: codes, then f16 scales)
FLAG_KV_Q8 = 2


def make_config(model: dict, page_size: int, num_pages: int, max_batch: int, max_pages_per_seq: int,
                watchdog_ms: int = 0, flags: int = 0) -> Config:
    c = Config()
    c.num_layers, c.hidden, c.num_q_heads = model["layers"], model["hidden"], model["n_q"]
    c.num_kv_heads, c.head_dim, c.num_experts = model["n_kv"], model["head_dim"], model["n_exp"]
    c.top_k, c.expert_ffn, c.vocab = model["top_k"], model["ffn"], model["vocab"]
    c.rope_theta, c.rms_eps = float(model["rope_theta"]), float(model["rms_eps"])
    c.page_size, c.num_pages, c.max_batch, c.max_pages_per_seq = page_size, num_pages, max_batch, max_pages_per_seq
    c.norm_topk = int(model.get("norm_topk", 1))
    c.flags = int(flags)
    c.watchdog_ms = int(watchdog_ms)
    return c


# ---------------------------------------------------------------- host-side planning (no GPU)
def plan_static(cfg: Config, n_ctas: int):
    info = PlanInfo()
    _check(lib().mk_plan_static(ctypes.byref(cfg), n_ctas, ctypes.byref(info), None, None))
    tasks = (Task * info.n_tasks)()
    off = np.zeros(n_ctas + 1, dtype=np.int32)
    _check(lib().mk_plan_static(ctypes.byref(cfg), n_ctas, ctypes.byref(info), tasks, off.ctypes.data))
    return info, list(tasks), off


def plan_attention(cfg: Config, n_ctas: int, seq_lens):
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    n = ctypes.c_int32(0)
    max_items = n_ctas + sl.size * cfg.num_kv_heads
    items = (AttnItem * max_items)()
    off = np.zeros(n_ctas + 1, dtype=np.int32)
    _check(lib().mk_plan_attention(ctypes.byref(cfg), n_ctas, sl.size, sl.ctypes.data, items, max_items,
                                   off.ctypes.data, ctypes.byref(n)))
    return list(items)[:n.value], off


def simulate(cfg: Config, n_ctas: int, seq_lens, routing_ids, seed: int = 0, lead: int = 6) -> SimResult:
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    ids = np.ascontiguousarray(routing_ids, dtype=np.int32)
    r = SimResult()
    _check(lib().mk_simulate(ctypes.byref(cfg), n_ctas, sl.size, sl.ctypes.data, ids.ctypes.data, seed, lead,
                             ctypes.byref(r)))
    return r


# ---------------------------------------------------------------- paged-KV block allocator
class KvPool:
    """Host-side page bookkeeping for continuous batching (``include/mk_kv.h``): a FIFO free
    list of pool pages and sequence slots, and the step's ``seq_lens`` / block tables."""

    def __init__(self, num_pages: int, page_size: int, max_slots: int, max_pages_per_seq: int, order=None):
        self.page_size, self.max_pages = page_size, max_pages_per_seq
        ptr = ctypes.c_void_p()
        o = None if order is None else np.ascontiguousarray(order, dtype=np.int32)
        _check(lib().mk_kv_pool_create(num_pages, page_size, max_slots, max_pages_per_seq,
                                       None if o is None else o.ctypes.data, ctypes.byref(ptr)))
        self.pool = ptr

    def admit(self, length: int) -> int:
        slot = ctypes.c_int32()
        _check(lib().mk_kv_admit(self.pool, int(length), ctypes.byref(slot)))
        return slot.value

    def reserve(self, slot: int, length: int):
        _check(lib().mk_kv_reserve(self.pool, int(slot), int(length)))

    def evict(self, slot: int):
        _check(lib().mk_kv_evict(self.pool, int(slot)))

    def fill(self, slots):
        sl = np.ascontiguousarray(slots, dtype=np.int32)
        lens = np.zeros(sl.size, dtype=np.int32)
        bt = np.zeros((sl.size, self.max_pages), dtype=np.int32)
        _check(lib().mk_kv_fill(self.pool, sl.ctypes.data, sl.size, lens.ctypes.data, bt.ctypes.data))
        return lens, bt

    def free_pages(self) -> int:
        return lib().mk_kv_free_pages(self.pool)

    def length(self, slot: int) -> int:
        return lib().mk_kv_len(self.pool, int(slot))

    def close(self):
        if self.pool:
            lib().mk_kv_pool_destroy(self.pool)
            self.pool = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ---------------------------------------------------------------- the engine
def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


class Engine:
    """One megakernel context on the current CUDA device.

    ``weights`` is the dict produced by ``workloads.make_weights`` (bf16 CUDA
    tensors; ``router_bias`` fp32 or None).  The tensors are borrowed and must
    outlive the engine (it keeps references).
    """

    def __init__(self, model: dict, weights: dict, page_size: int, num_pages: int, max_batch: int,
                 max_pages_per_seq: int, watchdog_ms: int = 0, flags: int = 0):
        import torch
        self.model = dict(model)
        self.cfg = make_config(model, page_size, num_pages, max_batch, max_pages_per_seq, watchdog_ms, flags)
        self._keep = weights
        L = model["layers"]
        lws = (LayerWeights * L)()
        for l, lw in enumerate(weights["layers"]):
            for name in ("attn_norm", "w_qkv", "w_o", "ffn_norm", "w_router", "w_gate_up", "w_down"):
                t = lw[name]
                assert t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous(), name
                setattr(lws[l], name, t.data_ptr())
            rb = lw.get("router_bias")
            if rb is not None:
                assert rb.is_cuda and rb.dtype == torch.float32 and rb.is_contiguous()
                lws[l].router_bias = rb.data_ptr()
        w = Weights()
        w.embed, w.final_norm, w.lm_head = (weights["embed"].data_ptr(), weights["final_norm"].data_ptr(),
                                            weights["lm_head"].data_ptr())
        w.layers = lws
        self._lws = lws
        self.ctx = ctypes.c_void_p()
        _check(lib().mk_create(ctypes.byref(self.cfg), ctypes.byref(w), ctypes.byref(self.ctx)))
        self.n_ctas = lib().mk_num_ctas(self.ctx)
        self._last_b = 0

    def step(self, tokens, seq_lens, block_tables, kv, logits=None, stream=None, greedy=False):
        """Enqueue one decode step on ``stream`` (default: torch's current stream).

        tokens: int32 CUDA [B]; seq_lens: host int32 sequence [B]; block_tables: int32
        CUDA [B, max_pages_per_seq]; kv: bf16 CUDA cache; logits: fp32 CUDA [B, V] or None.
        Returns the logits, or with ``greedy`` the tuple (logits, next_token int32 [B],
        margin fp32 [B]) selected on the device in the same launch.
        """
        import torch
        sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
        B = sl.size
        assert tokens.is_cuda and tokens.dtype == torch.int32 and tokens.numel() == B and tokens.is_contiguous()
        assert block_tables.is_cuda and block_tables.dtype == torch.int32 and block_tables.is_contiguous()
        assert block_tables.shape[-1] == self.cfg.max_pages_per_seq and block_tables.shape[0] >= B
        kv_dtype = torch.uint8 if (self.cfg.flags & FLAG_KV_Q8) else torch.bfloat16
        assert kv.is_cuda and kv.dtype == kv_dtype and kv.is_contiguous()
        if logits is None:
            logits = torch.empty(B, self.cfg.vocab, dtype=torch.float32, device=tokens.device)
        assert logits.is_cuda and logits.dtype == torch.float32 and logits.is_contiguous()
        if stream is None:
            stream = torch.cuda.current_stream()
        if greedy:
            nxt = torch.empty(B, dtype=torch.int32, device=tokens.device)
            mrg = torch.empty(B, dtype=torch.float32, device=tokens.device)
            _check(lib().mk_decode_step_greedy(self.ctx, B, _ptr(tokens), sl.ctypes.data, _ptr(block_tables),
                                               _ptr(kv), _ptr(logits), _ptr(nxt), _ptr(mrg),
                                               ctypes.c_void_p(stream.cuda_stream)))
            self._last_b = B
            return logits, nxt, mrg
        _check(lib().mk_decode_step(self.ctx, B, _ptr(tokens), sl.ctypes.data, _ptr(block_tables), _ptr(kv),
                                    _ptr(logits), ctypes.c_void_p(stream.cuda_stream)))
        self._last_b = B
        return logits

    def step_raw(self, batch: int, tokens_ptr: int, seq_lens_np, block_tables_ptr: int, kv_ptr: int,
                 logits_ptr: int, stream_ptr: int):
        """The C call with raw device pointers (for callers that manage their own buffers)."""
        sl = np.ascontiguousarray(seq_lens_np, dtype=np.int32)
        _check(lib().mk_decode_step(self.ctx, batch, ctypes.c_void_p(tokens_ptr), sl.ctypes.data,
                                    ctypes.c_void_p(block_tables_ptr), ctypes.c_void_p(kv_ptr),
                                    ctypes.c_void_p(logits_ptr), ctypes.c_void_p(stream_ptr)))

    def capture(self, tokens, block_tables, kv, logits):
        """A CUDA graph of one step over these fixed device buffers (``mk_graph_create``); the
        returned ``StepGraph`` launches it with each step's host lengths."""
        import torch
        B = tokens.numel()
        assert tokens.is_cuda and tokens.dtype == torch.int32 and tokens.is_contiguous()
        assert block_tables.is_cuda and block_tables.dtype == torch.int32 and block_tables.is_contiguous()
        assert logits.is_cuda and logits.dtype == torch.float32 and logits.is_contiguous() and logits.shape[0] == B
        g = ctypes.c_void_p()
        _check(lib().mk_graph_create(self.ctx, B, _ptr(tokens), _ptr(block_tables), _ptr(kv), _ptr(logits),
                                     ctypes.byref(g)))
        self._last_b = B
        return StepGraph(self, g, (tokens, block_tables, kv, logits))

    def status(self) -> dict:
        st = Status()
        rc = lib().mk_get_status(self.ctx, ctypes.byref(st))
        if rc not in (MK_OK, MK_ERR_TIMEOUT, MK_ERR_DEVICE_BOUNDS):
            raise MkError(rc, lib().mk_last_error().decode())
        return dict(code=st.code, op=OPS.get(st.op, st.op), layer=st.layer, cta=st.cta,
                    wait=WAITS.get(st.wait, st.wait), observed=st.observed, tag=st.tag, detail=st.detail)

    def check(self):
        st = self.status()
        if st["code"] != MK_OK:
            raise MkError(st["code"], f"device error {st}")

    def debug_read(self, what: str, layer: int = 0):
        B = self._last_b
        m, c = self.model, self.cfg
        L, H, E, K, F = m["layers"], m["hidden"], m["n_exp"], m["top_k"], m["ffn"]
        nqkv = (m["n_q"] + 2 * m["n_kv"]) * m["head_dim"]
        shapes = dict(x=((2 * L + 1, B, H), np.float32), qkv=((B, nqkv), np.float32),
                      attn=((B, m["n_q"] * m["head_dim"]), np.float32), router=((B, E), np.float32),
                      route_ids=((B, K), np.int32), route_w=((B, K), np.float32), h=((B, K, F), np.float32))
        shape, dt = shapes[what]
        out = np.empty(shape, dtype=dt)
        _check(lib().mk_debug_read(self.ctx, DBG[what], layer, out.ctypes.data, out.nbytes))
        return out

    def trace(self, enable: bool = True, events_per_cta: int = 2048):
        """Record the timeline of the following steps (a library built with MK_TRACE=1 only)."""
        self._trace_cap = events_per_cta if enable else 0
        _check(lib().mk_debug_trace(self.ctx, 1 if enable else 0, events_per_cta))

    def read_trace(self):
        out = np.zeros((self.n_ctas, self._trace_cap, 4), dtype=np.uint64)
        _check(lib().mk_debug_trace_read(self.ctx, out.ctypes.data, out.nbytes))
        return out

    def inject_stall(self, layer: int, watchdog_ms: int = 0):
        _check(lib().mk_debug_inject_stall(self.ctx, layer, watchdog_ms))

    def close(self):
        if self.ctx:
            lib().mk_destroy(self.ctx)
            self.ctx = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class StepGraph:
    """A captured decode step (``mk_graph_*``): ``launch(seq_lens)`` replays it on a stream."""

    def __init__(self, engine, handle, keep):
        self.engine, self.g, self._keep = engine, handle, keep

    def launch(self, seq_lens, stream=None):
        import torch
        sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
        if stream is None:
            stream = torch.cuda.current_stream()
        _check(lib().mk_graph_launch(self.g, sl.ctypes.data, ctypes.c_void_p(stream.cuda_stream)))

    def close(self):
        if self.g:
            lib().mk_graph_destroy(self.g)
            self.g = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
