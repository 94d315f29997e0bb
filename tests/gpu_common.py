"""Helpers for the GPU parity tests: move a host setup to the device, run the
library through its C ABI, and fetch weights lazily for the oracle."""
from __future__ import annotations

import numpy as np
import torch

import workloads as W
import persistent_moe_decode_megakernel_gb300 as mk

# "medium": the 30B head geometry (D=128, 8 query heads per KV head) at a size the
# oracle finishes in seconds, with tiles that span several shared-memory chunks.
MEDIUM = dict(layers=3, hidden=1024, n_q=16, n_kv=2, head_dim=128, n_exp=32, top_k=4, ffn=256, vocab=8192,
              rope_theta=1e4, rms_eps=1e-6, norm_topk=1)

TOL_LOGITS = 1e-2      # relative L2, the problem statement's bar (bf16 weights, fp32 accumulation)
MARGIN = 0.05          # greedy argmax must agree where the oracle's top-1/top-2 margin exceeds this


def to_device(w: dict, dev="cuda"):
    out = {k: v.to(dev) for k, v in w.items() if k != "layers"}
    out["layers"] = [{k: (None if v is None else v.to(dev)) for k, v in lw.items()} for lw in w["layers"]]
    return out


def engine_for(setup: dict, w_dev: dict, max_batch: int = 8, watchdog_ms: int = 0, flags: int = 0):
    return mk.Engine(setup["model"], w_dev, setup["page_size"], setup["num_pages"], max_batch, setup["max_pages"],
                     watchdog_ms=watchdog_ms, flags=flags)


def gpu_step(eng, tokens_np, seq_lens_np, bt_np, kv_dev):
    tok = torch.from_numpy(np.ascontiguousarray(tokens_np, dtype=np.int32)).cuda()
    bt = torch.from_numpy(np.ascontiguousarray(bt_np, dtype=np.int32)).cuda()
    logits = eng.step(tok, seq_lens_np, bt, kv_dev)
    torch.cuda.synchronize()
    eng.check()
    return logits.cpu().numpy()


def kv_to_device(kv_np):
    return torch.from_numpy(kv_np.view(np.int16).copy()).view(torch.bfloat16).cuda()


def route_mismatches(gpu_ids, orc_ids, orc_logits, K):
    """Rows whose expert SET differs; each must be an exact tie at the k-th place."""
    bad, ties = [], []
    for b in range(gpu_ids.shape[0]):
        if set(gpu_ids[b].tolist()) != set(orc_ids[b].tolist()):
            r = np.sort(orc_logits[b].astype(np.float64))[::-1]
            gap = r[K - 1] - r[K]
            (ties if gap <= 1e-4 * max(1.0, np.abs(r).max()) else bad).append((b, gap))
    return bad, ties


def own_topk_mismatches(ids, logits, K):
    """Rows whose routing ids are not exactly the top-k of the same implementation's own router
    logits: the k largest logits in descending order (softmax is monotone, so this is descending
    probability), equal logits taken lower expert index first.  Returns the row indices."""
    bad = []
    for b in range(ids.shape[0]):
        want = np.argsort(-np.asarray(logits[b], dtype=np.float32), kind="stable")[:K]
        if not np.array_equal(np.asarray(ids[b]), want):
            bad.append(b)
    return bad


def expected_appends(orc, dims, wn_layers, x_all, seq_lens, bt, kv_orig):
    """The cache with the oracle's appended k and v codes of every layer, each layer's computed
    from the GPU's own input to that layer (``x_all[2l]``, the engine's residual stream), so that
    a value compared with the GPU's append is one rounding away from it.  (Against an end-to-end
    oracle run, a value whose fp32 k or v lies within the GEMV's rounding error of a rounding
    boundary may round the other way; that allowed one-step difference changes the next layer's
    attention -- exactly, for a row whose attention covers that one position -- and so every
    later layer's input.)"""
    kv = np.array(kv_orig, copy=True)
    for l in range(len(wn_layers)):
        kvl = np.ascontiguousarray(kv_orig[l]).copy()
        orc.layer_trace(dims, wn_layers[l], x_all[2 * l], seq_lens, bt, kvl)
        kv[l] = kvl
    return kv


def check_rows(got, ref, tol=None, margin=None):
    """Per-row logits check: relative L2 of every row within ``tol``, and the same argmax
    wherever the oracle's top-1/top-2 margin exceeds ``margin``.  Returns the rows' errors."""
    from tests.helpers import rel_l2, top2_margin
    tol = TOL_LOGITS if tol is None else tol
    margin = MARGIN if margin is None else margin
    errs = []
    for b in range(ref.shape[0]):
        e = rel_l2(got[b], ref[b])
        assert e <= tol, ("row", b, e)
        if top2_margin(ref[b]) > margin:
            assert int(np.argmax(got[b])) == int(np.argmax(ref[b])), ("argmax", b)
        errs.append(e)
    return errs


class DeviceFetch:
    """Weights and KV of a torch-resident model (any device), copied to host arrays on
    demand (only the layer being computed and only the experts the oracle routed to).
    ``rows`` selects batch rows; their KV pages are gathered into a compact pool, page
    k of the pool being the k-th page of the selected rows in row order, with block
    tables ``self.bt`` that address it."""

    def __init__(self, w_dev: dict, kv_dev, bt_np, seq_lens, rows, page_size, model=None, num_pages=None):
        self.w, self.kv = w_dev, kv_dev
        self.rows = list(rows)
        ps = page_size
        self.page_size = ps
        self.model_for_q8, self.kv_num_pages = model, num_pages   # needed to split a q8_0 pool's planes
        pages = []
        for b in self.rows:
            n = (int(seq_lens[b]) + ps - 1) // ps
            pages.extend(int(p) for p in bt_np[b, :n])
        self.page_ids = torch.tensor(pages, dtype=torch.int64, device=kv_dev.device)
        maxp = max((int(seq_lens[b]) + ps - 1) // ps for b in self.rows)
        self.bt = np.full((len(self.rows), maxp), -1, dtype=np.int32)
        k = 0
        for i, b in enumerate(self.rows):
            n = (int(seq_lens[b]) + ps - 1) // ps
            self.bt[i, :n] = np.arange(k, k + n)
            k += n
        self.num_pages = k
        self.max_pages = maxp

    def embed_rows(self, tok):
        emb = self.w["embed"]
        return W.bf16_bits(emb[torch.as_tensor(tok, dtype=torch.int64, device=emb.device)])

    def layer(self, l):
        lw = self.w["layers"][l]
        d = {k: W.bf16_bits(lw[k]) for k in ("attn_norm", "w_qkv", "w_o", "ffn_norm", "w_router")}
        d["router_bias"] = None if lw.get("router_bias") is None else lw["router_bias"].cpu().numpy()
        return d

    def expert(self, l, e):
        lw = self.w["layers"][l]
        return W.bf16_bits(lw["w_gate_up"][e]), W.bf16_bits(lw["w_down"][e])

    def kv_layer(self, l):
        if self.kv.dtype == torch.uint8:   # q8_0 pool: compact the code plane and the scale plane alike
            m = self.model_for_q8
            codes, scales = W.kv_q8_planes(self.kv[l], m, self.kv_num_pages, self.page_size)
            c = codes.index_select(0, self.page_ids).contiguous().view(torch.uint8).reshape(-1)
            d = scales.index_select(0, self.page_ids).contiguous().view(torch.uint8).reshape(-1)
            return torch.cat([c, d]).cpu().numpy()
        return W.bf16_bits(self.kv[l].index_select(0, self.page_ids))

    def final(self):
        return W.bf16_bits(self.w["final_norm"]), W.bf16_bits(self.w["lm_head"])
