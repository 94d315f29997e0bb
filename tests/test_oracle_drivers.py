"""Pins for the oracle's Python drivers against its whole-step C entry point.

``Oracle.decode_step_lazy`` (the oracle of every full-size GPU test) and a chain
of ``Oracle.layer_trace`` calls closed by ``Oracle.final`` (the oracle of every
per-layer GPU check and of the CPU baseline) re-drive the C functions layer by
layer from Python: they map routed experts to weight pointers, fetch layers and
KV pages, and (through ``tests.gpu_common.DeviceFetch``) compact the pages of the
rows they check into a smaller pool with its own block tables.  Each must give
logits BIT-IDENTICAL to ``Oracle.decode_step``, which brute force and the planted
mutants of ``oracle.cpp`` already pin: the same C functions run in the same order
on the same values, and the oracle sums attention over positions in position
order whatever page holds them.  Rows are independent in a decode step, so a
reordered subset of rows must reproduce those rows exactly too.

The cases span the tiny model and the medium one (the 30B head geometry), batches
of 1, 3 and 8 with ragged lengths over shuffled pages, with and without a Zipf
router bias, and both router-weight readings (renormalised over the k, or the raw
softmax).  Two planted mistakes in the drivers' plumbing -- two routed experts'
pointers swapped, and one layer's weights fetched for another -- must be caught
("Image 2" paragraph of the page: MoE work depends on routing, so a wrong expert
or layer mapping changes the step)."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import Oracle, make_dims
from tests.gpu_common import MEDIUM, DeviceFetch
from tests.helpers import np_weights, rel_l2


class HostFetch:
    """Fetch interface of ``Oracle.decode_step_lazy`` over host arrays, without compaction."""

    def __init__(self, wn, kv):
        self.wn, self.kv = wn, kv

    def embed_rows(self, tok):
        return self.wn["embed"][np.asarray(tok, dtype=np.int64)]

    def layer(self, l):
        lw = self.wn["layers"][l]
        return {k: lw[k] for k in ("attn_norm", "w_qkv", "w_o", "ffn_norm", "w_router", "router_bias")}

    def expert(self, l, e):
        lw = self.wn["layers"][l]
        return lw["w_gate_up"][e], lw["w_down"][e]

    def kv_layer(self, l):
        return np.ascontiguousarray(self.kv[l]).copy()

    def final(self):
        return self.wn["final_norm"], self.wn["lm_head"]


def _setup(model, B, zipf, norm_topk, seed):
    m = dict(model, norm_topk=norm_topk)
    bias = W.zipf_router_bias(m, 1.1) if zipf else None
    wt = W.make_weights(m, "cpu", router_bias=bias)
    wn = np_weights(wt)
    ps = 16
    lens = W.lengths_uniform(B, 1, 300, seed=seed)
    max_pages = max((L + ps - 1) // ps for L in lens)
    num_pages = W.pages_needed(lens, ps) + 5
    bt, _ = W.make_block_tables(lens, ps, num_pages, max_pages, seed=seed + 100)
    kv = W.make_kv_random(m, num_pages, ps, "cpu", seed=seed + 200, used_pages=[int(p) for p in bt.flatten() if p >= 0])
    tokens = W.make_tokens(B, m["vocab"], seed=seed + 300).numpy()
    return dict(m=m, wt=wt, wn=wn, ps=ps, lens=np.array(lens, np.int32), bt=bt.numpy(), kv_t=kv,
                kv=W.bf16_bits(kv).copy(), tokens=tokens, num_pages=num_pages, max_pages=max_pages)


CASES = [(name, B, zipf, nt) for name in ("tiny", "medium") for B in (1, 3, 8) for zipf in (False, True)
         for nt in (1, 0)]


def _ids(c):
    return "%s-b%d-%s-norm%d" % (c[0], c[1], "zipf" if c[2] else "plain", c[3])


@pytest.fixture(scope="module")
def orc():
    return Oracle("f32")


@pytest.mark.parametrize("case", CASES, ids=[_ids(c) for c in CASES])
def test_drivers_bit_identical_to_decode_step(orc, case):
    name, B, zipf, nt = case
    s = _setup(W.TINY if name == "tiny" else MEDIUM, B, zipf, nt, seed=17 * B + 3 * zipf + nt)
    m = s["m"]
    dims = make_dims(m, s["ps"], s["num_pages"], s["max_pages"])
    ref = orc.decode_step(dims, s["wn"], s["tokens"], s["lens"], s["bt"], s["kv"].copy())
    assert np.isfinite(ref).all()

    # lazy driver over the caller's pool
    trace = {}
    lazy = orc.decode_step_lazy(dims, HostFetch(s["wn"], s["kv"]), s["tokens"], s["lens"], s["bt"], trace)
    assert np.array_equal(lazy.view(np.uint32), ref.view(np.uint32))
    assert len(trace["ids"]) == m["layers"] and trace["ids"][0].shape == (B, m["top_k"])

    # lazy driver over a compacted pool of a reordered subset of rows (the full-size tests' fetch)
    rows = list(range(B))[::-1] if B > 1 else [0]
    if B > 2:
        rows = rows[:-1]          # leave one row out
    fetch = DeviceFetch(s["wt"], s["kv_t"], s["bt"], s["lens"], rows, s["ps"])
    assert fetch.num_pages == sum((int(s["lens"][b]) + s["ps"] - 1) // s["ps"] for b in rows)
    dsub = make_dims(m, s["ps"], fetch.num_pages, fetch.max_pages)
    sub = orc.decode_step_lazy(dsub, fetch, s["tokens"][rows], s["lens"][rows], fetch.bt)
    assert np.array_equal(sub.view(np.uint32), ref[rows].view(np.uint32))

    # layer-by-layer trace chain closed by the final norm and LM head
    kv = s["kv"].copy()
    x = (s["wn"]["embed"][s["tokens"]].astype(np.uint32) << 16).view(np.float32)
    for l in range(m["layers"]):
        kvl = np.ascontiguousarray(kv[l])
        tr = orc.layer_trace(dims, s["wn"]["layers"][l], x, s["lens"], s["bt"], kvl)
        kv[l] = kvl
        assert np.array_equal(tr["ids"], trace["ids"][l])
        assert np.array_equal(tr["w"].view(np.uint32), trace["w"][l].view(np.uint32))
        assert np.array_equal(tr["router_logits"].view(np.uint32), trace["logits"][l].view(np.uint32))
        x = tr["x_out"]
    chain = orc.final(dims, s["wn"]["final_norm"], s["wn"]["lm_head"], x)
    assert np.array_equal(chain.view(np.uint32), ref.view(np.uint32))


def test_planted_expert_swap_in_lazy_driver_is_caught(orc, monkeypatch):
    s = _setup(W.TINY, 3, False, 1, seed=5)
    dims = make_dims(s["m"], s["ps"], s["num_pages"], s["max_pages"])
    ref = orc.decode_step(dims, s["wn"], s["tokens"], s["lens"], s["bt"], s["kv"].copy())
    good = Oracle._expert_ptrs

    def swapped(ids, expert):
        gu_p, dn_p = good(ids, expert)
        # row 0's first two routed experts trade places (both matrices)
        gu_p[0], gu_p[1] = gu_p[1], gu_p[0]
        dn_p[0], dn_p[1] = dn_p[1], dn_p[0]
        return gu_p, dn_p

    monkeypatch.setattr(Oracle, "_expert_ptrs", staticmethod(swapped))
    bad = orc.decode_step_lazy(dims, HostFetch(s["wn"], s["kv"]), s["tokens"], s["lens"], s["bt"])
    assert rel_l2(bad[0], ref[0]) > 1e-3          # the mistake changes row 0 ...
    assert np.array_equal(bad[1:].view(np.uint32), ref[1:].view(np.uint32))   # ... and nothing else


def test_planted_layer_mixup_in_fetch_is_caught(orc):
    s = _setup(W.TINY, 2, False, 1, seed=6)
    dims = make_dims(s["m"], s["ps"], s["num_pages"], s["max_pages"])
    ref = orc.decode_step(dims, s["wn"], s["tokens"], s["lens"], s["bt"], s["kv"].copy())

    class Mixed(HostFetch):
        def layer(self, l):          # layer 1 runs with layer 0's dense weights
            return super().layer(0)

    bad = orc.decode_step_lazy(dims, Mixed(s["wn"], s["kv"]), s["tokens"], s["lens"], s["bt"])
    assert rel_l2(bad, ref) > 1e-3


@pytest.mark.parametrize("name", ["tiny", "medium"])
def test_drivers_bit_identical_on_the_q8_cache(orc, name):
    # the same three drivers over a q8_0 cache: the compacting fetch moves the code plane and the
    # scale plane of the pages it keeps
    model = W.TINY if name == "tiny" else MEDIUM
    m = dict(model)
    B, ps = 3, 16
    wt = W.make_weights(m, "cpu")
    wn = np_weights(wt)
    lens = W.lengths_uniform(B, 1, 300, seed=41)
    max_pages = max((L + ps - 1) // ps for L in lens)
    P = W.pages_needed(lens, ps) + 5
    bt = W.make_block_tables(lens, ps, P, max_pages, seed=42)[0].numpy()
    kv_t = W.make_kv_q8_random(m, P, ps, "cpu", seed=43, used_pages=[int(p) for p in bt.flatten() if p >= 0])
    kv = kv_t.numpy().copy()
    tokens = W.make_tokens(B, m["vocab"], seed=44).numpy()
    sl = np.array(lens, np.int32)
    dims = make_dims(m, ps, P, max_pages, kv_q8=True)
    ref = orc.decode_step(dims, wn, tokens, sl, bt, kv.copy())
    lazy = orc.decode_step_lazy(dims, HostFetch(wn, kv), tokens, sl, bt)
    assert np.array_equal(lazy.view(np.uint32), ref.view(np.uint32))
    rows = [2, 0]
    fetch = DeviceFetch(wt, kv_t, bt, sl, rows, ps, model=m, num_pages=P)
    dsub = make_dims(m, ps, fetch.num_pages, fetch.max_pages, kv_q8=True)
    sub = orc.decode_step_lazy(dsub, fetch, tokens[rows], sl[rows], fetch.bt)
    assert np.array_equal(sub.view(np.uint32), ref[rows].view(np.uint32))
    x = (wn["embed"][tokens].astype(np.uint32) << 16).view(np.float32)
    kvc = kv.copy()
    for l in range(m["layers"]):
        kvl = np.ascontiguousarray(kvc[l])
        x = orc.layer_trace(dims, wn["layers"][l], x, sl, bt, kvl)["x_out"]
    chain = orc.final(dims, wn["final_norm"], wn["lm_head"], x)
    assert np.array_equal(chain.view(np.uint32), ref.view(np.uint32))
