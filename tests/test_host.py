"""Host-side tests of the CUDA library (no GPU needed): it loads and exports every
symbol the headers declare, rejects bad arguments before any launch, builds
plans that cover every tile exactly once in a dependency-respecting order, and
its data dependencies -- each record waiting for the writer tiles of exactly the
tagged words the device reads there -- run to completion without deadlock in the
CPU simulator."""
import ctypes
import os
import re

import numpy as np
import pytest

import workloads as W
import persistent_moe_decode_megakernel_gb300 as mk

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
N_CTAS = 152


@pytest.fixture(scope="module", autouse=True)
def built():
    mk.build()


def _declared():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            names |= set(re.findall(r"^[A-Za-z_][\w \*]*?\b(mk_\w+)\s*\(", src, flags=re.M))
    return names


def test_library_exports_every_declared_symbol():
    names = _declared()
    assert {"mk_create", "mk_decode_step", "mk_destroy", "mk_get_status", "mk_last_error"} <= names
    lib = ctypes.CDLL(mk.LIB_PATH)
    missing = [n for n in sorted(names) if not hasattr(lib, n)]
    assert missing == []
    assert set(mk.EXPORTS) == names


def _cfg(model=W.TINY, ps=16, pages=64, mb=8, mpp=32, **over):
    c = mk.make_config(model, ps, pages, mb, mpp)
    for k, v in over.items():
        setattr(c, k, v)
    return c


@pytest.mark.parametrize("field,value,code", [
    ("hidden", 0, mk.MK_ERR_INVALID_ARG), ("num_layers", -1, mk.MK_ERR_INVALID_ARG),
    ("num_q_heads", 3, mk.MK_ERR_INVALID_ARG), ("top_k", 9, mk.MK_ERR_INVALID_ARG),
    ("head_dim", 96, mk.MK_ERR_UNSUPPORTED), ("max_batch", 65, mk.MK_ERR_UNSUPPORTED),
    ("hidden", 4100, mk.MK_ERR_UNSUPPORTED), ("page_size", 512, mk.MK_ERR_UNSUPPORTED),
    ("norm_topk", 2, mk.MK_ERR_INVALID_ARG), ("flags", 4, mk.MK_ERR_INVALID_ARG),
    ("num_experts", 300, mk.MK_ERR_UNSUPPORTED),
    # a page of 264 positions fits half a ring slot at head_dim 64, but a chunk must hold whole
    # 16-position tiles and two such pages do not fit
    ("page_size", 264, mk.MK_ERR_UNSUPPORTED), ("page_size", 12, mk.MK_ERR_UNSUPPORTED),
])
def test_create_rejects_bad_config(field, value, code):
    c = _cfg(**{field: value})
    ctx = ctypes.c_void_p()
    w = mk.Weights()
    rc = mk.lib().mk_create(ctypes.byref(c), ctypes.byref(w), ctypes.byref(ctx))
    assert rc == code
    assert not ctx.value
    assert mk.lib().mk_last_error().decode() != ""


@pytest.mark.parametrize("ps", [8, 24, 64, 256])
def test_create_accepts_page_sizes_of_whole_tiles(ps):
    # page sizes that are multiples of 8 pass the configuration checks as long as a chunk can
    # hold whole 16-position tiles (at 8 and 24 a tile can span two pages); the call then stops
    # at the missing weights
    c = _cfg(ps=ps)
    ctx = ctypes.c_void_p()
    w = mk.Weights()
    rc = mk.lib().mk_create(ctypes.byref(c), ctypes.byref(w), ctypes.byref(ctx))
    assert rc == mk.MK_ERR_INVALID_ARG, mk.lib().mk_last_error().decode()
    assert "weights" in mk.lib().mk_last_error().decode()
    assert not ctx.value


def test_create_rejects_null_and_misaligned_weights():
    c = _cfg()
    ctx = ctypes.c_void_p()
    w = mk.Weights()
    assert mk.lib().mk_create(ctypes.byref(c), ctypes.byref(w), ctypes.byref(ctx)) == mk.MK_ERR_INVALID_ARG
    lws = (mk.LayerWeights * c.num_layers)()
    for l in range(c.num_layers):
        for n in ("attn_norm", "w_qkv", "w_o", "ffn_norm", "w_router", "w_gate_up", "w_down"):
            setattr(lws[l], n, 4096)
    w.embed, w.final_norm, w.lm_head, w.layers = 4096, 4096, 4096, lws
    lws[1].w_o = 4098   # not 16-byte aligned
    assert mk.lib().mk_create(ctypes.byref(c), ctypes.byref(w), ctypes.byref(ctx)) == mk.MK_ERR_INVALID_ARG
    assert "aligned" in mk.lib().mk_last_error().decode()


def test_step_rejects_null_context():
    sl = np.array([5], dtype=np.int32)
    rc = mk.lib().mk_decode_step(None, 1, None, sl.ctypes.data, None, None, None, None)
    assert rc == mk.MK_ERR_INVALID_ARG
    st = mk.Status()
    assert mk.lib().mk_get_status(None, ctypes.byref(st)) == mk.MK_ERR_INVALID_ARG
    mk.lib().mk_destroy(None)   # NULL is ignored


def _check_static_plan(cfg, n_ctas):
    info, tasks, off = mk.plan_static(cfg, n_ctas)
    m_rows = {2: (cfg.num_q_heads + 2 * cfg.num_kv_heads) * cfg.head_dim, 4: cfg.hidden, 5: cfg.num_experts,
              7: cfg.vocab, 1: cfg.hidden}
    cover = {}
    for i in range(n_ctas):
        lst = tasks[off[i]:off[i + 1]]
        assert lst[-1].op == 8                       # END closes every list
        L = cfg.num_layers
        order = [(-1, 0) if t.op == 1 else (L, 0) if t.op == 7 else (L + 1, 0) if t.op == 8 else (t.layer, t.op)
                 for t in lst]
        assert order == sorted(order)                # topological: layer by layer, phase by phase
        for t in lst:
            if t.op in m_rows:
                cover.setdefault((t.op, t.layer), []).append((t.lo, t.hi))
    for (op, layer), ranges in cover.items():
        ranges.sort()
        assert ranges[0][0] == 0 and ranges[-1][1] == m_rows[op]
        assert all(a[1] == b[0] for a, b in zip(ranges, ranges[1:]))   # each row exactly once
    assert info.n_qkv_tiles == len(cover[(2, 0)]) and info.n_head_tiles == len(cover[(7, cfg.num_layers)])
    return info


def test_static_plan_covers_every_row_once():
    _check_static_plan(_cfg(), N_CTAS)
    _check_static_plan(_cfg(), 7)
    info = _check_static_plan(mk.make_config(W.MOE30B, 16, 1000, 1, 600), N_CTAS)
    assert info.n_qkv_tiles == N_CTAS and info.n_router_tiles == 16   # 8 expert rows per router tile
    assert info.n_down_ranges == N_CTAS
    # engines sized for wide batches spread the router over the blocks: one expert row per tile
    info = _check_static_plan(mk.make_config(W.MOE30B, 16, 1000, 64, 600), N_CTAS)
    assert info.n_router_tiles == 128


@pytest.mark.parametrize("lens", [[65], [1], [16], [17], [512, 1, 33, 200, 16, 15, 100, 7], [8193],
                                  [int(x) for x in np.random.default_rng(7).integers(1, 2000, 64)]])
@pytest.mark.parametrize("model", [W.TINY, W.MOE30B])
def test_attention_plan_covers_pages_once(lens, model):
    cfg = _cfg(model, mb=max(8, len(lens)), mpp=1024, pages=8192) if max(lens) > 512 or len(lens) > 8 \
        else _cfg(model)
    items, off = mk.plan_attention(cfg, N_CTAS, lens)
    ps, Hkv = cfg.page_size, cfg.num_kv_heads
    seen = {}
    for i, it in enumerate(items):
        seen.setdefault((it.b, it.kvh), []).append((it.split, it.nsplit, it.page_lo, it.page_hi, i))
    for b, L in enumerate(lens):
        for h in range(Hkv):
            s = seen[(b, h)]
            npg = (L + ps - 1) // ps
            assert [x[0] for x in s] == list(range(len(s))) and all(x[1] == len(s) for x in s)
            assert s[0][2] == 0 and s[-1][3] == npg and all(a[3] == b_[2] for a, b_ in zip(s, s[1:]))
            assert [x[4] for x in s] == list(range(s[0][4], s[0][4] + len(s)))   # consecutive items
    # CSR over SMs, in order
    assert off[0] == 0 and off[-1] == len(items) and (np.diff(off) >= 0).all()
    loads = [sum(items[j].page_hi - items[j].page_lo for j in range(off[i], off[i + 1])) for i in range(N_CTAS)]
    total = sum(Hkv * ((L + ps - 1) // ps) for L in lens)
    assert sum(loads) == total
    npairs = len(lens) * Hkv
    if npairs <= N_CTAS:
        # one item per block at most; splits follow page counts, so the longest item is no
        # longer than an even cut of all pages over the blocks left after one per pair
        assert (np.diff(off) <= 1).all()
        assert max(loads) <= -(-total // max(1, N_CTAS - npairs))
        for (b, h), s in seen.items():
            sizes = [x[3] - x[2] for x in s]
            assert max(sizes) - min(sizes) <= 1
    else:
        assert max(loads) <= -(-total // N_CTAS)


def _random_routing(cfg, B, seed):
    rng = np.random.default_rng(seed)
    return np.stack([np.stack([rng.choice(cfg.num_experts, cfg.top_k, replace=False) for _ in range(B)])
                     for _ in range(cfg.num_layers)]).astype(np.int32)


@pytest.mark.parametrize("seed", range(6))
def test_simulated_step_completes_tiny(seed):
    cfg = _cfg()
    lens = [65, 1, 300, 17, 16, 512, 2, 90][: 1 + seed % 8]
    r = mk.simulate(cfg, N_CTAS if seed % 2 else 5, lens, _random_routing(cfg, len(lens), seed), seed=seed,
                    lead=1 + seed % 6)
    assert r.finished and not r.deadlocked and r.writes_ok and r.moe_units_ok


def test_simulated_step_completes_30b_shapes():
    cfg = mk.make_config(W.MOE30B, 16, 40000, 64, 2100)
    for B, seed in ((1, 1), (64, 2)):
        lens = W.lengths_loguniform(B, 512, 32768) if B > 1 else [8193]
        r = mk.simulate(cfg, N_CTAS, lens, _random_routing(cfg, B, seed), seed=seed, lead=6)
        assert r.finished and not r.deadlocked and r.writes_ok and r.moe_units_ok
        # every attention item ran
        assert r.tiles_run[3] == len(mk.plan_attention(cfg, N_CTAS, lens)[0]) * cfg.num_layers


@pytest.mark.parametrize("flags", [0, mk.FLAG_NO_DOWN_COPY])
@pytest.mark.parametrize("B", [1, 2, 3])
def test_simulated_moe_paths(B, flags):
    # the small-batch path (B <= 2 with the transposed copy) and the general path both cover
    # every gate/up unit and every down-projection element exactly once, without deadlock
    cfg = mk.make_config(W.MOE30B, 16, 40000, 64, 2100, flags=flags)
    for seed in range(3):
        lens = [8193, 700, 33][:B]
        r = mk.simulate(cfg, N_CTAS, lens, _random_routing(cfg, B, seed), seed=seed, lead=1 + seed)
        assert r.finished and not r.deadlocked and r.writes_ok and r.moe_units_ok


@pytest.mark.parametrize("B", [3, 7, 16])
def test_simulated_wide_batches_hidden_4096(B):
    # at hidden 4096 a register group holds three rows (their staged inputs fill the scratch), so
    # at B = 3 expert runs are streamed in ceil(rows / 3) passes; batches of 5 or more take the
    # tcgen05 path (gate/up runs, (expert, row block) down units, the per-slot sum); every unit is
    # still covered once
    m = W.scaled_model(W.MOE30B, hidden=4096, layers=2)
    cfg = mk.make_config(m, 16, 4000, 16, 200)
    rng = np.random.default_rng(B)
    lens = [int(x) for x in rng.integers(1, 2000, B)]
    r = mk.simulate(cfg, N_CTAS, lens, _random_routing(cfg, B, B), seed=B, lead=3)
    assert r.finished and not r.deadlocked and r.writes_ok and r.moe_units_ok


def test_router_tiles_follow_engine_width():
    # engines sized for batches of 8 or more take one expert row per router tile, smaller ones 8
    for mb, tiles in ((1, 16), (7, 16), (8, 128), (64, 128)):
        info, _, _ = mk.plan_static(mk.make_config(W.MOE30B, 16, 1000, mb, 600), N_CTAS)
        assert info.n_router_tiles == tiles, (mb, info.n_router_tiles)


@pytest.mark.parametrize("seed", range(24))
def test_simulated_step_random_shapes(seed):
    # random widths, expert counts, top-k, head geometry, page sizes, batches (1-64), grid sizes
    # and Zipf-skewed routing: the dependency graph finishes without deadlock, every tile that
    # writes data another SM reads runs exactly once and every MoE unit and down-projection
    # element is covered once
    rng = np.random.default_rng(1000 + seed)
    E = int(rng.choice([8, 32, 128]))
    K = min(int(rng.choice([1, 2, 4, 8])), E)
    nkv, G = int(rng.choice([1, 2, 4])), int(rng.choice([1, 2, 4, 8]))
    m = W.scaled_model(W.TINY, layers=2, hidden=int(rng.choice([256, 1024, 2048, 4096])), n_exp=E, top_k=K,
                       head_dim=int(rng.choice([64, 128])), n_kv=nkv, n_q=nkv * G,
                       ffn=int(rng.choice([128, 256, 768])), vocab=4096)
    B, ps = int(rng.integers(1, 65)), int(rng.choice([16, 64]))
    lens = [int(x) for x in rng.integers(1, 3000, B)]
    pages = [(L + ps - 1) // ps for L in lens]
    cfg = mk.make_config(m, ps, sum(pages) + 4, B, max(pages), flags=int(rng.integers(0, 2)))
    pop = 1.0 / np.arange(1, E + 1) ** 1.1
    perm = rng.permutation(E)
    ids = np.stack([np.stack([perm[rng.choice(E, K, replace=False, p=pop / pop.sum())] for _ in range(B)])
                    for _ in range(m["layers"])]).astype(np.int32)
    r = mk.simulate(cfg, int(rng.choice([7, 33, 152])), lens, ids, seed=seed, lead=int(rng.integers(1, 7)))
    assert r.finished and not r.deadlocked and r.writes_ok and r.moe_units_ok


def test_config_flags_are_checked():
    cfg = _cfg()
    cfg.flags = 4   # no such flag
    with pytest.raises(mk.MkError):
        mk.plan_static(cfg, 8)


def test_simulator_detects_a_missing_producer():
    # a routing table that names an out-of-range expert is rejected up front
    cfg = _cfg()
    bad = _random_routing(cfg, 1, 0)
    bad[0, 0, 0] = 99
    with pytest.raises(mk.MkError):
        mk.simulate(cfg, 8, [5], bad)


def test_graph_calls_check_their_arguments():
    # the captured-step calls reject missing arguments before touching a GPU
    L = mk.lib()
    out = ctypes.c_void_p()
    assert L.mk_graph_create(None, 1, None, None, None, None, ctypes.byref(out)) == mk.MK_ERR_INVALID_ARG
    assert L.mk_graph_launch(None, None, None) == mk.MK_ERR_INVALID_ARG
    L.mk_graph_destroy(None)   # NULL is ignored
