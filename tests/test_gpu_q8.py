"""GPU parity of the q8_0 KV cache (MK_FLAG_KV_Q8) against the oracle's q8_0 cache.

The reduced-byte cache of the Kinetic pages (the --cache-type-k/v option and the
paragraph on the quantized cache): keys and values kept as blocks of 32 int8
values with one f16 scale.  The step quantizes this token's k (after RoPE) and v
from their fp32 values, appends codes and scales, and attends over the codes.

Bars: logits of every row within relative L2 1e-2 of the oracle run on the same
q8_0 cache, the argmax where the oracle's margin exceeds 0.05, routing exactly the
top-k of the GPU's own router logits; per layer (each layer fed the GPU's own
input and reading the cache the GPU left) qkv 1e-5, attention 1e-4, x 1e-5.  The
appended codes (the oracle's computed from the GPU's own input to each layer,
tests.gpu_common.expected_appends): the quantizer rounds fp32 k and v that differ
from the oracle's by GEMV rounding, so a code may move by one and a scale by one f16
step; the decoded values must agree within 1.2 quantization steps."""
import numpy as np
import pytest
import torch

import workloads as W
import persistent_moe_decode_megakernel_gb300 as mk
from oracle import Oracle
from tests.gpu_common import (MEDIUM, check_rows, engine_for, expected_appends, gpu_step, own_topk_mismatches,
                              route_mismatches, to_device)
from tests.helpers import rel_l2, tiny_setup

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    mk.build()


def _decoded_token(kv_u8, m, P, ps, layer, page, slot):
    """Decoded K and V [2][Hkv][D] (fp64) and scales [2][Hkv][D/32] of one position of one layer."""
    codes, scales = W.kv_q8_planes(torch.from_numpy(np.ascontiguousarray(kv_u8[layer])), m, P, ps)
    c = codes[page, :, :, slot].numpy().astype(np.float64)
    sc = scales[page, :, :, slot].numpy().astype(np.float64)
    return c * np.repeat(sc, 32, axis=-1), sc, codes[page, :, :, slot].numpy().astype(np.int32), \
        scales[page, :, :, slot].numpy().view(np.uint16).astype(np.int32)


def _parity_q8(model, lens, ps=16, check_layers=True, max_batch=8):
    s = tiny_setup(model, lens, page_size=ps, kv_q8=True)
    m, P = s["model"], s["num_pages"]
    orc = Oracle("f32")
    w_dev = to_device(s["wt"])
    kv_dev = torch.from_numpy(s["kv"].copy()).cuda()
    eng = engine_for(s, w_dev, max_batch=max_batch, flags=mk.FLAG_KV_Q8)
    got = gpu_step(eng, s["tokens"], s["seq_lens"], s["bt"], kv_dev)
    kv_ref = s["kv"].copy()
    ref = orc.decode_step(s["dims"], s["wn"], s["tokens"], s["seq_lens"], s["bt"], kv_ref)
    check_rows(got, ref)
    for l in range(m["layers"]):
        assert not own_topk_mismatches(eng.debug_read("route_ids", l), eng.debug_read("router", l), m["top_k"])
    kv_after = kv_dev.cpu().numpy()
    if check_layers:
        x_all = eng.debug_read("x")
        for l in range(m["layers"]):
            tr = orc.layer_trace(s["dims"], s["wn"]["layers"][l], x_all[2 * l], s["seq_lens"], s["bt"],
                                 np.ascontiguousarray(kv_after[l]), append=False)
            assert rel_l2(eng.debug_read("qkv", l), tr["qkv"]) < 1e-5
            assert rel_l2(eng.debug_read("attn", l), tr["attn"]) < 1e-4, (l, rel_l2(eng.debug_read("attn", l), tr["attn"]))
            assert rel_l2(x_all[2 * l + 1], tr["x_mid"]) < 1e-5
            bad, ties = route_mismatches(eng.debug_read("route_ids", l), tr["ids"], tr["router_logits"], m["top_k"])
            assert not bad
            if not ties:
                assert rel_l2(x_all[2 * l + 2], tr["x_out"]) < 1e-5
    # the appended position of every row and layer
    kv_exp = expected_appends(orc, s["dims"], s["wn"]["layers"], eng.debug_read("x"), s["seq_lens"], s["bt"], s["kv"])
    moved = 0
    for b, L in enumerate(s["seq_lens"]):
        pos = int(L) - 1
        page, slot = int(s["bt"][b, pos // ps]), pos % ps
        for l in range(m["layers"]):
            vg, sg, cg, hg = _decoded_token(kv_after, m, P, ps, l, page, slot)
            vr, sr, cr, hr = _decoded_token(kv_exp, m, P, ps, l, page, slot)
            assert np.all(np.abs(hg - hr) <= 1), (b, l)                 # scales within one f16 step
            assert np.all(np.abs(cg - cr) <= 1), (b, l)                 # codes within one
            step = np.repeat(np.maximum(sg, sr), 32, axis=-1)
            assert np.all(np.abs(vg - vr) <= 1.2 * step + 1e-7), (b, l)
            moved += int((cg != cr).sum())
    print(f"q8 rows {len(lens)}: appended codes that moved by one: {moved}")
    eng.close()
    return got, ref


@pytest.mark.parametrize("lens", [[300], [1], [16], [17], [1000, 65, 1], [40, 3, 70, 1, 17, 33]])
def test_q8_cache_medium(lens):
    # head_dim 128 (the q8_0 path's geometry): single and wide batches, one-token and page-edge
    # lengths, items spanning several 256-position chunks
    _parity_q8(MEDIUM, lens, check_layers=len(lens) <= 3)


@pytest.mark.parametrize("lens", [[300, 700], [64, 1, 129]])
def test_q8_cache_page_64(lens):
    _parity_q8(MEDIUM, lens, ps=64)


def test_q8_cache_wide_batch_tensor_core_path():
    lens = [int(x) for x in np.random.default_rng(23).integers(1, 160, 20)]
    _parity_q8(MEDIUM, lens, check_layers=False, max_batch=24)


def test_q8_flag_needs_head_dim_128():
    s = tiny_setup(W.TINY, [5])
    with pytest.raises(mk.MkError) as e:
        engine_for(s, to_device(s["wt"]), flags=mk.FLAG_KV_Q8)
    assert e.value.code == mk.MK_ERR_UNSUPPORTED
