"""The allocation-free attention entry point (mk_paged_attention_noalloc) against
the CPU oracle's attention and against the attention that mk_decode_step itself
computed, through the C ABI.

Callers that cannot call cudaMalloc (code under another framework's allocator,
plug-ins handed only pre-allocated buffers) cannot create a context; this entry
point gives them one layer's paged GQA decode attention using only the
library's fixed device-resident scratch.  The test runs a decode step on a
normal context, takes that step's query vectors (rotated here with the same
fp64-angle RoPE table) and its KV cache after the step (which then holds every
position, the decoded one included), and checks that two calls in a row of the
scratch-only entry point reproduce, within the per-op attention tolerance the
parity tests use, the step's attention output of two layers and the oracle's
attention of those layers (the oracle fed the step's layer input and reading the
same cache, as the per-layer parity checks do).  A block table with entries
outside the pool must be reported through the status word, with those pages
skipped and a row that has no page in range left at zero.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W
import persistent_moe_decode_megakernel_gb300 as mk
from oracle import Oracle
from tests.gpu_common import MEDIUM, engine_for, gpu_step, kv_to_device, to_device
from tests.helpers import rel_l2, tiny_setup

pytestmark = pytest.mark.gpu

ATTN_TOL = 1e-4   # the per-op attention tolerance of tests/test_gpu_parity.py


def _fn():
    f = mk.lib().mk_paged_attention_noalloc
    i32, vp = ctypes.c_int32, ctypes.c_void_p
    f.argtypes = [i32, i32, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp]
    f.restype = ctypes.c_int
    return f


def _rotated_q(qkv, seq_lens, model):
    """q heads of the step's QKV output, NeoX rotate-half at pos = seq_len-1 (fp64 angles, fp32 cos/sin)."""
    Hq, D, theta = model["n_q"], model["head_dim"], model["rope_theta"]
    half = D // 2
    q = qkv[:, :Hq * D].reshape(-1, Hq, D).astype(np.float32)
    out = np.empty_like(q)
    inv = theta ** (-2.0 * np.arange(half) / D)
    for b, L in enumerate(seq_lens):
        ang = (L - 1) * inv
        c = np.cos(ang).astype(np.float32)
        s = np.sin(ang).astype(np.float32)
        a, z = q[b, :, :half], q[b, :, half:]
        out[b, :, :half] = a * c - z * s
        out[b, :, half:] = z * c + a * s
    return np.ascontiguousarray(out)


@pytest.mark.parametrize("model,lens", [(W.TINY, [65, 7, 300, 1]), (MEDIUM, [1000, 65, 1, 17])])
def test_noalloc_attention_matches_decode_step(model, lens):
    mk.build()
    s = tiny_setup(model, lens)
    w_dev = to_device(s["wt"])
    kv_dev = kv_to_device(s["kv"])
    eng = engine_for(s, w_dev)
    gpu_step(eng, s["tokens"], s["seq_lens"], s["bt"], kv_dev)
    f = _fn()
    bt = torch.from_numpy(s["bt"]).cuda()
    sl = np.ascontiguousarray(s["seq_lens"], dtype=np.int32)
    status = torch.full((1,), -99, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    m = s["model"]
    B, Hq, D = len(lens), m["n_q"], m["head_dim"]
    x_all = eng.debug_read("x")
    kv_after = W.bf16_bits(kv_dev)
    orc = Oracle("f32")
    for layer in (0, m["layers"] - 1):      # two calls in a row, sharing the scratch
        q = torch.from_numpy(_rotated_q(eng.debug_read("qkv", layer), lens, m)).cuda()
        out = torch.full((B, Hq * D), float("nan"), dtype=torch.float32, device="cuda")
        kv_layer = kv_dev[layer]
        assert kv_layer.is_contiguous()
        rc = f(B, Hq, m["n_kv"], D, s["page_size"], s["num_pages"], s["max_pages"], q.data_ptr(), sl.ctypes.data,
               bt.data_ptr(), kv_layer.data_ptr(), out.data_ptr(), status.data_ptr(),
               ctypes.c_void_p(stream.cuda_stream))
        assert rc == mk.MK_OK, mk.lib().mk_last_error().decode()
        torch.cuda.synchronize()
        assert int(status.item()) == mk.MK_OK
        got = out.cpu().numpy()
        ref = eng.debug_read("attn", layer)
        err = rel_l2(got, ref)
        assert err < ATTN_TOL, (layer, err)
        tr = orc.layer_trace(s["dims"], s["wn"]["layers"][layer], x_all[2 * layer], s["seq_lens"], s["bt"],
                             np.ascontiguousarray(kv_after[layer]), append=False)
        for b in range(B):
            err = rel_l2(got[b], tr["attn"][b])
            assert err < ATTN_TOL, ("oracle", layer, b, err)
    eng.close()


def test_noalloc_reports_pages_outside_the_pool():
    # The block table is read on the device and every entry is bounds-checked before a page
    # is touched: pages outside 0..num_pages-1 are skipped and reported, never read.
    mk.build()
    s = tiny_setup(W.TINY, [65, 40, 20])
    m = s["model"]
    kv_dev = kv_to_device(s["kv"])
    f = _fn()
    B, Hq, D = 3, m["n_q"], m["head_dim"]
    q = torch.randn(B, Hq, D, generator=torch.Generator().manual_seed(3)).cuda()
    sl = np.ascontiguousarray(s["seq_lens"], dtype=np.int32)
    stream = torch.cuda.current_stream()
    status = torch.full((1,), -99, dtype=torch.int32, device="cuda")

    def call(bt_np):
        out = torch.full((B, Hq * D), float("nan"), dtype=torch.float32, device="cuda")
        bt = torch.from_numpy(np.ascontiguousarray(bt_np, dtype=np.int32)).cuda()
        rc = f(B, Hq, m["n_kv"], D, s["page_size"], s["num_pages"], s["max_pages"], q.data_ptr(), sl.ctypes.data,
               bt.data_ptr(), kv_dev[0].data_ptr(), out.data_ptr(), status.data_ptr(),
               ctypes.c_void_p(stream.cuda_stream))
        assert rc == mk.MK_OK, mk.lib().mk_last_error().decode()
        torch.cuda.synchronize()
        return out.cpu().numpy(), int(status.item())

    good, st = call(s["bt"])
    assert st == mk.MK_OK and np.isfinite(good).all()
    bt = s["bt"].copy()
    bt[0, 1] = s["num_pages"] + 3           # one page of row 0 past the pool
    bt[2, :2] = -1                          # every page of row 2
    bad, st = call(bt)
    assert st == mk.MK_ERR_DEVICE_BOUNDS
    assert np.isfinite(bad).all()
    assert np.array_equal(bad[1].view(np.uint32), good[1].view(np.uint32))   # row 1 untouched
    assert not np.array_equal(bad[0], good[0])                                # row 0 lost a page
    assert np.all(bad[2] == 0.0)                                              # row 2 has no position
    # and the next clean call reports MK_OK again (the error word starts at zero every call)
    again, st = call(s["bt"])
    assert st == mk.MK_OK and np.array_equal(again.view(np.uint32), good.view(np.uint32))


def test_noalloc_rejects_shapes_beyond_its_scratch():
    mk.build()
    f = _fn()
    sl = np.full(64, 5, dtype=np.int32)
    buf = torch.zeros(16, dtype=torch.float32, device="cuda")
    p = buf.data_ptr()
    # 64 rows x 16 KV heads x 8 query heads per KV head x 130 floats > 4 MiB for a single range
    rc = f(64, 128, 16, 128, 16, 8, 1, p, sl.ctypes.data, p, p, p, None, None)
    assert rc == mk.MK_ERR_UNSUPPORTED
    assert "scratch" in mk.lib().mk_last_error().decode()
    rc = f(65, 8, 1, 128, 16, 8, 1, p, sl.ctypes.data, p, p, p, None, None)
    assert rc == mk.MK_ERR_INVALID_ARG
    # positions must stay below 2^30 on the device
    rc = f(1, 8, 1, 128, 64, 8, (1 << 24) + 1, p, sl.ctypes.data, p, p, p, None, None)
    assert rc == mk.MK_ERR_UNSUPPORTED
