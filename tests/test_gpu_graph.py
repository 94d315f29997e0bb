"""A decode step captured as a CUDA graph (mk_graph_create / mk_graph_launch): the host builds
each step's data (tag, lengths, RoPE rows, attention split plan) into pinned staging while the
previous step runs, and each launch is one replay.  Over ten consecutive greedy steps with
growing ragged lengths (rows crossing page boundaries take new pages from the block allocator,
so the block tables' contents change between replays) the replayed step must give logits
bit-identical to the plain step on the same inputs, and within the parity bar of the oracle."""
import numpy as np
import pytest
import torch

import workloads as W
import persistent_moe_decode_megakernel_gb300 as mk
from oracle import Oracle
from tests.gpu_common import check_rows, engine_for, gpu_step, kv_to_device, to_device
from tests.helpers import tiny_setup

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("lens", [[33, 5, 70], [15]])
def test_captured_step_replays_match_plain_steps(lens):
    mk.build()
    s = tiny_setup(W.TINY, lens, extra_pages=2)
    orc = Oracle("f32")
    w_dev = to_device(s["wt"])
    eng = engine_for(s, w_dev)
    B, ps = len(lens), s["page_size"]
    kv_g = kv_to_device(s["kv"])     # the graph's cache
    kv_p = kv_to_device(s["kv"])     # the plain step's cache
    kv_ref = s["kv"].copy()          # the oracle's
    tok = torch.zeros(B, dtype=torch.int32, device="cuda")
    bt = torch.zeros(B, s["max_pages"], dtype=torch.int32, device="cuda")
    logits = torch.zeros(B, W.TINY["vocab"], dtype=torch.float32, device="cuda")
    graph = eng.capture(tok, bt, kv_g, logits)
    order = np.concatenate([s["bt"][b, :-(-L // ps)] for b, L in enumerate(lens)] + [np.array(s["free"], np.int32)])
    pool = mk.KvPool(s["num_pages"], ps, B, s["max_pages"], order=order)
    slots = [pool.admit(L) for L in lens]
    tokens = s["tokens"].copy()
    seq = np.array(lens, dtype=np.int32)
    stream = torch.cuda.current_stream()
    for step in range(10):
        for b in range(B):
            pool.reserve(slots[b], int(seq[b]))
        lens_now, bt_now = pool.fill(slots)
        tok.copy_(torch.from_numpy(tokens))
        bt.copy_(torch.from_numpy(bt_now))
        graph.launch(lens_now, stream)
        torch.cuda.synchronize()
        eng.check()
        got_g = logits.cpu().numpy().copy()
        got_p = gpu_step(eng, tokens, lens_now, bt_now, kv_p)
        assert np.array_equal(got_g.view(np.uint32), got_p.view(np.uint32)), step
        ref = orc.decode_step(s["dims"], s["wn"], tokens, lens_now, bt_now, kv_ref)
        check_rows(got_g, ref)
        tokens = np.argmax(ref, axis=1).astype(np.int32)
        seq = seq + 1
    # the two caches the steps appended to are identical
    assert torch.equal(kv_g.view(torch.int16), kv_p.view(torch.int16))
    graph.close()
    pool.close()
    eng.close()
