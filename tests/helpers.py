"""Shared test helpers: host copies of the seeded workloads and oracle-driven prefill."""
from __future__ import annotations

import numpy as np
import torch

import workloads as W
from oracle import make_dims


def np_weights(w: dict) -> dict:
    """bf16 torch weights -> dict of numpy uint16 arrays (router_bias stays fp32 / None)."""
    out = {k: W.bf16_bits(v) for k, v in w.items() if k != "layers"}
    out["layers"] = []
    for lw in w["layers"]:
        d = {k: (W.bf16_bits(v) if (v is not None and k != "router_bias") else v) for k, v in lw.items()}
        if d.get("router_bias") is not None:
            d["router_bias"] = d["router_bias"].detach().cpu().numpy().astype(np.float32)
        out["layers"].append(d)
    return out


def tiny_setup(model: dict, lengths, page_size: int = 16, extra_pages: int = 0, seed_tokens: int = 11,
               kv_q8: bool = False):
    """Tiny model + a paged cache whose prefix is filled by teacher-forced oracle steps
    (``kv_q8``: a q8_0 cache, uint8 [L][layer_bytes], quantized by the oracle as it writes).

    Each row b gets ``lengths[b]-1`` random prefix tokens (seeded) decoded one at a
    time by the fp32 oracle; the row's next token is its last drawn token.  Returns
    a dict with host weights, dims, tokens, seq_lens, block tables and the KV cache.
    """
    from oracle import Oracle
    B = len(lengths)
    max_pages = max((L + page_size - 1) // page_size for L in lengths) + extra_pages
    num_pages = W.pages_needed(lengths, page_size) + B * extra_pages + 4
    wt = W.make_weights(model, "cpu")
    wn = np_weights(wt)
    bt, free = W.make_block_tables(lengths, page_size, num_pages, max_pages)
    if kv_q8:
        kv = np.zeros((model["layers"], W.kv_q8_layer_bytes(model, num_pages, page_size)), dtype=np.uint8)
    else:
        kv = np.zeros(W.kv_shape(model, num_pages, page_size), dtype=np.uint16)
    g = torch.Generator().manual_seed(seed_tokens)
    seqs = [torch.randint(0, model["vocab"], (L,), generator=g).numpy().astype(np.int32) for L in lengths]
    dims = make_dims(model, page_size, num_pages, max_pages, kv_q8=kv_q8)
    orc = Oracle("f32")
    # prefill: step t decodes token seqs[b][t] at seq_len t+1 for every row still in its prefix
    Tmax = max(lengths)
    for t in range(Tmax - 1):
        rows = [b for b in range(B) if t < lengths[b] - 1]
        if not rows:
            continue
        tok = np.array([seqs[b][t] for b in rows], dtype=np.int32)
        sl = np.array([t + 1 for _ in rows], dtype=np.int32)
        orc.decode_step(dims, wn, tok, sl, bt.numpy()[rows], kv)
    tokens = np.array([seqs[b][lengths[b] - 1] for b in range(B)], dtype=np.int32)
    return dict(model=model, wt=wt, wn=wn, dims=dims, tokens=tokens, seq_lens=np.array(lengths, dtype=np.int32),
                bt=bt.numpy(), kv=kv, free=free, num_pages=num_pages, max_pages=max_pages, page_size=page_size,
                seqs=seqs, kv_q8=kv_q8)


def rel_l2(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def top2_margin(logits_row):
    s = np.sort(np.asarray(logits_row, dtype=np.float64))
    return float(s[-1] - s[-2])
