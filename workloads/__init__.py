"""Seeded synthetic workloads shared by the tests, the smoke check and the benchmark.

This module only draws random numbers and lays out shapes; it holds none of the
decode step's arithmetic.  Both the CUDA path and the CPU oracle are fed from it.

Model shapes:
  * ``TINY``   -- 2 layers, hidden 256, 4 query / 2 KV heads of dim 64, 8 experts
    top-2 with expert FFN 128, vocab 1024, RoPE theta 1e4.
  * ``MOE30B`` -- the 30B-total / ~3.3B-active shape of the model described in
    "Inside the megakernel serving engine for North Mini Code" (intro and
    memory-bound paragraphs: 30B total, 3.3B active, BF16): 48 layers, hidden
    2048, 32 query / 4 KV heads of dim 128, 128 experts top-8 with expert FFN
    768, vocab 151936.  RoPE theta 1e4 (the pages give none; with random
    weights it does not change cost).

Workloads (each names its model, batch, lengths and page size):
  * ``tiny_bs1_ctx64``    -- batch 1, 64 cached tokens (seq_len 65), page 16.
  * ``tiny_bs8_ragged``   -- batch 8, lengths U{1..512}, page 16, shuffled pages,
    32 greedy steps with one admit/evict at step 16.
  * ``moe30b_bs1_ctx8k``  -- batch 1, 8192 cached tokens, page 16.
  * ``moe30b_bs1_ctx32k`` / ``_ctx128k`` / ``_ctx256k`` -- batch 1, page 64.
  * ``moe30b_bs64_ragged`` -- batch 64, lengths floor(exp(U(ln 512, ln 32768))),
    tokens uniform over the vocab, Zipf(1.1) router prior, page 16.
  * ``moe30b_bs1_ctx128k_q8`` / ``_ctx256k_q8`` -- batch 1, page 64, over a q8_0
    cache (the reduced-byte variant; not one of the bf16 workloads of the metric).

Random draws (seeds are fixed; each tensor of the model gets seed 1234 + its
index in a fixed tensor list):
  * weights ~ N(0, 0.02) rounded to bf16; RMSNorm gains = 1;
  * tokens: seed 1; lengths: seed 2; page shuffle: seed 3; KV values: seed 4;
    Zipf permutation: seed 5.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

TINY = dict(layers=2, hidden=256, n_q=4, n_kv=2, head_dim=64, n_exp=8, top_k=2, ffn=128, vocab=1024,
            rope_theta=1e4, rms_eps=1e-6, norm_topk=1)
MOE30B = dict(layers=48, hidden=2048, n_q=32, n_kv=4, head_dim=128, n_exp=128, top_k=8, ffn=768, vocab=151936,
              rope_theta=1e4, rms_eps=1e-6, norm_topk=1)

WEIGHT_SEED, TOKEN_SEED, LENGTH_SEED, PAGE_SEED, KV_SEED, ZIPF_SEED = 1234, 1, 2, 3, 4, 5
WEIGHT_STD = 0.02


@dataclass
class Workload:
    name: str
    model: dict
    batch: int
    page_size: int
    lengths: list = field(default_factory=list)   # seq_len per row (includes the token being decoded)
    zipf: float | None = None
    steps: int = 1
    admit_step: int | None = None
    kv_source: str = "random"    # "random": N(0,1) bf16 pages; "prefill": the tests run teacher-forced steps
    kv_q8: bool = False          # the cache holds q8_0 blocks (random codes and scales, see make_kv_q8_random)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def lengths_uniform(batch: int, lo: int, hi: int, seed: int = LENGTH_SEED):
    g = _gen(seed, "cpu")
    return [int(v) for v in torch.randint(lo, hi + 1, (batch,), generator=g)]


def lengths_loguniform(batch: int, lo: int, hi: int, seed: int = LENGTH_SEED):
    g = _gen(seed, "cpu")
    u = torch.rand(batch, generator=g, dtype=torch.float64)
    return [int(math.floor(math.exp(math.log(lo) + float(v) * (math.log(hi) - math.log(lo))))) for v in u]


def get(name: str) -> Workload:
    if name == "tiny_bs1_ctx64":
        return Workload(name, TINY, 1, 16, [65], kv_source="prefill")
    if name == "tiny_bs8_ragged":
        return Workload(name, TINY, 8, 16, lengths_uniform(8, 1, 512), steps=32, admit_step=16, kv_source="prefill")
    if name == "moe30b_bs1_ctx8k":
        return Workload(name, MOE30B, 1, 16, [8192 + 1])
    if name in ("moe30b_bs1_ctx32k", "moe30b_bs1_ctx128k", "moe30b_bs1_ctx256k"):
        ctx = {"moe30b_bs1_ctx32k": 32768, "moe30b_bs1_ctx128k": 131072, "moe30b_bs1_ctx256k": 262144}[name]
        return Workload(name, MOE30B, 1, 64, [ctx + 1])
    if name == "moe30b_bs64_ragged":
        return Workload(name, MOE30B, 64, 16, lengths_loguniform(64, 512, 32768), zipf=1.1)
    if name in ("moe30b_bs1_ctx128k_q8", "moe30b_bs1_ctx256k_q8"):
        ctx = 131072 if "128k" in name else 262144
        return Workload(name, MOE30B, 1, 64, [ctx + 1], kv_q8=True)
    raise KeyError(name)


NAMES = ("tiny_bs1_ctx64", "tiny_bs8_ragged", "moe30b_bs1_ctx8k", "moe30b_bs1_ctx32k", "moe30b_bs1_ctx128k",
         "moe30b_bs1_ctx256k", "moe30b_bs64_ragged", "moe30b_bs1_ctx128k_q8", "moe30b_bs1_ctx256k_q8")


def scaled_model(model: dict, **over) -> dict:
    """A copy of ``model`` with some fields replaced (e.g. fewer layers for a profile capture)."""
    m = dict(model)
    m.update(over)
    return m


# ---------------------------------------------------------------- weights

def weight_shapes(m: dict):
    """The fixed tensor list: (name, layer or None, shape).  Its order defines per-tensor seeds."""
    H, D, Hq, Hkv, E, F, V = m["hidden"], m["head_dim"], m["n_q"], m["n_kv"], m["n_exp"], m["ffn"], m["vocab"]
    out = [("embed", None, (V, H)), ("final_norm", None, (H,)), ("lm_head", None, (V, H))]
    for l in range(m["layers"]):
        out += [("attn_norm", l, (H,)), ("w_qkv", l, ((Hq + 2 * Hkv) * D, H)), ("w_o", l, (H, Hq * D)),
                ("ffn_norm", l, (H,)), ("w_router", l, (E, H)), ("w_gate_up", l, (E, 2 * F, H)),
                ("w_down", l, (E, H, F))]
    return out


def _normal_bf16(shape, seed, device, std=WEIGHT_STD):
    g = _gen(seed, device)
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(-1)
    n = flat.numel()
    step = 1 << 26   # draw in slices to bound the fp32 temporary
    for s in range(0, n, step):
        e = min(n, s + step)
        flat[s:e] = (torch.randn(e - s, generator=g, device=device, dtype=torch.float32) * std).to(torch.bfloat16)
    return out


def make_weights(m: dict, device="cpu", seed: int = WEIGHT_SEED, router_bias=None):
    """Random-init weights of model shape ``m``: a dict with ``embed``, ``final_norm``,
    ``lm_head`` and ``layers`` (a list of per-layer dicts), all bf16 tensors on ``device``."""
    w = {"layers": [dict() for _ in range(m["layers"])]}
    for idx, (name, layer, shape) in enumerate(weight_shapes(m)):
        if name.endswith("norm"):
            t = torch.ones(shape, dtype=torch.bfloat16, device=device)
        else:
            t = _normal_bf16(shape, seed + idx, device)
        if layer is None:
            w[name] = t
        else:
            w["layers"][layer][name] = t
    for l in range(m["layers"]):
        w["layers"][l]["router_bias"] = None if router_bias is None else router_bias[l].to(device)
    return w


def zipf_router_bias(m: dict, s: float = 1.1, seed: int = ZIPF_SEED):
    """Per-layer router bias b[l][e] = ln p(rank_l(e)), p proportional to rank^-s over a
    seeded per-layer permutation of the experts (fp32, [L, E])."""
    g = _gen(seed, "cpu")
    E = m["n_exp"]
    ranks = torch.arange(1, E + 1, dtype=torch.float64)
    p = ranks.pow(-s)
    logp = (p / p.sum()).log()
    out = torch.empty(m["layers"], E, dtype=torch.float32)
    for l in range(m["layers"]):
        perm = torch.randperm(E, generator=g)
        out[l, perm] = logp.to(torch.float32)
    return out


# ---------------------------------------------------------------- step inputs

def make_tokens(batch: int, vocab: int, seed: int = TOKEN_SEED):
    g = _gen(seed, "cpu")
    return torch.randint(0, vocab, (batch,), generator=g, dtype=torch.int64).to(torch.int32)


def pages_needed(lengths, page_size: int) -> int:
    return sum((int(L) + page_size - 1) // page_size for L in lengths)


def make_block_tables(lengths, page_size: int, num_pages: int, max_pages_per_seq: int, seed: int = PAGE_SEED):
    """Shuffled, non-contiguous page assignment: a seeded permutation of the page pool is
    dealt to the rows in order.  Unused table entries are -1.  Returns (tables [B, max_pages]
    int32, free list of the pages left over)."""
    g = _gen(seed, "cpu")
    perm = torch.randperm(num_pages, generator=g).to(torch.int32)
    B = len(lengths)
    bt = torch.full((B, max_pages_per_seq), -1, dtype=torch.int32)
    k = 0
    for b, L in enumerate(lengths):
        n = (int(L) + page_size - 1) // page_size
        if n > max_pages_per_seq or k + n > num_pages:
            raise ValueError("page pool too small for these lengths")
        bt[b, :n] = perm[k:k + n]
        k += n
    return bt, perm[k:].tolist()


def kv_shape(m: dict, num_pages: int, page_size: int):
    """Paged KV cache layout: [L][num_pages][2 (K, V)][Hkv][page_size][D], bf16."""
    return (m["layers"], num_pages, 2, m["n_kv"], page_size, m["head_dim"])


def make_kv_random(m: dict, num_pages: int, page_size: int, device="cpu", seed: int = KV_SEED, used_pages=None):
    """KV cache with every value ~ N(0, 1) rounded to bf16 (keys taken as already rotated).
    ``used_pages`` (a list of page ids) restricts the draw to those pages; the rest are zero."""
    shape = kv_shape(m, num_pages, page_size)
    kv = torch.zeros(shape, dtype=torch.bfloat16, device=device)
    g = _gen(seed, device)
    if used_pages is None:
        flat = kv.view(-1)
        step = 1 << 26
        for s in range(0, flat.numel(), step):
            e = min(flat.numel(), s + step)
            flat[s:e] = torch.randn(e - s, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
        return kv
    idx = torch.tensor(sorted(set(int(p) for p in used_pages)), dtype=torch.int64, device=device)
    per_page = kv[0, 0].numel()
    for l in range(m["layers"]):
        for s in range(0, idx.numel(), 4096):
            sel = idx[s:s + 4096]
            vals = torch.randn(sel.numel() * per_page, generator=g, device=device, dtype=torch.float32)
            kv[l].index_copy_(0, sel, vals.to(torch.bfloat16).view((sel.numel(),) + tuple(kv.shape[2:])))
    return kv


# ---------------------------------------------------------------- q8_0 KV cache layout
# Per layer: an int8 code plane [num_pages][2 (K, V)][Hkv][page_size][D] followed by an f16
# scale plane [num_pages][2][Hkv][page_size][D / 32] (one scale per 32 consecutive values of a
# K or V row).  The pool is a uint8 tensor [L][layer_bytes].

def kv_q8_layer_bytes(m: dict, num_pages: int, page_size: int) -> int:
    n = num_pages * 2 * m["n_kv"] * page_size * m["head_dim"]
    return n + (n // 32) * 2


def kv_q8_planes(layer_u8: torch.Tensor, m: dict, num_pages: int, page_size: int):
    """Views of one layer of a q8_0 pool: (codes int8 [P][2][Hkv][ps][D], scales f16 [P][2][Hkv][ps][D/32])."""
    D, Hkv = m["head_dim"], m["n_kv"]
    n = num_pages * 2 * Hkv * page_size * D
    codes = layer_u8[:n].view(torch.int8).view(num_pages, 2, Hkv, page_size, D)
    scales = layer_u8[n:n + (n // 32) * 2].view(torch.float16).view(num_pages, 2, Hkv, page_size, D // 32)
    return codes, scales


def make_kv_q8_random(m: dict, num_pages: int, page_size: int, device="cpu", seed: int = KV_SEED, used_pages=None):
    """q8_0 pool whose used pages hold random codes, round(N(0, 42^2)) clipped to [-127, 127], and
    random scales U(0.012, 0.024) stored as f16 (decoded values about N(0, 0.76^2)); other pages zero."""
    L = m["layers"]
    lb = kv_q8_layer_bytes(m, num_pages, page_size)
    kv = torch.zeros(L, lb, dtype=torch.uint8, device=device)
    g = _gen(seed, device)
    pages = range(num_pages) if used_pages is None else sorted(set(int(p) for p in used_pages))
    idx = torch.tensor(list(pages), dtype=torch.int64, device=device)
    for l in range(L):
        codes, scales = kv_q8_planes(kv[l], m, num_pages, page_size)
        for s in range(0, idx.numel(), 4096):
            sel = idx[s:s + 4096]
            c = torch.randn((sel.numel(),) + tuple(codes.shape[1:]), generator=g, device=device) * 42.0
            codes.index_copy_(0, sel, c.round().clamp_(-127, 127).to(torch.int8))
            d = torch.rand((sel.numel(),) + tuple(scales.shape[1:]), generator=g, device=device) * 0.012 + 0.012
            scales.index_copy_(0, sel, d.to(torch.float16))
    return kv


def bf16_bits(t: torch.Tensor):
    """Host numpy uint16 view of a bf16 tensor's bits (copies to host if needed)."""
    import numpy as np
    t = t.detach()
    if t.device.type != "cpu":
        t = t.cpu()
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)
