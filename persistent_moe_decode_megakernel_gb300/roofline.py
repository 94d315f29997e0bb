"""Algorithmic bytes of one decode step and the HBM speed-of-light (SoL) it implies.

"Inside the megakernel serving engine for North Mini Code" (memory-bound
paragraph) measures decode against SoL = HBM bandwidth / bytes moved per step,
where the bytes are the active weights plus the KV cache read.  This module
counts those bytes for a model shape and a batch:

* every non-expert weight of every layer (norm gains, fused QKV, O-proj,
  router and its bias) -- read once per step whatever the batch;
* the routed experts' gate/up and down matrices, once per distinct expert per
  layer (the *union* of the batch's choices);
* the final norm and the LM head;
* one embedding row per token (a step never reads the whole table);
* the KV read (every cached position of every row, K and V, all layers) and
  the KV append of the new token;
* the fp32 logits written.
"""
from __future__ import annotations


def kv_bytes_per_token(m: dict, kv_q8: bool = False) -> int:
    """Cache bytes of one position over all layers: bf16 K and V, or q8_0 (one int8 per value
    plus an f16 scale per 32 values: 34 bytes per 32 values)."""
    n = m["layers"] * 2 * m["n_kv"] * m["head_dim"]
    return n * 2 if not kv_q8 else n + (n // 32) * 2


def param_counts(m: dict) -> dict:
    H, D, Hq, Hkv, E, F, V, L = (m["hidden"], m["head_dim"], m["n_q"], m["n_kv"], m["n_exp"], m["ffn"],
                                 m["vocab"], m["layers"])
    per_layer_dense = 2 * H + (Hq + 2 * Hkv) * D * H + H * Hq * D + E * H
    per_expert = 3 * F * H
    vocab_tables = 2 * V * H + H      # embedding + LM head + final norm
    total = L * (per_layer_dense + E * per_expert) + vocab_tables
    active_with_tables = L * (per_layer_dense + m["top_k"] * per_expert) + vocab_tables
    return dict(per_layer_dense=per_layer_dense, per_expert=per_expert, total=total,
                active_with_tables=active_with_tables)


def step_bytes(m: dict, seq_lens, expert_union=None, router_bias: bool = False, kv_q8: bool = False) -> dict:
    """Algorithmic bytes for one step.  ``seq_lens`` includes the decoded token.
    ``expert_union``: distinct experts per layer (a list of L ints); defaults to
    min(E, B*k) per layer (exact at batch 1)."""
    H, D, Hq, Hkv, E, F, V, L = (m["hidden"], m["head_dim"], m["n_q"], m["n_kv"], m["n_exp"], m["ffn"],
                                 m["vocab"], m["layers"])
    B = len(seq_lens)
    pc = param_counts(m)
    if expert_union is None:
        expert_union = [min(E, B * m["top_k"])] * L
    dense = L * pc["per_layer_dense"] * 2 + (L * E * 4 if router_bias else 0)
    experts = sum(expert_union) * pc["per_expert"] * 2
    head = (V * H + H) * 2
    embed = B * H * 2
    kvt = kv_bytes_per_token(m, kv_q8)
    kv_read = sum(int(s) - 1 for s in seq_lens) * kvt     # cached positions; the new token comes from registers
    kv_write = B * kvt
    logits = B * V * 4
    total = dense + experts + head + embed + kv_read + kv_write + logits
    return dict(dense=dense, experts=experts, head=head, embed=embed, kv_read=kv_read, kv_write=kv_write,
                logits=logits, total=total)


def sol_tokens_per_s(bytes_per_step: float, hbm_bytes_per_s: float, batch: int = 1) -> float:
    return batch * hbm_bytes_per_s / bytes_per_step
