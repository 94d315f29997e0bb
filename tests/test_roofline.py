"""The SoL calculator and the byte model against the numbers the page prints
(tests/golden/pages_sol.json, with its citation) and the workload definitions."""
import json
import os

import pytest

import workloads as W
from persistent_moe_decode_megakernel_gb300 import roofline as R

G = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_sol.json")))


def test_sol_reproduces_page_numbers():
    sol = R.sol_tokens_per_s(G["weights_bytes_per_step"] + G["kv_bytes_8k"], G["h100_hbm_bytes_per_s"])
    assert round(sol, -1) == G["sol_tokens_per_s"]                      # ~470
    assert round(G["megakernel_tokens_per_s"] / sol, 2) == G["megakernel_frac_of_sol"]
    assert round(G["vllm_tokens_per_s"] / sol, 2) == G["vllm_frac_of_sol"]
    assert round(G["megakernel_tokens_per_s"] / G["vllm_tokens_per_s"], 2) == G["speedup_vs_vllm"]


def test_byte_model_matches_page_model_size():
    pc = R.param_counts(W.MOE30B)
    assert abs(pc["total"] / G["model_total_params"] - 1) < 0.03            # "30B total"
    # "3.3B active" counts both vocab tables; 6.6 GB of bf16 weights per step
    assert abs(pc["active_with_tables"] / G["model_active_params"] - 1) < 0.03
    assert abs(pc["active_with_tables"] * 2 / G["weights_bytes_per_step"] - 1) < 0.03


def test_step_bytes_bs1_8k():
    b = R.step_bytes(W.MOE30B, [8193])
    assert abs(b["dense"] + b["experts"] + b["head"] - 6.084e9) / 6.084e9 < 1e-3
    assert b["kv_read"] == 8192 * 98304
    assert R.kv_bytes_per_token(W.MOE30B) == 98304
    # "about 25 GB" of bf16 KV at 256K context
    assert 25e9 < 262144 * R.kv_bytes_per_token(W.MOE30B) < 26e9


def test_expert_union_default_and_explicit():
    m = W.MOE30B
    b1 = R.step_bytes(m, [100] * 64)
    assert b1["experts"] == m["layers"] * m["n_exp"] * R.param_counts(m)["per_expert"] * 2
    b2 = R.step_bytes(m, [100] * 64, expert_union=[10] * m["layers"])
    assert b2["experts"] == m["layers"] * 10 * R.param_counts(m)["per_expert"] * 2
