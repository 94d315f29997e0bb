"""Pins for the CPU oracle: each check ties it to something other than itself.

* brute force: a separately written full-causal-attention forward over the whole
  sequence (``tests/bruteforce.py``, numpy f64, no cache, no paging) must give the
  logits the incremental paged oracle produces step by step;
* paged vs contiguous storage: a shuffled block table must give bit-identical logits;
* one-token attention returns V exactly; special cases E=1/k=1 (dense SwiGLU) and
  k=E (dense soft mixture); softmax and top-k invariants and library routines;
  RoPE identities; the RMSNorm closed form; GEMV against an f64 dot product;
  bf16 rounding against torch's conversion.
"""
import numpy as np
import pytest
import scipy.special
import torch

import workloads as W
from oracle import make_dims
from tests import bruteforce as BF
from tests.helpers import np_weights, rel_l2, tiny_setup


def _model(**over):
    return W.scaled_model(W.TINY, **over)


def _incremental_logits(orc, model, wn, tokens, page_size=16, shuffle=True, seed=3):
    """Decode ``tokens`` one step at a time through the paged oracle; logits of every step."""
    T = len(tokens)
    max_pages = (T + page_size - 1) // page_size
    num_pages = max_pages + 3
    if shuffle:
        bt, _ = W.make_block_tables([T], page_size, num_pages, max_pages, seed=seed)
        bt = bt.numpy()
    else:
        bt = np.arange(max_pages, dtype=np.int32)[None, :]
    dims = make_dims(model, page_size, num_pages, max_pages)
    kv = np.zeros(W.kv_shape(model, num_pages, page_size), dtype=np.uint16)
    out = []
    for t in range(T):
        out.append(orc.decode_step(dims, wn, np.array([tokens[t]], np.int32), np.array([t + 1], np.int32), bt, kv)[0])
    return np.stack(out)


@pytest.fixture(scope="module")
def tiny_w():
    return np_weights(W.make_weights(W.TINY, "cpu"))


def test_incremental_paged_oracle_matches_bruteforce_f64(oracle64, tiny_w):
    tokens = torch.randint(0, W.TINY["vocab"], (40,), generator=torch.Generator().manual_seed(7)).numpy()
    inc = _incremental_logits(oracle64, W.TINY, tiny_w, tokens)
    ref, _ = BF.forward_sequence(W.TINY, tiny_w, tokens)
    assert inc.shape == ref.shape
    err = np.abs(inc - ref).max() / np.abs(ref).max()
    assert err < 1e-9, err


def test_fp32_oracle_close_to_bruteforce(oracle32, tiny_w):
    tokens = torch.randint(0, W.TINY["vocab"], (33,), generator=torch.Generator().manual_seed(8)).numpy()
    inc = _incremental_logits(oracle32, W.TINY, tiny_w, tokens)
    ref, _ = BF.forward_sequence(W.TINY, tiny_w, tokens)
    assert rel_l2(inc, ref) < 1e-4


def test_paged_equals_contiguous_bitwise(oracle32, tiny_w):
    tokens = torch.randint(0, W.TINY["vocab"], (37,), generator=torch.Generator().manual_seed(9)).numpy()
    a = _incremental_logits(oracle32, W.TINY, tiny_w, tokens, shuffle=True)
    b = _incremental_logits(oracle32, W.TINY, tiny_w, tokens, shuffle=False)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_page_size_does_not_change_result(oracle32, tiny_w):
    tokens = torch.randint(0, W.TINY["vocab"], (21,), generator=torch.Generator().manual_seed(10)).numpy()
    a = _incremental_logits(oracle32, W.TINY, tiny_w, tokens, page_size=16)
    b = _incremental_logits(oracle32, W.TINY, tiny_w, tokens, page_size=4)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_one_token_attention_returns_v(oracle32, tiny_w):
    m = W.TINY
    dims = make_dims(m, 16, 2, 1)
    x = np.random.default_rng(0).standard_normal((1, m["hidden"])).astype(np.float32)
    kv = np.zeros(W.kv_shape(dict(m, layers=1), 2, 16), dtype=np.uint16)[0]
    bt = np.array([[1]], dtype=np.int32)
    tr = oracle32.layer_trace(dims, tiny_w["layers"][0], x, [1], bt, kv)
    D, Hq, Hkv = m["head_dim"], m["n_q"], m["n_kv"]
    v = tr["qkv"][0, (Hq + Hkv) * D:].reshape(Hkv, D)
    v_bf16 = BF.round_bf16(v).astype(np.float32)
    attn = tr["attn"][0].reshape(Hq, D)
    for h in range(Hq):
        assert np.array_equal(attn[h], v_bf16[h // (Hq // Hkv)])
    # and the cache now holds exactly those bf16 values at page 1, slot 0
    cached = BF.bf16_to_f64(kv[1, 1, :, 0, :]).astype(np.float32)
    assert np.array_equal(cached, v_bf16)


def test_layer_trace_over_given_codes(oracle32, tiny_w):
    # append=False reads the current token's k and v from the cache instead of writing them: over
    # the codes an appending run left, every intermediate is bit-identical; with one appended v
    # code moved by one bf16 ulp, the one-token row's attention (which is v) moves by exactly that
    m = W.TINY
    dims = make_dims(m, 16, 4, 2)
    rng = np.random.default_rng(12)
    x = rng.standard_normal((2, m["hidden"])).astype(np.float32)
    kv = np.zeros(W.kv_shape(dict(m, layers=1), 4, 16), dtype=np.uint16)[0]
    prefix = rng.standard_normal((2, m["n_kv"], 3, m["head_dim"])).astype(np.float32).view(np.uint32).astype(np.uint64)
    kv[0, :, :, :3, :] = ((prefix + 0x7FFF + ((prefix >> 16) & 1)) >> 16).astype(np.uint16)   # bf16 codes (RNE)
    bt = np.array([[0, 1], [2, 3]], dtype=np.int32)
    a = oracle32.layer_trace(dims, tiny_w["layers"][0], x, [4, 1], bt, kv)   # appends into kv
    b = oracle32.layer_trace(dims, tiny_w["layers"][0], x, [4, 1], bt, kv.copy(), append=False)
    for k in ("qkv", "attn", "x_mid", "router_logits", "h", "x_out"):
        assert np.array_equal(a[k].view(np.uint32), b[k].view(np.uint32)), k
    moved = kv.copy()
    moved[2, 1, 0, 0, 5] += 1                  # row 1 (one token): page 2, V, KV head 0, slot 0, dim 5
    c = oracle32.layer_trace(dims, tiny_w["layers"][0], x, [4, 1], bt, moved, append=False)
    d_attn = c["attn"] - a["attn"]
    G, D = m["n_q"] // m["n_kv"], m["head_dim"]
    want = np.float32(BF.bf16_to_f64(moved[2, 1, 0, 0, 5]) - BF.bf16_to_f64(kv[2, 1, 0, 0, 5]))
    for h in range(m["n_q"]):
        for i in range(D):
            exp = want if (h // G == 0 and i == 5) else 0.0
            assert d_attn[1, h * D + i] == exp
    assert np.array_equal(c["attn"][0], a["attn"][0])


def test_single_expert_reduces_to_dense_swiglu(oracle64):
    m = _model(n_exp=1, top_k=1)
    wn = np_weights(W.make_weights(m, "cpu", seed=99))
    tokens = torch.randint(0, m["vocab"], (18,), generator=torch.Generator().manual_seed(12)).numpy()
    inc = _incremental_logits(oracle64, m, wn, tokens)
    ref, _ = BF.forward_sequence(m, wn, tokens, mlp="dense")
    assert np.abs(inc - ref).max() / np.abs(ref).max() < 1e-9


def test_topk_all_experts_is_soft_mixture(oracle64):
    m = _model(n_exp=4, top_k=4)
    wn = np_weights(W.make_weights(m, "cpu", seed=98))
    tokens = torch.randint(0, m["vocab"], (12,), generator=torch.Generator().manual_seed(13)).numpy()
    inc = _incremental_logits(oracle64, m, wn, tokens)
    ref, _ = BF.forward_sequence(m, wn, tokens, mlp="soft")
    assert np.abs(inc - ref).max() / np.abs(ref).max() < 1e-9


def test_router_bias_enters_routing(oracle64):
    m = _model()
    bias = W.zipf_router_bias(m, 1.1)
    wn = np_weights(W.make_weights(m, "cpu", router_bias=bias))
    tokens = torch.randint(0, m["vocab"], (10,), generator=torch.Generator().manual_seed(14)).numpy()
    inc = _incremental_logits(oracle64, m, wn, tokens)
    ref, _ = BF.forward_sequence(m, wn, tokens, router_bias=bias.numpy())
    assert np.abs(inc - ref).max() / np.abs(ref).max() < 1e-9
    ref_nobias, _ = BF.forward_sequence(m, wn, tokens)
    assert np.abs(inc - ref_nobias).max() > 1e-6   # the bias really changes something


def test_unnormalised_router_weights(oracle64):
    m = _model(norm_topk=0)
    wn = np_weights(W.make_weights(m, "cpu", seed=97))
    tokens = torch.randint(0, m["vocab"], (9,), generator=torch.Generator().manual_seed(15)).numpy()
    inc = _incremental_logits(oracle64, m, wn, tokens)
    ref, _ = BF.forward_sequence(m, wn, tokens)
    assert np.abs(inc - ref).max() / np.abs(ref).max() < 1e-9


def test_gemv_against_f64_dot(oracle32):
    rng = np.random.default_rng(1)
    Wf = rng.standard_normal((64, 2048)).astype(np.float32) * 0.02
    Wb = torch.from_numpy(Wf).to(torch.bfloat16)
    Wu = W.bf16_bits(Wb)
    x = rng.standard_normal(2048).astype(np.float32)
    y = oracle32.gemv(Wu, x)
    W64 = Wb.to(torch.float64).numpy()
    ref = W64 @ x.astype(np.float64)
    scale = np.abs(W64) @ np.abs(x.astype(np.float64))
    assert np.max(np.abs(y - ref) / scale) < 1e-6


def test_gemv_row_col_orientation(oracle64):
    # a transposed operand would mix rows: y[r] must depend only on row r
    Wu = W.bf16_bits(torch.zeros(3, 5, dtype=torch.bfloat16))
    Wu[1, 2] = W.bf16_bits(torch.tensor([2.0], dtype=torch.bfloat16))[0]
    y = oracle64.gemv(Wu, np.array([0, 0, 3.0, 0, 0]))
    assert list(y) == [0.0, 6.0, 0.0]


def test_rmsnorm_closed_form(oracle64):
    H = 256
    g = torch.linspace(0.5, 1.5, H).to(torch.bfloat16)
    gu = W.bf16_bits(g)
    c, eps = 0.37, 1e-6
    y = oracle64.rmsnorm(np.full(H, c), gu, eps)
    want = g.to(torch.float64).numpy() * c / np.sqrt(c * c + eps)
    assert np.allclose(y, want, rtol=1e-14, atol=0)


def test_rope_identities(oracle64):
    rng = np.random.default_rng(2)
    D, theta = 128, 1e4
    q, k = rng.standard_normal(D), rng.standard_normal(D)
    # position 0 is the identity
    assert np.array_equal(oracle64.rope(q, 0, theta), q)
    # rotation keeps the norm (cos/sin are fp32-rounded: |c^2+s^2-1| < 1e-7)
    for pos in (1, 17, 8191, 262143):
        assert abs(np.linalg.norm(oracle64.rope(q, pos, theta)) / np.linalg.norm(q) - 1) < 2e-7
    # q(m).k(n) depends only on m-n
    a = oracle64.rope(q, 100, theta) @ oracle64.rope(k, 90, theta)
    b = oracle64.rope(q, 1010, theta) @ oracle64.rope(k, 1000, theta)
    assert abs(a - b) < 1e-5 * np.linalg.norm(q) * np.linalg.norm(k)
    # complex-number form: (v_i + i v_{i+D/2}) * exp(i * pos * theta^(-2i/D))
    pos = 37
    z = q[:D // 2] + 1j * q[D // 2:]
    ang = pos * theta ** (-2.0 * np.arange(D // 2) / D)
    rot = z * (np.cos(ang).astype(np.float32) + 1j * np.sin(ang).astype(np.float32))
    got = oracle64.rope(q, pos, theta)
    assert np.allclose(got, np.concatenate([rot.real, rot.imag]), rtol=0, atol=1e-12)


def test_softmax_invariants(oracle32, oracle64):
    rng = np.random.default_rng(3)
    r = rng.standard_normal(128) * 3
    p = oracle64.softmax(r)
    assert abs(p.sum() - 1) < 1e-12 and (p >= 0).all()
    assert np.allclose(p, scipy.special.softmax(r), rtol=1e-12, atol=0)
    assert np.allclose(oracle64.softmax(r + 123.0), p, rtol=1e-10, atol=0)
    p32 = oracle32.softmax(r.astype(np.float32))
    assert abs(float(p32.sum()) - 1) < 1e-6


def test_topk_invariants(oracle32):
    rng = np.random.default_rng(4)
    for trial in range(20):
        r = rng.standard_normal(128).astype(np.float32)
        if trial % 2:
            r[rng.integers(0, 128, 10)] = r[5]   # plant exact ties
        k = int(rng.integers(1, 9))
        ids = oracle32.topk(r, k)
        assert list(ids) == list(np.argsort(-r, kind="stable")[:k])
        unsel = np.setdiff1d(np.arange(128), ids)
        assert r[ids].min() >= r[unsel].max()


def test_topk_ties_prefer_lower_index(oracle32):
    r = np.array([0.5, 1.0, 1.0, 0.2, 1.0], dtype=np.float32)
    assert list(oracle32.topk(r, 2)) == [1, 2]


def test_bf16_rounding_matches_torch(oracle32):
    rng = np.random.default_rng(5)
    vals = np.concatenate([rng.standard_normal(2000).astype(np.float32),
                           np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -1 - 2 ** -8, 0.0, -0.0, 1e-40, 3.4e38],
                                    dtype=np.float32)])
    want = W.bf16_bits(torch.from_numpy(vals).to(torch.bfloat16))
    got = np.array([oracle32.f32_to_bf16(v) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, want)
    assert oracle32.f32_to_bf16(1 + 2 ** -8) == 0x3F80        # tie -> even (down)
    assert oracle32.f32_to_bf16(1 + 3 * 2 ** -8) == 0x3F82    # tie -> even (up)


def test_router_weights_sum_to_one(oracle32, tiny_w):
    m = W.TINY
    dims = make_dims(m, 16, 4, 2)
    rng = np.random.default_rng(6)
    x = rng.standard_normal((3, m["hidden"])).astype(np.float32)
    kv = np.zeros(W.kv_shape(dict(m, layers=1), 4, 16), dtype=np.uint16)[0]
    bt = np.array([[0, 1], [2, 3], [1, 0]], dtype=np.int32)
    tr = oracle32.layer_trace(dims, tiny_w["layers"][0], x, [3, 5, 1], bt, kv)
    assert np.allclose(tr["w"].sum(axis=1), 1, atol=1e-6)
    for b in range(3):
        r = tr["router_logits"][b]
        assert list(tr["ids"][b]) == list(np.argsort(-r, kind="stable")[:m["top_k"]])


def test_tiny_prefill_setup_is_deterministic():
    a = tiny_setup(W.TINY, [5, 9])
    b = tiny_setup(W.TINY, [5, 9])
    assert np.array_equal(a["kv"], b["kv"]) and np.array_equal(a["tokens"], b["tokens"])
