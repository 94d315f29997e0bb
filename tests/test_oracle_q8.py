"""Pins for the oracle's q8_0 KV cache (the reduced-byte cache of the Kinetic pages: blocks of
32 int8 values with one f16 scale, 34 bytes where f16 takes 64).

* f16 scales: the oracle's fp32 -> f16 conversion equals numpy's IEEE half conversion on
  ties, subnormals, overflow and random values, and f16 -> fp32 is exact for every pattern;
* the block quantizer: codes within [-127, 127] with the largest magnitude at +-127, the
  round-trip error within half a step (plus the f16 rounding of the step), zero blocks,
  sign symmetry, exact scaling by powers of two, and idempotence (quantizing the decoded
  block gives back the same codes and scale);
* attention over the q8 cache: one-token attention returns the decoded V exactly; paged
  and contiguous storage give bit-identical logits; the incremental paged oracle matches a
  separately written full-causal forward whose cached k and v go through the same reading
  of the quantizer (``tests/bruteforce.py``);
* outputs stay close to the bf16 cache's but are not identical (the pages say as much).
"""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import Oracle, make_dims
from tests import bruteforce as BF
from tests.helpers import np_weights, rel_l2


@pytest.fixture(scope="module")
def tiny_w():
    return np_weights(W.make_weights(W.TINY, "cpu"))


def _f16_bits(x):
    with np.errstate(over="ignore"):   # values beyond the f16 range become infinities, as IEEE says
        return np.asarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def test_f16_conversion_matches_ieee_half(oracle32):
    one = np.float32(1.0)
    special = [0.0, -0.0, 1.0, 1 + 2 ** -11, 1 + 3 * 2 ** -11, 1 + 2 ** -11 + 2 ** -23, 65504.0, 65519.0, 65520.0,
               1e6, -1e6, 2 ** -14, 2 ** -24, 2 ** -25, 3 * 2 ** -25, 2 ** -26, 5e-8, 6e-8, 1.5 * 2 ** -24,
               2 ** -14 - 2 ** -25, 0.1, -0.3, 1 / 127, 2.2 / 127]
    rng = np.random.default_rng(0)
    vals = np.concatenate([np.array(special, np.float32),
                           (rng.standard_normal(4000) * np.exp2(rng.uniform(-28, 17, 4000))).astype(np.float32)])
    got = np.array([oracle32.f32_to_f16(float(v)) for v in vals], dtype=np.uint16)
    want = _f16_bits(vals)
    assert np.array_equal(got, want), vals[got != want][:5]
    assert oracle32.f32_to_f16(float(one)) == 0x3C00
    # every finite pattern decodes exactly
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    fin = np.isfinite(pats.view(np.float16))
    dec = np.array([oracle32.f16_to_f32(int(h)) for h in pats[fin]], dtype=np.float32)
    assert np.array_equal(dec.view(np.uint32), pats[fin].view(np.float16).astype(np.float32).view(np.uint32))


def _blocks(rng, n):
    scale = np.exp2(rng.uniform(-10, 6, (n, 1)))
    x = (rng.standard_normal((n, 32)) * scale).astype(np.float32)
    x[0] = 0.0                       # a block of zeros
    x[1, :5] = 0.0                   # zeros inside a block
    x[2] = np.abs(x[2])              # one-signed blocks
    x[3] = -np.abs(x[3])
    return x


def test_q8_block_quantizer_properties(oracle32):
    rng = np.random.default_rng(1)
    x = _blocks(rng, 400)
    q, dbits = oracle32.q8_quantize(x)
    q = q.reshape(-1, 32).astype(np.int32)
    d16 = dbits.view(np.float16).astype(np.float64)[:, None]
    d = (np.abs(x).max(axis=1, keepdims=True) / np.float32(127)).astype(np.float32).astype(np.float64)
    assert np.all(np.abs(q) <= 127)
    assert np.all(q[0] == 0) and dbits[0] == 0
    for b in range(1, len(x)):
        i = int(np.argmax(np.abs(x[b])))
        assert q[b, i] == (127 if x[b, i] > 0 else -127)
    err = np.abs(x.astype(np.float64) - q * d16)
    assert np.all(err <= 0.5 * d * (1 + 2 ** -20) + 127 * np.abs(d16 - d) + 1e-30)
    # sign symmetry and exact scaling by powers of two
    qn, dn = oracle32.q8_quantize(-x)
    assert np.array_equal(qn.reshape(-1, 32).astype(np.int32), -q) and np.array_equal(dn, dbits)
    # (for scales in f16's normal range, where multiplying by 4 is exact in f16 too)
    nrm = np.nonzero((d16[:, 0] >= 2.0 ** -14) & (d16[:, 0] * 4 <= 65504))[0]
    assert len(nrm) > 100
    q4, d4 = oracle32.q8_quantize(x[nrm] * np.float32(4.0))
    assert np.array_equal(q4.reshape(-1, 32).astype(np.int32), q[nrm])
    assert np.array_equal(d4.view(np.float16).astype(np.float64), 4 * d16[nrm, 0])
    # idempotence: the decoded block quantizes to the same codes and scale
    xd = (q * d16).astype(np.float32)
    q2, d2 = oracle32.q8_quantize(xd)
    assert np.array_equal(q2.reshape(-1, 32).astype(np.int32), q) and np.array_equal(d2, dbits)


def _decode_layer(kv_layer_u8, model, num_pages, ps):
    """fp64 K and V [P][2][Hkv][ps][D] of one q8_0 cache layer (code * scale)."""
    codes, scales = W.kv_q8_planes(torch.from_numpy(np.ascontiguousarray(kv_layer_u8)), model, num_pages, ps)
    c = codes.numpy().astype(np.float64)
    s = scales.numpy().astype(np.float64)
    return c * np.repeat(s, 32, axis=-1)


def test_one_token_attention_returns_decoded_v(oracle32, tiny_w):
    m, ps, P = W.TINY, 16, 3
    dims = make_dims(m, ps, P, 1, kv_q8=True)
    kv = np.zeros((m["layers"], W.kv_q8_layer_bytes(m, P, ps)), dtype=np.uint8)
    x = (tiny_w["embed"][[5, 77]].astype(np.uint32) << 16).view(np.float32)
    bt = np.array([[2], [0]], dtype=np.int32)
    kvl = np.ascontiguousarray(kv[0])
    tr = oracle32.layer_trace(dims, tiny_w["layers"][0], x, np.array([1, 1], np.int32), bt, kvl)
    dec = _decode_layer(kvl, m, P, ps)
    D, Hq, Hkv = m["head_dim"], m["n_q"], m["n_kv"]
    for b, page in enumerate((2, 0)):
        for h in range(Hq):
            v = dec[page, 1, h // (Hq // Hkv), 0]
            assert np.array_equal(tr["attn"][b, h * D:(h + 1) * D].astype(np.float64), v)
        # the appended v codes are the quantization of the layer's own fp32 v (round trip bound)
        vraw = tr["qkv"][b, (Hq + Hkv) * D:].reshape(Hkv, D).astype(np.float64)
        for g in range(Hkv):
            blk = vraw[g].reshape(-1, 32)
            dstep = np.abs(blk).max(axis=1, keepdims=True) / 127
            # half a step, plus the f16 rounding of the scale (at most 2^-11 of it, times 127)
            assert np.all(np.abs(blk - dec[page, 1, g, 0].reshape(-1, 32)) <= (0.5 + 127 * 2.0 ** -11) * dstep + 1e-7)


def _incremental(orc, model, wn, tokens, ps=16, shuffle=True, seed=3):
    T = len(tokens)
    mp = (T + ps - 1) // ps
    P = mp + 3
    if shuffle:
        bt = W.make_block_tables([T], ps, P, mp, seed=seed)[0].numpy()
    else:
        bt = np.arange(mp, dtype=np.int32)[None, :]
    dims = make_dims(model, ps, P, mp, kv_q8=True)
    kv = np.zeros((model["layers"], W.kv_q8_layer_bytes(model, P, ps)), dtype=np.uint8)
    return np.stack([orc.decode_step(dims, wn, np.array([tokens[t]], np.int32), np.array([t + 1], np.int32), bt,
                                     kv)[0] for t in range(T)])


def test_q8_paged_equals_contiguous_bitwise(oracle32, tiny_w):
    tokens = torch.randint(0, W.TINY["vocab"], (37,), generator=torch.Generator().manual_seed(9)).numpy()
    a = _incremental(oracle32, W.TINY, tiny_w, tokens, shuffle=True)
    b = _incremental(oracle32, W.TINY, tiny_w, tokens, shuffle=False)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_q8_incremental_matches_bruteforce_f64(oracle64, tiny_w):
    tokens = torch.randint(0, W.TINY["vocab"], (40,), generator=torch.Generator().manual_seed(7)).numpy()
    inc = _incremental(oracle64, W.TINY, tiny_w, tokens)
    ref, _ = BF.forward_sequence(W.TINY, tiny_w, tokens, kv_round="q8")
    err = np.abs(inc - ref).max() / np.abs(ref).max()
    assert err < 1e-9, err


def test_q8_logits_close_to_bf16_but_not_equal(oracle32, tiny_w):
    tokens = torch.randint(0, W.TINY["vocab"], (64,), generator=torch.Generator().manual_seed(11)).numpy()
    q8 = _incremental(oracle32, W.TINY, tiny_w, tokens)
    T = len(tokens)
    mp = (T + 15) // 16
    bt = W.make_block_tables([T], 16, mp + 3, mp, seed=3)[0].numpy()
    dims = make_dims(W.TINY, 16, mp + 3, mp)
    kv = np.zeros(W.kv_shape(W.TINY, mp + 3, 16), dtype=np.uint16)
    bf = np.stack([oracle32.decode_step(dims, tiny_w, np.array([tokens[t]], np.int32), np.array([t + 1], np.int32),
                                        bt, kv)[0] for t in range(T)])
    err = rel_l2(q8, bf)
    assert 0 < err < 5e-2, err
