"""The oracle's pins must catch plausible mistakes.

Each case copies ``oracle/oracle.cpp`` to a temporary directory, plants one
mistake by text replacement (CPU only), compiles it and runs the pin battery
below against the mutant.  A mutant that passes every pin is a hole in the
pins and fails this test.  The real oracle must pass the same battery.
"""
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest
import torch

import workloads as W
from oracle import Oracle, make_dims
from tests import bruteforce as BF
from tests.helpers import np_weights

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "oracle.cpp")

MUTANTS = [
    ("gqa head mapping", "const int g = h / G;", "const int g = h % Hkv;"),
    ("attention residual dropped", "xb[i] = xb[i] + o[i];", "xb[i] = o[i];"),
    ("rope sign", "v[i] = a * c - b * s;", "v[i] = a * c + b * s;"),
    ("attention scale missing", "s[t] = dot * scale;", "s[t] = dot;"),
    ("current token excluded", "for (int t = 0; t < Lc; ++t) {\n        const int pg = tab[t / d.page_size], sl = t % d.page_size;\n        T dot = 0;",
     "for (int t = 0; t < Lc - 1; ++t) {\n        const int pg = tab[t / d.page_size], sl = t % d.page_size;\n        T dot = 0;"),
    ("values read from key plane", "cache.get(pg, 1, g, sl, i)", "cache.get(pg, 0, g, sl, i)"),
    ("router not renormalised", "d.norm_topk ? p[ids[j]] / z : p[ids[j]]", "p[ids[j]]"),
    ("top-k tie to higher index", "if (best < 0 || r[i] > r[best]) best = i;",
     "if (best < 0 || r[i] >= r[best]) best = i;"),
    ("silu sign", "a / (static_cast<T>(1) + texp<T>(-a))", "a / (static_cast<T>(1) + texp<T>(a))"),
    ("gate and up swapped", "T a = gu[f];", "T a = gu[F + f];"),
    ("rmsnorm mean missing", "tsqrt<T>(ss / static_cast<T>(n) + static_cast<T>(eps))",
     "tsqrt<T>(ss + static_cast<T>(eps))"),
    ("gemv transposed", "const uint16_t* w = W + static_cast<size_t>(r) * cols;\n    T acc = 0;\n    for (int c = 0; c < cols; ++c) acc += static_cast<T>(bf16_to_f32(w[c])) * x[c];",
     "T acc = 0;\n    for (int c = 0; c < cols; ++c) acc += static_cast<T>(bf16_to_f32(W[static_cast<size_t>(c) * rows + r])) * x[c];"),
    ("combine weights ignored", "out[i] += wts[slot] * yj[i];", "out[i] += yj[i];"),
    ("final norm skipped", "rmsnorm<T>(d.hidden, x + static_cast<size_t>(b) * d.hidden, final_norm, d.rms_eps, y.data());",
     "for (int i = 0; i < d.hidden; ++i) y[i] = x[static_cast<size_t>(b) * d.hidden + i];"),
    ("kv written unrounded-then-truncated", "bits += 0x7fffu + lsb;", "bits += 0;"),
    ("rope pair offset", "T a = v[i], b = v[i + half];", "T a = v[i], b = v[half - 1 - i];"),
    ("router bias dropped", "r[e] = r[e] + static_cast<T>(w.router_bias[e]);", "r[e] = r[e];"),
    # the q8_0 cache
    ("q8 scale of the next block", "f16_to_f32(scales[o / 32 + i / 32])",
     "f16_to_f32(scales[o / 32 + (i / 32 + 1) % (d.head_dim / 32)])"),
    ("q8 codes truncated", "q[i] = static_cast<int8_t>(std::round(x[i] * id));",
     "q[i] = static_cast<int8_t>(std::trunc(x[i] * id));"),
    ("q8 max over half a block", "for (int i = 0; i < 32; ++i) amax", "for (int i = 0; i < 16; ++i) amax"),
    ("f16 scale truncated", "if (rem > half || (rem == half && (q & 1u))) ++q;", "(void)half;"),
    ("q8 scale step 1/128", "const float d = amax / 127.0f;", "const float d = amax / 128.0f;"),
]


def _battery(orc64: Oracle, orc32: Oracle, wn, wn_bias, bias, wn_nonorm) -> list:
    """Return the names of the pins that fail for this oracle build."""
    failed = []
    m = W.TINY

    def inc(orc, model, w, tokens):
        T = len(tokens)
        mp = (T + 15) // 16
        bt, _ = W.make_block_tables([T], 16, mp + 3, mp, seed=3)
        dims = make_dims(model, 16, mp + 3, mp)
        kv = np.zeros(W.kv_shape(model, mp + 3, 16), dtype=np.uint16)
        return np.stack([orc.decode_step(dims, w, np.array([tokens[t]], np.int32), np.array([t + 1], np.int32),
                                         bt.numpy(), kv)[0] for t in range(T)])

    def inc_q8(orc, model, w, tokens):
        T = len(tokens)
        mp = (T + 15) // 16
        bt, _ = W.make_block_tables([T], 16, mp + 3, mp, seed=3)
        dims = make_dims(model, 16, mp + 3, mp, kv_q8=True)
        kv = np.zeros((model["layers"], W.kv_q8_layer_bytes(model, mp + 3, 16)), dtype=np.uint8)
        return np.stack([orc.decode_step(dims, w, np.array([tokens[t]], np.int32), np.array([t + 1], np.int32),
                                         bt.numpy(), kv)[0] for t in range(T)])

    def close(a, b):
        return np.abs(a - b).max() / np.abs(b).max() < 1e-9

    tokens = torch.randint(0, m["vocab"], (20,), generator=torch.Generator().manual_seed(7)).numpy()
    try:
        if not close(inc(orc64, m, wn, tokens), BF.forward_sequence(m, wn, tokens)[0]):
            failed.append("bruteforce")
        if not close(inc(orc64, m, wn_bias, tokens), BF.forward_sequence(m, wn_bias, tokens, router_bias=bias)[0]):
            failed.append("bruteforce-bias")
        m0 = dict(m, norm_topk=0)
        if not close(inc(orc64, m0, wn_nonorm, tokens[:8]), BF.forward_sequence(m0, wn_nonorm, tokens[:8])[0]):
            failed.append("bruteforce-nonorm")
    except Exception:
        failed.append("bruteforce-error")
    # q8_0 cache: the paged incremental oracle against the brute force through the same reading
    try:
        if not close(inc_q8(orc64, m, wn, tokens[:12]), BF.forward_sequence(m, wn, tokens[:12], kv_round="q8")[0]):
            failed.append("bruteforce-q8")
    except Exception:
        failed.append("bruteforce-q8-error")
    with np.errstate(over="ignore"):
        f16 = np.array([1 + 2 ** -11, 1 + 3 * 2 ** -11, 65520.0, 3 * 2 ** -25, 0.1], np.float32)
        if [orc32.f32_to_f16(float(v)) for v in f16] != f16.astype(np.float16).view(np.uint16).tolist():
            failed.append("f16-rne")
    xb = np.linspace(-1.0, 0.9, 32).astype(np.float32)
    qb, db = orc32.q8_quantize(xb)
    step = np.float64(np.float32(1.0) / np.float32(127))
    if int(qb[0]) != -127 or np.abs(xb - qb.astype(np.float64) * db.view(np.float16).astype(np.float64)).max() > \
            (0.5 + 127 * 2.0 ** -11) * step:
        failed.append("q8-block")
    r = np.array([0.5, 1.0, 1.0, 0.2, 1.0], dtype=np.float32)
    if list(orc32.topk(r, 2)) != [1, 2]:
        failed.append("topk-ties")
    if orc32.f32_to_bf16(1 + 3 * 2 ** -8) != 0x3F82:
        failed.append("bf16-rne")
    Wu = W.bf16_bits(torch.zeros(3, 5, dtype=torch.bfloat16))
    Wu[1, 2] = 0x4000
    if list(orc64.gemv(Wu, np.array([0, 0, 3.0, 0, 0]))) != [0.0, 6.0, 0.0]:
        failed.append("gemv-orientation")
    return failed


@pytest.fixture(scope="module")
def weights():
    wn = np_weights(W.make_weights(W.TINY, "cpu"))
    bias = W.zipf_router_bias(W.TINY, 1.1)
    wn_bias = np_weights(W.make_weights(W.TINY, "cpu", router_bias=bias))
    wn_nonorm = np_weights(W.make_weights(dict(W.TINY, norm_topk=0), "cpu", seed=97))
    return wn, wn_bias, bias.numpy(), wn_nonorm


def test_real_oracle_passes_battery(weights):
    assert _battery(Oracle("f64"), Oracle("f32"), *weights) == []


def test_every_planted_mistake_is_caught(weights):
    src = open(SRC).read()
    tmp = tempfile.mkdtemp(prefix="orc_mut_")
    try:
        procs = []
        for i, (name, old, new) in enumerate(MUTANTS):
            assert src.count(old) == 1, f"mutation site not unique/present: {name}"
            path = os.path.join(tmp, f"m{i}.cpp")
            with open(path, "w") as f:
                f.write(src.replace(old, new))
            so = os.path.join(tmp, f"m{i}.so")
            procs.append((name, so, subprocess.Popen(
                ["g++", "-O1", "-std=c++17", "-fopenmp", "-ffp-contract=off", "-shared", "-fPIC", path, "-o", so])))
        survivors = []
        for name, so, p in procs:
            assert p.wait() == 0, f"mutant failed to compile: {name}"
            if not _battery(Oracle("f64", so), Oracle("f32", so), *weights):
                survivors.append(name)
        assert survivors == [], f"mutants not caught by any pin: {survivors}"
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
