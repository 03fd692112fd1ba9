"""Pins for the oracle's attention: the tutorial's worked example, absorbed ==
expanded, closed forms, a brute-force loop on tiny inputs, split invariance
and the empty context.

Tutorial: "DeepSeek的MLA技术：极致压缩KV Cache的创新方案" (juejin), sections
"角度3：具体数值例子", "步骤2", "完整的MLA注意力计算", "KV Cache的实现".
English report: "Absorbed MLA Cache Optimization on DeepSeek-V2-Lite —
Technical Report", §1.3 and §2.1.
"""

import math
import os

import numpy as np
import pytest

import synth
from oracle import attention as A
from oracle import quant as Q

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "p3_worked_example.txt")


def load_golden():
    vals = {}
    with open(GOLDEN, encoding="utf-8") as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            name, rest = line.split(None, 1)
            rows = [[float(v) for v in r.split()] for r in rest.split("|")]
            vals[name] = np.array(rows if len(rows) > 1 else rows[0])
    return vals


def test_worked_example_row_vector_convention():
    g = load_golden()
    c_kv = A.project_rows(g["X"], g["W_down"])
    assert np.allclose(c_kv, g["C_KV"], atol=1e-12)
    k1 = A.project_rows(g["C_KV"], g["W_1_up"])
    assert np.allclose(k1, g["K_1"], atol=1e-12)


def tiny_inputs(T=256, H=16, seed=3, layer=0):
    cos, sin = synth.rope_tables(T)
    c = synth.bf16_to_f32(synth.latent_bf16(seed, layer, 0, 0, T))
    k = synth.bf16_to_f32(synth.kpe_bf16(seed, layer, 0, 0, T, cos, sin))
    qn = synth.bf16_to_f32(synth.q_nope_bf16(seed, layer, 1, H))[0]
    qp = synth.bf16_to_f32(synth.q_pe_bf16(seed, layer, 1, H))[0]
    wuk = synth.bf16_to_f32(synth.w_uk_bf16(seed, layer, H))
    wuv = synth.bf16_to_f32(synth.w_uv_bf16(seed, layer, H))
    return c, k, qn, qp, wuk, wuv


@pytest.mark.parametrize("fmt", [Q.FMT_BF16, Q.FMT_INT8, Q.FMT_INT4])
@pytest.mark.parametrize("kfmt", [Q.FMT_BF16, Q.FMT_INT8])
def test_absorbed_equals_expanded(fmt, kfmt):
    """The tiny workload: absorbed attention == re-expanded attention within
    1e-5 in fp64, on the same dequantized latent."""
    c, k, qn, qp, wuk, wuv = tiny_inputs()
    d = Q.quantize_token_rows(c, k, fmt, kfmt)
    _, o_lat, lse, o = A.absorbed_decode_full(qn, qp, wuk, wuv, d["c_hat"], d["kpe_hat"])
    o_exp, lse_exp = A.expanded_decode(qn, qp, wuk, wuv, d["c_hat"], d["kpe_hat"])
    assert A.max_rel_error(o, o_exp) < 1e-5
    assert np.max(np.abs(lse - lse_exp)) < 1e-9


def test_single_token_closed_form():
    """T = 1: softmax weight 1, so o_lat is that token's latent and lse its score."""
    c, k, qn, qp, wuk, wuv = tiny_inputs(T=1)
    q_lat = A.absorb_q(qn, wuk)
    o_lat, lse = A.absorbed_decode(q_lat, qp, c, k)
    assert np.array_equal(o_lat, np.repeat(c.astype(np.float64), 16, axis=0))
    s = (q_lat @ c[0].astype(np.float64) + qp.astype(np.float64) @ k[0]) / math.sqrt(192)
    assert np.allclose(lse, s, rtol=0, atol=1e-12)


def test_equal_scores_give_mean():
    """Zero queries make every score 0: o_lat is the mean latent, lse = ln T."""
    c, k, qn, qp, wuk, wuv = tiny_inputs(T=100)
    o_lat, lse = A.absorbed_decode(np.zeros((4, 512)), np.zeros((4, 64)), c, k)
    assert np.allclose(o_lat, np.broadcast_to(c.astype(np.float64).mean(axis=0), (4, 512)), atol=1e-12)
    assert np.allclose(lse, math.log(100), atol=1e-12)


def test_brute_force_loops_tiny():
    """Pure-Python loops with math.exp on H=2, T=5, reduced dims."""
    rng = np.random.default_rng(9)
    H, T, D, R = 2, 5, 6, 4
    q_lat, q_pe = rng.standard_normal((H, D)), rng.standard_normal((H, R))
    c, k = rng.standard_normal((T, D)), rng.standard_normal((T, R))
    scale = 0.37
    o_lat, lse = A.absorbed_decode(q_lat, q_pe, c, k, softmax_scale=scale)
    for h in range(H):
        s = []
        for t in range(T):
            acc = 0.0
            for i in range(D):
                acc += q_lat[h, i] * c[t, i]
            for i in range(R):
                acc += q_pe[h, i] * k[t, i]
            s.append(acc * scale)
        mx = max(s)
        w = [math.exp(v - mx) for v in s]
        tot = sum(w)
        for i in range(D):
            ref = sum(w[t] * c[t, i] for t in range(T)) / tot
            assert abs(o_lat[h, i] - ref) < 1e-12
        assert abs(lse[h] - (mx + math.log(tot))) < 1e-12


@pytest.mark.parametrize("bounds", [[0, 256], [0, 64, 128, 192, 256], [0, 1, 2, 255, 256],
                                    [0, 100, 100, 256], [0, 37, 64, 65, 200, 256]])
def test_split_partials_combine_equal_unsplit(bounds):
    c, k, qn, qp, wuk, wuv = tiny_inputs()
    q_lat = A.absorb_q(qn, wuk)
    o_ref, lse_ref = A.absorbed_decode(q_lat, qp, c, k)
    m, l, o = A.split_partials(q_lat, qp, c, k, bounds)
    o_lat, lse = A.lse_combine(m, l, o)
    assert A.max_rel_error(o_lat, o_ref) < 1e-12
    assert np.max(np.abs(lse - lse_ref)) < 1e-12


def test_empty_context():
    H = 3
    o_lat, lse = A.absorbed_decode(np.ones((H, 512)), np.ones((H, 64)), np.zeros((0, 512)), np.zeros((0, 64)))
    assert np.all(o_lat == 0) and np.all(np.isneginf(lse))
    m, l, o = A.split_partials(np.ones((H, 512)), np.ones((H, 64)), np.zeros((0, 512)), np.zeros((0, 64)), [0, 0])
    o2, lse2 = A.lse_combine(m, l, o)
    assert np.all(o2 == 0) and np.all(np.isneginf(lse2))


def test_absorb_unabsorb_against_explicit_loops():
    rng = np.random.default_rng(5)
    qn = rng.standard_normal((2, 128))
    wuk = rng.standard_normal((2, 128, 512))
    q_lat = A.absorb_q(qn, wuk)
    for h in range(2):
        for n in (0, 17, 511):
            assert abs(q_lat[h, n] - sum(qn[h, kk] * wuk[h, kk, n] for kk in range(128))) < 1e-10
    o_lat = rng.standard_normal((2, 512))
    wuv = rng.standard_normal((2, 512, 128))
    o = A.unabsorb_o(o_lat, wuv)
    for h in range(2):
        for v in (0, 64, 127):
            assert abs(o[h, v] - sum(o_lat[h, cc] * wuv[h, cc, v] for cc in range(512))) < 1e-10


def test_max_rel_error_metric():
    ref = np.array([[1.0, -4.0, 2.0], [0.5, 0.25, 0.0]])
    x = ref + np.array([[0.004, 0.0, 0.0], [0.0, 0.0005, 0.0]])
    # row 0: 0.004 / 4 = 1e-3; row 1: 0.0005 / 0.5 = 1e-3
    assert abs(A.max_rel_error(x, ref) - 1e-3) < 1e-15
