"""Pins for the oracle's causal prefill attention (queries of just-appended
tokens attending to the positions up to their own): the absorbed per-query
form against the textbook masked score matrix on re-expanded K/V, the first
query's closed form, causality, a chunk computed by hand, and planted
mistakes that each pin has to catch.

English report "Absorbed MLA Cache Optimization on DeepSeek-V2-Lite —
Technical Report" §2.1 (attention from the cached latent); tutorial
"DeepSeek的MLA技术：极致压缩KV Cache的创新方案", "步骤2" and "完整的MLA注意力计算"
(per-head softmax(Q K^T / sqrt(d)) V on the re-expanded K, V).
"""

import math

import numpy as np
import pytest

import synth
from oracle import attention as A
from oracle import quant as Q


def chunk_inputs(n, ctx_before, H=16, seed=5, layer=0, fmt=Q.FMT_INT8, kfmt=Q.FMT_INT8):
    T = ctx_before + n
    cos, sin = synth.rope_tables(T)
    c = synth.bf16_to_f32(synth.latent_bf16(seed, layer, 0, 0, T))
    k = synth.bf16_to_f32(synth.kpe_bf16(seed, layer, 0, 0, T, cos, sin))
    d = Q.quantize_token_rows(c, k, fmt, kfmt)
    qn = synth.bf16_to_f32(synth.q_nope_bf16(seed, layer, n, H))
    qp = synth.bf16_to_f32(synth.q_pe_bf16(seed, layer, n, H))
    wuk = synth.bf16_to_f32(synth.w_uk_bf16(seed, layer, H))
    wuv = synth.bf16_to_f32(synth.w_uv_bf16(seed, layer, H))
    q_lat = np.stack([A.absorb_q(qn[i], wuk) for i in range(n)])
    return d["c_hat"], d["kpe_hat"], qn, qp, q_lat, wuk, wuv


@pytest.mark.parametrize("ctx_before", [0, 7, 64])
def test_prefill_absorbed_equals_expanded_masked(ctx_before):
    """Absorbed per-query prefixes == the expanded masked score matrix (o and
    lse), fp64, on dequantized INT8 latents."""
    n = 12
    c_hat, kpe_hat, qn, qp, q_lat, wuk, wuv = chunk_inputs(n, ctx_before)
    o_lat, lse = A.absorbed_prefill(q_lat, qp, c_hat, kpe_hat, ctx_before)
    o = np.stack([A.unabsorb_o(o_lat[i], wuv) for i in range(n)])
    o_exp, lse_exp = A.expanded_prefill(qn, qp, wuk, wuv, c_hat, kpe_hat, ctx_before)
    assert A.max_rel_error(o, o_exp) < 1e-9
    assert np.max(np.abs(lse - lse_exp)) < 1e-9


def test_prefill_first_query_closed_form():
    """With no earlier context, query 0 sees only its own token: o_lat is that
    token's latent and lse its score."""
    c_hat, kpe_hat, qn, qp, q_lat, wuk, wuv = chunk_inputs(3, 0)
    o_lat, lse = A.absorbed_prefill(q_lat, qp, c_hat, kpe_hat, 0)
    for h in range(q_lat.shape[1]):
        assert np.array_equal(o_lat[0, h], c_hat[0].astype(np.float64))
        s = (q_lat[0, h] @ c_hat[0].astype(np.float64) + qp[0, h].astype(np.float64) @ kpe_hat[0].astype(np.float64))
        assert abs(lse[0, h] - s * A.DEFAULT_SOFTMAX_SCALE) < 1e-12


def test_prefill_causality():
    """Changing the tokens after position p leaves the queries at or before p
    unchanged and changes the later ones."""
    n, ctx_before, p = 10, 4, 8
    c_hat, kpe_hat, qn, qp, q_lat, wuk, wuv = chunk_inputs(n, ctx_before)
    o1, l1 = A.absorbed_prefill(q_lat, qp, c_hat, kpe_hat, ctx_before)
    c2, k2 = c_hat.copy(), kpe_hat.copy()
    c2[p + 1:] *= -3.0
    k2[p + 1:] += 1.0
    o2, l2 = A.absorbed_prefill(q_lat, qp, c2, k2, ctx_before)
    first_later = p - ctx_before + 1
    assert np.array_equal(o1[:first_later], o2[:first_later]) and np.array_equal(l1[:first_later], l2[:first_later])
    assert all(not np.allclose(o1[i], o2[i]) for i in range(first_later, n))


def test_prefill_hand_computed_chunk():
    """One head, 2-wide latent, 1-wide rope, unit softmax scale, ctx_before = 1:
    keys c = (1, 0), (0, 1), (1, 1) with k_pe 0, 0, 1; queries q_lat = (2, 0)
    and (0, 1), q_pe = 0 and 1.  Query 0 (position 1) scores 2, 0; query 1
    (position 2) scores 0, 1, 1 + 1 = 2."""
    c = np.array([[1.0, 0.0], [0.0, 1.0], [1.0, 1.0]])
    k = np.array([[0.0], [0.0], [1.0]])
    q_lat = np.array([[[2.0, 0.0]], [[0.0, 1.0]]])
    q_pe = np.array([[[0.0]], [[1.0]]])
    o_lat, lse = A.absorbed_prefill(q_lat, q_pe, c, k, 1, softmax_scale=1.0)
    e2 = math.exp(2.0)
    want0 = np.array([e2 * 1.0 + 1.0 * 0.0, e2 * 0.0 + 1.0 * 1.0]) / (e2 + 1.0)
    assert np.allclose(o_lat[0, 0], want0, atol=1e-15)
    assert abs(lse[0, 0] - math.log(e2 + 1.0)) < 1e-15
    e1 = math.exp(1.0)
    den = 1.0 + e1 + e2
    want1 = np.array([1.0 + e2, e1 + e2]) / den
    assert np.allclose(o_lat[1, 0], want1, atol=1e-15)
    assert abs(lse[1, 0] - math.log(den)) < 1e-15


def _excludes_own_token(q_lat, q_pe, c_hat, kpe_hat, ctx_before, softmax_scale=A.DEFAULT_SOFTMAX_SCALE):
    outs, lses = [], []
    for i in range(np.asarray(q_lat).shape[0]):
        t = ctx_before + i
        o, l = A.absorbed_decode(q_lat[i], q_pe[i], c_hat[:t], kpe_hat[:t], softmax_scale)
        outs.append(o)
        lses.append(l)
    return np.stack(outs), np.stack(lses)


def _ignores_ctx_before(q_lat, q_pe, c_hat, kpe_hat, ctx_before, softmax_scale=A.DEFAULT_SOFTMAX_SCALE):
    outs, lses = [], []
    for i in range(np.asarray(q_lat).shape[0]):
        o, l = A.absorbed_decode(q_lat[i], q_pe[i], c_hat[:i + 1], kpe_hat[:i + 1], softmax_scale)
        outs.append(o)
        lses.append(l)
    return np.stack(outs), np.stack(lses)


def _sees_whole_chunk(q_lat, q_pe, c_hat, kpe_hat, ctx_before, softmax_scale=A.DEFAULT_SOFTMAX_SCALE):
    n = np.asarray(q_lat).shape[0]
    outs, lses = [], []
    for i in range(n):
        o, l = A.absorbed_decode(q_lat[i], q_pe[i], c_hat[:ctx_before + n], kpe_hat[:ctx_before + n], softmax_scale)
        outs.append(o)
        lses.append(l)
    return np.stack(outs), np.stack(lses)


@pytest.mark.parametrize("bad", [_excludes_own_token, _ignores_ctx_before, _sees_whole_chunk],
                         ids=["excludes-own-token", "ignores-ctx-before", "no-causal-mask"])
def test_planted_prefill_mistake_fails_a_pin(monkeypatch, bad):
    monkeypatch.setattr(A, "absorbed_prefill", bad)
    pins = [lambda: test_prefill_absorbed_equals_expanded_masked(7), test_prefill_first_query_closed_form,
            test_prefill_causality, test_prefill_hand_computed_chunk]
    failed = 0
    for pin in pins:
        try:
            pin()
        except (AssertionError, ValueError, IndexError):
            failed += 1
    assert failed >= 1
