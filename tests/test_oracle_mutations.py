"""Planted mistakes: each plausible slip in the oracle must fail a pin.

Every case monkeypatches one oracle function with a wrong variant (on the CPU,
never on a GPU) and runs an existing pin, which has to raise.
"""

import numpy as np
import pytest

from oracle import attention as A
from oracle import quant as Q
import tests.test_oracle_attention as TA
import tests.test_oracle_quant as TQ

F32 = np.float32


def _int8_floor(x, group):
    g = Q._groups(x, group)
    s = np.max(np.abs(g), axis=2) / F32(127)
    safe = np.where(s > 0, s, F32(1)).astype(np.float32)
    q = np.clip(np.floor(g / safe[..., None]), -127, 127)
    return q.astype(np.int8).reshape(x.shape[0], -1), s.astype(np.float32)


def _int8_over_128(x, group):
    g = Q._groups(x, group)
    s = (np.max(np.abs(g), axis=2) / F32(128)).astype(np.float32)
    safe = np.where(s > 0, s, F32(1)).astype(np.float32)
    q = np.clip(np.rint(g / safe[..., None]), -127, 127)
    return q.astype(np.int8).reshape(x.shape[0], -1), s


def _int4_zero_sign(x, group=16):
    q, s, z = Q.__dict__["_orig_int4"](x, group)
    return q, s, (-z).astype(np.float32)


def _sym_int4_over_8(x, group=16):
    g = Q._groups(x, group)
    s = (np.max(np.abs(g), axis=2) / F32(8)).astype(np.float32)
    safe = np.where(s > 0, s, F32(1)).astype(np.float32)
    q = np.clip(np.rint(g / safe[..., None]), -7, 7)
    return q.astype(np.int8).reshape(x.shape[0], -1), s


def _decode_no_rope(q_lat, q_pe, c_hat, kpe_hat, softmax_scale=A.DEFAULT_SOFTMAX_SCALE):
    return A.__dict__["_orig_decode"](q_lat, np.zeros_like(np.asarray(q_pe, np.float64)), c_hat, kpe_hat,
                                      softmax_scale)


def _absorb_wrong_head(q_nope, w_uk):
    q_nope, w_uk = np.asarray(q_nope, np.float64), np.asarray(w_uk, np.float64)
    H = q_nope.shape[0]
    return np.stack([q_nope[h] @ w_uk[(h + 1) % H] for h in range(H)])


def _combine_without_l(m, l, o):
    return A.__dict__["_orig_combine"](m, np.ones_like(l), o)


def _project_rows_reversed(x, w):
    return np.asarray(x, np.float64) @ np.asarray(w, np.float64)[::-1]


CASES = [
    ("int8 rounds by floor", Q, "quantize_sym_int8", _int8_floor,
     lambda: TQ.test_int8_codes_are_nearest_levels_brute_force(16)),
    ("int8 scale absmax/128", Q, "quantize_sym_int8", _int8_over_128,
     TQ.test_int8_scale_is_absmax_over_127),
    ("int4 zero-point sign flipped", Q, "quantize_asym_int4", _int4_zero_sign,
     TQ.test_int4_scale_zero_and_endpoints),
    ("sym int4 scale absmax/8", Q, "quantize_sym_int4", _sym_int4_over_8,
     TQ.test_sym_int4_scale_absmax_over_7_ties_and_zero_group),
    ("decode drops the q_pe.k_pe term", A, "absorbed_decode", _decode_no_rope,
     lambda: TA.test_absorbed_equals_expanded(Q.FMT_INT8, Q.FMT_INT8)),
    ("absorb uses the wrong head's W_UK", A, "absorb_q", _absorb_wrong_head,
     lambda: TA.test_absorbed_equals_expanded(Q.FMT_BF16, Q.FMT_BF16)),
    ("combine ignores the partial sums l", A, "lse_combine", _combine_without_l,
     lambda: TA.test_split_partials_combine_equal_unsplit([0, 64, 128, 192, 256])),
    ("projection reads W rows reversed", A, "project_rows", _project_rows_reversed,
     TA.test_worked_example_row_vector_convention),
]


@pytest.mark.parametrize("name,mod,attr,bad,pin", CASES, ids=[c[0] for c in CASES])
def test_planted_mistake_fails_a_pin(monkeypatch, name, mod, attr, bad, pin):
    monkeypatch.setitem(Q.__dict__, "_orig_int4", Q.quantize_asym_int4)
    monkeypatch.setitem(A.__dict__, "_orig_decode", A.absorbed_decode)
    monkeypatch.setitem(A.__dict__, "_orig_combine", A.lse_combine)
    pin()                                   # the pin passes on the real oracle
    monkeypatch.setattr(mod, attr, bad)
    with pytest.raises(AssertionError):
        pin()


def test_wrong_softmax_scale_fails_closed_form(monkeypatch):
    TA.test_single_token_closed_form()
    monkeypatch.setattr(A, "DEFAULT_SOFTMAX_SCALE", 1.0 / np.sqrt(128.0))
    orig = A.absorbed_decode
    monkeypatch.setattr(A, "absorbed_decode",
                        lambda q, p, c, k, softmax_scale=A.DEFAULT_SOFTMAX_SCALE: orig(q, p, c, k, softmax_scale))
    with pytest.raises(AssertionError):
        TA.test_single_token_closed_form()
