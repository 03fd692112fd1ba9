"""Pins for the oracle's quantizers.

They tie the oracle to what the pages and arithmetic fix, not to itself:
brute-force nearest level, hand-built half-way ties with literal expected
codes, degenerate groups, the round-trip bound, and the error ordering of the
Chinese report's §3.2 table ("DeepSeek-V2-Lite MLA 吸收式 KV 缓存优化 — 完整实验报告")
and the English report's §4.2 / §5.1.
"""

import numpy as np
import pytest

import synth
from oracle import quant as Q

RNG = np.random.default_rng(1234)


def ulp32(x):
    x = np.abs(np.asarray(x, np.float32))
    return np.spacing(x).astype(np.float64)


def synth_latent(T=512, layer=0, seed=7):
    return synth.bf16_to_f32(synth.latent_bf16(seed, layer, 0, 0, T))


def synth_kpe(T=512, layer=0, seed=7):
    cos, sin = synth.rope_tables(T)
    return synth.bf16_to_f32(synth.kpe_bf16(seed, layer, 0, 0, T, cos, sin))


# --------------------------------------------------------------- INT8 --------

@pytest.mark.parametrize("group", [16, 8, 32, 64, 512])
def test_int8_codes_are_nearest_levels_brute_force(group):
    w = max(128, group)
    x = np.concatenate([synth_latent(64)[:, :w], RNG.standard_normal((64, w)).astype(np.float32) * 3])
    q, s = Q.quantize_sym_int8(x, group)
    assert q.dtype == np.int8 and s.dtype == np.float32
    sg = np.repeat(s, group, axis=1)
    ratio = (x / sg).astype(np.float64)          # the fp32 quotient the definition rounds
    levels = np.arange(-127, 128, dtype=np.float64)
    d = np.abs(ratio[..., None] - levels)        # distance to every code
    best = d.min(axis=-1)
    chosen = np.abs(ratio - q.astype(np.float64))
    assert np.all(chosen == best)
    # exact ties go to the even code
    tie = np.sum(d == best[..., None], axis=-1) > 1
    assert np.all(q[tie] % 2 == 0)


def test_int8_scale_is_absmax_over_127():
    x = synth_latent(32)
    q, s = Q.quantize_sym_int8(x, 16)
    a = np.abs(x).reshape(32, 32, 16).max(axis=2).astype(np.float64)
    assert np.all(np.abs(s.astype(np.float64) * 127 - a) <= 2 * ulp32(a))
    # the absmax element of every group codes to +-127
    g = np.abs(q.reshape(32, 32, 16).astype(np.int32)).max(axis=2)
    assert np.all(g == 127)


def test_int8_half_even_ties_literal():
    # s = 127 / 127 = 1 exactly, so x / s = x and the ties are exact.
    row = np.array([127, 0.5, 1.5, 2.5, 3.5, -0.5, -1.5, -2.5, 126.5, -126.5, 0, 7, -7, 0.25, 0.75, 100.49],
                   np.float32)[None, :]
    q, s = Q.quantize_sym_int8(row, 16)
    assert s[0, 0] == np.float32(1.0)
    expect = [127, 0, 2, 2, 4, 0, -2, -2, 126, -126, 0, 7, -7, 0, 1, 100]
    assert q[0].tolist() == expect


def test_int8_degenerate_and_extreme_groups():
    rows = np.zeros((4, 16), np.float32)
    rows[1, :] = 3.25                         # constant group
    rows[2, 0] = -1000.0                      # single outlier, rest tiny
    rows[2, 1:] = 1e-3
    rows[3, :] = np.array([127, -127] * 8, np.float32)
    q, s = Q.quantize_sym_int8(rows, 16)
    assert s[0, 0] == 0 and np.all(q[0] == 0)                       # all-zero group
    assert np.all(q[1] == 127)
    x_hat = Q.dequantize_sym_int8(q, s, 16)
    assert np.all(np.abs(x_hat[1] - 3.25) <= 2 * ulp32(3.25))
    assert q[2, 0] == -127 and np.all(q[2, 1:] == 0)
    assert q[3].tolist() == [127, -127] * 8


@pytest.mark.parametrize("group", [16, 8])
def test_int8_round_trip_bound(group):
    x = np.concatenate([synth_latent(256), synth_latent(256, layer=3)])[:, :512]
    q, s = Q.quantize_sym_int8(x, group)
    x_hat = Q.dequantize_sym_int8(q, s, group)
    sg = np.repeat(s, group, axis=1).astype(np.float64)
    ag = np.repeat(np.abs(x).reshape(x.shape[0], -1, group).max(axis=2), group, axis=1)
    err = np.abs(x.astype(np.float64) - x_hat)
    # 0.5 scale in exact arithmetic; a few fp32 ulps of the group absmax for
    # the rounded quotient and product.
    assert np.all(err <= 0.5 * sg + 4 * ulp32(ag))


# --------------------------------------------------------------- INT4 --------

def test_int4_codes_are_nearest_levels_brute_force():
    x = np.concatenate([synth_latent(64), RNG.standard_normal((64, 512)).astype(np.float32) + 2.0])
    q, s, z = Q.quantize_asym_int4(x, 16)
    assert q.dtype == np.uint8 and q.max() <= 15
    sg = np.repeat(s, 16, axis=1)
    zg = np.repeat(z, 16, axis=1).astype(np.float64)
    ratio = (x / sg).astype(np.float64)
    levels = np.arange(16, dtype=np.float64)
    d = np.abs(ratio[..., None] - (levels - zg[..., None]))
    best = d.min(axis=-1)
    chosen = np.abs(ratio - (q.astype(np.float64) - zg))
    assert np.all(chosen == best)
    tie = np.sum(d == best[..., None], axis=-1) > 1
    assert np.all((q[tie].astype(np.int64) - zg[tie].astype(np.int64)) % 2 == 0)


def test_int4_scale_zero_and_endpoints():
    x = synth_latent(64)
    q, s, z = Q.quantize_asym_int4(x, 16)
    g = x.reshape(64, 32, 16).astype(np.float64)
    mn, mx = g.min(axis=2), g.max(axis=2)
    assert np.all(np.abs(s * 15.0 - (mx - mn)) <= 4 * ulp32(np.maximum(np.abs(mx), np.abs(mn))))
    assert np.all(z == np.round(z)) and z.dtype == np.float32
    qg = q.reshape(64, 32, 16)
    imin, imax = g.argmin(axis=2), g.argmax(axis=2)
    qmin = np.take_along_axis(qg, imin[..., None], 2)[..., 0]
    qmax = np.take_along_axis(qg, imax[..., None], 2)[..., 0]
    assert np.all(qmin <= 1) and np.all(qmax >= 14)
    # groups straddling zero have their zero-point inside the code range
    straddle = (mn < 0) & (mx > 0)
    assert np.all((z[straddle] >= 0) & (z[straddle] <= 15))


def test_int4_degenerate_groups_reconstruct_exactly():
    rows = np.zeros((4, 16), np.float32)
    rows[1, :] = 2.5
    rows[2, :] = -0.75
    rows[3, :8] = 1.0
    rows[3, 8:] = 4.0
    q, s, z = Q.quantize_asym_int4(rows, 16)
    assert s[0, 0] == 0 and z[0, 0] == 0 and np.all(q[0] == 0)
    assert s[1, 0] == 2.5 and z[1, 0] == -1 and np.all(q[1] == 0)
    assert s[2, 0] == 0.75 and z[2, 0] == 1 and np.all(q[2] == 0)
    x_hat = Q.dequantize_asym_int4(q, s, z, 16)
    assert np.array_equal(x_hat[:3], rows[:3])
    # two-level group: min 1 -> code 0, max 4 -> code 15, s = 0.2, z = -5
    assert np.isclose(s[3, 0], 0.2) and z[3, 0] == -5
    assert np.all(q[3, :8] == 0) and np.all(q[3, 8:] == 15)


def test_int4_half_even_tie_literal():
    # min = -1, max = 14 -> s = 1, z = 1; x / s = 2.5 -> rint 2 (even) -> q = 3
    row = np.array([-1, 14, 2.5, 3.5, -0.5, 0.5, 0, 13.5, 1, 1, 1, 1, 1, 1, 1, 1], np.float32)[None, :]
    q, s, z = Q.quantize_asym_int4(row, 16)
    assert s[0, 0] == 1 and z[0, 0] == 1
    assert q[0, :8].tolist() == [0, 15, 3, 5, 1, 1, 1, 15]


def test_int4_round_trip_bound():
    x = np.concatenate([synth_latent(256), RNG.standard_normal((64, 512)).astype(np.float32) * 50 + 100])
    q, s, z = Q.quantize_asym_int4(x, 16)
    x_hat = Q.dequantize_asym_int4(q, s, z, 16)
    sg = np.repeat(s, 16, axis=1).astype(np.float64)
    ag = np.repeat(np.abs(x).reshape(x.shape[0], -1, 16).max(axis=2), 16, axis=1)
    err = np.abs(x.astype(np.float64) - x_hat)
    assert np.all(err <= 0.5 * sg + 8 * ulp32(ag))


# ----------------------------------------------------------- symmetric INT4 --

@pytest.mark.parametrize("group", [16, 8])
def test_sym_int4_codes_are_nearest_levels_brute_force(group):
    x = np.concatenate([synth_latent(64)[:, :128], RNG.standard_normal((64, 128)).astype(np.float32) * 3])
    q, s = Q.quantize_sym_int4(x, group)
    assert q.dtype == np.int8 and q.min() >= -7 and q.max() <= 7
    sg = np.repeat(s, group, axis=1)
    ratio = (x / sg).astype(np.float64)
    levels = np.arange(-7, 8, dtype=np.float64)
    d = np.abs(ratio[..., None] - levels)
    best = d.min(axis=-1)
    assert np.all(np.abs(ratio - q.astype(np.float64)) == best)
    tie = np.sum(d == best[..., None], axis=-1) > 1
    assert np.all(q[tie] % 2 == 0)


def test_sym_int4_scale_absmax_over_7_ties_and_zero_group():
    x = synth_kpe(32)
    q, s = Q.quantize_sym_int4(x, 8)
    a = np.abs(x).reshape(32, 8, 8).max(axis=2).astype(np.float64)
    assert np.all(np.abs(s.astype(np.float64) * 7 - a) <= 2 * ulp32(a))
    assert np.all(np.abs(q.reshape(32, 8, 8).astype(np.int32)).max(axis=2) == 7)
    # absmax 7 -> s = 1: 2.5 -> 2, 3.5 -> 4, -0.5 -> 0, 6.5 -> 6 (half even); a zero group stays zero
    row = np.array([[7, 2.5, 3.5, -0.5, 6.5, -6.5, 1.5, 0, 0, 0, 0, 0, 0, 0, 0, 0]], np.float32)
    q, s = Q.quantize_sym_int4(row, 8)
    assert s[0].tolist() == [1.0, 0.0]
    assert q[0].tolist() == [7, 2, 4, 0, 6, -6, 2, 0] + [0] * 8


def test_token_rows_int8_block_count_formats():
    c, k = synth_latent(16), synth_kpe(16)
    for fmt, g in ((Q.FMT_INT8_G8, 8), (Q.FMT_INT8_G32, 32), (Q.FMT_INT8_G64, 64), (Q.FMT_INT8_TOKEN, 512)):
        d = Q.quantize_token_rows(c, k, fmt, Q.FMT_INT8)
        q, s = Q.quantize_sym_int8(c, g)
        assert d["c_scale"].shape == (16, 512 // g)
        assert np.array_equal(d["c_codes"], q) and np.array_equal(d["c_scale"], s)
    # one block per token is the report's per-token row
    q1, s1 = Q.quantize_per_token_int8(c)
    d = Q.quantize_token_rows(c, k, Q.FMT_INT8_TOKEN, Q.FMT_INT8)
    assert np.array_equal(d["c_codes"], q1) and np.array_equal(d["c_scale"][:, 0], s1[:, 0])


def test_sym_int4_round_trip_bound():
    x = np.concatenate([synth_latent(128), synth_kpe(128)[:, :64].repeat(8, axis=1)])
    for group in (16, 8):
        q, s = Q.quantize_sym_int4(x, group)
        x_hat = Q.dequantize_sym_int4(q, s, group)
        sg = np.repeat(s, group, axis=1).astype(np.float64)
        ag = np.repeat(np.abs(x).reshape(x.shape[0], -1, group).max(axis=2), group, axis=1)
        assert np.all(np.abs(x.astype(np.float64) - x_hat) <= 0.5 * sg + 4 * ulp32(ag))


def test_token_rows_sym_int4_fields():
    c, k = synth_latent(16), synth_kpe(16)
    d = Q.quantize_token_rows(c, k, Q.FMT_INT4_SYM, Q.FMT_INT4_SYM)
    assert d["c_codes"].shape == (16, 512) and d["c_scale"].shape == (16, 32) and "c_zero" not in d
    assert d["kpe_codes"].shape == (16, 64) and d["kpe_scale"].shape == (16, 8)
    assert np.array_equal(d["c_hat"], Q.dequantize_sym_int4(*Q.quantize_sym_int4(c, 16), 16))


# ------------------------------------------------- the pages' error ordering --

def test_error_ordering_per_group_per_token_per_tensor():
    """CN §3.2 / EN §4.2: per-group (0.0109) < per-token (0.0636) < per-tensor
    (0.2979) on a latent with per-channel outliers."""
    x = synth_latent(512)
    e_group = Q.relative_error(x, Q.dequantize_sym_int8(*Q.quantize_sym_int8(x, 16), 16))[0]
    qt, st = Q.quantize_per_token_int8(x)
    e_token = Q.relative_error(x, Q.dequantize_sym_int8(qt, st, 512))[0]
    qa, sa = Q.quantize_per_tensor_int8(x)
    e_tensor = Q.relative_error(x, qa.astype(np.float32) * sa)[0]
    assert e_group < e_token < e_tensor
    assert e_tensor / e_group > 5


def test_error_more_groups_is_better():
    """EN §5.1: 8 blocks worse than 32 blocks worse than 64 blocks."""
    x = synth_latent(512)
    errs = [Q.relative_error(x, Q.dequantize_sym_int8(*Q.quantize_sym_int8(x, 512 // n), 512 // n))[0]
            for n in (8, 32, 64)]
    assert errs[0] > errs[1] > errs[2]


def test_error_asym_int4_beats_sym_int4():
    """CN §3.2: asymmetric INT4 (0.0786) better than symmetric INT4 (0.1116)."""
    x = synth_latent(512)
    q, s, z = Q.quantize_asym_int4(x, 16)
    e_asym = Q.relative_error(x, Q.dequantize_asym_int4(q, s, z, 16))[0]
    qs, ss = Q.quantize_sym_int4(x, 16)
    e_sym = Q.relative_error(x, Q.dequantize_sym_int8(qs, ss, 16))[0]
    assert e_asym < e_sym


def test_error_kpe_int8_below_latent_int8():
    """CN §3.2: k_pe INT8 in 8 blocks (0.0051) beats the latent INT8 (0.0109)."""
    x = synth_latent(512)
    k = synth_kpe(512)
    e_lat = Q.relative_error(x, Q.dequantize_sym_int8(*Q.quantize_sym_int8(x, 16), 16))[0]
    e_kpe = Q.relative_error(k, Q.dequantize_sym_int8(*Q.quantize_sym_int8(k, 8), 8))[0]
    assert e_kpe < e_lat


def test_relative_error_literal_values():
    """The error metric behind the ordering checks, pinned by hand-computed
    values: mean |x - x_hat| / mean |x| and max |x - x_hat| / mean |x|."""
    # e = [0.5, 0]; mean|x| = 1.5 -> mean 0.25 / 1.5 = 1/6, max 0.5 / 1.5 = 1/3
    m, mx = Q.relative_error([1.0, 2.0], [1.5, 2.0])
    assert m == pytest.approx(1 / 6, rel=1e-15) and mx == pytest.approx(1 / 3, rel=1e-15)
    # signs do not matter; a denominator of max|x| (= 3) would give 1/6, not 1/4
    m, mx = Q.relative_error([-1.0, -3.0], [-1.0, -2.0])
    assert m == pytest.approx(0.25, rel=1e-15) and mx == pytest.approx(0.5, rel=1e-15)
    # the mean runs over every element of a 2-D tensor: e = [0, 0, 0, 2],
    # mean|x| = 10 / 4 -> mean 0.5 / 2.5 = 0.2, max 2 / 2.5 = 0.8
    m, mx = Q.relative_error([[1.0, 2.0], [3.0, 4.0]], [[1.0, 2.0], [3.0, 2.0]])
    assert m == pytest.approx(0.2, rel=1e-15) and mx == pytest.approx(0.8, rel=1e-15)
    # no error at all
    assert Q.relative_error([0.5, -7.0, 3.0], [0.5, -7.0, 3.0]) == (0.0, 0.0)


# ---------------------------------------------------------------------------
# The stored per-token bound M_t (the decode's weight of its fp16 P V terms)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("fmt", [Q.FMT_INT8, Q.FMT_INT8_G8, Q.FMT_INT8_G32, Q.FMT_INT8_G64, Q.FMT_INT8_TOKEN,
                                 Q.FMT_INT4_SYM])
def test_bound_is_the_largest_dequantized_magnitude_symmetric(fmt):
    """Symmetric formats: every group's largest input maps to the extreme
    code, so M_t is exactly max_c |x_hat[c]| (bit for bit), outliers or not."""
    c = synth_latent(T=256)
    c[7, 100:116] = 0.0                                   # an all-zero group
    c[9] = 0.0                                            # an all-zero token: bound 0
    d = Q.quantize_token_rows(c, synth_kpe(T=256), fmt, Q.FMT_INT8)
    exp = np.max(np.abs(d["c_hat"]), axis=1).astype(np.float32)
    assert np.array_equal(d["c_bound"].view(np.uint32), exp.view(np.uint32))
    assert d["c_bound"][9] == 0.0


def test_bound_asymmetric_int4_covers_both_ends():
    """Asymmetric INT4: M_t = max_g s (|z - 7.5| + 7.5) >= max |x_hat|, equal
    to it when a group's min and max map to codes 0 and 15, and never more
    than one step s above it."""
    c = synth_latent(T=256)
    d = Q.quantize_token_rows(c, synth_kpe(T=256), Q.FMT_INT4, Q.FMT_INT8)
    m = np.max(np.abs(d["c_hat"]), axis=1)
    b = d["c_bound"].astype(np.float64)
    assert np.all(b >= m * (1 - 2.0 ** -23))
    assert np.all(b <= m + np.max(d["c_scale"], axis=1) * (1 + 2.0 ** -20))
    # literal: one group [-3, 5, 0 ...]: s = 8/15, z = rint(3 / s) = rint(5.625) = 6;
    # codes 0 (x = -3) and 15 (x = 5): x_hat = -6 s and 9 s; the bound is 9 s,
    # the larger end, where |z| alone (6 s) would be wrong
    x = np.zeros((1, 512), np.float32)
    x[0, 0], x[0, 1] = -3.0, 5.0
    q, s, z = Q.quantize_asym_int4(x)
    assert z[0, 0] == 6.0 and s[0, 0] == np.float32(8.0) / np.float32(15.0)
    bound = Q.latent_bound(s, z)
    assert bound[0] == np.float32(s[0, 0] * np.float32(9.0))
    assert bound[0] == np.max(np.abs(Q.dequantize_asym_int4(q, s, z)))
    # a group with min > 0 has z < 0: the far end 15 - z dominates
    y = np.zeros((1, 512), np.float32)
    y[0, :16] = np.linspace(10.0, 11.0, 16, dtype=np.float32)
    q, s, z = Q.quantize_asym_int4(y)
    assert z[0, 0] < 0
    assert Q.latent_bound(s, z)[0] == np.float32(s[0, 0] * (np.float32(15.0) - z[0, 0]))
    # the bound takes the largest group, not the first
    w = np.zeros((1, 512), np.float32)
    w[0, 0:2] = [-1.0, 1.0]
    w[0, 496:498] = [-4.0, 4.0]
    q, s, z = Q.quantize_asym_int4(w)
    assert Q.latent_bound(s, z)[0] == np.max(s * (np.abs(z - np.float32(7.5)) + np.float32(7.5)))
    assert Q.latent_bound(s, z)[0] >= 4.0 * (1 - 2.0 ** -22)


# ---------------------------------------------------------------------------
# Outlier-protected mixed precision (English report §4.3 row C)
# ---------------------------------------------------------------------------

def test_select_outlier_channels_brute_force():
    x = np.zeros((3, 512), np.float32)
    big = [3, 40, 41, 200, 511]
    for i, c in enumerate(big):
        x[i % 3, c] = -(10.0 + i)                         # sign does not matter
    x[1, 7] = x[2, 9] = 2.0                               # a tie: the lower index goes first
    x[0, 100] = 1.5
    got = Q.select_outlier_channels(x, k=7)
    assert got.tolist() == sorted(big + [7, 9])
    assert Q.select_outlier_channels(x, k=6).tolist() == sorted(big + [7])
    # brute force on random data: the chosen set holds the k largest maxima
    r = RNG.standard_normal((16, 512)).astype(np.float32)
    sel = Q.select_outlier_channels(r)
    a = np.max(np.abs(r), axis=0)
    assert len(sel) == Q.OUTLIER_CHANNELS == 25 and np.all(np.diff(sel) > 0)
    assert np.min(a[sel]) >= np.max(np.delete(a, sel))


def test_outlier_format_literal_group():
    """Group 0 holds a protected channel of 100 and inliers 1, -1, 0.25: the
    scale comes from the inliers alone (1 / 127), the protected value is kept
    exactly; plain per-group INT8 would quantize 1.0 to a single step of
    100 / 127."""
    x = np.zeros((1, 512), np.float32)
    x[0, :4] = [100.0, 1.0, -1.0, 0.25]
    q, s, v = Q.quantize_int8_outlier(x, [0] + list(range(400, 424)))
    assert s[0, 0] == np.float32(1.0) / np.float32(127.0)
    assert q[0, :4].tolist() == [0, 127, -127, 32]        # 0.25 * 127 = 31.75 -> 32
    assert v[0, 0] == 100.0 and v.shape == (1, 25)
    xh = Q.dequantize_int8_outlier(q, s, v, [0] + list(range(400, 424)))
    assert xh[0, 0] == 100.0 and xh[0, 1] == np.float32(127) * s[0, 0]
    q8, s8 = Q.quantize_sym_int8(x, 16)
    assert q8[0, 1] == 1 and s8[0, 0] == np.float32(100.0) / np.float32(127.0)


def test_outlier_format_exact_channels_and_nearest_levels():
    c = synth_latent(T=64)
    o = Q.select_outlier_channels(c)
    d = Q.quantize_token_rows(c, synth_kpe(T=64), Q.FMT_INT8_OUTLIER, Q.FMT_BF16, outliers=o)
    assert np.array_equal(d["c_hat"][:, o], c[:, o]) and np.all(d["c_codes"][:, o] == 0)
    inl = np.setdiff1d(np.arange(512), o)
    levels = np.arange(-127, 128, dtype=np.float64)
    for t in range(0, 64, 9):
        for g in range(32):
            ch = [k for k in range(16 * g, 16 * g + 16) if k in set(inl.tolist())]
            a = max((abs(float(c[t, k])) for k in ch), default=0.0)
            s = np.float32(np.float32(a) / np.float32(127.0))
            assert d["c_scale"][t, g] == s
            for k in ch:
                if s == 0:
                    assert d["c_codes"][t, k] == 0
                    continue
                qf = np.float64(np.float32(c[t, k]) / s)       # the fp32 quotient, then nearest level
                best = levels[np.argmin(np.abs(levels - qf))]
                assert abs(d["c_codes"][t, k] - best) <= (1 if abs(abs(qf - best) - 0.5) < 1e-6 else 0)
    exp = np.max(np.abs(d["c_hat"]), axis=1).astype(np.float32)
    assert np.array_equal(d["c_bound"].view(np.uint32), exp.view(np.uint32))


def test_error_outlier_protection_beats_per_group_int8():
    """English report §4.3: row C (mixed, outlier-protected) 0.007 below row A
    (per-group INT8) 0.011 - on the synthetic latent, whose outlier channels
    the calibration finds."""
    c = synth_latent(T=512, layer=3)
    o = Q.select_outlier_channels(c[:128])                  # calibrated on a prefix
    d = Q.quantize_token_rows(c, synth_kpe(T=512, layer=3), Q.FMT_INT8_OUTLIER, Q.FMT_BF16, outliers=o)
    q8, s8 = Q.quantize_sym_int8(c, 16)
    e_mixed = Q.relative_error(c, d["c_hat"])[0]
    e_int8 = Q.relative_error(c, Q.dequantize_sym_int8(q8, s8, 16))[0]
    assert e_mixed < 0.8 * e_int8
