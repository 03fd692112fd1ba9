"""The range-split oracle used by the full-size parity tests equals the
direct oracle: tokens regenerated per range match the whole-sequence
generator, and merged range partials match the unsplit absorbed decode."""

import numpy as np

import synth
from oracle import attention as A
from oracle import quant as Q
from tests._oracle_pool import make_pool, oracle_outputs, tokens_bf16


def test_ranges_regenerate_the_same_tokens():
    seed, layer, b, T = 5, 3, 2, 300
    cos, sin = synth.rope_tables(T)
    stats = synth.channel_stats(seed, layer)
    c, k = synth.sequence_bf16(seed, layer, b, T, cos, sin, stats=stats)
    for t0, t1 in [(0, 64), (100, 299), (250, 300), (299, 300)]:
        cc, kk = tokens_bf16(seed, layer, b, T, t0, t1, stats, cos, sin)
        assert np.array_equal(cc, c[t0:t1]) and np.array_equal(kk, k[t0:t1])


def test_merged_ranges_equal_direct_oracle():
    seed, H, lens = 9, 16, [700, 129, 64]
    lf, kf = Q.FMT_INT4, Q.FMT_INT8
    pool = make_pool(2)
    try:
        got = oracle_outputs(pool, seed, [0, 1], range(len(lens)), lens, H, lf, kf, span=256)
    finally:
        pool.close()
        pool.join()
    for l in (0, 1):
        qn = synth.bf16_to_f32(synth.q_nope_bf16(seed, l, len(lens), H))
        qp = synth.bf16_to_f32(synth.q_pe_bf16(seed, l, len(lens), H))
        wuk = synth.bf16_to_f32(synth.w_uk_bf16(seed, l, H))
        wuv = synth.bf16_to_f32(synth.w_uv_bf16(seed, l, H))
        for b, T in enumerate(lens):
            cos, sin = synth.rope_tables(T)
            c, k = synth.sequence_bf16(seed, l, b, T, cos, sin, stats=synth.channel_stats(seed, l))
            d = Q.quantize_token_rows(synth.bf16_to_f32(c), synth.bf16_to_f32(k), lf, kf)
            _, ol, lse, o = A.absorbed_decode_full(qn[b], qp[b], wuk, wuv, d["c_hat"], d["kpe_hat"])
            g_ol, g_lse, g_o = got[(l, b)]
            assert A.max_rel_error(g_ol, ol) < 1e-12
            assert A.max_rel_error(g_o, o) < 1e-12
            assert np.max(np.abs(g_lse - lse)) < 1e-12
