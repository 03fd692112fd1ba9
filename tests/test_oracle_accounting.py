"""Pins for the byte accounting against the figures the two reports print.

Chinese report "DeepSeek-V2-Lite MLA 吸收式 KV 缓存优化 — 完整实验报告" §1.2, §1.3,
§3.1, §4.1; English report "Absorbed MLA Cache Optimization on DeepSeek-V2-Lite
— Technical Report" §1.3, §2.2, §4.3.
"""

from oracle import accounting as acc

B16, I8, I4 = acc.FMT_BF16, acc.FMT_INT8, acc.FMT_INT4


def r1(x):
    return round(x, 1)


def test_expanded_bytes():
    # EN §1.3: (192+128) x 16 heads x 2 B = 10,240 B per layer; 270 KB per token.
    assert acc.expanded_layer_bytes() == 10240
    assert acc.token_bytes(acc.expanded_layer_bytes()) == 276480   # CN §1.2
    assert acc.kib(276480) == 270.0


def test_mla_theoretical_row():
    # CN §1.2 / EN §1.2: (512+64+128) x 27 = 19,008 B = 18.6 KB, 14.5x.
    assert acc.mla_theoretical_token_bytes() == 19008
    assert r1(acc.kib(19008)) == 18.6
    assert r1(acc.ratio(276480, 19008)) == 14.5


def test_absorbed_latent_bf16():
    # EN §2.2: (512+64) x 2 = 1,152 B per layer, 30.4 KB; CN §3.1: 8.9x.
    per_layer = acc.layer_bytes(B16, B16)
    assert per_layer == 1152
    tok = acc.token_bytes(per_layer)
    assert tok == 31104
    assert r1(acc.kib(tok)) == 30.4
    assert r1(acc.ratio(276480, tok)) == 8.9


def test_code_only_quantized_rows():
    # EN §2.2: latent8 + kpe16 = 512 + 128 = 640 B, 16.9 KB (16x, EN §4.3).
    assert acc.layer_bytes(I8, B16) == 640
    assert r1(acc.kib(acc.token_bytes(640))) == 16.9
    assert acc.ratio(276480, acc.token_bytes(640)) == 16.0
    # CN §4.1 / EN §4.3 row A: latent8 + kpe8 -> 15.2 KB, 17.8x.
    t8 = acc.token_bytes(acc.layer_bytes(I8, I8))
    assert acc.layer_bytes(I8, I8) == 576
    assert r1(acc.kib(t8)) == 15.2 and r1(acc.ratio(276480, t8)) == 17.8
    # EN §4.3 row D: INT4 + kpe8 -> 8.4 KB, 32x.
    t4 = acc.token_bytes(acc.layer_bytes(I4, I8))
    assert acc.layer_bytes(I4, I8) == 320
    assert r1(acc.kib(t4)) == 8.4 and acc.ratio(276480, t4) == 32.0
    # CN §4.1 extreme row: 7.6 KB, 35.6x needs k_pe at 4 bits as well
    # (288 B per layer); recorded as the pages' inconsistency with EN's 8.4 KB.
    t44 = acc.token_bytes(acc.layer_bytes(I4, I4))
    assert acc.layer_bytes(I4, I4) == 288
    assert r1(acc.kib(t44)) == 7.6 and r1(acc.ratio(276480, t44)) == 35.6


def test_metadata_overhead_reported_on_top():
    # fp32 scale per 16-channel group (32) and per 8-channel k_pe group (8),
    # plus fp32 zero-points for asymmetric INT4.
    assert acc.layer_bytes(I8, I8, metadata=True) == 512 + 64 + 4 * 32 + 4 * 8 == 736
    assert acc.layer_bytes(I4, I8, metadata=True) == 256 + 64 + 8 * 32 + 4 * 8 == 608
    assert acc.layer_bytes(B16, B16, metadata=True) == 1152
    assert acc.token_bytes(736) == 19872 and r1(acc.kib(19872)) == 19.4
    assert acc.token_bytes(608) == 16416 and r1(acc.kib(16416)) == 16.0


def test_symmetric_int4_formats_metadata():
    # the 7.6 KB scheme as stored: asymmetric INT4 latent (scale + zero) and
    # symmetric INT4 k_pe (scale only): 288 B of codes + 288 B of metadata
    I4S = acc.FMT_INT4_SYM
    assert acc.layer_bytes(I4, I4S) == 288
    assert acc.layer_bytes(I4, I4S, metadata=True) == 256 + 32 + 8 * 32 + 4 * 8 == 576
    assert acc.layer_bytes(I4S, I8, metadata=True) == 256 + 64 + 4 * 32 + 4 * 8 == 480
    assert acc.layer_bytes(I4S, I4S, metadata=True) == 256 + 32 + 4 * 32 + 4 * 8 == 448


def test_int8_block_count_formats_metadata():
    # EN §5.1 sweep (8 / 32 / 64 blocks) and CN §3.2 per-token: same 512 B of
    # codes, one fp32 scale per block
    assert acc.layer_bytes(acc.FMT_INT8_G64, I8, metadata=True) == 512 + 4 * 8 + 96 == 640
    assert acc.layer_bytes(acc.FMT_INT8_G32, I8, metadata=True) == 512 + 4 * 16 + 96 == 672
    assert acc.layer_bytes(I8, I8, metadata=True) == 736
    assert acc.layer_bytes(acc.FMT_INT8_G8, I8, metadata=True) == 512 + 4 * 64 + 96 == 864
    assert acc.layer_bytes(acc.FMT_INT8_TOKEN, I8, metadata=True) == 512 + 4 + 96 == 612
    assert acc.layer_bytes(acc.FMT_INT8_G8, I8) == acc.layer_bytes(I8, I8) == 576


def test_capacity_in_10gb():
    # CN §4.1: INT8 69万 tokens, INT4 138万 tokens; EN §4.3: 39K / 690K / 620K / 1.24M.
    cap = lambda per_layer: acc.capacity_tokens(acc.token_bytes(per_layer))
    assert acc.capacity_tokens(276480) == 38836            # "39K"
    assert cap(576) == 690420                              # "690K" / 69万
    assert cap(640) == 621378                              # "620K"
    assert cap(320) == 1242756                             # "1.24M"
    assert cap(288) == 1380840                             # 138万
    # EN §4.3 prints 340K for the bf16 latent; the arithmetic gives 345,210
    # (a 1.5 % discrepancy on the page, recorded, not reproduced).
    assert cap(1152) == 345210


def test_outlier_protected_row():
    # EN §4.3 row C: 18.2 KB, 14.8x, 580K tokens in 10 GB.  Read as INT8
    # latent + 25 protected bf16 channels + bf16 k_pe = 690 B per layer.
    I8O = acc.FMT_INT8_OUTLIER
    assert acc.layer_bytes(I8O, B16) == 512 + 2 * 25 + 128 == 690
    t = acc.token_bytes(690)
    assert r1(acc.kib(t)) == 18.2 and r1(acc.ratio(276480, t)) == 14.8
    assert acc.capacity_tokens(t) == 576350 and round(acc.capacity_tokens(t), -4) == 580000
    # 24 or 26 protected channels miss one of the three printed figures
    for k in (24, 26):
        tk = acc.token_bytes(512 + 2 * k + 128)
        assert not (r1(acc.kib(tk)) == 18.2 and r1(acc.ratio(276480, tk)) == 14.8
                    and round(acc.capacity_tokens(tk), -4) == 580000)
    assert acc.layer_bytes(I8O, B16, metadata=True) == 690 + 4 * 32
    assert acc.layer_bytes(I8O, I8, metadata=True) == 512 + 50 + 64 + 4 * 32 + 4 * 8
