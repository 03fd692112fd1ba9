"""The outlier-protected mixed-precision format (INT8 latent with 25
protected bf16 channels per layer; English report §4.3 row C) on the GPU:
the calibration call against the oracle's selection, quantize-on-write bit
for bit (codes, scales, protected values, bound), and the decode step
against the oracle's attention over the same dequantized latents."""

import numpy as np
import pytest
import torch

import synth
import mla_latent_kv_append_gb300 as mla
from oracle import quant as Q
from synth.workload import Workload
from tests._helpers import F_I8OUT, assert_fields_match, read_tokens
from tests.test_gpu_decode import run_and_check

pytestmark = pytest.mark.gpu


def to_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


@pytest.mark.parametrize("layer", [0, 5, 26])
def test_calibration_matches_the_oracle(layer):
    c = synth.latent_bf16(31, layer, 0, 0, 700, stats=synth.channel_stats(31, layer))
    got = mla.mla_select_outlier_channels(to_dev(c)).cpu().numpy()
    exp = Q.select_outlier_channels(synth.bf16_to_f32(c))
    assert np.array_equal(got, exp)
    # the synthetic latent's five outlier channels are among them
    big = np.argsort(-np.abs(synth.bf16_to_f32(c)).max(axis=0))[:5]
    assert set(big.tolist()) <= set(got.tolist())


def test_calibration_ties_and_a_single_row():
    x = np.zeros((1, 512), np.float32)
    x[0, [3, 9, 400, 511]] = [-2.0, 2.0, 2.0, 5.0]              # ties at 2.0: lower index first
    x[0, 100:121] = 1.0                                          # 21 equal channels fill the rest
    c = synth.bf16_rne(x)
    got = mla.mla_select_outlier_channels(to_dev(c)).cpu().numpy()
    assert np.array_equal(got, Q.select_outlier_channels(synth.bf16_to_f32(c)))
    assert got.tolist() == sorted([3, 9, 400, 511] + list(range(100, 121)))


def edge_rows(outl):
    """Rows with protected channels in every role: a group made only of
    protected channels (its inlier scale is 0), a protected channel far
    larger than its group, negative protected values, zeros."""
    rows = np.zeros((6, 512), np.float32)
    rows[1] = 0.5
    rows[1, outl] = -300.0
    rows[2] = np.tile(np.linspace(-3, 3, 16, dtype=np.float32), 32)
    rows[2, outl] = 1e4
    rows[3, outl] = np.linspace(-7, 7, len(outl), dtype=np.float32)
    rows[4] = -1.0
    rows[5] = np.tile(np.array([127, -127] * 8, np.float32), 32)
    rows[5, outl[::2]] = 0.0
    return synth.bf16_rne(rows)


@pytest.mark.parametrize("kf", [mla.FMT_BF16, mla.FMT_INT8_SYM], ids=["kpe-bf16", "kpe-int8"])
def test_append_bit_exact(kf):
    n, pages = 300, 8
    cos, sin = synth.rope_tables(n)
    c = synth.latent_bf16(23, 1, 0, 0, n, stats=synth.channel_stats(23, 1))
    k = synth.kpe_bf16(23, 1, 0, 0, n, cos, sin)
    # the protected set: the 16 channels of group 3 plus 9 others (group 3
    # keeps no inlier at all)
    outl = sorted(set(range(48, 64)) | {0, 1, 100, 101, 250, 333, 334, 400, 511})
    assert len(outl) == 25
    sp = edge_rows(np.array(outl))
    c[:len(sp)] = sp
    slots = np.random.default_rng(kf).permutation(pages * 64)[:n].astype(np.int32)
    cache = mla.CacheLayer(pages, F_I8OUT, kf, outlier_channels=outl)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.mla_cache_append(cache, to_dev(c), to_dev(k), torch.from_numpy(slots).cuda(), err)
    torch.cuda.synchronize()
    assert err.item() == 0
    got = read_tokens(cache.pool.cpu().numpy(), cache.layout, F_I8OUT, kf, slots)
    assert_fields_match(got, c, k, F_I8OUT, kf, outliers=outl)
    assert np.all(got["c_codes"][:, outl] == 0)
    assert np.all(got["c_scale"][:, 3] == 0)                     # group 3 is all protected


@pytest.mark.parametrize("kf", [mla.FMT_BF16, mla.FMT_INT8_SYM], ids=["kpe-bf16", "kpe-int8"])
def test_decode_against_the_oracle(kf):
    """Lengths for the split path and the short exact path, several splits
    per sequence; the workload's calibration must equal the oracle's."""
    lens = [5000, 300, 64, 1, 257, 0, 2049]
    wl = Workload(2, 16, lens, F_I8OUT, kf, seed=91)
    from tests._helpers import OracleCache
    oc = OracleCache(wl)
    for l in range(wl.L):
        assert np.array_equal(np.array(wl.outliers[l]), oc.outliers(l))
    _, worst = run_and_check(wl)
    assert worst < 2e-3


def test_decode_64_heads_and_split_counts():
    wl = Workload(1, 64, [3000, 700], F_I8OUT, mla.FMT_BF16, seed=92)
    run_and_check(wl)
    wl = Workload(1, 16, [4100], F_I8OUT, mla.FMT_BF16, seed=93)
    for ns in (1, 7, 150):
        run_and_check(wl, num_splits=ns)
