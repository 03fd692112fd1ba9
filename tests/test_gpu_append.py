"""mla_cache_append on the GPU against the oracle's quantizers: codes, scales
and zero-points bit-exact, for every format pair, including degenerate and
half-way groups, skipped and out-of-range slots, and a prefill-sized append."""

import numpy as np
import pytest
import torch

import synth
import mla_latent_kv_append_gb300 as mla
from tests._helpers import ALL_FORMATS, FMT_NAME, assert_fields_match, read_tokens

pytestmark = pytest.mark.gpu


def special_rows():
    """Hand-built latent rows: zeros, constants, half-way ties, +-127 multiples,
    a single outlier, a narrow all-positive range (large zero-point)."""
    rows = np.zeros((8, 512), np.float32)
    rows[1] = 3.25
    rows[2] = -0.75
    tie = np.array([127, 0.5, 1.5, 2.5, 3.5, -0.5, -1.5, -2.5, 126.5, -126.5, 0, 7, -7, 0.25, 0.75, 100.5], np.float32)
    rows[3] = np.tile(tie, 32)
    rows[4] = np.tile(np.array([127, -127] * 8, np.float32), 32)
    rows[5, ::16] = -1000.0
    rows[5, 1::16] = 1e-3
    rows[6] = 100.0 + np.arange(512, dtype=np.float32) % 16 * 0.0625
    rows[7] = np.tile(np.array([-1, 14, 2.5, 3.5, -0.5, 0.5, 0, 13.5, 1, 1, 1, 1, 1, 1, 1, 1], np.float32), 32)
    return synth.bf16_rne(rows)


def make_tokens(n, seed=21):
    cos, sin = synth.rope_tables(n)
    c = synth.latent_bf16(seed, 0, 0, 0, n)
    k = synth.kpe_bf16(seed, 0, 0, 0, n, cos, sin)
    sp = special_rows()[:n]
    c[:len(sp)] = sp
    k[:len(sp)] = sp[:, :64]
    return c, k


def to_dev(bits):
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()


@pytest.mark.parametrize("lf,kf", ALL_FORMATS, ids=["%s-%s" % (FMT_NAME[a], FMT_NAME[b]) for a, b in ALL_FORMATS])
def test_append_bit_exact(lf, kf):
    n, pages = 300, 8
    c, k = make_tokens(n)
    rng = np.random.default_rng(lf * 10 + kf)
    slots = rng.permutation(pages * 64)[:n].astype(np.int32)
    cache = mla.CacheLayer(pages, lf, kf)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.mla_cache_append(cache, to_dev(c), to_dev(k), torch.from_numpy(slots).cuda(), err)
    torch.cuda.synchronize()
    assert err.item() == 0
    got = read_tokens(cache.pool.cpu().numpy(), cache.layout, lf, kf, slots)
    assert_fields_match(got, c, k, lf, kf)


def test_append_skips_minus_one_and_flags_out_of_range():
    lf, kf = mla.FMT_INT8_SYM, mla.FMT_INT8_SYM
    c, k = make_tokens(6)
    cache = mla.CacheLayer(2, lf, kf)
    before = cache.pool.clone()
    slots = torch.tensor([-1, 128, -5, 1 << 30, -1, 127], dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.mla_cache_append(cache, to_dev(c), to_dev(k), slots, err)
    torch.cuda.synchronize()
    assert err.item() == mla.DEVERR_SLOT
    after = cache.pool.cpu().numpy()
    changed = np.nonzero(after != before.cpu().numpy())[0]
    # only the token at slot 127 (page 1, offset 63) was written
    got = read_tokens(after, cache.layout, lf, kf, [127])
    assert_fields_match(got, c[5:6], k[5:6], lf, kf)
    assert changed.min() >= cache.layout.page_bytes


def test_append_empty_is_noop():
    cache = mla.CacheLayer(1, mla.FMT_INT4_ASYM, mla.FMT_INT8_SYM)
    z = torch.empty((0, 512), dtype=torch.bfloat16, device="cuda")
    mla.mla_cache_append(cache, z, torch.empty((0, 64), dtype=torch.bfloat16, device="cuda"),
                         torch.empty(0, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert int(cache.pool.sum().item()) == 0


@pytest.mark.parametrize("lf", [mla.FMT_INT8_SYM, mla.FMT_INT4_ASYM])
def test_prefill_sized_append(lf):
    """An 8192-token append (the mixed serving step's prefill) into scattered pages."""
    n = 8192
    c, k = make_tokens(n, seed=5)
    pages = n // 64 + 3
    perm = synth.page_permutation(99, pages)
    t = np.arange(n)
    slots = (perm[t // 64].astype(np.int64) * 64 + t % 64).astype(np.int32)
    cache = mla.CacheLayer(pages, lf, mla.FMT_INT8_SYM)
    mla.mla_cache_append(cache, to_dev(c), to_dev(k), torch.from_numpy(slots).cuda())
    torch.cuda.synchronize()
    got = read_tokens(cache.pool.cpu().numpy(), cache.layout, lf, mla.FMT_INT8_SYM, slots)
    assert_fields_match(got, c, k, lf, mla.FMT_INT8_SYM)


def near_tie_rows(n_rows, lf, seed=123):
    """Latent rows whose per-group quotients x / s sit at or within a few fp32
    ulps of half-integers (the cases where a division that is not correctly
    rounded would change a code).  Each group holds its extreme values, so
    the scale is known on the host."""
    rng = np.random.default_rng(seed)
    b16 = lambda v: np.float32(synth.bf16_to_f32(synth.bf16_rne(np.array([v], np.float32)))[0])
    rows = np.zeros((n_rows, 512), np.float32)
    for i in range(n_rows):
        for g in range(32):
            if lf == mla.FMT_INT8_SYM:
                a = b16(abs(rng.standard_normal()) * 2.0 ** rng.integers(-20, 20)) or np.float32(1)
                s = np.float32(a / np.float32(127))
                vals, lo, hi = [a], -a, a
            else:
                mn = b16(rng.standard_normal() * 2.0 ** rng.integers(-10, 10))
                mx = b16(mn + abs(rng.standard_normal()) * 2.0 ** rng.integers(-8, 8))
                if mx <= mn:
                    mx = b16(mn + abs(mn) * 0.05 + 1e-3)
                s = np.float32(np.float32(mx - mn) / np.float32(15))
                vals, lo, hi = [mn, mx], mn, mx
            k0 = int(np.floor(lo / np.float64(s)))
            tries = 0
            while len(vals) < 16 and tries < 200:
                tries += 1
                k = rng.integers(k0, k0 + 255 if lf == mla.FMT_INT8_SYM else k0 + 16)
                x = b16((k + 0.5) * np.float64(s))
                if lo <= x <= hi:
                    vals.append(x)
            vals += [lo] * (16 - len(vals))
            rows[i, 16 * g:16 * g + 16] = rng.permutation(np.array(vals, np.float32))
    return synth.bf16_rne(rows)


@pytest.mark.parametrize("lf", [mla.FMT_INT8_SYM, mla.FMT_INT4_ASYM])
def test_near_tie_quotients_bit_exact(lf):
    n = 256
    c = near_tie_rows(n, lf)
    k = c[:, :64].copy()
    slots = np.arange(n, dtype=np.int32)
    cache = mla.CacheLayer(n // 64, lf, mla.FMT_INT8_SYM)
    mla.mla_cache_append(cache, to_dev(c), to_dev(k), torch.from_numpy(slots).cuda())
    torch.cuda.synchronize()
    got = read_tokens(cache.pool.cpu().numpy(), cache.layout, lf, mla.FMT_INT8_SYM, slots)
    assert_fields_match(got, c, k, lf, mla.FMT_INT8_SYM)
