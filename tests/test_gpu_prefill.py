"""mla_prefill_absorbed on the GPU against the oracle: the queries of a chunk
of just-appended tokens of one sequence attend causally to the positions up
to their own.  Per query row: o_lat and o within max relative error 2e-3,
lse within 2e-3 absolute, on the same codes (the cache is written by the
library's append and quantized by the oracle from the same bf16 tokens)."""

import numpy as np
import pytest
import torch

import mla_latent_kv_append_gb300 as mla
import synth
import synth.device as sd
from oracle import attention as A
from oracle import quant as Q
from tests._helpers import ATTN_TOL, FMT_NAME

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, params=["decode_kernels", "auto"])
def prefill_path(request):
    """Every test runs on the decode-kernel path and on the automatic choice
    (the tensor cores for prefixes of 257 to 65536 tokens and 8192 rows or
    more, or 2048 rows or more once the prefixes reach 4096 tokens)."""
    prev = mla.mla_set_prefill_path(mla.PREFILL_DECODE_KERNELS if request.param == "decode_kernels"
                                    else mla.PREFILL_AUTO)
    yield request.param
    mla.mla_set_prefill_path(prev)


class Chunk:
    """One sequence of T = ctx_before + n tokens in a paged cache (pages in a
    seeded order, the pool's other bytes 0xFF), plus the chunk's queries."""

    def __init__(self, lf, kf, ctx_before, n, H, seed, layer=0, spare_pages=3):
        self.lf, self.kf, self.ctx_before, self.n, self.H, self.seed, self.layer = lf, kf, ctx_before, n, H, seed, layer
        self.T = T = ctx_before + n
        pages = (T + 63) // 64
        outl = None
        if lf == mla.FMT_INT8_OUTLIER:     # the library's calibration on the workload's sample rows
            sample = torch.empty((synth.CALIBRATION_TOKENS, synth.D_C), dtype=torch.bfloat16, device="cuda")
            sd.latent_into(sample, seed, layer, 0, 0, sd.LayerStats(seed, layer))
            outl = mla.mla_select_outlier_channels(sample).cpu().tolist()
        self.cache = mla.CacheLayer(pages + spare_pages, lf, kf, outlier_channels=outl)
        self.cache.pool.fill_(0xFF)
        perm = synth.page_permutation(seed, pages + spare_pages)[:pages].astype(np.int32)
        self.block_table = torch.from_numpy(perm).cuda()
        st = sd.LayerStats(seed, layer)
        rope = sd.RopeTables(max(1, T))
        c = torch.empty((T, synth.D_C), dtype=torch.bfloat16, device="cuda")
        k = torch.empty((T, synth.D_R), dtype=torch.bfloat16, device="cuda")
        sd.latent_into(c, seed, layer, 0, 0, st)
        sd.kpe_into(k, seed, layer, 0, 0, rope)
        t = np.arange(T)
        slots = torch.from_numpy((perm[t // 64].astype(np.int64) * 64 + t % 64).astype(np.int32)).cuda()
        mla.mla_cache_append(self.cache, c, k, slots)
        self.q_nope = sd.prefill_q_nope(seed, layer, n, H)
        self.q_pe = sd.prefill_q_pe(seed, layer, n, H)
        self.w_uk = sd.w_uk(seed, layer, H)
        self.w_uv = sd.w_uv(seed, layer, H)

    def run(self):
        n, H = self.n, self.H
        q_lat = torch.empty((n, H, 512), dtype=torch.float32, device="cuda")
        mla.mla_q_absorb(self.q_nope, self.w_uk, q_lat)
        ws = torch.empty(mla.mla_prefill_workspace_bytes(n, H), dtype=torch.uint8, device="cuda")
        o_lat = torch.empty((n, H, 512), dtype=torch.float32, device="cuda")
        lse = torch.empty((n, H), dtype=torch.float32, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        mla.mla_prefill_absorbed(self.cache, q_lat, self.q_pe, self.block_table, self.ctx_before, ws, o_lat, lse, err)
        o = torch.empty((n, H, 128), dtype=torch.float32, device="cuda")
        mla.mla_out_unabsorb(o_lat, self.w_uv, o)
        torch.cuda.synchronize()
        assert err.item() == 0
        return o_lat.cpu().numpy(), lse.cpu().numpy(), o.cpu().numpy()

    def oracle(self, rows):
        """(o_lat, lse, o) of the oracle for the chunk's query rows `rows`."""
        seed, layer, H = self.seed, self.layer, self.H
        cos, sin = synth.rope_tables(max(1, self.T))
        c = synth.latent_bf16(seed, layer, 0, 0, self.T, stats=synth.channel_stats(seed, layer))
        k = synth.kpe_bf16(seed, layer, 0, 0, self.T, cos, sin)
        outl = None
        if self.lf == Q.FMT_INT8_OUTLIER:  # the oracle's own calibration
            outl = Q.select_outlier_channels(synth.bf16_to_f32(synth.calibration_latent_bf16(seed, layer)))
        d = Q.quantize_token_rows(synth.bf16_to_f32(c), synth.bf16_to_f32(k), self.lf, self.kf, outliers=outl)
        qn = synth.bf16_to_f32(synth.prefill_q_nope_bf16(seed, layer, rows, H))
        qp = synth.bf16_to_f32(synth.prefill_q_pe_bf16(seed, layer, rows, H))
        wuk = synth.bf16_to_f32(synth.w_uk_bf16(seed, layer, H))
        wuv = synth.bf16_to_f32(synth.w_uv_bf16(seed, layer, H))
        out = []
        for a, i in enumerate(rows):
            t = self.ctx_before + int(i) + 1
            q_lat = A.absorb_q(qn[a], wuk)
            o_lat, lse = A.absorbed_decode(q_lat, qp[a], d["c_hat"][:t], d["kpe_hat"][:t])
            out.append((o_lat, lse, A.unabsorb_o(o_lat, wuv)))
        return out


def check(ch, rows=None):
    o_lat, lse, o = ch.run()
    rows = list(range(ch.n)) if rows is None else rows
    worst = 0.0
    for i, (ol_ref, lse_ref, o_ref) in zip(rows, ch.oracle(rows)):
        e1 = A.max_rel_error(o_lat[i], ol_ref)
        e2 = A.max_rel_error(o[i], o_ref)
        e3 = float(np.max(np.abs(lse[i] - lse_ref)))
        worst = max(worst, e1, e2)
        assert e1 < ATTN_TOL and e2 < ATTN_TOL and e3 < ATTN_TOL, (i, e1, e2, e3)
    return worst


FORMATS = [(mla.FMT_INT8_SYM, mla.FMT_INT8_SYM), (mla.FMT_INT4_ASYM, mla.FMT_INT8_SYM), (mla.FMT_BF16, mla.FMT_BF16),
           (mla.FMT_INT4_SYM, mla.FMT_INT4_SYM), (mla.FMT_INT8_G8, mla.FMT_INT8_SYM),
           (mla.FMT_INT8_TOKEN, mla.FMT_INT8_SYM), (mla.FMT_INT8_G32, mla.FMT_INT8_SYM),
           (mla.FMT_INT8_G64, mla.FMT_INT8_SYM), (mla.FMT_INT4_ASYM, mla.FMT_INT4_SYM),
           (mla.FMT_BF16, mla.FMT_INT8_SYM), (mla.FMT_INT8_OUTLIER, mla.FMT_BF16)]


@pytest.mark.parametrize("lf,kf", FORMATS, ids=["%s-%s" % (FMT_NAME[a], FMT_NAME[b]) for a, b in FORMATS])
def test_prefill_from_empty(lf, kf):
    """A 200-token prompt into an empty sequence, every query row."""
    check(Chunk(lf, kf, 0, 200, 16, seed=90))


@pytest.mark.parametrize("ctx_before,n", [(1, 1), (63, 65), (100, 77), (640, 33)])
def test_chunked_prefill_after_context(ctx_before, n):
    """A chunk appended after ctx_before cached tokens (page and chunk
    boundaries on both sides), every query row."""
    check(Chunk(mla.FMT_INT8_SYM, mla.FMT_INT8_SYM, ctx_before, n, 16, seed=91))


def test_prefill_64_heads():
    check(Chunk(mla.FMT_INT4_ASYM, mla.FMT_INT8_SYM, 30, 150, 64, seed=92))


def test_prefill_slices():
    """2100 queries: two slices of the query batch; rows around the slice
    boundary, the first and last rows and a sample are compared."""
    ch = Chunk(mla.FMT_INT8_SYM, mla.FMT_INT8_SYM, 5, 2100, 16, seed=93)
    rng = np.random.default_rng(93)
    rows = sorted(set([0, 1, 2045, 2046, 2047, 2048, 2049, 2099] + [int(r) for r in rng.integers(0, 2100, 12)]))
    check(ch, rows)


def test_prefill_bad_page_is_flagged():
    ch = Chunk(mla.FMT_INT8_SYM, mla.FMT_INT8_SYM, 0, 100, 16, seed=94)
    ch.block_table[1] = ch.cache.num_pages + 3
    q_lat = torch.zeros((100, 16, 512), dtype=torch.float32, device="cuda")
    ws = torch.empty(mla.mla_prefill_workspace_bytes(100, 16), dtype=torch.uint8, device="cuda")
    o_lat = torch.empty((100, 16, 512), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.mla_prefill_absorbed(ch.cache, q_lat, ch.q_pe, ch.block_table, 0, ws, o_lat, None, err)
    torch.cuda.synchronize()
    assert err.item() == mla.DEVERR_PAGE
    assert np.all(np.isfinite(o_lat.cpu().numpy()))


@pytest.mark.parametrize("name", ["mixed_h64_int8", "mixed_h64_int4", "mixed_h64_bf16"])
def test_full_size_prefill_sampled(name):
    """The 64-head serving workload's 8192-token prefill chunk, through the
    workload's own step (its append, then the chunk's attention): query rows
    at the page, chunk and slice boundaries plus a seeded sample, each
    against the oracle over its prefix."""
    import gc
    import bench
    from synth.workload import DecodeStep, PrefillStep, Workload
    gc.collect()
    torch.cuda.empty_cache()
    cfg = bench.CONFIGS[name]
    seq = bench.seq_lens_for(cfg, bench.SEED)
    lf, kf = bench.FMT[cfg["latent"]], bench.FMT[cfg["kpe"]]
    wl = Workload(1, cfg["heads"], seq, lf, kf, bench.SEED, prefill=cfg["prefill"])
    DecodeStep(wl).run()                      # appends the prefill chunk
    pre = PrefillStep(wl)
    keep = torch.empty((1, wl.prefill, wl.H, 512), dtype=torch.float32, device="cuda")
    o = pre.run(keep_o_lat=keep)
    torch.cuda.synchronize()
    assert pre.dev_err.item() == 0
    P, H = wl.prefill, wl.H
    rng = np.random.default_rng(len(name))
    rows = sorted(set([0, 1, 31, 32, 63, 64, 2047, 2048, 4095, P - 1] + [int(r) for r in rng.integers(0, P, 14)]))
    c_bits, k_bits = wl.host_prefill(0)
    d = Q.quantize_token_rows(synth.bf16_to_f32(c_bits), synth.bf16_to_f32(k_bits), lf, kf)
    qn = synth.bf16_to_f32(synth.prefill_q_nope_bf16(bench.SEED, 0, rows, H))
    qp = synth.bf16_to_f32(synth.prefill_q_pe_bf16(bench.SEED, 0, rows, H))
    wuk = synth.bf16_to_f32(synth.w_uk_bf16(bench.SEED, 0, H))
    wuv = synth.bf16_to_f32(synth.w_uv_bf16(bench.SEED, 0, H))
    ol_h, lse_h, o_h = keep[0].cpu().numpy(), pre.lse[0].cpu().numpy(), o[0].cpu().numpy()
    worst = 0.0
    for a, i in enumerate(rows):
        q_lat = A.absorb_q(qn[a], wuk)
        ol_ref, lse_ref = A.absorbed_decode(q_lat, qp[a], d["c_hat"][:i + 1], d["kpe_hat"][:i + 1])
        o_ref = A.unabsorb_o(ol_ref, wuv)
        e1 = A.max_rel_error(ol_h[i], ol_ref)
        e2 = A.max_rel_error(o_h[i], o_ref)
        e3 = float(np.max(np.abs(lse_h[i] - lse_ref)))
        worst = max(worst, e1, e2)
        assert e1 < ATTN_TOL and e2 < ATTN_TOL and e3 < ATTN_TOL, (name, i, e1, e2, e3)
    print("%s prefill: %d rows compared, worst max-rel error %.2e" % (name, len(rows), worst))


def test_prefill_outlier_format_past_the_exact_length():
    """The outlier-protected format with prefixes long enough for the split
    path (query rows at 301 .. 700 tokens), 32 heads."""
    check(Chunk(mla.FMT_INT8_OUTLIER, mla.FMT_INT8_SYM, 300, 400, 32, seed=91),
          rows=list(range(0, 400, 7)) + [399])
