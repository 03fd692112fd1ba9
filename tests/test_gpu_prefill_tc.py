"""The tensor-core prefill path (mla_set_prefill_path(PREFILL_TENSOR_CORES))
against the oracle, on prefixes long enough (> 256 tokens) that its own
output is what the call returns: every format pair, ragged row and key
tiles (n H not a multiple of 128, key counts off the 128-key tile, head
counts that do not divide 128), the query-slice boundary, and rows below
256 tokens that the exact recomputation takes over.  Per query row: o_lat
and o within max relative error 2e-3, lse within 2e-3 absolute."""

import numpy as np
import pytest

import mla_latent_kv_append_gb300 as mla
from tests._helpers import FMT_NAME
from tests.test_gpu_prefill import Chunk, check

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def tensor_core_path():
    prev = mla.mla_set_prefill_path(mla.PREFILL_TENSOR_CORES)
    yield
    mla.mla_set_prefill_path(prev)


# every (latent, k_pe) pair the library supports: the key pass is compiled per pair
ALL_PAIRS = ([(lf, kf) for lf in (mla.FMT_BF16, mla.FMT_INT8_SYM, mla.FMT_INT4_ASYM, mla.FMT_INT4_SYM)
              for kf in (mla.FMT_BF16, mla.FMT_INT8_SYM, mla.FMT_INT4_SYM)] +
             [(lf, mla.FMT_INT8_SYM) for lf in (mla.FMT_INT8_G8, mla.FMT_INT8_G32, mla.FMT_INT8_G64,
                                                mla.FMT_INT8_TOKEN)] +
             [(mla.FMT_INT8_OUTLIER, mla.FMT_BF16), (mla.FMT_INT8_OUTLIER, mla.FMT_INT8_SYM)])


@pytest.mark.parametrize("lf,kf", ALL_PAIRS, ids=["%s-%s" % (FMT_NAME[a], FMT_NAME[b]) for a, b in ALL_PAIRS])
def test_tc_prefill_formats(lf, kf):
    """100 queries after 260 cached tokens (prefixes 261 .. 360: three key
    tiles, the causal edge inside the third), every query row."""
    check(Chunk(lf, kf, 260, 100, 16, seed=95))


@pytest.mark.parametrize("ctx_before,n,H", [(0, 700, 16), (200, 129, 48), (1000, 300, 128), (127, 129, 32),
                                            (383, 1, 16)])
def test_tc_prefill_shapes(ctx_before, n, H):
    """Row tiles that end mid-token (H = 48), a single query, 128 heads (one
    token per row tile), key counts on and off the tile edge; rows below 256
    tokens (ctx_before = 0) come from the exact recomputation."""
    ch = Chunk(mla.FMT_INT8_SYM, mla.FMT_INT8_SYM, ctx_before, n, H, seed=96)
    rng = np.random.default_rng(ctx_before + n + H)
    rows = sorted(set([0, n - 1, n // 2] + [int(r) for r in rng.integers(0, n, 24)]))
    check(ch, rows)


def test_tc_prefill_slices():
    """4200 queries: two slices of 4096 query tokens; rows around the
    boundary, the first and the last, and a sample."""
    ch = Chunk(mla.FMT_INT4_ASYM, mla.FMT_INT8_SYM, 10, 4200, 16, seed=97)
    rng = np.random.default_rng(97)
    rows = sorted(set([0, 1, 4094, 4095, 4096, 4097, 4199] + [int(r) for r in rng.integers(0, 4200, 12)]))
    check(ch, rows)


def test_tc_prefill_too_long_is_unsupported():
    """The key tiles hold 65536 positions: a longer prefix is refused
    before anything is launched."""
    import torch
    ch = Chunk(mla.FMT_INT8_SYM, mla.FMT_INT8_SYM, 0, 64, 16, seed=98)
    bt = torch.zeros(1100, dtype=torch.int32, device="cuda")
    q_lat = torch.zeros((64, 16, 512), dtype=torch.float32, device="cuda")
    ws = torch.empty(mla.mla_prefill_workspace_bytes(64, 16), dtype=torch.uint8, device="cuda")
    o_lat = torch.empty((64, 16, 512), dtype=torch.float32, device="cuda")
    with pytest.raises(RuntimeError, match="unsupported"):
        mla.mla_prefill_absorbed(ch.cache, q_lat, ch.q_pe, bt, 65536 - 63, ws, o_lat)


@pytest.mark.parametrize("lf", [mla.FMT_INT8_SYM, mla.FMT_INT4_ASYM], ids=["int8", "int4"])
def test_tc_prefill_peaked_softmax_over_cancelling_latents(lf):
    """512 queries (16 heads: 8192 rows) after 3584 cached tokens whose
    softmax puts most of its weight on 32 hot tokens in cancelling pairs
    (the decode's peaked construction, tests/test_gpu_peaked.py): the rows
    whose fp16 P and V roundings would exceed the bound must be caught by
    the precision check and recomputed exactly."""
    import torch
    import synth
    from oracle import attention as A
    from oracle import quant as Q
    from tests._helpers import ATTN_TOL
    from tests.test_gpu_peaked import _build
    T, n = 4096, 512
    wl, c, k, _, q_pe1, pos = _build(T, lf, "spread", seed=7100 + lf)
    rng = np.random.default_rng(7100 + lf)
    q_lat = (rng.standard_normal((n, 16, 512)) * 1e-4).astype(np.float32)
    q_pe = np.broadcast_to(q_pe1[0], (n, 16, 64)).astype(np.float32)
    q_lat_d = torch.from_numpy(q_lat).cuda()
    q_pe_d = torch.from_numpy(synth.bf16_rne(q_pe).view(np.int16)).cuda().view(torch.bfloat16)
    ws = torch.empty(mla.mla_prefill_workspace_bytes(n, 16), dtype=torch.uint8, device="cuda")
    o = torch.empty((n, 16, 512), dtype=torch.float32, device="cuda")
    lse = torch.empty((n, 16), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bt = wl.block_table[0].contiguous()
    mla.mla_prefill_absorbed(wl.caches[0], q_lat_d, q_pe_d, bt, T - n, ws, o, lse, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    d = Q.quantize_token_rows(c, k, lf, Q.FMT_INT8)
    o_h, lse_h = o.cpu().numpy(), lse.cpu().numpy()
    # the last query sees every hot token: >= 90 % of its mass on them and a
    # residual well below the hot terms
    s_last = A.scores(q_lat[n - 1], q_pe[n - 1], d["c_hat"], d["kpe_hat"])
    _, lse_last = A.absorbed_decode(q_lat[n - 1], q_pe[n - 1], d["c_hat"], d["kpe_hat"])
    p = np.exp(s_last - lse_last[:, None])
    assert np.all(p[:, pos].sum(axis=1) > 0.9)
    rows = sorted(set([0, n // 2, n - 1] + [int(r) for r in rng.integers(0, n, 9)]))
    for i in rows:
        t = T - n + i + 1
        ol_ref, lse_ref = A.absorbed_decode(q_lat[i], q_pe[i], d["c_hat"][:t], d["kpe_hat"][:t])
        e = A.max_rel_error(o_h[i], ol_ref)
        e_lse = float(np.max(np.abs(lse_h[i] - lse_ref)))
        assert e < ATTN_TOL and e_lse < ATTN_TOL, (i, e, e_lse)


def test_tc_prefill_zero_wait_limit_gives_up_cleanly():
    """The tensor-core kernel's bounded waits made to run out through the
    wait-limit hook (no fault, no trap): MLA_DEVERR_TIMEOUT, finite outputs,
    and the next call with the default limit on the same stream and buffers
    gives the full result again, bit for bit."""
    import torch
    ch = Chunk(mla.FMT_INT8_SYM, mla.FMT_INT8_SYM, 700, 600, 16, seed=99)
    ref_ol, ref_lse, _ = ch.run()
    q_lat = torch.empty((ch.n, 16, 512), dtype=torch.float32, device="cuda")
    mla.mla_q_absorb(ch.q_nope, ch.w_uk, q_lat)
    ws = torch.empty(mla.mla_prefill_workspace_bytes(ch.n, 16), dtype=torch.uint8, device="cuda")
    hits = 0
    prev = mla.mla_set_wait_limit_ns(0)
    try:
        for _ in range(3):
            o = torch.full((ch.n, 16, 512), float("nan"), dtype=torch.float32, device="cuda")
            lse = torch.full((ch.n, 16), float("nan"), dtype=torch.float32, device="cuda")
            err = torch.zeros(1, dtype=torch.int32, device="cuda")
            mla.mla_prefill_absorbed(ch.cache, q_lat, ch.q_pe, ch.block_table, ch.ctx_before, ws, o, lse, err)
            torch.cuda.synchronize()
            assert err.item() & ~8 == 0
            hits += bool(err.item() & 8)
            assert torch.isfinite(o).all()
            assert not torch.isnan(lse).any() and not (lse == float("inf")).any()
    finally:
        assert mla.mla_set_wait_limit_ns(prev) == 0
    assert hits > 0
    o = torch.full((ch.n, 16, 512), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((ch.n, 16), float("nan"), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.mla_prefill_absorbed(ch.cache, q_lat, ch.q_pe, ch.block_table, ch.ctx_before, ws, o, lse, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert np.array_equal(o.cpu().numpy(), ref_ol) and np.array_equal(lse.cpu().numpy(), ref_lse)


def test_tc_prefill_at_the_key_limit():
    """Prefixes that end exactly at the key tiles' 65536 positions (all 512
    key tiles, the last query's row tile sweeping every one): sampled rows,
    the last query included."""
    ch = Chunk(mla.FMT_INT4_ASYM, mla.FMT_INT8_SYM, 65536 - 40, 40, 16, seed=100)
    check(ch, [0, 1, 17, 38, 39])


def test_tc_prefill_bad_page_is_flagged():
    """A page id outside the pool in the sequence's block table: the key pass
    reports MLA_DEVERR_PAGE and reads that page's tokens as 0; the call
    completes and every output stays finite."""
    import torch
    ch = Chunk(mla.FMT_INT8_SYM, mla.FMT_INT8_SYM, 300, 200, 16, seed=101)
    ch.block_table[2] = ch.cache.num_pages + 5
    q_lat = torch.empty((200, 16, 512), dtype=torch.float32, device="cuda")
    mla.mla_q_absorb(ch.q_nope, ch.w_uk, q_lat)
    ws = torch.empty(mla.mla_prefill_workspace_bytes(200, 16), dtype=torch.uint8, device="cuda")
    o_lat = torch.full((200, 16, 512), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((200, 16), float("nan"), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.mla_prefill_absorbed(ch.cache, q_lat, ch.q_pe, ch.block_table, 300, ws, o_lat, lse, err)
    torch.cuda.synchronize()
    assert err.item() == mla.DEVERR_PAGE
    assert torch.isfinite(o_lat).all() and torch.isfinite(lse).all()
