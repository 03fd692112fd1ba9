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
from tests.test_gpu_prefill import FORMATS, Chunk, check

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def tensor_core_path():
    prev = mla.mla_set_prefill_path(mla.PREFILL_TENSOR_CORES)
    yield
    mla.mla_set_prefill_path(prev)


@pytest.mark.parametrize("lf,kf", FORMATS, ids=["%s-%s" % (FMT_NAME[a], FMT_NAME[b]) for a, b in FORMATS])
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
    """1100 queries: two slices of 1024 query tokens; rows around the
    boundary, the first and the last, and a sample."""
    ch = Chunk(mla.FMT_INT4_ASYM, mla.FMT_INT8_SYM, 10, 1100, 16, seed=97)
    rng = np.random.default_rng(97)
    rows = sorted(set([0, 1, 1022, 1023, 1024, 1025, 1099] + [int(r) for r in rng.integers(0, 1100, 12)]))
    check(ch, rows)


def test_tc_prefill_too_long_is_unsupported():
    """The key tiles hold 16384 positions: a longer prefix is refused
    before anything is launched."""
    import torch
    ch = Chunk(mla.FMT_INT8_SYM, mla.FMT_INT8_SYM, 0, 64, 16, seed=98)
    bt = torch.zeros(300, dtype=torch.int32, device="cuda")
    q_lat = torch.zeros((64, 16, 512), dtype=torch.float32, device="cuda")
    ws = torch.empty(mla.mla_prefill_workspace_bytes(64, 16), dtype=torch.uint8, device="cuda")
    o_lat = torch.empty((64, 16, 512), dtype=torch.float32, device="cuda")
    with pytest.raises(RuntimeError, match="unsupported"):
        mla.mla_prefill_absorbed(ch.cache, q_lat, ch.q_pe, bt, 16384 - 63, ws, o_lat)
