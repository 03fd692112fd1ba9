"""mla_q_absorb / mla_out_unabsorb on the GPU against the oracle's fp64
projections (row-vector convention pinned by the tutorial's worked example)."""

import numpy as np
import pytest
import torch

import synth
import synth.device as sd
import mla_latent_kv_append_gb300 as mla
from oracle import attention as A

pytestmark = pytest.mark.gpu

# fp32 accumulation of exact products over 128 / 512 terms
TOL = 1e-5


@pytest.mark.parametrize("B,H", [(1, 16), (8, 16), (17, 16), (64, 64), (3, 128)])
def test_q_absorb(B, H):
    seed, layer = 4, 1
    qn = sd.q_nope(seed, layer, B, H)
    wuk = sd.w_uk(seed, layer, H)
    q_lat = torch.empty((B, H, 512), dtype=torch.float32, device="cuda")
    mla.mla_q_absorb(qn, wuk, q_lat)
    torch.cuda.synchronize()
    qn_h = synth.bf16_to_f32(synth.q_nope_bf16(seed, layer, B, H))
    wuk_h = synth.bf16_to_f32(synth.w_uk_bf16(seed, layer, H))
    got = q_lat.cpu().numpy()
    for b in range(B):
        ref = A.absorb_q(qn_h[b], wuk_h)
        assert A.max_rel_error(got[b], ref) < TOL


@pytest.mark.parametrize("B,H", [(1, 16), (8, 16), (9, 16), (64, 64), (2, 128)])
def test_out_unabsorb(B, H):
    seed, layer = 6, 2
    rng = np.random.default_rng(B * 1000 + H)
    o_lat_h = (rng.standard_normal((B, H, 512)) * 3).astype(np.float32)
    wuv = sd.w_uv(seed, layer, H)
    o = torch.empty((B, H, 128), dtype=torch.float32, device="cuda")
    mla.mla_out_unabsorb(torch.from_numpy(o_lat_h).cuda(), wuv, o)
    torch.cuda.synchronize()
    wuv_h = synth.bf16_to_f32(synth.w_uv_bf16(seed, layer, H))
    got = o.cpu().numpy()
    for b in range(B):
        assert A.max_rel_error(got[b], A.unabsorb_o(o_lat_h[b], wuv_h)) < TOL


def test_zero_batch_is_noop():
    q = torch.empty((0, 16, 128), dtype=torch.bfloat16, device="cuda")
    mla.mla_q_absorb(q, torch.zeros((16, 128, 512), dtype=torch.bfloat16, device="cuda"),
                     torch.empty((0, 16, 512), dtype=torch.float32, device="cuda"))
    mla.mla_out_unabsorb(torch.empty((0, 16, 512), dtype=torch.float32, device="cuda"),
                         torch.zeros((16, 512, 128), dtype=torch.bfloat16, device="cuda"),
                         torch.empty((0, 16, 128), dtype=torch.float32, device="cuda"))
    torch.cuda.synchronize()


@pytest.mark.parametrize("B,H", [(1000, 16), (4100, 16), (600, 64), (513, 128), (2432, 64), (2048, 128)])
def test_large_batches_split_over_the_grid(B, H):
    """Prefill-sized batches (512 rows and more: a CTA keeps a head's whole
    weight, each warp takes whole 16-row tiles; a ragged last tile
    included); sampled rows of both projections against the oracle.  Grids:
    16 heads split every head over 9 CTAs; 600 x 64 and 513 x 128 run the
    absorb on one CTA per SM with ranges crossing head boundaries and the
    unabsorb head-aligned; 2432 x 64 and 2048 x 128 cross head boundaries in
    both."""
    seed, layer = 7, 0
    rng = np.random.default_rng(B)
    rows = sorted(set([0, 15, 16, B - 17, B - 1] + [int(r) for r in rng.integers(0, B, 20)]))
    qn = sd.q_nope(seed, layer, B, H)
    wuk = sd.w_uk(seed, layer, H)
    q_lat = torch.empty((B, H, 512), dtype=torch.float32, device="cuda")
    mla.mla_q_absorb(qn, wuk, q_lat)
    wuv = sd.w_uv(seed, layer, H)
    o = torch.empty((B, H, 128), dtype=torch.float32, device="cuda")
    mla.mla_out_unabsorb(q_lat, wuv, o)
    torch.cuda.synchronize()
    qn_h = synth.bf16_to_f32(synth.q_nope_bf16(seed, layer, B, H))
    wuk_h = synth.bf16_to_f32(synth.w_uk_bf16(seed, layer, H))
    wuv_h = synth.bf16_to_f32(synth.w_uv_bf16(seed, layer, H))
    ql, oo = q_lat.cpu().numpy(), o.cpu().numpy()
    for b in rows:
        assert A.max_rel_error(ql[b], A.absorb_q(qn_h[b], wuk_h)) < TOL
        assert A.max_rel_error(oo[b], A.unabsorb_o(ql[b], wuv_h)) < TOL
