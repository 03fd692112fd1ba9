"""Context-sharded decode on one GPU: the ranks' local decodes run one after
another over their page ranges (the local block-table views the sharded path
builds), their (o_lat, lse) results are stacked as the all-gather would
stack them, and mla_lse_merge must give the oracle's attention over the
whole context (and agree with the unsharded decode)."""

import numpy as np
import pytest
import torch

import mla_latent_kv_append_gb300 as mla
from mla_latent_kv_append_gb300 import sharded
from oracle import attention as A
from synth.workload import DecodeStep, Workload
from tests._helpers import ATTN_TOL, OracleCache

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("lens,world", [([5000, 700, 64], 3), ([4096], 8), ([300, 1], 4), ([9000], 2)])
def test_sharded_parts_merge_to_the_whole(lens, world):
    wl = Workload(1, 16, lens, mla.FMT_INT4_ASYM, mla.FMT_INT8_SYM, seed=90)
    step = DecodeStep(wl)
    step.run()                                   # appends the new token; full decode for reference
    torch.cuda.synchronize()
    full_o, full_lse = step.o_lat.clone(), step.lse[0].clone()
    B, H = wl.B, wl.H
    parts_o = torch.empty((world, B, H, 512), dtype=torch.float32, device="cuda")
    parts_l = torch.empty((world, B, H), dtype=torch.float32, device="cuda")
    per_seq = [sharded.context_ranges(T, world) for T in wl.seq_lens]
    for r in range(world):
        bt, lens_r = sharded.local_block_table(wl.block_table, wl.seq_lens_dev, [rs[r] for rs in per_seq])
        mla.mla_decode_absorbed(wl.caches[0], step.q_lat, wl.q_pe[0], bt, lens_r, step.workspace, parts_o[r],
                                parts_l[r], step.dev_err)
    o_lat = torch.empty((B, H, 512), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, H), dtype=torch.float32, device="cuda")
    mla.mla_lse_merge(parts_o, parts_l, o_lat, lse)
    torch.cuda.synchronize()
    assert step.dev_err.item() == 0
    oc = OracleCache(wl)
    got, got_lse = o_lat.cpu().numpy(), lse.cpu().numpy()
    for b in range(B):
        _, ol_ref, lse_ref, _ = oc.decode(0, b)
        assert A.max_rel_error(got[b], ol_ref) < ATTN_TOL
        assert np.max(np.abs(got_lse[b] - lse_ref)) < ATTN_TOL
    # the split changes only the rounding of the fp16 P tiles and the merge order
    assert A.max_rel_error(got, full_o.cpu().numpy()) < 1e-3


def test_merge_empty_parts_and_single_part():
    B, H = 3, 16
    rng = np.random.default_rng(3)
    on = rng.standard_normal((2, B, H, 512)).astype(np.float32)
    ln = rng.standard_normal((2, B, H)).astype(np.float32)
    ln[1, 0] = -np.inf                           # sequence 0: the second part is empty
    ln[:, 1] = -np.inf                           # sequence 1: every part is empty
    o, l = torch.from_numpy(on).cuda(), torch.from_numpy(ln).cuda()
    out = torch.empty((B, H, 512), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, H), dtype=torch.float32, device="cuda")
    mla.mla_lse_merge(o, l, out, lse)
    one, one_lse = torch.empty_like(out), torch.empty_like(lse)
    mla.mla_lse_merge(o[:1].contiguous(), l[:1].contiguous(), one, one_lse)
    torch.cuda.synchronize()
    got, got_lse = out.cpu().numpy(), lse.cpu().numpy()
    for b in (0, 2):
        exp_o, exp_l = A.lse_combine(ln[:, b], np.ones((2, H)), on[:, b])
        assert A.max_rel_error(got[b], exp_o) < 1e-6
        assert np.max(np.abs(got_lse[b] - exp_l)) < 1e-5
    assert A.max_rel_error(got[0], on[0, 0]) < 1e-6 and np.max(np.abs(got_lse[0] - ln[0, 0])) < 1e-6
    assert np.all(got[1] == 0) and np.all(np.isneginf(got_lse[1]))
    assert A.max_rel_error(one.cpu().numpy()[[0, 2]], on[0][[0, 2]]) < 1e-6
    assert np.max(np.abs(one_lse.cpu().numpy()[[0, 2]] - ln[0][[0, 2]])) < 1e-6


def test_sharded_decode_on_a_side_stream():
    """sharded_decode with a stream that is not torch's current one, in a
    one-rank NCCL group: the decode, the all-gather and the merge must all be
    ordered on that stream, and the result equals the plain decode."""
    import datetime
    import os
    import socket

    import torch.distributed as dist

    wl = Workload(1, 16, [5000, 300], mla.FMT_INT8_SYM, mla.FMT_INT8_SYM, seed=91)
    step = DecodeStep(wl)
    step.run()
    torch.cuda.synchronize()
    ref_o, ref_lse = step.o_lat.clone(), step.lse[0].clone()
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    os.environ.setdefault("NCCL_NVLS_ENABLE", "0")
    dist.init_process_group("nccl", init_method="tcp://127.0.0.1:%d" % port, rank=0, world_size=1,
                            timeout=datetime.timedelta(seconds=120))
    try:
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        o_lat = torch.full_like(ref_o, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        for _ in range(3):
            sharded.sharded_decode(wl.caches[0], step.q_lat, wl.q_pe[0], wl.block_table, wl.seq_lens_dev,
                                   step.workspace, o_lat, lse, dev_err=step.dev_err, stream=side)
        side.synchronize()
        torch.cuda.synchronize()
    finally:
        dist.destroy_process_group()
    assert step.dev_err.item() == 0
    # one part: the merge of a single part reproduces it up to the lse rounding
    assert A.max_rel_error(o_lat.cpu().numpy(), ref_o.cpu().numpy()) < 1e-5
    assert np.max(np.abs(lse.cpu().numpy() - ref_lse.cpu().numpy())) < 1e-5
