"""mla_decode_absorbed_noalloc, the decode entry point for callers that cannot
allocate device memory (plugins handed only their buffers, code running during
CUDA-graph capture, serving loops that forbid allocation after start-up).

It is called here through the C ABI (ctypes) twice in a row and compared with
mla_decode_absorbed, which takes a caller-allocated workspace.  Both calls run
the same kernels over the same partition of the context, so their outputs
must agree bit for bit: any difference means the scratch array was read
before it was written or shared with something else.  This file sorts last so that a run
stopping at the first failure has already run every other test; it also
passes when run alone in a fresh process."""

import ctypes

import pytest
import torch

import mla_latent_kv_append_gb300 as mla
from synth.workload import DecodeStep, Workload

pytestmark = pytest.mark.gpu


def _noalloc(wl, q_lat, layer, o_lat, lse, err, batch=None, heads=None, num_splits=0):
    cs = wl.caches[layer].c_struct()
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    return mla.lib.mla_decode_absorbed_noalloc(
        ctypes.byref(cs), p(q_lat), p(wl.q_pe[layer]), p(wl.block_table), wl.block_table.shape[1],
        p(wl.seq_lens_dev), wl.B if batch is None else batch, wl.H if heads is None else heads,
        ctypes.c_float(mla.DEFAULT_SOFTMAX_SCALE), num_splits, p(o_lat), p(lse), p(err),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("lf", [mla.FMT_INT8_SYM, mla.FMT_INT4_ASYM])
def test_noalloc_matches_workspace_call_twice(lf):
    wl = Workload(1, 16, [300, 1000, 64, 5], lf, mla.FMT_INT8_SYM, seed=31)
    step = DecodeStep(wl)
    mla.mla_q_absorb(wl.q_nope[0], wl.w_uk[0], step.q_lat)
    ref_o = torch.empty_like(step.o_lat)
    ref_lse = torch.empty((wl.B, wl.H), dtype=torch.float32, device="cuda")
    mla.mla_decode_absorbed(wl.caches[0], step.q_lat, wl.q_pe[0], wl.block_table, wl.seq_lens_dev,
                            step.workspace, ref_o, ref_lse, step.dev_err)
    torch.cuda.synchronize()
    for _ in range(2):
        o = torch.full_like(ref_o, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        assert _noalloc(wl, step.q_lat, 0, o, lse, err) == 0
        torch.cuda.synchronize()
        assert err.item() == 0
        assert torch.equal(o, ref_o)
        assert torch.equal(lse, ref_lse)


def test_noalloc_rejects_requests_beyond_its_scratch():
    wl = Workload(1, 128, [64], mla.FMT_INT8_SYM, mla.FMT_INT8_SYM, seed=32)
    q_lat = torch.zeros((wl.B, 128, 512), dtype=torch.float32, device="cuda")
    o = torch.empty_like(q_lat)
    lse = torch.empty((wl.B, 128), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    # 128 heads with 4000 splits needs ~(4000 + 1) * 128 * 2 KiB > the scratch size
    assert _noalloc(wl, q_lat, 0, o, lse, err, num_splits=4000) == 1
