"""The decode kernel's bounded waits, made to run out on purpose through the
wait-limit hook (no fault, no trap): with a limit of 0 ns the blocks give up
at their first wait that is not already satisfied, report MLA_DEVERR_TIMEOUT,
write empty partials for the rest of their share and leave only after their
own bulk copies have landed.  The outputs stay finite; the next call with the
default limit, on the same stream, gives the full result again."""

import pytest
import torch

import mla_latent_kv_append_gb300 as mla
from synth.workload import DecodeStep, Workload
from tests._helpers import ATTN_TOL, OracleCache
from oracle import attention as A

pytestmark = pytest.mark.gpu

MLA_DEVERR_TIMEOUT = 8


@pytest.mark.parametrize("lf", [mla.FMT_INT8_SYM, mla.FMT_INT4_ASYM])
def test_zero_wait_limit_gives_up_cleanly(lf):
    wl = Workload(1, 16, [20000, 3000, 700, 64], lf, mla.FMT_INT8_SYM, seed=61)
    step = DecodeStep(wl)
    step.run()
    torch.cuda.synchronize()
    assert step.dev_err.item() == 0
    ref_o, ref_lse = step.o_lat.clone(), step.lse[0].clone()
    args = (wl.caches[0], step.q_lat, wl.q_pe[0], wl.block_table, wl.seq_lens_dev, step.workspace)
    hits = 0
    prev = mla.mla_set_wait_limit_ns(0)
    try:
        for _ in range(5):
            o = torch.full_like(ref_o, float("nan"))
            lse = torch.full_like(ref_lse, float("nan"))
            err = torch.zeros(1, dtype=torch.int32, device="cuda")
            mla.mla_decode_absorbed(*args, o, lse, err)
            torch.cuda.synchronize()
            assert err.item() & ~MLA_DEVERR_TIMEOUT == 0
            hits += bool(err.item() & MLA_DEVERR_TIMEOUT)
            assert torch.isfinite(o).all()
            assert not torch.isnan(lse).any() and not (lse == float("inf")).any()
    finally:
        assert mla.mla_set_wait_limit_ns(prev) == 0
    assert hits > 0
    # the default limit again, same stream, same buffers: the full result
    o = torch.full_like(ref_o, float("nan"))
    lse = torch.full_like(ref_lse, float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.mla_decode_absorbed(*args, o, lse, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert torch.equal(o, ref_o) and torch.equal(lse, ref_lse)
    oc = OracleCache(wl)
    for b in range(wl.B):
        _, ol_ref, _, _ = oc.decode(0, b)
        assert A.max_rel_error(o[b].cpu().numpy(), ol_ref) < ATTN_TOL

