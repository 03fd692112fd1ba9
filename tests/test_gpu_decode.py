"""mla_decode_absorbed (with the full per-layer step: append -> absorb ->
decode -> unabsorb) on the GPU against the oracle: max relative error 2e-3
per row of o_lat and o, lse within 2e-3 absolute, on the same codes."""

import numpy as np
import pytest
import torch

import mla_latent_kv_append_gb300 as mla
from oracle import attention as A
from synth.workload import DecodeStep, Workload
from tests._helpers import ALL_FORMATS, ATTN_TOL, FMT_NAME, OracleCache

pytestmark = pytest.mark.gpu


def run_and_check(wl, num_splits=0, layers=None, seqs=None, tol=ATTN_TOL):
    step = DecodeStep(wl, num_splits=num_splits)
    keep = torch.empty((wl.L, wl.B, wl.H, 512), dtype=torch.float32, device="cuda")
    o = step.run(keep_o_lat=keep)
    torch.cuda.synchronize()
    assert step.dev_err.item() == 0
    oc = OracleCache(wl)
    o_h, ol_h, lse_h = o.cpu().numpy(), keep.cpu().numpy(), step.lse.cpu().numpy()
    worst = 0.0
    for l in (layers if layers is not None else range(wl.L)):
        for b in (seqs if seqs is not None else range(wl.B)):
            _, ol_ref, lse_ref, o_ref = oc.decode(l, b)
            if wl.seq_lens[b] == 0:
                assert np.all(ol_h[l, b] == 0) and np.all(o_h[l, b] == 0) and np.all(np.isneginf(lse_h[l, b]))
                continue
            e1 = A.max_rel_error(ol_h[l, b], ol_ref)
            e2 = A.max_rel_error(o_h[l, b], o_ref)
            e3 = float(np.max(np.abs(lse_h[l, b] - lse_ref)))
            worst = max(worst, e1, e2)
            assert e1 < tol and e2 < tol and e3 < tol, (l, b, e1, e2, e3)
    return o_h, worst


@pytest.mark.parametrize("lf,kf", ALL_FORMATS, ids=["%s-%s" % (FMT_NAME[a], FMT_NAME[b]) for a, b in ALL_FORMATS])
def test_tiny_config(lf, kf):
    """1 layer, 16 heads, batch 1, context 256 (paged, 64-token pages)."""
    wl = Workload(1, 16, [256], lf, kf, seed=0x4D4C41)
    run_and_check(wl)


RAGGED_FORMATS = [(mla.FMT_BF16, mla.FMT_INT8_SYM), (mla.FMT_INT8_SYM, mla.FMT_INT8_SYM),
                  (mla.FMT_INT4_ASYM, mla.FMT_INT8_SYM), (mla.FMT_INT4_SYM, mla.FMT_INT8_SYM),
                  (mla.FMT_INT4_ASYM, mla.FMT_INT4_SYM)]


@pytest.mark.parametrize("lf,kf", RAGGED_FORMATS, ids=["%s-%s" % (FMT_NAME[a], FMT_NAME[b]) for a, b in RAGGED_FORMATS])
def test_ragged_batch_edges(lf, kf):
    """Context lengths around page and chunk boundaries, plus an empty sequence."""
    lens = [1, 31, 32, 33, 63, 64, 65, 100, 0, 257, 129]
    wl = Workload(1, 16, lens, lf, kf, seed=77)
    run_and_check(wl)


def test_split_invariance_and_counts():
    lens = [700, 5, 1300, 64, 2049]
    wl = Workload(2, 16, lens, mla.FMT_INT8_SYM, mla.FMT_INT8_SYM, seed=78)
    outs = []
    for ns in (1, 2, 3, 7, 40, 0, 400):
        o, _ = run_and_check(wl, num_splits=ns, layers=[1])
        outs.append(o)
    # every split count is within 2e-3 of the oracle (run_and_check); between
    # split counts the results differ only by the fp16 rounding of P and of
    # the scaled P, taken relative to different running maxima (~2^-11)
    for o in outs[1:]:
        assert A.max_rel_error(o, outs[0]) < 1e-3


@pytest.mark.parametrize("ns", [16, 64, 128, 512], ids=["grouped", "per-head", "sliced-2", "sliced-8"])
def test_combine_grids(ns):
    """The combine's three grids, chosen from the batch (4) and the split
    count: eight heads per block (G < 8 B), one head per block
    (8 B <= G < 32 B), and one head's channels sliced over 2 or 8 blocks
    (G >= 32 B).  The batch holds an empty sequence, a short one (recomputed
    exactly) and long ones spread over up to ~250 slots; 32 heads (four head
    groups)."""
    lens = [3000, 0, 150, 4100]
    wl = Workload(1, 32, lens, mla.FMT_INT8_SYM, mla.FMT_INT8_SYM, seed=81)
    run_and_check(wl, num_splits=ns)


def _slot_counts(lens, G):
    """Slots per sequence under the split kernel's partition (split x takes
    chunks [C x / Ge, C (x + 1) / Ge), Ge = min(G, C)): the splits holding
    a sequence's first through last 32-token chunk."""
    chunks = [(t + 31) // 32 for t in lens]
    C = sum(chunks)
    Ge = min(G, C)
    def split(c):
        return ((c + 1) * Ge + C - 1) // C - 1
    out, c0 = [], 0
    for n in chunks:
        out.append(split(c0 + n - 1) - split(c0) + 1 if n else 0)
        c0 += n
    return out


def test_combine_slot_reduction_boundary():
    """The per-head combine reduces the slot figures in one warp when a
    sequence has at most 32 slots and across the block otherwise: one call
    with a 32-slot and a 33-slot sequence (and a 4-slot one), against the
    oracle."""
    lens, G = [2472, 2536, 300], 67
    assert _slot_counts(lens, G) == [32, 33, 4]
    wl = Workload(1, 16, lens, mla.FMT_INT8_SYM, mla.FMT_INT8_SYM, seed=83)
    run_and_check(wl, num_splits=G)


def test_64_heads_mixed_lengths():
    wl = Workload(1, 64, [1000, 37, 2500], mla.FMT_INT8_SYM, mla.FMT_INT8_SYM, seed=79)
    run_and_check(wl)


def test_int4_longer_context():
    wl = Workload(1, 16, [4096, 3000], mla.FMT_INT4_ASYM, mla.FMT_INT8_SYM, seed=80)
    run_and_check(wl)


def test_bad_page_and_bad_length_are_flagged_not_faulted():
    wl = Workload(1, 16, [200, 100], mla.FMT_INT8_SYM, mla.FMT_INT8_SYM, seed=81)
    step = DecodeStep(wl)
    step.run()
    torch.cuda.synchronize()
    assert step.dev_err.item() == 0
    # corrupt one block-table entry of sequence 0, and make sequence 1 too long
    bt = wl.block_table.clone()
    bt[0, 1] = wl.num_pages + 5
    lens = wl.seq_lens_dev.clone()
    lens[1] = wl.max_pages * 64 + 1
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.mla_decode_absorbed(wl.caches[0], step.q_lat, wl.q_pe[0], bt, lens, step.workspace, step.o_lat,
                            step.lse[0], err)
    torch.cuda.synchronize()
    assert err.item() == mla.DEVERR_PAGE | mla.DEVERR_SEQLEN
    ol = step.o_lat.cpu().numpy()
    assert np.all(np.isfinite(ol))
    assert np.all(ol[1] == 0) and np.all(np.isneginf(step.lse[0, 1].cpu().numpy()))


def test_most_heads():
    """128 heads (eight head tiles), the largest head count the ABI takes."""
    wl = Workload(1, 128, [300, 65, 1], mla.FMT_INT8_SYM, mla.FMT_INT8_SYM, seed=82)
    run_and_check(wl)


def test_largest_batch():
    """B = 4096 (the ABI's limit) short sequences: the chunk prefix sums fill
    the shared-memory reserve; sampled sequences against the oracle."""
    rng = np.random.default_rng(83)
    lens = [int(t) for t in rng.integers(0, 80, 4096)]
    wl = Workload(1, 16, lens, mla.FMT_INT4_ASYM, mla.FMT_INT8_SYM, seed=83)
    seqs = sorted(set([0, 4095] + [int(b) for b in rng.integers(0, 4096, 48)]))
    run_and_check(wl, seqs=seqs)


POISON_FORMATS = [(mla.FMT_BF16, mla.FMT_BF16), (mla.FMT_INT8_SYM, mla.FMT_INT8_SYM),
                  (mla.FMT_INT4_ASYM, mla.FMT_INT8_SYM), (mla.FMT_INT4_SYM, mla.FMT_INT4_SYM),
                  (mla.FMT_INT8_G8, mla.FMT_INT8_SYM), (mla.FMT_INT8_G32, mla.FMT_INT8_SYM),
                  (mla.FMT_INT8_G64, mla.FMT_INT8_SYM), (mla.FMT_INT8_TOKEN, mla.FMT_INT8_SYM),
                  (mla.FMT_INT4_ASYM, mla.FMT_BF16)]


@pytest.mark.parametrize("lf,kf", POISON_FORMATS, ids=["%s-%s" % (FMT_NAME[a], FMT_NAME[b]) for a, b in POISON_FORMATS])
def test_poisoned_page_tails(lf, kf):
    """Every pool byte starts as 0xFF (NaN scales and zero-points, extreme
    codes), so the slots past each sequence's end hold garbage: the decode
    must read only the first seq_len tokens and stay finite."""
    lens = [1, 31, 33, 64, 65, 100, 129, 250]
    wl = Workload(1, 16, lens, lf, kf, seed=84, fill=False)
    for c in wl.caches:
        c.pool.fill_(0xFF)
    wl.fill()
    run_and_check(wl)


@pytest.mark.parametrize("lens,H", [([4096] * 8, 16), ([4096, 100, 0, 3000], 32), ([300] * 40, 16), ([70000], 16)],
                         ids=["per-head-grid", "short-and-empty", "grouped-grid", "one-long"])
def test_decode_with_unabsorb_matches_the_two_calls(lens, H):
    """mla_decode_absorbed_unabsorb against mla_decode_absorbed followed by
    mla_out_unabsorb: o_lat and lse bit for bit (the same kernels), o within
    fp32 summation order, in each combine grid (the per-head grid projects
    inside the combine, including rows of the exact path)."""
    wl = Workload(1, H, lens, mla.FMT_INT8_SYM, mla.FMT_INT8_SYM, seed=17)
    step = DecodeStep(wl)
    step.run()
    torch.cuda.synchronize()
    o_f, ol_f, lse_f = step.o[0].clone(), step.o_lat.clone(), step.lse[0].clone()
    mla.mla_decode_absorbed(wl.caches[0], step.q_lat, wl.q_pe[0], wl.block_table, wl.seq_lens_dev, step.workspace,
                            step.o_lat, step.lse[0], step.dev_err)
    o_s = torch.empty_like(o_f)
    mla.mla_out_unabsorb(step.o_lat, wl.w_uv[0], o_s)
    torch.cuda.synchronize()
    assert step.dev_err.item() == 0
    assert torch.equal(ol_f, step.o_lat) and torch.equal(lse_f, step.lse[0])
    scale = o_s.abs().amax(dim=-1, keepdim=True).clamp_min(1e-30)
    assert float(((o_f - o_s).abs() / scale).max()) < 1e-5
    for b, T in enumerate(lens):
        if T == 0:
            assert torch.all(o_f[b] == 0)
