"""Host side of the context-sharded decode, on CPU: the page-aligned range
plan, the local block-table view, and the (o_lat, lse) all-gather between
two gloo ranks.  Each rank's local result is the oracle's decode over its
range (standing in for its GPU), and the gathered parts merged by the
oracle's log-sum-exp rule must equal the oracle's decode over the whole
context."""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as tmp

import synth
from oracle import attention as A
from oracle import quant as Q
from mla_latent_kv_append_gb300 import sharded


@pytest.mark.parametrize("T,world", [(1, 2), (64, 2), (65, 2), (1000, 3), (4096, 8), (100, 4), (130, 8)])
def test_context_ranges_cover_once_page_aligned(T, world):
    rs = sharded.context_ranges(T, world)
    assert len(rs) == world
    covered = np.zeros(T, int)
    for t0, t1 in rs:
        assert 0 <= t0 <= t1 <= T
        assert t0 % 64 == 0 or t0 == T
        covered[t0:t1] += 1
    assert np.all(covered == 1)
    sizes = [((t1 - t0) + 63) // 64 for t0, t1 in rs]
    assert max(sizes) - min(sizes) <= 1


def test_local_block_table_view():
    bt = torch.arange(2 * 10, dtype=torch.int32).reshape(2, 10)
    lens = torch.tensor([600, 130], dtype=torch.int32)
    ranges = [(128, 600), (64, 130)]
    lbt, llen = sharded.local_block_table(bt, lens, ranges)
    assert llen.tolist() == [472, 66]
    assert lbt[0, :8].tolist() == list(range(2, 10)) and lbt[1, :2].tolist() == [11, 12]
    assert torch.all(lbt[1, 2:] == -1)
    with pytest.raises(ValueError):
        sharded.local_block_table(bt, lens, [(10, 600), (0, 130)])


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, T, lf, kf):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        seed, layer, H = 11, 0, 16
        cos, sin = synth.rope_tables(T)
        c_bits, k_bits = synth.sequence_bf16(seed, layer, 0, T, cos, sin)
        d = Q.quantize_token_rows(synth.bf16_to_f32(c_bits), synth.bf16_to_f32(k_bits), lf, kf)
        qn = synth.bf16_to_f32(synth.q_nope_bf16(seed, layer, 1, H))[0]
        qp = synth.bf16_to_f32(synth.q_pe_bf16(seed, layer, 1, H))[0]
        q_lat = A.absorb_q(qn, synth.bf16_to_f32(synth.w_uk_bf16(seed, layer, H)))
        t0, t1 = sharded.context_ranges(T, world)[rank]
        o_r, lse_r = A.absorbed_decode(q_lat, qp, d["c_hat"][t0:t1], d["kpe_hat"][t0:t1])
        o_parts, l_parts = sharded.gather_partials(torch.from_numpy(o_r[None].astype(np.float32)),
                                                   torch.from_numpy(lse_r[None].astype(np.float32)))
        assert tuple(o_parts.shape) == (world, 1, H, 512) and tuple(l_parts.shape) == (world, 1, H)
        o_m, lse_m = A.lse_combine(l_parts[:, 0].numpy(), np.ones((world, H)), o_parts[:, 0].numpy())
        o_full, lse_full = A.absorbed_decode(q_lat, qp, d["c_hat"], d["kpe_hat"])
        assert A.max_rel_error(o_m, o_full) < 1e-6, A.max_rel_error(o_m, o_full)
        assert np.max(np.abs(lse_m - lse_full)) < 1e-5
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("T,world", [(700, 2), (100, 2), (1000, 3)])
def test_two_rank_exchange_equals_unsharded(T, world):
    tmp.spawn(_rank_main, args=(world, _free_port(), T, Q.FMT_INT8, Q.FMT_INT8), nprocs=world, join=True)
