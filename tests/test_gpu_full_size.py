"""Parity at the benchmark's full sizes, in the launch configuration bench.py
times (same workloads, same seed, automatic split count, whole decode step:
append -> absorb -> decode + combine -> unabsorb for every layer).

Attention outputs of every layer and sequence are compared for the 4096-token
INT8 workload and the 64-head mixed-length workloads; for the 32K, 256K and
1M-token workloads layers {0, 13, 26} and every sequence are compared.  The
oracle works through each sequence in 32K-token ranges in spawned host
processes and merges the ranges with its log-sum-exp combine.  Stored codes,
scales and zero-points are compared bit for bit on sampled token windows
(first, last, and random ones) of the compared layers; the mixed serving
step's 8192-token prefill append is compared in full.
"""

import gc

import numpy as np
import pytest
import torch

import bench
import synth
from oracle import attention as A
from synth.workload import DecodeStep, Workload
from tests._helpers import ATTN_TOL, assert_fields_match, read_tokens
from tests._oracle_pool import make_pool, oracle_outliers, oracle_outputs, tokens_bf16

pytestmark = pytest.mark.gpu

SAMPLED = (0, 13, 26)
CASES = [
    ("v2lite_int8", None),
    ("v2lite_int4_32k", SAMPLED),
    ("v2lite_int8_32k", (0, 26)),
    ("v2lite_int4_kpe4_32k", (0, 26)),
    ("v2lite_int8_per_token", (0, 13, 26)),
    ("v2lite_int8_64blocks", (0, 26)),
    ("v2lite_int8_outlier", (0, 13, 26)),
    ("long_int4_1m", SAMPLED),
    ("long_bf16_256k", SAMPLED),
    ("mixed_h64_int8", None),
    ("mixed_h64_int4", None),
    ("mixed_h64_bf16", None),
]


@pytest.fixture(scope="module")
def pool():
    p = make_pool()
    yield p
    p.close()
    p.join()


def check_stored_windows(wl, layers, rng, seqs_per_layer=3, windows=6, width=64):
    lf, kf = wl.latent_fmt, wl.kpe_fmt
    for l in layers:
        pool_np = wl.caches[l].pool.cpu().numpy()
        stats = synth.channel_stats(wl.seed, l)
        seqs = sorted(set([0, wl.B - 1] + list(rng.integers(0, wl.B, seqs_per_layer))))
        for b in seqs:
            T = wl.seq_lens[b]
            cos, sin = synth.rope_tables(T)
            starts = {0, max(0, T - width)} | set(int(s) for s in rng.integers(0, max(1, T - width), windows))
            for t0 in sorted(starts):
                t1 = min(T, t0 + width)
                c, k = tokens_bf16(wl.seed, l, b, T, t0, t1, stats, cos, sin)
                got = read_tokens(pool_np, wl.caches[l].layout, lf, kf, wl.slots(b, t0, t1))
                assert_fields_match(got, c, k, lf, kf, outliers=oracle_outliers(wl.seed, l, lf))
        del pool_np


@pytest.mark.parametrize("name,layers", CASES, ids=[c[0] for c in CASES])
def test_full_size_parity(pool, name, layers):
    cfg = bench.CONFIGS[name]
    seed = bench.SEED
    seq_lens = bench.seq_lens_for(cfg, seed)
    L, H = cfg["layers"], cfg["heads"]
    lf, kf = bench.FMT[cfg["latent"]], bench.FMT[cfg["kpe"]]
    layers = list(range(L)) if layers is None else [l for l in layers if l < L]
    gc.collect()
    torch.cuda.empty_cache()                      # the previous workload's cache pools
    wl = Workload(L, H, seq_lens, lf, kf, seed, prefill=cfg.get("prefill", 0))
    step = DecodeStep(wl)                         # automatic split count, as timed by the bench
    keep = torch.empty((L, wl.B, H, synth.D_C), dtype=torch.float32, device="cuda")
    o = step.run(keep_o_lat=keep)
    torch.cuda.synchronize()
    assert step.dev_err.item() == 0
    o_h, ol_h, lse_h = o.cpu().numpy(), keep.cpu().numpy(), step.lse.cpu().numpy()
    ref = oracle_outputs(pool, seed, layers, range(wl.B), seq_lens, H, lf, kf)
    assert len(ref) == len(layers) * wl.B
    worst = 0.0
    for (l, b), (ol_ref, lse_ref, o_ref) in sorted(ref.items()):
        e1 = A.max_rel_error(ol_h[l, b], ol_ref)
        e2 = A.max_rel_error(o_h[l, b], o_ref)
        e3 = float(np.max(np.abs(lse_h[l, b] - lse_ref)))
        worst = max(worst, e1, e2)
        assert e1 < ATTN_TOL and e2 < ATTN_TOL and e3 < ATTN_TOL, (name, l, b, e1, e2, e3)
    print("%s: %d (layer, sequence) pairs compared, worst max-rel error %.2e" % (name, len(ref), worst))
    check_stored_windows(wl, layers[:1] + layers[-1:], np.random.default_rng(len(name)))
    if wl.prefill:                    # the serving step's prefill append, every token
        for l in layers[:1] + layers[-1:]:
            c, k = wl.host_prefill(l)
            got = read_tokens(wl.caches[l].pool.cpu().numpy(), wl.caches[l].layout, lf, kf, wl.slot_pre_host)
            assert_fields_match(got, c, k, lf, kf, outliers=oracle_outliers(wl.seed, l, lf))
