"""Oracle work for the full-size parity tests, run in spawned host processes.

Only NumPy, the host generator and the oracle are imported here (no torch, no
CUDA), so the worker processes start quickly and never touch the GPU.  A
sequence is cut into context ranges; each worker regenerates its range from
the seeded generator, quantizes it with the oracle and returns the oracle's
split-K partials (m, l, o) for that range, which the parent merges with the
oracle's log-sum-exp combine (the combine equals the unsplit decode: pinned
by the oracle's own split tests).
"""

import os

import numpy as np

import synth
from oracle import attention as A
from oracle import quant as Q


def tokens_bf16(seed, layer, b, T, t0, t1, stats, cos, sin):
    """bf16 bits of tokens [t0, t1) of the T-token sequence b, laid out as the
    workload writes them: positions below T-1 are the prefilled context and
    position T-1 is the token the decode step appends (its own stream)."""
    cs, ks = [], []
    e = min(t1, T - 1)
    if e > t0:
        cs.append(synth.latent_bf16(seed, layer, b, t0, e, stats=stats))
        ks.append(synth.kpe_bf16(seed, layer, b, t0, e, cos, sin))
    if t0 <= T - 1 < t1:
        cs.append(synth.latent_bf16(seed, layer, b, T - 1, T, kind=synth.KIND_NEW_LATENT, stats=stats))
        ks.append(synth.kpe_bf16(seed, layer, b, T - 1, T, cos, sin, kind=synth.KIND_NEW_KPE))
    return np.concatenate(cs), np.concatenate(ks)


def oracle_outliers(seed, layer, lf):
    """The oracle's calibration of a layer's protected channels (outlier format only)."""
    if lf != Q.FMT_INT8_OUTLIER:
        return None
    return Q.select_outlier_channels(synth.bf16_to_f32(synth.calibration_latent_bf16(seed, layer)))


def range_partials(task):
    """(layer, b, m [H], l [H], o [H, 512]) of the oracle over tokens [t0, t1)."""
    seed, layer, b, B, T, H, lf, kf, t0, t1 = task
    stats = synth.channel_stats(seed, layer)
    cos, sin = synth.rope_tables(t1)
    c, k = tokens_bf16(seed, layer, b, T, t0, t1, stats, cos, sin)
    d = Q.quantize_token_rows(synth.bf16_to_f32(c), synth.bf16_to_f32(k), lf, kf,
                              outliers=oracle_outliers(seed, layer, lf))
    qn = synth.bf16_to_f32(synth.q_nope_bf16(seed, layer, B, H))[b]
    qp = synth.bf16_to_f32(synth.q_pe_bf16(seed, layer, B, H))[b]
    wuk = synth.bf16_to_f32(synth.w_uk_bf16(seed, layer, H))
    q_lat = A.absorb_q(qn, wuk)
    m, l, o = A.split_partials(q_lat, qp, d["c_hat"], d["kpe_hat"], [0, t1 - t0])
    return layer, b, m[0], l[0], o[0]


def make_pool(n=None):
    """Spawned worker pool (spawn, so it is safe after CUDA was initialised),
    one BLAS thread per worker."""
    import multiprocessing as mp
    os.environ["OPENBLAS_NUM_THREADS"] = "1"
    os.environ["OMP_NUM_THREADS"] = "1"
    n = n or max(1, min(16, os.cpu_count() or 1))
    return mp.get_context("spawn").Pool(n)


def oracle_outputs(pool, seed, layers, seqs, seq_lens, H, lf, kf, span=32768):
    """{(layer, b): (o_lat [H, 512], lse [H], o [H, 128])} from the oracle."""
    B = len(seq_lens)
    tasks = []
    for l in layers:
        for b in seqs:
            T = int(seq_lens[b])
            for t0 in range(0, T, span):
                tasks.append((seed, l, b, B, T, H, lf, kf, t0, min(T, t0 + span)))
    parts = {}
    for l, b, m, lsum, o in pool.imap_unordered(range_partials, tasks, chunksize=1):
        parts.setdefault((l, b), []).append((m, lsum, o))
    out = {}
    wuv = {l: synth.bf16_to_f32(synth.w_uv_bf16(seed, l, H)) for l in layers}
    for (l, b), ps in parts.items():
        m = np.stack([p[0] for p in ps])
        lsum = np.stack([p[1] for p in ps])
        o = np.stack([p[2] for p in ps])
        o_lat, lse = A.lse_combine(m, lsum, o)
        out[(l, b)] = (o_lat, lse, A.unabsorb_o(o_lat, wuv[l]))
    return out
