"""The seeded input generator: determinism, the bf16 rounding it uses, and the
value distributions of the workload description."""

import numpy as np
import torch

import synth


def test_bf16_rne_matches_torch_conversion():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 10 ** rng.uniform(-5, 5, 100000),
                        np.array([0.0, -0.0, 1.0, 1.00390625, 1.005859375, 65504.0, -3.0e38], np.float32)])
    x = x.astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(synth.bf16_rne(x), ref)
    assert np.array_equal(synth.bf16_to_f32(ref), torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).float().numpy())


def test_deterministic_and_prefix_consistent():
    a = synth.latent_bf16(5, 2, 3, 0, 300)
    b = synth.latent_bf16(5, 2, 3, 100, 300)
    assert np.array_equal(a[100:], b)
    assert not np.array_equal(a, synth.latent_bf16(5, 2, 4, 0, 300))
    assert not np.array_equal(a, synth.latent_bf16(6, 2, 3, 0, 300))


def test_normal_moments():
    z = synth.normal_from_hash(synth.hash_at(synth.stream_key(1, 0, 3), np.arange(1 << 20)))
    assert abs(z.mean()) < 5e-3 and abs(z.std() - 1.0) < 5e-3
    assert np.abs(z).max() <= 3.47


def test_channel_stats_recipe():
    mu, sigma = synth.channel_stats(11, 4)
    big = sigma > 10.0
    assert big.sum() <= 5
    base = ~(np.abs(mu) > 1.0) & ~(sigma > 10.0)
    assert np.all((sigma[base] >= 0.1 - 1e-7) & (sigma[base] <= 10.0 + 1e-6))
    assert np.sum((np.abs(mu) > 1.0) | (sigma > 10.0)) <= 5


def test_rope_preserves_pair_norms():
    cos, sin = synth.rope_tables(64)
    z = synth.bf16_to_f32(synth.kpe_bf16(1, 0, 0, 0, 64, cos, np.zeros_like(sin) * 0 + sin))
    assert z.shape == (64, 64)
    # rotation by position 0 is the identity on the underlying normals
    key = synth.stream_key(1, 0, synth.KIND_KPE)
    raw = synth.normal_from_hash(synth.hash_at(key, synth.token_index(0, np.arange(1), np.arange(64))))
    assert np.array_equal(z[0], synth.bf16_to_f32(synth.bf16_rne(raw[0])))


def test_row_subset_matches_full_grid():
    """normal_rows_bf16 gives exactly the selected rows of normal3_bf16."""
    full = synth.normal3_bf16(4, 2, synth.KIND_PRE_QNOPE, 40, 16, synth.D_NOPE, synth.UNIT_SCALE)
    rows = [39, 0, 17, 17, 5]
    assert np.array_equal(synth.prefill_q_nope_bf16(4, 2, rows, 16), full[rows])
    pe = synth.normal3_bf16(4, 2, synth.KIND_PRE_QPE, 40, 16, synth.D_R, synth.UNIT_SCALE)
    assert np.array_equal(synth.prefill_q_pe_bf16(4, 2, rows, 16), pe[rows])
    # the prefill queries are streams of their own, not the decode queries
    assert not np.array_equal(full[:5], synth.q_nope_bf16(4, 2, 5, 16))
