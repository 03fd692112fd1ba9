"""The device generator reproduces the host generator bit for bit."""

import numpy as np
import pytest
import torch

import synth
import synth.device as sd

pytestmark = pytest.mark.gpu


def bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def test_latent_and_kpe_match_host():
    seed, layer, b = 123, 5, 7
    st = sd.LayerStats(seed, layer)
    rope = sd.RopeTables(3000)
    c = torch.empty((1000, 512), dtype=torch.bfloat16, device="cuda")
    k = torch.empty((1000, 64), dtype=torch.bfloat16, device="cuda")
    sd.latent_into(c, seed, layer, b, 2000, st)
    sd.kpe_into(k, seed, layer, b, 2000, rope)
    cos, sin = synth.rope_tables(3000)
    assert np.array_equal(bits(c), synth.latent_bf16(seed, layer, b, 2000, 3000))
    assert np.array_equal(bits(k), synth.kpe_bf16(seed, layer, b, 2000, 3000, cos, sin))


def test_queries_and_weights_match_host():
    seed, layer = 9, 3
    assert np.array_equal(bits(sd.q_nope(seed, layer, 5, 16)), synth.q_nope_bf16(seed, layer, 5, 16))
    assert np.array_equal(bits(sd.q_pe(seed, layer, 5, 64)), synth.q_pe_bf16(seed, layer, 5, 64))
    assert np.array_equal(bits(sd.w_uk(seed, layer, 16)), synth.w_uk_bf16(seed, layer, 16))
    assert np.array_equal(bits(sd.w_uv(seed, layer, 16)), synth.w_uv_bf16(seed, layer, 16))
    rows = [0, 3, 299]
    assert np.array_equal(bits(sd.prefill_q_nope(seed, layer, 300, 16))[rows],
                          synth.prefill_q_nope_bf16(seed, layer, rows, 16))
    assert np.array_equal(bits(sd.prefill_q_pe(seed, layer, 300, 64))[rows], synth.prefill_q_pe_bf16(seed, layer, rows, 64))
