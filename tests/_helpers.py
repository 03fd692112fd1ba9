"""Shared test helpers: read cache fields back through the published page
layout, and run the oracle for one (layer, sequence) of a workload."""

import numpy as np

import synth
from oracle import attention as A
from oracle import quant as Q

F_BF16, F_INT8, F_INT4 = 0, 1, 2
ALL_FORMATS = [(F_BF16, F_BF16), (F_BF16, F_INT8), (F_INT8, F_BF16), (F_INT8, F_INT8), (F_INT4, F_BF16),
               (F_INT4, F_INT8)]
FMT_NAME = {F_BF16: "bf16", F_INT8: "int8", F_INT4: "int4"}

ATTN_TOL = 2e-3          # max relative error of attention outputs (per row, inf-norm)


def read_tokens(pool_np, layout, latent_fmt, kpe_fmt, slots):
    """Stored fields of the tokens at `slots` (numpy int array)."""
    slots = np.asarray(slots, np.int64)
    page, off = slots // 64, slots % 64
    base = page * layout.page_bytes
    out = {}
    rows = pool_np[(base + layout.codes_off + off * layout.codes_row_bytes)[:, None]
                   + np.arange(layout.codes_row_bytes)[None, :]]
    if latent_fmt == F_BF16:
        out["c_bits"] = rows.copy().view(np.uint16)
    else:
        gi = np.arange(32)[None, :] * 64 + off[:, None]
        scale = pool_np[(base + layout.scale_off)[:, None, None] + (gi * 4)[..., None] + np.arange(4)]
        out["c_scale"] = scale.reshape(len(slots), 32, 4).copy().view(np.float32)[..., 0]
        if latent_fmt == F_INT8:
            out["c_codes"] = rows.view(np.int8).copy()
        else:
            lo, hi = rows & 15, rows >> 4
            out["c_codes"] = np.stack([lo, hi], axis=2).reshape(len(slots), 512).astype(np.uint8)
            zero = pool_np[(base + layout.zero_off)[:, None, None] + (gi * 4)[..., None] + np.arange(4)]
            out["c_zero"] = zero.reshape(len(slots), 32, 4).copy().view(np.float32)[..., 0]
    krows = pool_np[(base + layout.kpe_off + off * layout.kpe_row_bytes)[:, None]
                    + np.arange(layout.kpe_row_bytes)[None, :]]
    if kpe_fmt == F_BF16:
        out["kpe_bits"] = krows.copy().view(np.uint16)
    else:
        out["kpe_codes"] = krows.view(np.int8).copy()
        gi = np.arange(8)[None, :] * 64 + off[:, None]
        ks = pool_np[(base + layout.kpe_scale_off)[:, None, None] + (gi * 4)[..., None] + np.arange(4)]
        out["kpe_scale"] = ks.reshape(len(slots), 8, 4).copy().view(np.float32)[..., 0]
    return out


def assert_fields_match(got, c_bits, k_bits, latent_fmt, kpe_fmt):
    """Bit-exact comparison of stored fields with the oracle's quantization."""
    exp = Q.quantize_token_rows(synth.bf16_to_f32(c_bits), synth.bf16_to_f32(k_bits), latent_fmt, kpe_fmt)
    if latent_fmt == F_BF16:
        assert np.array_equal(got["c_bits"], c_bits)
    else:
        assert np.array_equal(got["c_codes"], exp["c_codes"]), "latent codes differ"
        assert np.array_equal(got["c_scale"].view(np.uint32), exp["c_scale"].view(np.uint32)), "scales differ"
        if latent_fmt == F_INT4:
            assert np.array_equal(got["c_zero"].view(np.uint32), exp["c_zero"].view(np.uint32)), "zeros differ"
    if kpe_fmt == F_BF16:
        assert np.array_equal(got["kpe_bits"], k_bits)
    else:
        assert np.array_equal(got["kpe_codes"], exp["kpe_codes"]), "k_pe codes differ"
        assert np.array_equal(got["kpe_scale"].view(np.uint32), exp["kpe_scale"].view(np.uint32))


class OracleCache:
    """Per-layer oracle inputs of a workload (host generator only)."""

    def __init__(self, wl):
        self.wl = wl
        self._q = {}

    def query(self, layer):
        if layer not in self._q:
            self._q[layer] = [synth.bf16_to_f32(a) for a in self.wl.host_query(layer)]
        return self._q[layer]

    def sequence(self, layer, b):
        c_bits, k_bits = self.wl.host_sequence(layer, b)
        return c_bits, k_bits

    def decode(self, layer, b):
        """(q_lat, o_lat, lse, o) of the oracle for sequence b of `layer`."""
        qn, qp, wuk, wuv = self.query(layer)
        c_bits, k_bits = self.sequence(layer, b)
        d = Q.quantize_token_rows(synth.bf16_to_f32(c_bits), synth.bf16_to_f32(k_bits), self.wl.latent_fmt,
                                  self.wl.kpe_fmt)
        return A.absorbed_decode_full(qn[b], qp[b], wuk, wuv, d["c_hat"], d["kpe_hat"])
