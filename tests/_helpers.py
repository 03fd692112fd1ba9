"""Shared test helpers: read cache fields back through the published page
layout, and run the oracle for one (layer, sequence) of a workload."""

import numpy as np

import synth
from oracle import attention as A
from oracle import quant as Q

F_BF16, F_INT8, F_INT4, F_INT4S = 0, 1, 2, 3
F_I8G8, F_I8G32, F_I8G64, F_I8TOK = 4, 5, 6, 7
F_I8OUT = 8
INT8_GROUP = {F_INT8: 16, F_I8G8: 8, F_I8G32: 32, F_I8G64: 64, F_I8TOK: 512, F_I8OUT: 16}
ALL_FORMATS = ([(lf, kf) for lf in (F_BF16, F_INT8, F_INT4, F_INT4S) for kf in (F_BF16, F_INT8, F_INT4S)] +
               [(lf, F_INT8) for lf in (F_I8G8, F_I8G32, F_I8G64, F_I8TOK)])
FMT_NAME = {F_BF16: "bf16", F_INT8: "int8", F_INT4: "int4", F_INT4S: "int4sym", F_I8G8: "int8g8",
            F_I8G32: "int8g32", F_I8G64: "int8g64", F_I8TOK: "int8tok", F_I8OUT: "int8out"}

ATTN_TOL = 2e-3          # max relative error of attention outputs (per row, inf-norm)


def _int4_channel(j, k):
    """Channel (0..31 within a chunk) of nibble k of word j, as mla.h documents."""
    grp = (k >> 1) & 1
    return grp * 16 + 4 * j + (2 if k & 1 else 0) + (k >> 2)


def read_tokens(pool_np, layout, latent_fmt, kpe_fmt, slots):
    """Stored fields of the tokens at `slots` (numpy int array), decoded from
    the byte layout that include/mla.h documents (32-token blocks, swizzled
    16-byte chunks, interleaved 4-bit nibbles, symmetric 4-bit codes stored
    as code + 8)."""
    slots = np.asarray(slots, np.int64)
    n = len(slots)
    page, tok = slots // 64, slots % 64
    u = tok % 32
    base = page * layout.page_bytes + (tok // 32) * layout.block_bytes
    out = {}

    def gather(off, nbytes):
        return pool_np[(base + off)[:, None] + np.arange(nbytes)[None, :]]

    def fp32_field(off, groups):
        idx = (base + off)[:, None, None] + ((np.arange(groups)[None, :] * 32 + u[:, None]) * 4)[..., None] \
            + np.arange(4)
        return pool_np[idx].reshape(n, groups, 4).copy().view(np.float32)[..., 0]

    row = layout.codes_row_bytes
    nchunk = row // 16
    phys = gather(layout.codes_off + u * row, row).reshape(n, nchunk, 16)
    c = np.arange(nchunk)[None, :]
    pos = (c & ~7) | ((c ^ u[:, None]) & 7)
    logical = np.take_along_axis(phys, pos[..., None], axis=1)           # [n, nchunk, 16]
    if latent_fmt == F_BF16:
        out["c_bits"] = logical.reshape(n, row).copy().view(np.uint16)
    else:
        out["c_scale"] = fp32_field(layout.scale_off, 512 // INT8_GROUP.get(latent_fmt, 16))
        out["c_bound"] = fp32_field(layout.bound_off, 1)[:, 0]
        if latent_fmt == F_I8OUT:
            idx = (base + layout.outlier_off)[:, None, None] + ((np.arange(25)[None, :] * 32 + u[:, None]) * 2)[..., None] \
                + np.arange(2)
            out["c_outlier_bits"] = pool_np[idx].reshape(n, 25, 2).copy().view(np.uint16)[..., 0]
        if latent_fmt in INT8_GROUP:
            codes = logical.reshape(n, row).view(np.int8).copy()
            if latent_fmt == F_I8G8:         # word j of a chunk: channels 2j, 2j+1, 8+2j, 8+2j+1
                perm = np.array([0, 1, 8, 9, 2, 3, 10, 11, 4, 5, 12, 13, 6, 7, 14, 15])
                fixed = np.empty_like(codes)
                for c in range(row // 16):
                    fixed[:, 16 * c + perm] = codes[:, 16 * c:16 * c + 16]
                codes = fixed
            out["c_codes"] = codes
        else:
            codes = _nibbles(logical, n, nchunk)
            if latent_fmt == F_INT4:
                out["c_codes"] = codes
                out["c_zero"] = fp32_field(layout.zero_off, 32)
            else:
                out["c_codes"] = (codes.astype(np.int16) - 8).astype(np.int8)
    krow = layout.kpe_row_bytes
    kch = krow // 16
    kphys = gather(layout.kpe_off + u * krow, krow).reshape(n, kch, 16)
    c = np.arange(kch)[None, :]
    if kpe_fmt == F_BF16:
        kpos = c ^ (u[:, None] & 7)
    elif kpe_fmt == F_INT8:
        kpos = c ^ ((u[:, None] >> 1) & 3)
    else:
        kpos = c ^ ((u[:, None] >> 2) & 1)
    klog = np.take_along_axis(kphys, kpos[..., None], axis=1)
    if kpe_fmt == F_BF16:
        out["kpe_bits"] = klog.reshape(n, krow).copy().view(np.uint16)
    elif kpe_fmt == F_INT8:
        out["kpe_codes"] = klog.reshape(n, krow).view(np.int8).copy()
        out["kpe_scale"] = fp32_field(layout.kpe_scale_off, 8)
    else:
        out["kpe_codes"] = (_nibbles(klog, n, kch, channels=64).astype(np.int16) - 8).astype(np.int8)
        out["kpe_scale"] = fp32_field(layout.kpe_scale_off, 8)
    return out


def _nibbles(logical, n, nchunk, channels=512):
    """4-bit values of [n, nchunk, 16] logical chunk bytes (the documented
    word / nibble order) -> uint8 [n, channels]."""
    words = logical.reshape(n, nchunk, 4, 4).astype(np.uint32)
    words = words[..., 0] | (words[..., 1] << 8) | (words[..., 2] << 16) | (words[..., 3] << 24)
    codes = np.zeros((n, channels), np.uint8)
    for j in range(4):
        for k in range(8):
            ch = np.arange(nchunk) * 32 + _int4_channel(j, k)
            codes[:, ch] = (words[:, :, j] >> (4 * k)) & 15
    return codes


def assert_fields_match(got, c_bits, k_bits, latent_fmt, kpe_fmt, outliers=None):
    """Bit-exact comparison of stored fields with the oracle's quantization."""
    exp = Q.quantize_token_rows(synth.bf16_to_f32(c_bits), synth.bf16_to_f32(k_bits), latent_fmt, kpe_fmt,
                                outliers=outliers)
    if latent_fmt == F_BF16:
        assert np.array_equal(got["c_bits"], c_bits)
    else:
        assert np.array_equal(got["c_codes"].astype(np.int16), exp["c_codes"].astype(np.int16)), "latent codes differ"
        assert np.array_equal(got["c_scale"].view(np.uint32), exp["c_scale"].view(np.uint32)), "scales differ"
        assert np.array_equal(got["c_bound"].view(np.uint32), exp["c_bound"].view(np.uint32)), "bounds differ"
        if latent_fmt == F_I8OUT:
            assert np.array_equal(got["c_outlier_bits"], c_bits[:, np.asarray(outliers)]), "protected values differ"
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

    def outliers(self, layer):
        """The oracle's own calibration of the protected channels (outlier format)."""
        if self.wl.latent_fmt != F_I8OUT:
            return None
        return Q.select_outlier_channels(synth.bf16_to_f32(synth.calibration_latent_bf16(self.wl.seed, layer)))

    def decode(self, layer, b):
        """(q_lat, o_lat, lse, o) of the oracle for sequence b of `layer`."""
        qn, qp, wuk, wuv = self.query(layer)
        c_bits, k_bits = self.sequence(layer, b)
        d = Q.quantize_token_rows(synth.bf16_to_f32(c_bits), synth.bf16_to_f32(k_bits), self.wl.latent_fmt,
                                  self.wl.kpe_fmt, outliers=self.outliers(layer))
        return A.absorbed_decode_full(qn[b], qp[b], wuk, wuv, d["c_hat"], d["kpe_hat"])
