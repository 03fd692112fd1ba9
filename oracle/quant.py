"""Latent-cache quantizers (oracle; test infrastructure only).

Sources (page title, section):

* "DeepSeek-V2-Lite MLA 吸收式 KV 缓存优化 — 完整实验报告" (the Chinese report),
  §3.2 "量化方案对比": per-channel INT8 in 32 blocks, per-tensor INT8,
  per-token INT8, symmetric and asymmetric INT4 in 32 blocks, k_pe INT8 in
  8 blocks, k_pe symmetric INT4 in 8 blocks.
* "Absorbed MLA Cache Optimization on DeepSeek-V2-Lite — Technical Report"
  (the English report), §4.2 "Quantization Error Comparison" and §5.1
  (more blocks give lower error; 32 blocks recommended).
* "DeepSeek的MLA技术：极致压缩KV Cache的创新方案" (the juejin tutorial),
  section "量化压缩": scale = absmax / 127, code = round(x / scale),
  x_hat = code * scale.

Readings taken where the pages are open:

* "32 blocks" of the 512-dim latent are 32 groups of 16 consecutive channels
  with one scale per (token, group): a scale computed across future tokens is
  impossible when quantizing on write.
* Symmetric INT8: s = absmax / 127 in fp32, q = clamp(rint(x / s), -127, 127).
  A group whose absmax is 0 gets s = 0 and q = 0.
* Asymmetric INT4: s = (max - min) / 15 (one fp32 subtraction, one fp32
  division), z = rint(-min / s) stored as an integer-valued fp32,
  q = clamp(rint(x / s) + z, 0, 15).  x_hat = (q - z) * s.  When s comes out
  0: if min == 0 then s = z = q = 0; otherwise s = |min|, z = rint(-min / s)
  (= -1 or +1) and q = 0, which reconstructs the constant group exactly.
* The block count of INT8 is a format choice: the English report's §5.1
  compares 8, 32 and 64 blocks (groups of 64, 16 and 8 channels) and the
  Chinese report's §3.2 a per-token row (one block of 512); each is a cache
  format here (same rule, group size 8 / 16 / 32 / 64 / 512).
* Symmetric INT4 (the report's "对称 INT4 (32块)" latent row and "k_pe 对称
  INT4 (8块)" row): s = absmax / 7, q = clamp(rint(x / s), -7, 7), the
  INT8 rule with 7 levels a side; x_hat = q * s.  Used as a cache format
  for the latent and for k_pe (the report's 7.6 KB scheme pairs asymmetric
  INT4 latent codes with 4-bit k_pe).
* Outlier-protected mixed precision (the English report's §4.3 row "C:
  Mixed precision (outlier-protected)", 18.2 KB per token, 14.8x, 580K
  tokens in 10 GB; no mechanism is given): a fixed set of K = 25 latent
  channels per layer (5 % of 512, rounded down) keeps its bf16 input
  exactly; every other channel takes per-group symmetric INT8 (32 groups of
  16) with the protected channels left out of their group's absmax (their
  codes are 0); k_pe stays bf16, as in the row "B: latent8+kpe16" it
  extends.  512 + 2 x 25 + 128 = 690 code bytes per layer reproduce all
  three printed figures, which 24 or 26 channels do not (INT8 k_pe would
  need 57 protected channels, 11 %, for the same bytes; a whole 5 % with
  row B's bf16 k_pe is the plainer reading).  The protected set comes from
  calibration: the K channels with the largest max |x| over a sample of
  rows (ties to the lower index).
* All arithmetic is IEEE fp32 with round-half-even (NumPy float32 ops and
  ``np.rint``); no fused multiply-add.

Parity status: pinned (round-trip bound, brute-force nearest level,
hand-built half-way ties, degenerate groups, the pages' error ordering; the
outlier-protected format by exact protected channels, brute-force levels of
the rest, a literal group, brute-force channel selection and its error
ordering against per-group INT8).
"""

import numpy as np

F32 = np.float32


def _groups(x, group):
    x = np.asarray(x, dtype=np.float32)
    if x.ndim != 2 or x.shape[1] % group:
        raise ValueError("x must be [rows, channels] with channels % group == 0")
    return x.reshape(x.shape[0], x.shape[1] // group, group)


def quantize_sym_int8(x, group):
    """Symmetric INT8 with one fp32 scale per (row, group of `group` channels).

    Chinese report §3.2 row "per-channel INT8 (32块)" (group 16 on the
    512-dim latent) and row "k_pe INT8 (8块)" (group 8 on the 64-dim k_pe);
    tutorial "量化压缩" for scale = absmax/127 and code = round(x/scale).

    Returns (codes int8 [rows, channels], scale float32 [rows, groups]).
    """
    g = _groups(x, group)
    a = np.max(np.abs(g), axis=2)
    s = a / F32(127)
    live = s > 0
    safe = np.where(live, s, F32(1)).astype(np.float32)
    q = np.rint(g / safe[..., None])
    q = np.clip(q, -127, 127)
    q = np.where(live[..., None], q, F32(0))
    return q.astype(np.int8).reshape(x.shape), s.astype(np.float32)


def dequantize_sym_int8(codes, scale, group):
    """x_hat = float(code) * scale in fp32 (tutorial "量化压缩", dequantize line)."""
    codes = np.asarray(codes)
    rows, ch = codes.shape
    q = codes.astype(np.float32).reshape(rows, ch // group, group)
    return (q * np.asarray(scale, np.float32)[..., None]).reshape(rows, ch)


def quantize_asym_int4(x, group=16):
    """Asymmetric INT4 with fp32 scale and zero-point per (row, group).

    Chinese report §3.2 row "非对称 INT4 (32块)" and §4.1 (the 7.6 KB scheme);
    the scale / zero formulas are the plain affine min-max rule
    s = (max - min) / 15, z = round(-min / s).

    Returns (codes uint8 in [0, 15] [rows, channels] - one code per channel,
    not packed; scale float32 [rows, groups]; zero float32 [rows, groups]).
    """
    g = _groups(x, group)
    mn = np.min(g, axis=2)
    mx = np.max(g, axis=2)
    s = ((mx - mn).astype(np.float32) / F32(15)).astype(np.float32)
    deg = s == 0
    # degenerate group: s = |min| (or 0 when min == 0)
    s = np.where(deg, np.abs(mn), s).astype(np.float32)
    live = s > 0
    safe = np.where(live, s, F32(1)).astype(np.float32)
    z = np.rint(-mn / safe)
    z = np.where(live, z, F32(0)).astype(np.float32)
    r = np.rint(g / safe[..., None]).astype(np.float32)
    q = np.clip(r + z[..., None], 0, 15)
    q = np.where(live[..., None], q, F32(0))
    return q.astype(np.uint8).reshape(x.shape), s, z


def dequantize_asym_int4(codes, scale, zero, group=16):
    """x_hat = (float(code) - zero) * scale, both steps in fp32."""
    codes = np.asarray(codes)
    rows, ch = codes.shape
    q = codes.astype(np.float32).reshape(rows, ch // group, group)
    d = q - np.asarray(zero, np.float32)[..., None]
    return (d * np.asarray(scale, np.float32)[..., None]).reshape(rows, ch)


# ---------------------------------------------------------------------------
# Comparison quantizers: rows of the pages' error tables that the cache does
# not store, used only to pin the ordering the tables state.
# ---------------------------------------------------------------------------

def quantize_per_tensor_int8(x):
    """One scale for the whole tensor: Chinese report §3.2 "per-tensor INT8";
    tutorial "量化压缩" (its code takes abs().max() over the whole tensor)."""
    x = np.asarray(x, np.float32)
    s = np.max(np.abs(x)) / F32(127)
    if s == 0:
        return np.zeros(x.shape, np.int8), F32(0)
    q = np.clip(np.rint(x / s), -127, 127)
    return q.astype(np.int8), F32(s)


def quantize_per_token_int8(x):
    """One scale per row (token): Chinese report §3.2 "per-token INT8"."""
    x = np.asarray(x, np.float32)
    return quantize_sym_int8(x, x.shape[1])


def quantize_sym_int4(x, group=16):
    """Symmetric INT4, s = absmax / 7, codes in [-7, 7]: Chinese report §3.2
    rows "对称 INT4 (32块)" (group 16 on the latent; the row the asymmetric
    scheme is said to beat) and "k_pe 对称 INT4 (8块)" (group 8 on k_pe).

    Returns (codes int8 in [-7, 7] [rows, channels], scale float32 [rows, groups]).
    """
    g = _groups(x, group)
    a = np.max(np.abs(g), axis=2)
    s = (a / F32(7)).astype(np.float32)
    live = s > 0
    safe = np.where(live, s, F32(1)).astype(np.float32)
    q = np.clip(np.rint(g / safe[..., None]), -7, 7)
    q = np.where(live[..., None], q, F32(0))
    return q.astype(np.int8).reshape(x.shape), s


def dequantize_sym_int4(codes, scale, group):
    """x_hat = float(code) * scale in fp32 (same as the INT8 rule)."""
    return dequantize_sym_int8(codes, scale, group)


OUTLIER_CHANNELS = 25


def select_outlier_channels(sample, k=OUTLIER_CHANNELS):
    """Calibration of the protected set: the k channels with the largest
    max |x| over the sample rows [rows, 512], ties to the lower channel
    index; returned in increasing order (int32 [k])."""
    a = np.max(np.abs(np.asarray(sample, np.float32)), axis=0)
    order = sorted(range(a.shape[0]), key=lambda c: (-float(a[c]), c))
    return np.array(sorted(order[:k]), np.int32)


def quantize_int8_outlier(x, outliers, group=16):
    """Outlier-protected mixed precision (English report §4.3 row C, read as
    above): per-group symmetric INT8 of the channels outside `outliers`,
    whose absmax leaves the protected channels out; the protected channels
    keep their (bf16) input values and get code 0.

    Returns (codes int8 [rows, 512], scale float32 [rows, groups],
    values float32 [rows, k] of the protected channels in `outliers` order).
    """
    x = np.asarray(x, np.float32)
    o = np.asarray(outliers, np.int64)
    inl = x.copy()
    inl[:, o] = 0.0
    q, s = quantize_sym_int8(inl, group)
    return q, s, x[:, o].copy()


def dequantize_int8_outlier(codes, scale, values, outliers, group=16):
    """x_hat = code * scale on the INT8 channels, the stored value on the
    protected ones."""
    xh = dequantize_sym_int8(codes, scale, group)
    xh[:, np.asarray(outliers, np.int64)] = np.asarray(values, np.float32)
    return xh


def latent_bound(scale, zero=None, levels=127):
    """Per-token bound M_t on the dequantized latent: the largest magnitude a
    code of the token can dequantize to, the maximum over its groups of
    levels * s (symmetric formats: 127 levels a side for INT8, 7 for INT4)
    or of s * (|z - 7.5| + 7.5) (asymmetric INT4, where q - z ranges over
    -z .. 15 - z).  fp32, one rounding per product; the maximum skips NaN.

    Not a quantity of the pages: the cache stores it beside the scales so
    that the decode can weigh its fp16 P V roundings (the rows it recomputes
    exactly).  For the symmetric formats it equals max_c |x_hat[c]|, since
    each group's largest input maps to the extreme code.

    scale, zero: float32 [rows, groups].  Returns float32 [rows].
    """
    s = np.asarray(scale, np.float32)
    if zero is None:
        per_group = s * F32(levels)
    else:
        z = np.asarray(zero, np.float32)
        per_group = s * (np.abs(z - F32(7.5)) + F32(7.5))
    return np.fmax.reduce(per_group.astype(np.float32), axis=1).astype(np.float32)


def relative_error(x, x_hat):
    """Mean and max of |x - x_hat| / mean|x| over the tensor.

    The pages' error column ("平均误差 / Mean Relative Error") is not defined
    on them; this is the reading used for the ordering checks.
    """
    x = np.asarray(x, np.float64)
    e = np.abs(x - np.asarray(x_hat, np.float64))
    denom = np.mean(np.abs(x))
    return float(np.mean(e) / denom), float(np.max(e) / denom)


# ---------------------------------------------------------------------------
# Whole-token helpers used by tests: latent (512) + k_pe (64) in one call.
# ---------------------------------------------------------------------------

FMT_BF16, FMT_INT8, FMT_INT4, FMT_INT4_SYM = 0, 1, 2, 3
FMT_INT8_G8, FMT_INT8_G32, FMT_INT8_G64, FMT_INT8_TOKEN = 4, 5, 6, 7
FMT_INT8_OUTLIER = 8
LATENT_GROUP, KPE_GROUP = 16, 8
# symmetric INT8 latent formats -> channels per group (English report §5.1
# block-count sweep: 64, 16, 8 blocks; Chinese report §3.2 per-token row)
INT8_GROUP = {FMT_INT8: 16, FMT_INT8_G8: 8, FMT_INT8_G32: 32, FMT_INT8_G64: 64, FMT_INT8_TOKEN: 512}


def quantize_token_rows(c, kpe, latent_fmt, kpe_fmt, outliers=None):
    """Quantize latent rows c [N, 512] and k_pe rows kpe [N, 64] as the cache
    stores them (`outliers`: the protected channels of FMT_INT8_OUTLIER).
    Returns a dict of the stored fields plus the dequantized fp32 values the
    attention reads ("c_hat", "kpe_hat")."""
    c = np.asarray(c, np.float32)
    kpe = np.asarray(kpe, np.float32)
    out = {}
    if latent_fmt == FMT_BF16:
        out["c_hat"] = c.copy()
    elif latent_fmt in INT8_GROUP:
        g = INT8_GROUP[latent_fmt]
        q, s = quantize_sym_int8(c, g)
        out.update(c_codes=q, c_scale=s, c_hat=dequantize_sym_int8(q, s, g), c_bound=latent_bound(s))
    elif latent_fmt == FMT_INT4:
        q, s, z = quantize_asym_int4(c, LATENT_GROUP)
        out.update(c_codes=q, c_scale=s, c_zero=z,
                   c_hat=dequantize_asym_int4(q, s, z, LATENT_GROUP), c_bound=latent_bound(s, z))
    elif latent_fmt == FMT_INT4_SYM:
        q, s = quantize_sym_int4(c, LATENT_GROUP)
        out.update(c_codes=q, c_scale=s, c_hat=dequantize_sym_int4(q, s, LATENT_GROUP),
                   c_bound=latent_bound(s, levels=7))
    elif latent_fmt == FMT_INT8_OUTLIER:
        q, s, v = quantize_int8_outlier(c, outliers, LATENT_GROUP)
        vmax = np.fmax.reduce(np.abs(v), axis=1).astype(np.float32)
        out.update(c_codes=q, c_scale=s, c_outlier=v,
                   c_hat=dequantize_int8_outlier(q, s, v, outliers, LATENT_GROUP),
                   c_bound=np.fmax(latent_bound(s), vmax).astype(np.float32))
    else:
        raise ValueError("latent_fmt")
    if kpe_fmt == FMT_BF16:
        out["kpe_hat"] = kpe.copy()
    elif kpe_fmt == FMT_INT8:
        q, s = quantize_sym_int8(kpe, KPE_GROUP)
        out.update(kpe_codes=q, kpe_scale=s, kpe_hat=dequantize_sym_int8(q, s, KPE_GROUP))
    elif kpe_fmt == FMT_INT4_SYM:
        q, s = quantize_sym_int4(kpe, KPE_GROUP)
        out.update(kpe_codes=q, kpe_scale=s, kpe_hat=dequantize_sym_int4(q, s, KPE_GROUP))
    else:
        raise ValueError("kpe_fmt")
    return out
