"""Seeded synthetic inputs for absorbed MLA decode (host side).

This module serves both the oracle (tests, bench baseline) and the CUDA path
(bench, tests): it holds the input recipe only and none of the method's
arithmetic (no quantization, no attention, no projection).  Its device twin,
``synth_gen.cu``, produces bit-identical values on the GPU so that full-size
caches can be filled quickly while the oracle regenerates any sampled
sequence on the host.

Recipe (the DeepSeek-V2-Lite shapes of the reports; value distributions of
the workload description):

* latent c[t, ch] = bf16( mu[ch] + sigma[ch] * z ), mu ~ U(-1, 1),
  sigma log-uniform on [0.1, 10], and round(1% of 512) = 5 outlier channels
  per layer whose mu and sigma are multiplied by 20;
* k_pe[t] = RoPE(z, position t): pairs (i, i + 32), base 10000, rotation
  done in fp32 with tabulated fp32 cos / sin;
* q_nope, q_pe = bf16(z); W_UK, W_UV = bf16(z / sqrt(512)) (variance 1/512);
  the queries of a prefill chunk come from their own streams, indexed like
  the decode queries with the token's index in the chunk in place of b.

z is an approximately standard normal variate built from a counter-based
generator: h = mix64(key + i * GOLDEN) with the splitmix64 finaliser
(Steele, Lea and Flood, "Fast splittable pseudorandom number generators",
2014), and z = (sum of the four 16-bit fields of h - 131070) / sqrt((2^32-1)/3)
(Irwin-Hall with n = 4: mean 0, variance 1, support +-3.46).  Every step is
exact integer arithmetic followed by one fp32 multiply, one fp32 add and one
round-to-nearest-even to bf16, so host and device agree bit for bit.

Element index i within a stream: latent / k_pe use ((b << 22 | t) << 10 | ch),
queries ((b << 10 | h) << 10 | k), weights ((h << 10 | row) << 10 | col).
A stream key is mix64-folded from (seed, layer, kind).
"""

import numpy as np

MASK64 = (1 << 64) - 1
GOLDEN = 0x9E3779B97F4A7C15
KIND_MUL = 0xD1B54A32D192ED03

KIND_LATENT, KIND_KPE, KIND_QNOPE, KIND_QPE, KIND_WUK, KIND_WUV, KIND_STATS = 1, 2, 3, 4, 5, 6, 7
KIND_NEW_LATENT, KIND_NEW_KPE = 8, 9
KIND_PRE_QNOPE, KIND_PRE_QPE = 10, 11          # queries of a prefill chunk

D_C, D_R, D_NOPE, D_V = 512, 64, 128, 128
ROPE_BASE = 10000.0

NORMAL_SCALE = np.float32(1.0 / np.sqrt((65536.0 ** 2 - 1.0) / 3.0))
WEIGHT_SCALE = np.float32(1.0 / np.sqrt(512.0))
UNIT_SCALE = np.float32(1.0)

_U64 = np.uint64


def mix64_int(z):
    """splitmix64 finaliser on a Python int (mod 2^64)."""
    z &= MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return z ^ (z >> 31)


def mix64(z):
    """splitmix64 finaliser on a uint64 array (wrap-around multiply)."""
    z = np.asarray(z, dtype=_U64)
    z = (z ^ (z >> _U64(30))) * _U64(0xBF58476D1CE4E5B9)
    z = (z ^ (z >> _U64(27))) * _U64(0x94D049BB133111EB)
    return z ^ (z >> _U64(31))


def stream_key(seed, layer, kind):
    k = mix64_int(seed & MASK64)
    k = mix64_int(k ^ ((layer * GOLDEN) & MASK64))
    return mix64_int(k ^ ((kind * KIND_MUL) & MASK64))


def hash_at(key, idx):
    idx = np.asarray(idx, dtype=_U64)
    with np.errstate(over="ignore"):
        return mix64(_U64(key) + idx * _U64(GOLDEN))


def normal_from_hash(h):
    m = _U64(0xFFFF)
    s = (h & m) + ((h >> _U64(16)) & m) + ((h >> _U64(32)) & m) + (h >> _U64(48))
    return (s.astype(np.int64) - 131070).astype(np.float32) * NORMAL_SCALE


def bf16_rne(x):
    """fp32 -> bf16 bits, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def bf16_to_f32(b):
    b = np.asarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------------------
# per-layer parameters (small; computed on the host and uploaded)
# ---------------------------------------------------------------------------

def channel_stats(seed, layer, n_outliers=5):
    """(mu, sigma) float32 [512] for one layer's latent channels."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, layer, KIND_STATS])))
    mu = rng.uniform(-1.0, 1.0, D_C)
    sigma = 0.1 * 100.0 ** rng.uniform(0.0, 1.0, D_C)
    out = rng.permutation(D_C)[:n_outliers]
    mu[out] *= 20.0
    sigma[out] *= 20.0
    return mu.astype(np.float32), sigma.astype(np.float32)


def rope_tables(n_pos):
    """fp32 cos / sin tables [n_pos, 32] for positions 0..n_pos-1."""
    inv = ROPE_BASE ** (-np.arange(0, D_R, 2, dtype=np.float64) / D_R)
    ang = np.arange(n_pos, dtype=np.float64)[:, None] * inv[None, :]
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)


def token_index(b, t, ch):
    return ((_U64(b) << _U64(22) | np.asarray(t, _U64)[:, None]) << _U64(10)) | np.asarray(ch, _U64)[None, :]


# ---------------------------------------------------------------------------
# bulk generators (host).  All return bf16 bits as uint16.
# ---------------------------------------------------------------------------

def latent_bf16(seed, layer, b, t0, t1, kind=KIND_LATENT, stats=None):
    """Latent rows c[t0:t1] of sequence b in `layer` -> uint16 [t1-t0, 512]."""
    mu, sigma = stats if stats is not None else channel_stats(seed, layer)
    key = stream_key(seed, layer, kind)
    out = np.empty((t1 - t0, D_C), np.uint16)
    step = 4096
    ch = np.arange(D_C)
    for a in range(t0, t1, step):
        e = min(t1, a + step)
        z = normal_from_hash(hash_at(key, token_index(b, np.arange(a, e), ch)))
        out[a - t0:e - t0] = bf16_rne(mu[None, :] + sigma[None, :] * z)
    return out


# The rows a layer's protected channels (outlier-protected format) are
# calibrated on: the first CALIBRATION_TOKENS latent rows of sequence 0.
CALIBRATION_TOKENS = 256


def calibration_latent_bf16(seed, layer):
    return latent_bf16(seed, layer, 0, 0, CALIBRATION_TOKENS, stats=channel_stats(seed, layer))


def kpe_bf16(seed, layer, b, t0, t1, cos_tab, sin_tab, kind=KIND_KPE):
    """k_pe rows of sequence b, positions t0..t1-1 -> uint16 [t1-t0, 64]."""
    key = stream_key(seed, layer, kind)
    out = np.empty((t1 - t0, D_R), np.uint16)
    step = 8192
    ch = np.arange(D_R)
    half = D_R // 2
    for a in range(t0, t1, step):
        e = min(t1, a + step)
        z = normal_from_hash(hash_at(key, token_index(b, np.arange(a, e), ch)))
        c, s = cos_tab[a:e], sin_tab[a:e]
        z1, z2 = z[:, :half], z[:, half:]
        lo = z1 * c - z2 * s
        hi = z1 * s + z2 * c
        out[a - t0:e - t0] = bf16_rne(np.concatenate([lo, hi], axis=1))
    return out


def _grid3(d0, d1, d2):
    i0 = np.arange(d0, dtype=_U64)[:, None, None]
    i1 = np.arange(d1, dtype=_U64)[None, :, None]
    i2 = np.arange(d2, dtype=_U64)[None, None, :]
    return ((i0 << _U64(10) | i1) << _U64(10)) | i2


def normal3_bf16(seed, layer, kind, d0, d1, d2, mul):
    """bf16(z * mul) on a [d0, d1, d2] grid indexed ((i0<<10|i1)<<10|i2)."""
    z = normal_from_hash(hash_at(stream_key(seed, layer, kind), _grid3(d0, d1, d2)))
    return bf16_rne(z * np.float32(mul))


def q_nope_bf16(seed, layer, B, H):
    return normal3_bf16(seed, layer, KIND_QNOPE, B, H, D_NOPE, UNIT_SCALE)


def q_pe_bf16(seed, layer, B, H):
    return normal3_bf16(seed, layer, KIND_QPE, B, H, D_R, UNIT_SCALE)


def normal_rows_bf16(seed, layer, kind, rows, d1, d2, mul):
    """Rows `rows` (any subset, any order) of the [*, d1, d2] grid of
    normal3_bf16: the same values, without generating the other rows."""
    i0 = np.asarray(rows, dtype=_U64)[:, None, None]
    i1 = np.arange(d1, dtype=_U64)[None, :, None]
    i2 = np.arange(d2, dtype=_U64)[None, None, :]
    z = normal_from_hash(hash_at(stream_key(seed, layer, kind), ((i0 << _U64(10) | i1) << _U64(10)) | i2))
    return bf16_rne(z * np.float32(mul))


def prefill_q_nope_bf16(seed, layer, rows, H):
    """q_nope of the prefill chunk's query tokens `rows` (index within the chunk)."""
    return normal_rows_bf16(seed, layer, KIND_PRE_QNOPE, rows, H, D_NOPE, UNIT_SCALE)


def prefill_q_pe_bf16(seed, layer, rows, H):
    return normal_rows_bf16(seed, layer, KIND_PRE_QPE, rows, H, D_R, UNIT_SCALE)


def w_uk_bf16(seed, layer, H):
    return normal3_bf16(seed, layer, KIND_WUK, H, D_NOPE, D_C, WEIGHT_SCALE)


def w_uv_bf16(seed, layer, H):
    return normal3_bf16(seed, layer, KIND_WUV, H, D_C, D_V, WEIGHT_SCALE)


def sequence_bf16(seed, layer, b, T, cos_tab, sin_tab, stats=None):
    """All T cached tokens of sequence b: the first T-1 are the prefilled
    context and token T-1 is the one appended by the decode step (its own
    stream), as the bench lays them out."""
    c = np.empty((T, D_C), np.uint16)
    k = np.empty((T, D_R), np.uint16)
    if T > 1:
        c[:T - 1] = latent_bf16(seed, layer, b, 0, T - 1, stats=stats)
        k[:T - 1] = kpe_bf16(seed, layer, b, 0, T - 1, cos_tab, sin_tab)
    if T > 0:
        c[T - 1:] = latent_bf16(seed, layer, b, T - 1, T, kind=KIND_NEW_LATENT, stats=stats)
        k[T - 1:] = kpe_bf16(seed, layer, b, T - 1, T, cos_tab, sin_tab, kind=KIND_NEW_KPE)
    return c, k


def page_permutation(seed, num_pages):
    """Seeded permutation of physical page ids (block tables are scattered)."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 0xB10C])))
    return rng.permutation(num_pages).astype(np.int32)


def log_uniform_lengths(seed, B, lo, hi):
    """Per-sequence context lengths round(exp(U(ln lo, ln hi)))."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 0x1E45])))
    return np.rint(np.exp(rng.uniform(np.log(lo), np.log(hi), B))).astype(np.int64)
