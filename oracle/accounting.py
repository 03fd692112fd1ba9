"""KV-cache byte accounting and capacity (oracle; test infrastructure).

Sources (page title, section):

* "DeepSeek-V2-Lite MLA 吸收式 KV 缓存优化 — 完整实验报告": §1.2 理论压缩率
  (2x16x(128+64+128)x27 = 276,480 B; (512+64+128)x27 = 19,008 B; 14.5x),
  §1.3 (10,240 B/layer, 270 KB), §3.1 (30.4 KB, 8.9x), §4.1 (15.2 KB 17.8x,
  7.6 KB 35.6x, 10 GB holds 690K / 1.38M tokens).
* "Absorbed MLA Cache Optimization on DeepSeek-V2-Lite — Technical Report":
  §1.3 ((192+128) x 16 heads x 2 B = 10,240 B), §2.2 ((512+64)x2 = 1,152 B;
  512x1 + 64x2 = 640 B, 16.9 KB), §4.3 (39K / 340K / 690K / 620K / 1.24M
  tokens in 10 GB; 8.4 KB for INT4 + k_pe INT8, 32x; row C, mixed precision
  (outlier-protected), 18.2 KB, 14.8x, 580K tokens).

Conventions the pages' numbers fix: "KB" is 1024 bytes (276,480 B is printed
as 270 KB), "10 GB" is 10 x 2^30 bytes (39K, 690K, 620K, 1.24M and 1.38M all
come out of it), and the code-only figures count 1 byte per INT8 element,
half a byte per INT4 element and 2 bytes per bf16 element.

The cache this library builds stores fp32 scales (and fp32 zero-points for
asymmetric INT4) on top of the codes; ``layer_bytes(..., metadata=True)``
reports those bytes explicitly.

Parity status: pinned (every printed figure is reproduced as an exact integer
or to the printed rounding, in tests/test_oracle_accounting.py).
"""

FMT_BF16, FMT_INT8, FMT_INT4, FMT_INT4_SYM = 0, 1, 2, 3
FMT_INT8_G8, FMT_INT8_G32, FMT_INT8_G64, FMT_INT8_TOKEN = 4, 5, 6, 7
FMT_INT8_OUTLIER = 8
OUTLIER_CHANNELS = 25       # protected bf16 channels of FMT_INT8_OUTLIER
INT8_GROUP = {FMT_INT8: 16, FMT_INT8_G8: 8, FMT_INT8_G32: 32, FMT_INT8_G64: 64, FMT_INT8_TOKEN: 512}

KV_LORA_RANK = 512
ROPE_DIM = 64
QK_NOPE_DIM = 128
V_DIM = 128
V2_LITE_LAYERS = 27
V2_LITE_HEADS = 16
LATENT_GROUP = 16
KPE_GROUP = 8
KIB = 1024
TEN_GB = 10 * 2 ** 30


def expanded_layer_bytes(heads=V2_LITE_HEADS, elem_bytes=2):
    """Expanded K (nope + rope = 192) and V (128) per head, bf16."""
    return (QK_NOPE_DIM + ROPE_DIM + V_DIM) * heads * elem_bytes


def mla_theoretical_token_bytes(layers=V2_LITE_LAYERS):
    """The reports' "MLA theoretical" row, reproduced as printed:
    (512 + 64 + 128) x layers at one byte per element."""
    return (KV_LORA_RANK + ROPE_DIM + 128) * layers


def _elem_bytes(fmt, n):
    if fmt == FMT_BF16:
        return 2 * n
    if fmt in INT8_GROUP:
        return n
    if fmt == FMT_INT8_OUTLIER:           # int8 codes plus the protected channels in bf16
        return n + 2 * OUTLIER_CHANNELS
    if fmt in (FMT_INT4, FMT_INT4_SYM):
        return n // 2
    raise ValueError(fmt)


def layer_bytes(latent_fmt, kpe_fmt, metadata=False):
    """Bytes per token per layer of the absorbed cache.

    metadata=False gives the pages' code-only figure; metadata=True adds one
    fp32 scale per group (and one fp32 zero-point per latent group for
    asymmetric INT4), which is what the cache here actually stores.  4-bit
    k_pe is symmetric (FMT_INT4_SYM; FMT_INT4 gives the same code-only
    figure), as in the Chinese report's "k_pe 对称 INT4 (8块)" row.
    """
    b = _elem_bytes(latent_fmt, KV_LORA_RANK) + _elem_bytes(kpe_fmt, ROPE_DIM)
    if metadata:
        lg = KV_LORA_RANK // LATENT_GROUP
        kg = ROPE_DIM // KPE_GROUP
        if latent_fmt in INT8_GROUP:
            b += 4 * (KV_LORA_RANK // INT8_GROUP[latent_fmt])
        elif latent_fmt == FMT_INT8_OUTLIER:
            b += 4 * lg
        elif latent_fmt == FMT_INT4:
            b += 8 * lg
        elif latent_fmt == FMT_INT4_SYM:
            b += 4 * lg
        if kpe_fmt in (FMT_INT8, FMT_INT4, FMT_INT4_SYM):
            b += 4 * kg
    return b


def token_bytes(per_layer, layers=V2_LITE_LAYERS):
    return per_layer * layers


def kib(nbytes):
    return nbytes / KIB


def ratio(baseline_bytes, nbytes):
    return baseline_bytes / nbytes


def capacity_tokens(bytes_per_token, budget=TEN_GB):
    """Whole tokens that fit in `budget` bytes."""
    return budget // bytes_per_token
