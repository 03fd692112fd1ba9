/*
 * mla.h - C ABI of the absorbed Multi-head Latent Attention (MLA) decode
 * library for NVIDIA GB300 (sm_103a).
 *
 * What it computes.  A decode step of MLA attention runs directly against a
 * cache that keeps, per token and layer, one 512-dim compressed latent
 * ("compressed_kv") and one 64-dim RoPE key ("k_pe"), and never the per-head
 * K/V.  Sources (page title, section):
 *   [CN] "DeepSeek-V2-Lite MLA 吸收式 KV 缓存优化 — 完整实验报告"
 *        §1.1 (compressed_kv = kv_a_proj(h); K, V = kv_b_proj(compressed)),
 *        §3.1 (cache the 576-dim latent), §3.2 (per-group INT8 in 32 blocks,
 *        asymmetric INT4 in 32 blocks, k_pe INT8 in 8 blocks).
 *   [EN] "Absorbed MLA Cache Optimization on DeepSeek-V2-Lite — Technical
 *        Report" §1.3 (expanded K is nope 128 + rope 64, V is 128), §2.1
 *        (store(layer, compressed_kv, k_pe) quantizes on write; get()
 *        dequantizes and projects at compute time).
 *   [TU] "DeepSeek的MLA技术：极致压缩KV Cache的创新方案" (juejin tutorial),
 *        "步骤2" (K_i = C^KV W_i^upK, V_i = C^KV W_i^upV), "KV Cache的实现"
 *        (append the latent every step), "量化压缩" (scale = absmax / 127).
 * Per sequence b and head h, with c_hat / kpe_hat the dequantized cache:
 *   q_lat[h] = q_nope[h] @ W_UK[h]                         (mla_q_absorb)
 *   s[t]     = (q_lat[h] . c_hat[t] + q_pe[h] . kpe_hat[t]) * softmax_scale
 *   o_lat[h] = sum_t softmax(s)[t] c_hat[t];  lse[h] = log sum_t exp(s[t])
 *                                                          (mla_decode_absorbed)
 *   o[h]     = o_lat[h] @ W_UV[h]                          (mla_out_unabsorb)
 * Moving W_UK onto the query and W_UV onto the output is the algebraic
 * identity q.(W c) = (q W).c; it lets every cached byte be read once for all
 * heads.
 *
 * Conventions for every call.
 *   - Ownership: the caller allocates and frees all memory (device memory
 *     unless stated).  The library never allocates, frees or synchronizes;
 *     it keeps no state between calls apart from a per-device attribute
 *     cache.  Calls are thread-safe and re-entrant.
 *   - Execution: every call enqueues its kernels on `stream` (NULL = the
 *     legacy default stream) and returns without waiting.  The kernels use
 *     programmatic dependent launch: each may start while the previous
 *     kernels of the stream still run, and waits for them (griddepcontrol.wait,
 *     which also makes their stores visible) before touching data a kernel
 *     may have produced.  The few arrays read before that wait are named
 *     below ("read during the launch overlap"): no kernel enqueued on the
 *     stream since its last full ordering point (a host synchronisation, a
 *     cudaStreamWaitEvent, a memory copy) may write them, whether or not
 *     that kernel triggers its dependents early.
 *   - Layout: arrays are row-major and contiguous with the shapes given.
 *     bf16 values are passed as their 16-bit patterns (uint16_t).
 *   - Errors: arguments are checked on the host before any launch; a bad
 *     argument returns MLA_ERR_INVALID_ARG (or MLA_ERR_UNSUPPORTED for a
 *     valid but unimplemented shape) and launches nothing.  A failed launch
 *     returns MLA_ERR_CUDA.  Data-dependent faults found on the device (a
 *     slot, page id or sequence length out of range) never trap: the kernel
 *     skips the affected work and ORs a MLA_DEVERR_* bit into *dev_err when
 *     dev_err is not NULL.  The caller reads dev_err after the stream
 *     completes; a non-zero value means MLA_ERR_DEVICE_BOUNDS.
 *   - Heads: H is a multiple of 16 and at most 128.  Dimensions are fixed at
 *     the DeepSeek-V2 values: kv_lora_rank 512, rope 64, qk_nope 128, v 128.
 */
#ifndef MLA_GB300_H
#define MLA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;                       /* cudaStream_t is struct CUstream_st* */
typedef struct CUstream_st* mla_stream_t;

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1,
  MLA_ERR_UNSUPPORTED = 2,
  MLA_ERR_CUDA = 3,
  MLA_ERR_DEVICE_BOUNDS = 4
} mla_status;

typedef enum {
  MLA_FMT_BF16 = 0,        /* values stored as bf16, no scale */
  MLA_FMT_INT8_SYM = 1,    /* int8 code, fp32 scale per (token, group) */
  MLA_FMT_INT4_ASYM = 2,   /* 4-bit code, fp32 scale and zero per (token, group) */
  MLA_FMT_INT4_SYM = 3,    /* 4-bit code in [-7, 7], fp32 scale per (token, group) */
  /* INT8_SYM latent with another block count ([EN] §5.1 sweep of 8 / 32 /
   * 64 blocks, [CN] §3.2 per-token row); latent only, with INT8 k_pe */
  MLA_FMT_INT8_G8 = 4,     /* 64 blocks of 8 channels */
  MLA_FMT_INT8_G32 = 5,    /* 16 blocks of 32 channels */
  MLA_FMT_INT8_G64 = 6,    /* 8 blocks of 64 channels */
  MLA_FMT_INT8_TOKEN = 7,  /* one block of 512 channels (per-token scale) */
  /* outlier-protected mixed precision ([EN] §4.3 row "C: Mixed precision
   * (outlier-protected)", 18.2 KB per token, 14.8x, 580K tokens in 10 GB;
   * the page gives no mechanism, this is the reading): INT8_SYM latent
   * (32 groups of 16) except MLA_OUTLIER_CHANNELS protected channels per
   * layer, kept as their bf16 input and left out of their group's absmax
   * (their codes are 0).  512 + 2 x 25 code bytes plus bf16 k_pe give the
   * row's 690 B per layer.  k_pe: MLA_FMT_BF16 (the row) or INT8_SYM. */
  MLA_FMT_INT8_OUTLIER = 8
} mla_fmt;

/* Bits ORed into *dev_err. */
#define MLA_DEVERR_SLOT    1  /* append: slot not in [0, num_pages*64) and not -1 */
#define MLA_DEVERR_PAGE    2  /* decode: block_table entry not in [0, num_pages)   */
#define MLA_DEVERR_SEQLEN  4  /* decode: seq_len < 0 or > max_pages*64            */
#define MLA_DEVERR_TIMEOUT 8  /* a bounded wait inside a kernel gave up           */

#define MLA_KV_LORA_RANK 512
#define MLA_ROPE_DIM 64
#define MLA_QK_NOPE_DIM 128
#define MLA_V_DIM 128
#define MLA_PAGE_TOKENS 64
#define MLA_LATENT_GROUP 16      /* 512 channels = 32 groups ([CN] §3.2 "32块") */
#define MLA_KPE_GROUP 8          /* 64 channels = 8 groups ([CN] §3.2 "8块")   */
#define MLA_OUTLIER_CHANNELS 25  /* protected channels of MLA_FMT_INT8_OUTLIER (5 % of 512) */

/*
 * One layer's paged latent cache.  The pool holds num_pages pages of 64
 * tokens; a token's physical slot is page * 64 + offset.  Which pages belong
 * to which sequence is the caller's business (block tables below).
 *   latent_fmt: any mla_fmt.  kpe_fmt: MLA_FMT_BF16, MLA_FMT_INT8_SYM or
 *   MLA_FMT_INT4_SYM; the INT8_G* / INT8_TOKEN latent formats take
 *   MLA_FMT_INT8_SYM k_pe only, INT8_OUTLIER takes BF16 or INT8_SYM.
 *   pool: device memory of mla_cache_pool_bytes() bytes, 256-byte aligned,
 *         owned by the caller.
 *   outlier_channels: INT8_OUTLIER only (NULL for every other format): HOST
 *         memory holding the layer's MLA_OUTLIER_CHANNELS protected latent
 *         channels, strictly increasing, in [0, 512) (for instance from
 *         mla_select_outlier_channels); read during each call, by value.
 *         Every call on a layer must pass the same set; a violation of
 *         these rules is MLA_ERR_INVALID_ARG.
 */
typedef struct {
  int32_t num_pages;
  int32_t latent_fmt;
  int32_t kpe_fmt;
  int32_t reserved;        /* must be 0 */
  void* pool;
  const int32_t* outlier_channels;
} mla_cache_layer;

/*
 * Byte layout of one page.  A page of 64 tokens is two contiguous blocks of
 * 32 tokens (token t of a page lives in block t / 32 as block token
 * u = t % 32), so that one bulk copy moves a whole 32-token work unit.
 * Inside a block, structure of arrays; offsets are from the block start,
 * every field starts on a 128-byte boundary, -1 marks a field the format
 * does not have:
 *   codes      [32][codes_row_bytes]: bf16 values (1024 B), int8 codes
 *              (512 B) or 4-bit codes (256 B).  The row is a sequence of
 *              16-byte chunks; logical chunk c of block token u is stored at
 *              chunk position (c & ~7) | ((c ^ u) & 7).  An int8 chunk is 16
 *              channels in channel order (INT8_G8: its 32-bit word j holds
 *              channels 2j, 2j+1, 8+2j, 8+2j+1); a bf16 chunk is 8 channels.
 *              A 4-bit chunk c holds groups A = 2c and B = 2c + 1; its 32-bit
 *              word j (j = 0..3) packs, from the least significant nibble,
 *              A[4j], A[4j+2], B[4j], B[4j+2], A[4j+1], A[4j+3], B[4j+1],
 *              B[4j+3] (X[i] = nibble of channel i of group X).  A nibble is
 *              the code (INT4_ASYM, 0..15) or the code + 8 (INT4_SYM, 1..15).
 *   scale      fp32 [G groups][32 block tokens]    (int8 / 4-bit latent; G = 32,
 *              or 64 / 16 / 8 / 1 for INT8_G8 / G32 / G64 / TOKEN)
 *   zero       fp32 [32 groups][32 block tokens]   (INT4_ASYM latent; integer-valued)
 *   outlier    bf16 [25 protected channels][32 block tokens], in the order
 *              of outlier_channels, padded to 1664 bytes (INT8_OUTLIER)
 *   kpe        [32][kpe_row_bytes]: bf16 (128 B = 8 chunks of 8 channels,
 *              chunk c of token u at position c ^ (u & 7)), int8 (64 B =
 *              4 chunks of two 8-channel groups, chunk c at c ^ ((u >> 1) & 3))
 *              or INT4_SYM (32 B = 2 chunks of 32 channels, chunk c at
 *              c ^ ((u >> 2) & 1); chunk c packs its halves A = channels
 *              32c .. 32c+15 and B = 32c+16 .. 32c+31 like a 4-bit latent
 *              chunk, nibble = code + 8)
 *   kpe_scale  fp32 [8 groups][32 block tokens]    (int8 / INT4_SYM k_pe)
 *   bound      fp32 [32 block tokens]              (int8 / 4-bit latent)
 *              M_t, the largest magnitude a code of the token's latent can
 *              dequantize to: 127 max_g s_g (INT8 formats), 7 max_g s_g
 *              (INT4_SYM), max_g s_g (|z_g - 7.5| + 7.5) (INT4_ASYM), in
 *              fp32 with one rounding per product; INT8_OUTLIER also takes
 *              the protected values' magnitudes into the maximum.  For INT8
 *              and INT4_SYM formats it equals max_c |c_hat[c]|.  Written by mla_cache_append;
 *              the decode reads it to find the rows it recomputes exactly
 *              (see mla_decode_absorbed).
 * page_bytes = 2 * block_bytes = 64 x (1152, 740, 612 or 580) bytes for
 * bf16/bf16, int8/int8, int4/int8 and int4/int4-sym (the last is [CN]
 * §4.1's 7.6 KB-per-token scheme: 288 B of codes per layer plus scales,
 * zero-points and the bound).  The swizzles spread the rows of eight consecutive tokens
 * over all shared-memory banks when a block is copied verbatim into shared
 * memory.
 */
typedef struct {
  int64_t page_bytes, block_bytes;
  int64_t codes_off, codes_row_bytes;
  int64_t scale_off, zero_off;
  int64_t kpe_off, kpe_row_bytes;
  int64_t kpe_scale_off;
  int64_t bound_off;
  int64_t outlier_off;
} mla_page_layout;

/* Fills *out for the cache's formats.  MLA_ERR_INVALID_ARG on a bad format. */
mla_status mla_cache_page_layout(const mla_cache_layer* cache, mla_page_layout* out);

/* num_pages * page_bytes, or 0 for an invalid descriptor. */
size_t mla_cache_pool_bytes(const mla_cache_layer* cache);

/*
 * mla_cache_append - quantize-on-write of n new tokens into the paged cache.
 * [EN] §2.1 store(): compressed_kv [seq, 512] is quantized, k_pe [seq, 64]
 * stored; [CN] §3.2 for the formats.  Quantization rules, all IEEE fp32 with
 * round-half-even and no fused multiply-add:
 *   INT8_SYM  (groups of 16 latent channels - 8, 32, 64 or 512 for the
 *             INT8_G8 / G32 / G64 / TOKEN formats - or 8 k_pe channels):
 *       s = max|x| / 127;  q = clamp(rint(x / s), -127, 127);  s = 0 -> q = 0
 *   INT4_ASYM (groups of 16): s = (max - min) / 15;  z = rint(-min / s);
 *       q = clamp(rint(x / s) + z, 0, 15); if s == 0: s = |min|, z = rint(-min/s)
 *       (or s = z = 0 when min == 0) and q = 0.
 *   INT4_SYM  (groups of 16 latent channels, or 8 k_pe channels; [CN] §3.2
 *       "对称 INT4" rows): s = max|x| / 7;  q = clamp(rint(x / s), -7, 7);
 *       s = 0 -> q = 0.
 *   INT8_OUTLIER: the protected channels' input bits are stored, their
 *       codes are 0, and the INT8_SYM rule runs on the other channels with
 *       the protected ones counted as 0 in their group's max|x|.
 *   BF16: the input bits are copied.
 *   A quantized latent also gets its bound M_t (see mla_page_layout).
 *   c_new   bf16 [n][512]     kpe_new bf16 [n][64]
 *   slot    int32 [n]: physical slot (page * 64 + offset) of each token;
 *           -1 skips the token silently; any other value outside
 *           [0, num_pages * 64) skips it and sets MLA_DEVERR_SLOT.
 *   Two tokens with the same slot in one call race; the result is one of them.
 *   n == 0 is a no-op.  dev_err may be NULL.
 */
mla_status mla_cache_append(const mla_cache_layer* cache, const uint16_t* c_new,
                            const uint16_t* kpe_new, const int32_t* slot, int32_t n,
                            int32_t* dev_err, mla_stream_t stream);

/*
 * mla_select_outlier_channels - calibration of MLA_FMT_INT8_OUTLIER's
 * protected set ([EN] §4.3 row C, read as in mla_fmt): the
 * MLA_OUTLIER_CHANNELS latent channels with the largest max |x| over n
 * sample rows, ties to the lower channel index, written in increasing
 * order.  NaN inputs are skipped by the maximum.
 *   c_sample     device bf16 [n][512], 16-byte aligned; n >= 1
 *   channels_out device int32 [MLA_OUTLIER_CHANNELS], 4-byte aligned
 */
mla_status mla_select_outlier_channels(const uint16_t* c_sample, int32_t n, int32_t* channels_out,
                                       mla_stream_t stream);

/*
 * mla_q_absorb - q_lat[b][h] = q_nope[b][h] @ W_UK[h]   (the query side of
 * weight absorption; [TU] "步骤2" K_i = C^KV W_i^upK with W_UK[h] = (W_i^upK)^T).
 *   q_nope bf16 [B][H][128]   W_UK bf16 [H][128][512]   q_lat fp32 [B][H][512]
 *   fp32 accumulation of exact bf16 products.  B == 0 is a no-op.
 *   W_UK is read during the launch overlap (see Execution above).
 */
mla_status mla_q_absorb(const uint16_t* q_nope, const uint16_t* w_uk, float* q_lat,
                        int32_t batch, int32_t heads, mla_stream_t stream);

/*
 * mla_decode_workspace_bytes - bytes of device workspace mla_decode_absorbed
 * needs for this batch, head count and num_splits (0 = automatic).  The
 * workspace holds the split-K partials (per split and head, fp32: running
 * max, running sum, the weight of the fp16 P V products and the
 * unnormalised 512-wide latent output).
 */
size_t mla_decode_workspace_bytes(int32_t batch, int32_t heads, int32_t num_splits);

/*
 * mla_decode_absorbed - absorbed attention of one decode query per sequence
 * against its cached latents ([EN] §2.1 get(): attention computed from the
 * latent; flash-decode split over context chunks with a log-sum-exp
 * combine).  Dequantization is fused into the tile loads: x_hat = q * s for
 * INT8 and INT4_SYM, (q - z) * s for INT4_ASYM.
 *   q_lat       fp32 [B][H][512]   (from mla_q_absorb)
 *   q_pe        bf16 [B][H][64]
 *   block_table int32 [B][max_pages]: page id of each sequence's logical page
 *   seq_lens    int32 [B]: tokens attended (positions 0..len-1, the newly
 *               appended token included).  0 gives o_lat = 0 and lse = -inf.
 *   softmax_scale: typically 1 / sqrt(128 + 64).
 *   num_splits: ranges the context work is divided into, 1 .. 65535
 *               (0 = automatic: SMs / (H / 16), so that the H / 16 head
 *               tiles of every range run side by side, one CTA per SM, and
 *               read the range's pages once between them).  Work is split
 *               evenly over all sequences' 32-token chunks.
 *   workspace:  device, >= mla_decode_workspace_bytes(B, H, num_splits)
 *               bytes, 256-byte aligned; contents are scratch.
 *   o_lat fp32 [B][H][512]      lse fp32 [B][H] (natural log; may be NULL)
 *   Precision, against attention in fp64 over the same dequantized values:
 *   the scores use exact products (q_lat split into two fp16 parts against
 *   the exact codes); P enters the P V products as fp16 times the fp16
 *   group scale, which costs ~2-6e-4 relative error over long contexts.
 *   Two kinds of rows are recomputed in fp32 from the cache instead:
 *   sequences shorter than 256 tokens, and rows whose output is a small
 *   residual of heavily weighted tokens (latents that cancel), detected
 *   from the partials as sqrt(sum_t (w_t M_t)^2) > 4 |o_lat row|_inf, with
 *   w_t the softmax weights and M_t a bound on token t's |c_hat| from its
 *   scales (and zero-points).
 *   Every row is tested to a max relative error below 2e-3 (o_lat) and
 *   2e-3 absolute (lse).
 *   A page id outside [0, num_pages) contributes nothing and sets
 *   MLA_DEVERR_PAGE; seq_len outside [0, max_pages*64] is treated as 0 and
 *   sets MLA_DEVERR_SEQLEN.  B == 0 is a no-op.  B <= 4096, and
 *   B * max_pages * 2 (the batch's 32-token chunk capacity) < 2^31, else
 *   MLA_ERR_INVALID_ARG.
 *   seq_lens is read during the launch overlap (see Execution above).
 */
mla_status mla_decode_absorbed(const mla_cache_layer* cache, const float* q_lat,
                               const uint16_t* q_pe, const int32_t* block_table,
                               int32_t max_pages, const int32_t* seq_lens, int32_t batch,
                               int32_t heads, float softmax_scale, int32_t num_splits,
                               void* workspace, size_t workspace_bytes, float* o_lat,
                               float* lse, int32_t* dev_err, mla_stream_t stream);

/*
 * mla_decode_absorbed_unabsorb - mla_decode_absorbed followed by
 * mla_out_unabsorb on its o_lat, in one call: o[b][h] = o_lat[b][h] @ W_UV[h]
 * ([TU] "步骤2", V_i = C^KV W_i^upV, the output side of the absorption).
 * The arguments are mla_decode_absorbed's plus
 *   w_uv  device bf16 [H][512][128], 16-byte aligned (as mla_out_unabsorb)
 *   o     device fp32 [B][H][128], 16-byte aligned
 * Both must be non-NULL (MLA_ERR_INVALID_ARG otherwise).  o_lat and lse are
 * written as by mla_decode_absorbed.  When the batch takes the combine's
 * one-block-per-(sequence, head) grid (about 8 to 32 context splits per
 * sequence, e.g. a few sequences of a few thousand tokens), that block
 * projects its row right after merging it (fp32 multiply-adds over bf16
 * W_UV), which removes a kernel from the decode step's critical path;
 * otherwise the call launches the unabsorb kernel after the combine.  The
 * two ways differ only in the order of the fp32 sums.
 */
/*
 * mla_decode_kernel_count - how many kernels one mla_decode_absorbed call
 * (with_unabsorb = 0) or mla_decode_absorbed_unabsorb call (1) launches for
 * this batch shape: the split kernel and the combine, plus the unabsorb
 * kernel when the combine's grid does not project the rows itself.  0 for
 * batch 0, -1 for arguments the calls would reject.  Host only.
 */
int32_t mla_decode_kernel_count(const mla_cache_layer* cache, int32_t batch, int32_t heads, int32_t num_splits,
                                int32_t with_unabsorb);

mla_status mla_decode_absorbed_unabsorb(const mla_cache_layer* cache, const float* q_lat,
                                        const uint16_t* q_pe, const int32_t* block_table,
                                        int32_t max_pages, const int32_t* seq_lens, int32_t batch,
                                        int32_t heads, float softmax_scale, int32_t num_splits,
                                        void* workspace, size_t workspace_bytes, float* o_lat,
                                        float* lse, const uint16_t* w_uv, float* o, int32_t* dev_err,
                                        mla_stream_t stream);

/*
 * mla_decode_absorbed_noalloc - the same decode as mla_decode_absorbed for
 * callers that cannot allocate device memory: a plugin handed only its input
 * and output buffers, code running during CUDA-graph capture (cudaMalloc is
 * not capturable there), or a serving loop that forbids allocation after
 * start-up.  The source pages have no counterpart; this is a deployment
 * variant of the call above.
 *   Arguments and results are those of mla_decode_absorbed, without the
 *   workspace: the split-K partials go to a scratch array of
 *   MLA_NOALLOC_SCRATCH_BYTES compiled into the library, which every device
 *   that loads the library holds until the process exits.  It calls no
 *   allocator (no cudaMalloc, cudaFree or allocating library routine).
 *   Returns MLA_ERR_INVALID_ARG when mla_decode_workspace_bytes(batch, heads,
 *   num_splits) exceeds MLA_NOALLOC_SCRATCH_BYTES (e.g. 64 heads at batch 64
 *   with the automatic split count fits; pass a smaller num_splits
 *   otherwise).
 *   The first call on a device looks up the array's device address (with
 *   that device current) and caches it; make that first call before any
 *   stream capture.  All calls share the array and it keeps the last call's
 *   contents (nothing in it needs to start at zero), so calls that overlap
 *   on the GPU - on different streams or from different host threads - race.
 */
#define MLA_NOALLOC_SCRATCH_BYTES (32u << 20)
mla_status mla_decode_absorbed_noalloc(const mla_cache_layer* cache, const float* q_lat,
                                       const uint16_t* q_pe, const int32_t* block_table,
                                       int32_t max_pages, const int32_t* seq_lens, int32_t batch,
                                       int32_t heads, float softmax_scale, int32_t num_splits,
                                       float* o_lat, float* lse, int32_t* dev_err, mla_stream_t stream);

/*
 * mla_prefill_workspace_bytes - bytes of device workspace mla_prefill_absorbed
 * needs for a chunk of n query tokens and this head count under the current
 * prefill path setting (0 for invalid arguments).  Bounded in n: queries are
 * processed in slices of 2048 (decode kernels) or 4096 (tensor cores: 288 KB
 * of query tiles per 128 rows, ~600 MB at 64 heads); the tensor-core path
 * adds the key tiles of up to 65536 positions (~151 MB).
 */
size_t mla_prefill_workspace_bytes(int32_t n, int32_t heads);

/*
 * Prefill implementations (mla_set_prefill_path):
 *   MLA_PREFILL_AUTO           tensor cores when 256 < ctx_before + n <=
 *                              65536 and either n * heads >= 8192, or
 *                              n * heads >= 2048 and ctx_before + n >= 4096;
 *                              else the decode kernels (the default)
 *   MLA_PREFILL_DECODE_KERNELS always the split-K decode kernels
 *   MLA_PREFILL_TENSOR_CORES   always tensor cores; a call with
 *                              ctx_before + n > 65536 returns
 *                              MLA_ERR_UNSUPPORTED
 * Both compute the same attention within the same bound (§ prefill below).
 */
#define MLA_PREFILL_AUTO 0
#define MLA_PREFILL_DECODE_KERNELS 1
#define MLA_PREFILL_TENSOR_CORES 2

/*
 * mla_set_prefill_path - selects the implementation of the prefill calls this
 * process makes afterwards (and the size mla_prefill_workspace_bytes
 * returns); returns the previous setting, or -1 (nothing changed) for an
 * unknown value.
 */
int32_t mla_set_prefill_path(int32_t path);

/*
 * mla_prefill_path_taken - the implementation (MLA_PREFILL_DECODE_KERNELS or
 * MLA_PREFILL_TENSOR_CORES) a prefill call with these sizes takes under the
 * current setting; -1 for invalid sizes.
 */
int32_t mla_prefill_path_taken(int32_t ctx_before, int32_t n, int32_t heads);

/*
 * mla_prefill_absorbed - causal absorbed attention of a prefill chunk: the
 * queries of n tokens of one sequence that were just appended to the cache
 * (chunked prefill when ctx_before > 0).  Query i sits at position
 * ctx_before + i and attends to the cached positions 0 .. ctx_before + i,
 * its own token included; per query this is the decode of [EN] §2.1 over
 * that prefix.  Tensor-core path: the cached tokens are dequantized once
 * into fp16 (hi, lo) key tiles and a tcgen05 kernel runs 128 query rows
 * against 128 keys at a time (scores from three fp16 products, P and V in
 * fp16, fp32 accumulation); decode-kernel path: the split-K decode kernels
 * with the queries as the batch.  On both, rows that see fewer than 256
 * tokens, and rows whose softmax weight sits on tokens whose latents cancel
 * (the decode's precision check), are recomputed exactly in fp32.
 *   q_lat       fp32 [n][H][512]  (mla_q_absorb with batch = n)
 *   q_pe        bf16 [n][H][64]
 *   block_table int32 [max_pages]: the sequence's page ids; positions up to
 *               ctx_before + n - 1 must have been appended.
 *   workspace:  device, >= mla_prefill_workspace_bytes(n, H) bytes,
 *               256-byte aligned; contents are scratch.
 *   o_lat fp32 [n][H][512]      lse fp32 [n][H] (natural log; may be NULL)
 *   n == 0 is a no-op.  ctx_before >= 0 and ctx_before + n <= max_pages * 64,
 *   else MLA_ERR_INVALID_ARG.  A page id outside [0, num_pages) contributes
 *   nothing and sets MLA_DEVERR_PAGE.
 */
mla_status mla_prefill_absorbed(const mla_cache_layer* cache, const float* q_lat, const uint16_t* q_pe,
                                const int32_t* block_table, int32_t max_pages, int32_t ctx_before, int32_t n,
                                int32_t heads, float softmax_scale, void* workspace, size_t workspace_bytes,
                                float* o_lat, float* lse, int32_t* dev_err, mla_stream_t stream);

/*
 * mla_out_unabsorb - o[b][h] = o_lat[b][h] @ W_UV[h]   (the output side of
 * weight absorption; [TU] "步骤2" V_i = C^KV W_i^upV with W_UV[h] = W_i^upV).
 *   o_lat fp32 [B][H][512]   W_UV bf16 [H][512][128]   o fp32 [B][H][128]
 *   B == 0 is a no-op.  W_UV is read during the launch overlap (see
 *   Execution above).
 */
mla_status mla_out_unabsorb(const float* o_lat, const uint16_t* w_uv, float* o,
                            int32_t batch, int32_t heads, mla_stream_t stream);

/*
 * mla_lse_merge - attention over the union of disjoint context parts of the
 * same sequences, from the parts' own results: the exchange step of a
 * context-sharded decode (each GPU runs mla_decode_absorbed over its own
 * pages of a sequence; the (o_lat, lse) pairs are gathered and merged here).
 * With M = max_r lse_r and w_r = exp(lse_r - M):
 *   o_lat = sum_r w_r o_r / sum_r w_r,   lse = M + ln sum_r w_r
 * which is exactly the softmax attention of [EN] §2.1 over the union.
 *   o_parts  fp32 [R][B][H][512]   lse_parts fp32 [R][B][H]  (natural log;
 *            -inf marks an empty part, weight 0)
 *   o_lat    fp32 [B][H][512]      lse fp32 [B][H] (may be NULL)
 *   All parts empty gives o_lat = 0 and lse = -inf.  1 <= R <= 4096,
 *   B <= 4096, H as for the decode; B == 0 is a no-op.  Arrays 16-byte
 *   aligned; o_lat must not overlap o_parts.
 */
mla_status mla_lse_merge(const float* o_parts, const float* lse_parts, int32_t parts, int32_t batch,
                         int32_t heads, float* o_lat, float* lse, mla_stream_t stream);

/* Static string for a status code. */
const char* mla_status_string(mla_status status);

/* Text of the CUDA error behind the calling thread's most recent
 * MLA_ERR_CUDA ("no error" if none); a static string, not to be freed. */
const char* mla_last_cuda_error(void);

/*
 * mla_set_wait_limit_ns - bound, in nanoseconds, on every wait inside the
 * decode kernels (stage arrivals, the hand-offs between the block's warp
 * roles) of the decode and prefill calls this process launches afterwards;
 * returns the previous bound, or -1 (nothing changed) for ns < 0.  The
 * default is 10 s.  A test and diagnostic hook, not part of the pages'
 * method: a wait that runs out sets MLA_DEVERR_TIMEOUT in *dev_err, and its
 * block writes empty partials (weight 0) for the rest of its share of the
 * context and leaves once its own bulk copies have landed.  Nothing traps
 * and the outputs stay finite, but they miss that share of the context.
 * With ns = 0 a wait polls without suspending and gives up once the GPU's
 * global timer has advanced (within about a microsecond) without completion.
 */
int64_t mla_set_wait_limit_ns(int64_t ns);

/* ABI version (major * 100 + minor). */
int32_t mla_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MLA_GB300_H */
