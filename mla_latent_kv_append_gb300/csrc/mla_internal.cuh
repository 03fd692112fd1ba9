// Internal helpers shared by the library's translation units (device code and
// host-side launch plumbing).  Not part of the C ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/mla.h"

namespace mla {

constexpr int kDc = MLA_KV_LORA_RANK;      // 512 latent channels
constexpr int kDr = MLA_ROPE_DIM;          // 64 rope channels
constexpr int kDn = MLA_QK_NOPE_DIM;       // 128
constexpr int kDv = MLA_V_DIM;             // 128
constexpr int kPage = MLA_PAGE_TOKENS;     // 64 tokens per page
constexpr int kLG = MLA_LATENT_GROUP;      // 16
constexpr int kKG = MLA_KPE_GROUP;         // 8
constexpr int kNLG = kDc / kLG;            // 32 latent groups
constexpr int kNKG = kDr / kKG;            // 8 k_pe groups
constexpr int kNOut = MLA_OUTLIER_CHANNELS;  // 25 protected channels (INT8_OUTLIER)
constexpr int kOutSlots = 32;              // their slots in the decode kernel (8 warps x 4)
constexpr int kOutFieldBytes = 1664;       // bf16 [25][32 tokens] = 1600 B, padded to 128
constexpr int kChunk = 32;                 // decode work unit: 32 tokens
constexpr int kMaxBatch = 4096;
constexpr int kMaxSplits = 65535;          // decode grid dimension y
constexpr int kMaxMergeParts = 4096;         // mla_lse_merge: most parts per call

// Byte layout of one page; see mla_page_layout in mla.h.  A page is two
// contiguous blocks of 32 tokens; offsets are within a block.
constexpr int kBlockTokens = 32;

struct PageLayout {
  int64_t page_bytes, block_bytes;
  int64_t codes_off, codes_row;
  int64_t scale_off, zero_off;
  int64_t kpe_off, kpe_row;
  int64_t kpe_scale_off;
  int64_t bound_off;
  int64_t outlier_off;
};

// The protected channels of an INT8_OUTLIER layer, passed to the kernels by
// value: slot k < 25 holds channel ch[k] (increasing), slots 25..31 hold -1;
// bit c of mask is set for a protected channel c.
struct OutlierSet {
  int16_t ch[kOutSlots];
  uint32_t mask[kDc / 32];
};

// Channels per scale group of a quantized latent format (16 unless one of
// the INT8 block-count variants).
__host__ __device__ constexpr int latent_group_size(int latent_fmt) {
  return latent_fmt == MLA_FMT_INT8_G8 ? 8
         : latent_fmt == MLA_FMT_INT8_G32 ? 32
         : latent_fmt == MLA_FMT_INT8_G64 ? 64
         : latent_fmt == MLA_FMT_INT8_TOKEN ? kDc : kLG;
}
__host__ __device__ constexpr bool is_int8_latent(int latent_fmt) {
  return latent_fmt == MLA_FMT_INT8_SYM || (latent_fmt >= MLA_FMT_INT8_G8 && latent_fmt <= MLA_FMT_INT8_OUTLIER);
}

__host__ __device__ inline bool compute_layout(int latent_fmt, int kpe_fmt, PageLayout* L) {
  int64_t row;
  switch (latent_fmt) {
    case MLA_FMT_BF16: row = 2 * kDc; break;
    case MLA_FMT_INT8_G8:
    case MLA_FMT_INT8_G32:
    case MLA_FMT_INT8_G64:
    case MLA_FMT_INT8_TOKEN:
      if (kpe_fmt != MLA_FMT_INT8_SYM) return false;
      row = kDc;
      break;
    case MLA_FMT_INT8_SYM: row = kDc; break;
    case MLA_FMT_INT8_OUTLIER:
      if (kpe_fmt != MLA_FMT_BF16 && kpe_fmt != MLA_FMT_INT8_SYM) return false;
      row = kDc;
      break;
    case MLA_FMT_INT4_ASYM:
    case MLA_FMT_INT4_SYM: row = kDc / 2; break;
    default: return false;
  }
  if (kpe_fmt != MLA_FMT_BF16 && kpe_fmt != MLA_FMT_INT8_SYM && kpe_fmt != MLA_FMT_INT4_SYM) return false;
  int64_t off = 0;
  L->codes_off = off;
  L->codes_row = row;
  off += kBlockTokens * row;
  L->scale_off = L->zero_off = -1;
  if (latent_fmt != MLA_FMT_BF16) {
    L->scale_off = off;
    off += (int64_t)(kDc / latent_group_size(latent_fmt)) * kBlockTokens * 4;
  }
  if (latent_fmt == MLA_FMT_INT4_ASYM) { L->zero_off = off; off += (int64_t)kNLG * kBlockTokens * 4; }
  L->outlier_off = -1;
  if (latent_fmt == MLA_FMT_INT8_OUTLIER) { L->outlier_off = off; off += kOutFieldBytes; }
  L->kpe_off = off;
  L->kpe_row = kpe_fmt == MLA_FMT_BF16 ? 2 * kDr : (kpe_fmt == MLA_FMT_INT8_SYM ? kDr : kDr / 2);
  off += kBlockTokens * L->kpe_row;
  L->kpe_scale_off = -1;
  if (kpe_fmt != MLA_FMT_BF16) { L->kpe_scale_off = off; off += (int64_t)kNKG * kBlockTokens * 4; }
  L->bound_off = -1;
  if (latent_fmt != MLA_FMT_BF16) { L->bound_off = off; off += kBlockTokens * 4; }
  L->block_bytes = off;
  L->page_bytes = 2 * off;
  return true;
}

// Stored position of 16-byte chunk c of a latent code row of token t (t =
// token index within its 32-token block): the low three bits of the chunk
// index are XORed with t, so that eight consecutive tokens' copies of one
// logical chunk fall in eight different shared-memory bank groups.
__host__ __device__ __forceinline__ int latent_chunk_pos(int c, int t) { return (c & ~7) | ((c ^ t) & 7); }
// Same for the k_pe row: 8 chunks (bf16), 4 chunks (int8) or 2 chunks
// (4-bit) per token.
__host__ __device__ __forceinline__ int kpe_chunk_pos(int c, int t, int kpe_fmt) {
  return kpe_fmt == MLA_FMT_BF16 ? (c ^ (t & 7)) : (kpe_fmt == MLA_FMT_INT8_SYM ? (c ^ ((t >> 1) & 3)) : (c ^ ((t >> 2) & 1)));
}
// INT4 chunk c holds latent groups A = 2c and B = 2c + 1 (16 channels each).
// Its 32-bit word j (j = 0..3) packs, from the least significant nibble:
// A[4j], A[4j+2], B[4j], B[4j+2], A[4j+1], A[4j+3], B[4j+1], B[4j+3].
// Returns (group_in_chunk * 16 + channel_in_group) of nibble k of word j.
__host__ __device__ __forceinline__ int int4_nibble_channel(int j, int k) {
  const int grp = (k >> 1) & 1;                       // nibbles 2,3,6,7 -> group B
  const int idx = 4 * j + ((k & 1) ? 2 : 0) + (k >> 2);
  return grp * 16 + idx;
}

// ---------------------------------------------------------------------------
// bf16 bit helpers (exact widening; rounding narrowing is RNE)
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf16f(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }

__device__ __forceinline__ void set_err(int32_t* dev_err, int bit) {
  if (dev_err) atomicOr(dev_err, bit);
}

// Split-K partial workspace:
//   [cum: B+1 int32 | span: 2B int32 | m: slots*H | l: slots*H | e2: slots*H | o: slots*H*512]
// span[2b], span[2b+1] = first and last split (CTA column) that worked on sequence b.
// e2: per partial and head, sum_t (p_t M_t)^2 over its tokens (p_t in the
// partial's scale, M_t a bound on |c_hat_t|): the weight of the split kernel's
// fp16 P V products, which the combine compares with the merged output.
struct Workspace {
  int32_t* cum;
  int32_t* span;
  float* m;
  float* l;
  float* e2;
  float* o;
};

__host__ __device__ inline int64_t align256(int64_t x) { return (x + 255) & ~(int64_t)255; }

__host__ __device__ inline int64_t workspace_bytes(int B, int H, int G) {
  int64_t slots = (int64_t)G + B;
  return align256((int64_t)(B + 1) * 4) + align256((int64_t)2 * B * 4) + 3 * align256(slots * H * 4) +
         slots * H * kDc * 4;
}

__host__ __device__ inline Workspace carve_workspace(void* base, int B, int H, int G) {
  char* p = (char*)base;
  int64_t slots = (int64_t)G + B;
  Workspace w;
  w.cum = (int32_t*)p;
  p += align256((int64_t)(B + 1) * 4);
  w.span = (int32_t*)p;
  p += align256((int64_t)2 * B * 4);
  w.m = (float*)p;
  p += align256(slots * H * 4);
  w.l = (float*)p;
  p += align256(slots * H * 4);
  w.e2 = (float*)p;
  p += align256(slots * H * 4);
  w.o = (float*)p;
  return w;
}

// Context partition: the total C chunks (32 tokens each) of all sequences are
// cut into Ge = min(G, C) contiguous, non-empty ranges, range x =
// [C*x/Ge, C*(x+1)/Ge); CTAs x >= Ge have no work.  Partials of sequence b
// computed by CTA x go to slot x + b, which is unique because two sequences
// share at most a boundary CTA.  The CTAs that hold a sequence's first and
// last chunk record themselves in span[], so the combine needs no division.
__host__ __device__ inline int64_t range_lo(int64_t C, int x, int G) { return C * x / G; }

// Programmatic dependent launch.  Every kernel of the library lets the next
// kernel in the stream begin launching as soon as all of its own blocks are
// running (pdl_launch_dependents), and waits for the previous kernel to
// complete and its memory to be visible (pdl_wait) before its first global
// memory access, in every block.  The exceptions are call inputs that no
// kernel of the library writes and that the API forbids any kernel in flight
// to write: the absorb and unabsorb kernels fetch their weight tile, and the
// decode kernel reads the sequence lengths, before the wait (not the
// prefill's per-row lengths, which a kernel writes just before).  Only the
// wait makes a previous kernel's stores visible, triggered early or not.
// Results are ordered as in plain stream order; the next grid's launch and
// block scheduling overlap this grid's tail.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Host side launch helpers (api.cu)
int device_sm_count();
// Checks a layer descriptor (pool, formats, protected channels) and fills its
// page layout and protected set (empty unless INT8_OUTLIER).
bool cache_check(const mla_cache_layer* c, PageLayout* L, OutlierSet* o);
uint64_t wait_limit_ns();                // set by mla_set_wait_limit_ns
mla_status launch_status();
mla_status cuda_status(cudaError_t e);   // records the error string on failure

// Launchers implemented in the kernel translation units.
mla_status launch_append(const mla_cache_layer* cache, const PageLayout& L, const OutlierSet& outl,
                         const uint16_t* c_new, const uint16_t* kpe_new, const int32_t* slot, int n,
                         int32_t* dev_err, cudaStream_t stream);
mla_status launch_select_outliers(const uint16_t* c_sample, int n, int32_t* out, cudaStream_t stream);
mla_status launch_q_absorb(const uint16_t* q_nope, const uint16_t* w_uk, float* q_lat, int B, int H,
                           cudaStream_t stream);
mla_status launch_out_unabsorb(const float* o_lat, const uint16_t* w_uv, float* o, int B, int H,
                               cudaStream_t stream);
mla_status launch_lse_merge(const float* o_parts, const float* lse_parts, int R, int B, int H, float* o_lat,
                            float* lse, cudaStream_t stream);
struct DecodeParams {
  const uint8_t* pool;
  PageLayout L;
  int latent_fmt, kpe_fmt;
  int num_pages;
  const float* q_lat;
  const uint16_t* q_pe;
  const int32_t* block_table;
  int max_pages;
  int bt_stride;          // block-table row stride: max_pages, or 0 when every row is row 0 (prefill)
  const int32_t* seq_lens;
  int lens_after_wait;    // 1: seq_lens is written by the kernel launched just before (the
                          // prefill's lengths): read it only after waiting on that kernel
  int B, H, G;
  float scale_log2;       // softmax_scale * log2(e)
  OutlierSet outl;        // INT8_OUTLIER: the protected channels
  uint64_t wait_ns;       // bound on every wait inside the decode kernel (wait_limit_ns())
  Workspace ws;
  float* o_lat;
  float* lse;
  const uint16_t* w_uv;   // with o: the output projection follows the merge (nullptr: not requested)
  float* o;
  int32_t* dev_err;
};
mla_status launch_decode(const DecodeParams& p, cudaStream_t stream);
int combine_grid(int latent_fmt, int B, int G);   // decode.cu
mla_status launch_decode_mma(const DecodeParams& p, cudaStream_t stream);   // decode kernel only

// Tensor-core prefill support (decode.cu): the key tiles of tokens 0 .. len - 1
// of block-table row 0 (fp16 hi / lo pairs, 128 tokens x 9 channel blocks x
// 2 x 16 KB per tile, swizzled) with the tokens' bounds mt[len rounded up to
// 128] and, if table is not null, x_hat of tokens 0 .. 255 in fp32
// ([token][576]); and the exact fp32 recomputation of the rows that need it
// (with skip_short, not the rows shorter than 256 positions).
mla_status launch_prefill_keys(const DecodeParams& p, int len, void* kws, float* mt, float* table,
                               cudaStream_t stream);
// The long rows the fixup hands to the split recomputation: *count items
// (b, h0, row mask, length), each recomputed over kSplitParts token ranges
// whose partial states (8 heads x (max, sum, 512 channels)) go to parts;
// done[i] counts the finished ranges of item i.  count and done start at 0.
constexpr int kSplitCap = 64;
constexpr int kSplitParts = 32;
struct SplitQueue {
  int32_t* count;
  int32_t* done;      // [kSplitCap]
  int32_t* items;     // [kSplitCap][4]
  float* parts;       // [kSplitCap][kSplitParts][8][2 + 512]
};
__host__ __device__ inline int64_t split_queue_bytes() {
  return align256((int64_t)(1 + kSplitCap) * 4) + align256((int64_t)kSplitCap * 16) +
         (int64_t)kSplitCap * kSplitParts * 8 * (2 + kDc) * 4;
}
__host__ __device__ inline SplitQueue carve_split_queue(void* base) {
  char* c = (char*)base;
  SplitQueue q;
  q.count = (int32_t*)c;
  q.done = q.count + 1;
  c += align256((int64_t)(1 + kSplitCap) * 4);
  q.items = (int32_t*)c;
  c += align256((int64_t)kSplitCap * 16);
  q.parts = (float*)c;
  return q;
}
mla_status launch_exact_fixup(const DecodeParams& p, const float* risk, const float* omax, const SplitQueue& q,
                              int skip_short, cudaStream_t stream);

// Tensor-core prefill (prefill_tc.cu).  A tile holds 128 rows (queries or
// keys) x 9 channel blocks x (hi, lo) x 16 KB.
constexpr int kTcTileBytes = 9 * 2 * 16384;
struct TcParams {
  const uint8_t* qws;     // [row tile][kb][hi, lo][16 KB]
  const uint8_t* kws;     // [key tile][kb][hi, lo][16 KB]
  const float* mt;        // [key tiles * 128] bound on |x_hat| per token
  int R;                  // query rows of the slice (token-major: r = i H + h)
  int H;
  int qpos0;              // position of the slice's first query token
  int n_rt;               // row tiles, ceil(R / 128)
  float scale_log2;
  int risk;               // record the precision check (quantized latents)
  float* o_lat;           // [R][512]
  float* lse;             // [R] or nullptr
  float* risk_out;        // [R]: sqrt(sum_t (w_t M_t)^2)
  float* omax;            // [R][2]: |o_lat|_inf of each 256-channel half
  int32_t* dev_err;
  uint64_t wait_ns;
};
mla_status launch_q_split(const float* q_lat, const uint16_t* q_pe, int R, int n_rt, uint8_t* qws,
                          cudaStream_t stream);
mla_status launch_prefill_tc(const TcParams& p, cudaStream_t stream);
// The exact fp32 attention of query tokens 0 .. n_short - 1 of a slice (their
// positions qpos0 + i all below 255), every head, from the fp32 x_hat table.
mla_status launch_short_rows(const float* table, const float* q_lat, const uint16_t* q_pe, int H, int n_short,
                             int qpos0, float scale_log2, float* o_lat, float* lse, cudaStream_t stream);

}  // namespace mla
