// Tensor-core split-K decode kernel for mla_decode_absorbed (sm_103a).
//
// Computes, for a tile of 16 heads and the 32-token chunks of the CTA's share
// of the batch (same partition and partial-slot scheme as decode.cu), the
// online-softmax partials of
//   s[h,t] = (q_lat[h] . c_hat[t] + q_pe[h] . kpe_hat[t]) * softmax_scale
//   o[h]   = sum_t exp(s - m) c_hat[t]
// (English report "Absorbed MLA Cache Optimization on DeepSeek-V2-Lite —
// Technical Report" §2.1: attention straight from the cached latent; juejin
// tutorial "步骤2" for the absorbed up-projections).
//
// Structure (one CTA per SM, 12 warps, warp-specialized):
//  * Compute warps 0..7: warp w owns latent groups 4w..4w+3 (64 channels)
//    and k_pe group w.  Each code byte is read from shared memory once
//    (ldmatrix) and turned into exact fp16 integers; the same registers serve
//    QK^T and, after a movmatrix transpose, PV.
//  * QK^T per 16-channel group: mma.m16n8k16 (M = 16 heads, N = 8 tokens,
//    K = the group's 16 channels) of q_lat split into fp16 hi + lo against
//    the exact integer codes (INT4: code - zero, formed exactly in fp16),
//    then one fp32 FMA per element applies the group's per-token scale.
//    This keeps every product exact, which the 2e-3 bound needs: scores here
//    have a spread of ~10, so a rounding of the latent or the query to 11
//    bits would already cost ~1e-3.
//  * Softmax warpgroup (warps 8..11, 128 threads, 8 per head row): sums the
//    8 compute warps' partial scores of a chunk through shared memory, runs
//    the online softmax (max / sum by shuffles over the row's 8 threads) and
//    publishes P in fp16 (bf16 hi + lo for a bf16 latent) with the rescale
//    factor.  Its first thread is the loader: it streams 32-token blocks
//    (one contiguous cp.async.bulk each, mbarrier-signalled) into a ring of
//    shared-memory stages and refills a stage once every compute warp has
//    handed in the chunk it held.
//  * PV: o[16 heads][the warp's 64 channels] += (P scaled per token by the
//    group's scale) x (the same exact codes, transposed with movmatrix),
//    one chunk behind QK^T, so a compute warp's QK^T of chunk i overlaps
//    the softmax of chunk i - 1.  P * s is one fp16 product of fp16 P and
//    fp16 s; over long contexts its roundings average out (~3e-4 of the
//    output).  Sequences shorter than 256 tokens, where they need not, are
//    recomputed exactly by the combine kernel (decode.cu).
//  * bf16 latent: q_lat is split into bf16 hi + lo against the exact bf16
//    values, one accumulator over all groups, P split into bf16 hi + lo.
#include <cuda_fp16.h>
#include <math.h>

#include "mla_internal.cuh"

namespace mla {

namespace {

constexpr int kCW = 8;                         // compute warps
constexpr int kThreads = kCW * 32;
constexpr int kHT = 16;                        // heads per CTA
constexpr int kPStride = 40;                   // row stride (16-bit elements) of the P tile: 80 B, conflict-free ldmatrix
constexpr int kXStride = 20;                   // row stride (float2) of a warp's partial-score tile: 160 B, conflict-free

template <int LF, int KF>
struct Fmt {
  static constexpr bool kLatBf16 = LF == MLA_FMT_BF16;
  static constexpr bool kLatInt4 = LF == MLA_FMT_INT4_ASYM || LF == MLA_FMT_INT4_SYM;
  static constexpr bool kLatSym4 = LF == MLA_FMT_INT4_SYM;       // zero-point fixed at 8 (nibble = code + 8)
  static constexpr bool kLatOut = LF == MLA_FMT_INT8_OUTLIER;    // INT8 plus 25 protected bf16 channels
  static constexpr bool kKpeBf16 = KF == MLA_FMT_BF16;
  static constexpr bool kKpeInt4 = KF == MLA_FMT_INT4_SYM;
  static constexpr int kRow = kLatBf16 ? 1024 : (is_int8_latent(LF) ? 512 : 256);
  static constexpr int kKRow = kKpeBf16 ? 128 : (kKpeInt4 ? 32 : 64);
  static constexpr int kGS = latent_group_size(LF);             // channels per scale group
  static constexpr bool kLatG8 = kGS == 8;                       // two scale groups per 16-channel MMA step
  static constexpr int kSPG = kLatG8 ? 1 : kGS / 16;             // 16-channel MMA steps per scale group
  // operand layout: standard m16n8k16 fragments (thread j holds channels 2j,
  // 2j+1 and 8+2j, 8+2j+1) for bf16 and 8-channel groups, else permuted
  // (thread j holds channels 4j .. 4j+3)
  static constexpr bool kStdLayout = kLatBf16 || kLatG8;
  // quantized latents: the softmax warps also accumulate, per head row, the
  // weight of the fp16 P V products (sum of (p_t M_t)^2, M_t the token's
  // stored bound on |c_hat|), from which the combine decides whether the row
  // needs the exact fp32 recomputation
  static constexpr bool kRisk = !kLatBf16;
  static constexpr int kScaleOff = kBlockTokens * kRow;
  static constexpr int kZeroOff = kScaleOff + (kLatBf16 ? 0 : (kDc / kGS) * kBlockTokens * 4);
  static constexpr int kOutOff = kZeroOff + (LF == MLA_FMT_INT4_ASYM ? kNLG * kBlockTokens * 4 : 0);
  static constexpr int kKpeOff = kOutOff + (kLatOut ? kOutFieldBytes : 0);
  static constexpr int kKScaleOff = kKpeOff + kBlockTokens * kKRow;
  static constexpr int kBoundOff = kKScaleOff + (kKpeBf16 ? 0 : kNKG * kBlockTokens * 4);
  static constexpr int kBlock = kBoundOff + (kLatBf16 ? 0 : kBlockTokens * 4);
  static constexpr int kStages = kBlock <= 24 * 1024 ? 6 : (kBlock <= 40 * 1024 ? 4 : 3);
  static constexpr int kXPartBytes = 2 * kCW * kHT * kXStride * 8;   // partial scores [buf][warp][row][pair]
  // P tiles per buffer: fp16 P (bf16 hi for a bf16 latent), bf16 lo; with
  // protected channels also bf16 hi and lo of P for their P V products
  static constexpr int kPTiles = kLatOut ? 4 : 2;
  static constexpr int kPBytes = 2 * kPTiles * kHT * kPStride * 2;    // [buf][tile][16][kPStride]
  static constexpr int kFixed = kStages * kBlock + kXPartBytes + kPBytes + (2 * kHT + kCW) * 4 + kStages * 8 + kStages * 4;
  // shared-memory offsets that vector accesses rely on: stages and the P
  // tiles (16 B), the bounds array after alpha / amax (float4 reads)
  static_assert(kBlock % 128 == 0 && kXPartBytes % 16 == 0 && kPBytes % 16 == 0, "stage / tile alignment");
  static_assert((kStages * kBlock + kXPartBytes + kPBytes + (2 * kHT + kCW) * 4) % 16 == 0, "bounds alignment");
};

// ---------------------------------------------------------------------------
// PTX helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.shared::cta.b64 st, [%0];\n}\n" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}\n" ::"r"(bar),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait on an mbarrier phase.  Returns false once limit_ns have
// passed without completion (checked every 256 polls, or at every poll when
// the limit is 0, which also polls without suspending); the caller records
// MLA_DEVERR_TIMEOUT and gives up its work.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  uint32_t done = 0;
  uint64_t t0 = 0;
  for (uint32_t it = 0;; ++it) {
    if (limit_ns == 0) {     // no wait at all: the non-blocking probe (try_wait may suspend until completion)
      asm volatile(
          "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
          : "=r"(done)
          : "r"(bar), "r"(parity)
          : "memory");
    } else {
      asm volatile(
          "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
          : "=r"(done)
          : "r"(bar), "r"(parity)
          : "memory");
    }
    if (done) return true;
    if (it == 0) t0 = global_ns();
    else if (((it & 255) == 0 || limit_ns == 0) && global_ns() - t0 > limit_ns) return false;
  }
}

// mbar_wait by every lane of a warp, with a warp-uniform answer: a lane
// that gave up makes the whole warp give up, so that the warp leaves its
// loops together (its mma.sync, ldmatrix and shuffles need all lanes).
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, limit_ns));
}

// Limit of the loader's final wait for its own bulk copies: those land within
// microseconds unless the memory system itself is stuck.
constexpr uint64_t kDrainLimitNs = 10000000000ull;

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// Register-only instructions are not volatile so that the compiler may
// interleave independent MMA chains; shared-memory reads (ldmatrix) stay
// volatile to keep them after the barrier waits that guard them.
__device__ __forceinline__ uint32_t movt(uint32_t a) {
  uint32_t d;
  asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(d) : "r"(a));
  return d;
}

// d = a * b + c, fp16 inputs, fp32 accumulate (c and d may alias)
__device__ __forceinline__ void mma_f16(float* d, const uint32_t* a, uint32_t b0, uint32_t b1, const float* c) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%11,%12,%13};\n"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]),
        "f"(c[3]));
}

// d = a * b + c for m16n8k8 (two A registers, one B register)
__device__ __forceinline__ void mma_f16_k8(float* d, uint32_t a0, uint32_t a1, uint32_t b0, const float* c) {
  asm("mma.sync.aligned.m16n8k8.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5}, {%6}, {%7,%8,%9,%10};\n"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(b0), "f"(c[0]), "f"(c[1]), "f"(c[2]), "f"(c[3]));
}

// d = a * b + c for m16n8k8 bf16
__device__ __forceinline__ void mma_bf16_k8(float* d, uint32_t a0, uint32_t a1, uint32_t b0, const float* c) {
  asm("mma.sync.aligned.m16n8k8.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5}, {%6}, {%7,%8,%9,%10};\n"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(b0), "f"(c[0]), "f"(c[1]), "f"(c[2]), "f"(c[3]));
}

__device__ __forceinline__ void mma_bf16(float* d, const uint32_t* a, uint32_t b0, uint32_t b1, const float* c) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%11,%12,%13};\n"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]),
        "f"(c[3]));
}

// acc[0..1] += d[0..1] * s and acc[2..3] += d[2..3] * s (C-fragment rows r and
// r + 8 of one n-tile against its two tokens' scales) as two packed f32x2 FMAs
__device__ __forceinline__ void scale_acc(float* acc, const float* d, float2 s) {
  const float2 a = __ffma2_rn(make_float2(d[0], d[1]), s, make_float2(acc[0], acc[1]));
  const float2 b = __ffma2_rn(make_float2(d[2], d[3]), s, make_float2(acc[2], acc[3]));
  acc[0] = a.x;
  acc[1] = a.y;
  acc[2] = b.x;
  acc[3] = b.y;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 bits_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

__device__ __forceinline__ uint32_t pack_f16(float a, float b) { return h2_bits(__floats2half2_rn(a, b)); }

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;\n" : "=r"(r) : "f"(b), "f"(a));
  return r;
}

__device__ __forceinline__ float bf16_lo_f(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi_f(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

// fp32 pair -> (hi, lo) split in fp16 (hi = rn(x), lo = rn(x - hi)); x already scaled into range
__device__ __forceinline__ void split_f16(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(a, b);
  const float2 hf = __half22float2(h);
  hi = h2_bits(h);
  lo = pack_f16(a - hf.x, b - hf.y);
}

__device__ __forceinline__ void split_bf16(float a, float b, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf16(a, b);
  lo = pack_bf16(a - bf16_lo_f(hi), b - bf16_hi_f(hi));
}

// 4 int8 codes (one 32-bit word) -> two f16x2 holding the codes exactly:
// the bytes become 1024 + (code + 128) by bit placement, then 1152 is
// subtracted in fp16 (exact: integers below 2048)
__device__ __forceinline__ void i8x4_to_f16(uint32_t w, uint32_t& r0, uint32_t& r1) {
  const __half2 bias = __floats2half2_rn(1152.f, 1152.f);
  const uint32_t x = w ^ 0x80808080u;
  r0 = h2_bits(__hsub2(bits_h2(__byte_perm(x, 0x64646464u, 0x4140)), bias));
  r1 = h2_bits(__hsub2(bits_h2(__byte_perm(x, 0x64646464u, 0x4342)), bias));
}

// one int4 word (layout in mla_internal.cuh) -> group A regs (a0, a1) and
// group B regs (b0, b1), each f16x2 holding code - zero exactly: the nibbles
// become 1024 + code (or 1024 + 16 code) by bit placement; zo = (1024 + zA,
// 1024 + zB) and zc = (-64 - zA, -64 - zB) (f16x2, exact for |z| < 960), and
// one exact fp16 subtract or fma with the broadcast half removes both offsets
__device__ __forceinline__ void i4x8_to_f16(uint32_t w, __half2 zo, __half2 zc, uint32_t& a0, uint32_t& a1,
                                            uint32_t& b0, uint32_t& b1) {
  const __half2 k16 = __floats2half2_rn(0.0625f, 0.0625f);
  a0 = h2_bits(__hsub2(bits_h2((w & 0x000F000Fu) | 0x64006400u), __low2half2(zo)));
  a1 = h2_bits(__hfma2(bits_h2((w & 0x00F000F0u) | 0x64006400u), k16, __low2half2(zc)));
  const uint32_t v = w >> 8;
  b0 = h2_bits(__hsub2(bits_h2((v & 0x000F000Fu) | 0x64006400u), __high2half2(zo)));
  b1 = h2_bits(__hfma2(bits_h2((v & 0x00F000F0u) | 0x64006400u), k16, __high2half2(zc)));
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ int checked_len(const DecodeParams& p, int b, bool report) {
  int len = p.seq_lens[b];
  if (len < 0 || (int64_t)len > (int64_t)p.max_pages * kPage) {
    if (report) set_err(p.dev_err, MLA_DEVERR_SEQLEN);
    len = 0;
  }
  return len;
}

__device__ __forceinline__ int seq_of_chunk(const int32_t* cum, int B, int c) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cum[mid] <= c) lo = mid; else hi = mid - 1;
  }
  while (lo + 1 < B && cum[lo + 1] <= c) ++lo;
  return lo;
}

// ---------------------------------------------------------------------------
// Per-warp query state for one (sequence, head tile)
// ---------------------------------------------------------------------------
struct QueryRaw {            // this thread's fp32 query values, before range scaling
  float4 x[4][2];            // q_lat: [group][row r / r+8], the 4 channels this thread feeds
  float kx[2][4];            // q_pe: [row][4 channels]
  float ox[2][2];            // protected channels (INT8_OUTLIER): [row][slot 4w + 2j + e]
};

struct ChunkRegs {           // one chunk's B operands, kept from QK^T for PV
  uint32_t bq[4][4][2];      // exact codes (or code - zero): [group][ntile][reg]
  uint32_t s2h[4][4];        // fp16 scale pairs of the C-fragment tokens: [group][ntile]
  uint32_t ov[2][2];         // protected values (bf16 token pairs of slot 4w + r): [k step][reg]
};

struct Query {
  uint32_t hi[4][4], lo[4][4];   // A fragments of q_lat (hi + lo split) for the warp's 4 groups
  uint32_t ka[4];                // A fragment of q_pe for the warp's k_pe group / chunk
  uint32_t oh[2], ol[2];         // m16n8k8 A fragments (bf16 hi + lo) of the warp's protected channels
};

// Loads this thread's share of q_lat / q_pe and returns its largest magnitude.
template <int LF, int KF>
__device__ __forceinline__ float load_query_raw(const DecodeParams& p, int b, int h0, int w, int lane, QueryRaw& q) {
  using F = Fmt<LF, KF>;
  const int r = lane >> 2, j = lane & 3;
  const float* ql0 = p.q_lat + ((size_t)b * p.H + h0 + r) * kDc;
  const float* ql1 = ql0 + 8 * kDc;
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    const int gg = 4 * w + g;
    if (F::kStdLayout) {
      // standard layout: channels 2j, 2j+1 and 8+2j, 8+2j+1 of the 16 channels
      const float2 a0 = *reinterpret_cast<const float2*>(ql0 + 16 * gg + 2 * j);
      const float2 a1 = *reinterpret_cast<const float2*>(ql0 + 16 * gg + 8 + 2 * j);
      const float2 b0 = *reinterpret_cast<const float2*>(ql1 + 16 * gg + 2 * j);
      const float2 b1 = *reinterpret_cast<const float2*>(ql1 + 16 * gg + 8 + 2 * j);
      q.x[g][0] = make_float4(a0.x, a0.y, a1.x, a1.y);
      q.x[g][1] = make_float4(b0.x, b0.y, b1.x, b1.y);
    } else {
      // permuted layout: thread j feeds channels 4j .. 4j+3 of the group
      q.x[g][0] = *reinterpret_cast<const float4*>(ql0 + 16 * gg + 4 * j);
      q.x[g][1] = *reinterpret_cast<const float4*>(ql1 + 16 * gg + 4 * j);
    }
  }
  const uint16_t* qp0 = p.q_pe + ((size_t)b * p.H + h0 + r) * kDr;
  const uint16_t* qp1 = qp0 + 8 * kDr;
  if (F::kKpeBf16) {
    // warp w: k16 chunk w % 4 (channels 16(w%4) .. +15), standard layout
    const int c0 = 16 * (w & 3);
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const uint16_t* qp = rr ? qp1 : qp0;
      q.kx[rr][0] = bf16f(qp[c0 + 2 * j]);
      q.kx[rr][1] = bf16f(qp[c0 + 2 * j + 1]);
      q.kx[rr][2] = bf16f(qp[c0 + 8 + 2 * j]);
      q.kx[rr][3] = bf16f(qp[c0 + 8 + 2 * j + 1]);
    }
  } else {
    // warp w: k_pe group w inside 16-channel chunk w/2; thread j feeds channels
    // 4j..4j+3 of the chunk, which belong to the group only when j/2 == w%2
    const bool act = (j >> 1) == (w & 1);
    const int c0 = 16 * (w >> 1) + 4 * j;
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const uint16_t* qp = rr ? qp1 : qp0;
#pragma unroll
      for (int e = 0; e < 4; ++e) q.kx[rr][e] = act ? bf16f(qp[c0 + e]) : 0.f;
    }
  }
  float amax = 0.f;
  if (F::kLatOut) {
    // the warp's protected slots 4w .. 4w+3 (k = slot - 4w of an m16n8k8 step;
    // threads j = 0, 1 feed k = 2j, 2j + 1, threads 2, 3 the zero half)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int sl = 4 * w + 2 * j + e;
      const int ch = (j < 2 && sl < kNOut) ? p.outl.ch[sl] : -1;
      q.ox[0][e] = ch >= 0 ? ql0[ch] : 0.f;
      q.ox[1][e] = ch >= 0 ? ql1[ch] : 0.f;
      amax = fmaxf(amax, fmaxf(fabsf(q.ox[0][e]), fabsf(q.ox[1][e])));
    }
  }
#pragma unroll
  for (int g = 0; g < 4; ++g)
#pragma unroll
    for (int rr = 0; rr < 2; ++rr)
      amax = fmaxf(amax, fmaxf(fmaxf(fabsf(q.x[g][rr].x), fabsf(q.x[g][rr].y)),
                               fmaxf(fabsf(q.x[g][rr].z), fabsf(q.x[g][rr].w))));
#pragma unroll
  for (int rr = 0; rr < 2; ++rr)
#pragma unroll
    for (int e = 0; e < 4; ++e) amax = fmaxf(amax, fabsf(q.kx[rr][e]));
  return amax;
}

// Scales by 2^e (exact) and splits into the MMA A fragments.
template <int LF, int KF>
__device__ __forceinline__ void finish_query(const QueryRaw& raw, float up, Query& q) {
  using F = Fmt<LF, KF>;
#pragma unroll
  for (int g = 0; g < 4; ++g)
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const float4 v = raw.x[g][rr];
      uint32_t h01, l01, h23, l23;
      if (F::kLatBf16) {
        split_bf16(v.x, v.y, h01, l01);
        split_bf16(v.z, v.w, h23, l23);
      } else {
        split_f16(v.x * up, v.y * up, h01, l01);
        split_f16(v.z * up, v.w * up, h23, l23);
      }
      // A fragment: reg0 = row r (k 0..7 half), reg1 = row r+8, reg2 = row r (k 8..15), reg3 = row r+8
      q.hi[g][rr] = h01;
      q.hi[g][rr + 2] = h23;
      q.lo[g][rr] = l01;
      q.lo[g][rr + 2] = l23;
    }
  if (F::kLatOut) {
    split_bf16(raw.ox[0][0] * up, raw.ox[0][1] * up, q.oh[0], q.ol[0]);
    split_bf16(raw.ox[1][0] * up, raw.ox[1][1] * up, q.oh[1], q.ol[1]);
  }
  if (F::kKpeBf16) {
    q.ka[0] = pack_bf16(raw.kx[0][0] * up, raw.kx[0][1] * up);
    q.ka[1] = pack_bf16(raw.kx[1][0] * up, raw.kx[1][1] * up);
    q.ka[2] = pack_bf16(raw.kx[0][2] * up, raw.kx[0][3] * up);
    q.ka[3] = pack_bf16(raw.kx[1][2] * up, raw.kx[1][3] * up);
  } else {
    q.ka[0] = pack_f16(raw.kx[0][0] * up, raw.kx[0][1] * up);
    q.ka[1] = pack_f16(raw.kx[1][0] * up, raw.kx[1][1] * up);
    q.ka[2] = pack_f16(raw.kx[0][2] * up, raw.kx[0][3] * up);
    q.ka[3] = pack_f16(raw.kx[1][2] * up, raw.kx[1][3] * up);
  }
}

// Step A of one chunk for warp w (latent groups 4w .. 4w+3): B operands
// (exact codes, or code - zero) into bq, the fp16 PV scale pairs into s2h,
// and the warp's partial scores (QK^T over its channels plus its k_pe part)
// into acc [ntile][C fragment].  st: the chunk's block in shared memory;
// nv: its valid tokens.
template <int LF, int KF>
__device__ __forceinline__ void qk_chunk(const uint8_t* st, int nv, int w, int lane, const Query& q,
                                         uint32_t (&bq)[4][4][2], uint32_t (&s2h)[4][4], uint32_t (&ov)[2][2],
                                         float (&acc)[4][4]) {
  using F = Fmt<LF, KF>;
  const int r = lane >> 2, j = lane & 3;
  // Tokens past nv (nv may be 0: no data, everything masked) hold stale or
  // unwritten bytes.  Their scores need no mask
  // here (the softmax replaces them with -inf by selection), but everything
  // PV multiplies with their zero P must be finite: their scales and
  // zero-points are masked bitwise.  mc[n]: the C-fragment token pair
  // (8n + 2j, 8n + 2j + 1), as f16x2 lanes; mb[n]: the B-operand token 8n + r.
  // The masks are applied to full chunks too: one branch-free instance of
  // this step measured faster (32K INT4 call 0.282 against 0.295 ms) than
  // either a run-time test or a separate instance for full chunks.
  uint32_t mc[4], mb[4];
#pragma unroll
  for (int n = 0; n < 4; ++n) {
    mc[n] = (8 * n + 2 * j < nv ? 0x0000FFFFu : 0u) | (8 * n + 2 * j + 1 < nv ? 0xFFFF0000u : 0u);
    mb[n] = 8 * n + r < nv ? ~0u : 0u;
  }
  const uint32_t st_a = smem_u32(st);
  const float* sc = reinterpret_cast<const float*>(st + F::kScaleOff);
  // ---- step A: B operands (exact codes, or code - zero) and QK^T of chunk i
  if (F::kLatBf16) {
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const int ch = 2 * (4 * w + g);
      uint32_t t0, t1, t2, t3;
      ldsm_x4(st_a + lane * F::kRow + latent_chunk_pos(ch, lane) * 16, t0, t1, t2, t3);
      bq[g][0][0] = t0; bq[g][1][0] = t1; bq[g][2][0] = t2; bq[g][3][0] = t3;
      ldsm_x4(st_a + lane * F::kRow + latent_chunk_pos(ch + 1, lane) * 16, t0, t1, t2, t3);
      bq[g][0][1] = t0; bq[g][1][1] = t1; bq[g][2][1] = t2; bq[g][3][1] = t3;
    }
    // PV reads these values: zero the tokens past the end
#pragma unroll
    for (int n = 0; n < 4; ++n)
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        bq[g][n][0] &= mb[n];
        bq[g][n][1] &= mb[n];
      }
  } else if (F::kLatInt4) {
    const float* zp = reinterpret_cast<const float*>(st + F::kZeroOff);
    const __half2 k1024 = __floats2half2_rn(1024.f, 1024.f), km64 = __floats2half2_rn(-64.f, -64.f);
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      uint32_t t[4];
      ldsm_x4(st_a + lane * F::kRow + latent_chunk_pos(2 * w + cc, lane) * 16, t[0], t[1], t[2], t[3]);
#pragma unroll
      for (int n = 0; n < 4; ++n) {
        __half2 zz;
        if (F::kLatSym4) {
          zz = __floats2half2_rn(8.f, 8.f);                         // nibble = code + 8
        } else {
          // zero-points of this thread's B token (8n + r) for groups A and B of the chunk
          const float za = zp[(4 * w + 2 * cc) * kBlockTokens + 8 * n + r];
          const float zb = zp[(4 * w + 2 * cc + 1) * kBlockTokens + 8 * n + r];
          zz = bits_h2(h2_bits(__floats2half2_rn(za, zb)) & mb[n]);   // exact (integer zero-points)
        }
        i4x8_to_f16(t[n], __hadd2(zz, k1024), __hsub2(km64, zz), bq[2 * cc][n][0], bq[2 * cc][n][1],
                    bq[2 * cc + 1][n][0], bq[2 * cc + 1][n][1]);
      }
    }
  } else {
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      uint32_t t[4];
      ldsm_x4(st_a + lane * F::kRow + latent_chunk_pos(4 * w + g, lane) * 16, t[0], t[1], t[2], t[3]);
#pragma unroll
      for (int n = 0; n < 4; ++n) i8x4_to_f16(t[n], bq[g][n][0], bq[g][n][1]);
    }
  }
  // bf16 k_pe: warp w takes 16-channel chunk w % 4 and n-tiles 2 (w / 4),
  // 2 (w / 4) + 1 (bk[0..1]); quantized k_pe: group w, all four n-tiles
  uint32_t bk[4][2];
  if (F::kKpeBf16) {
    const int nh = w >> 2, kc = w & 3;
    uint32_t t[4], u[4];
    ldsm_x4(st_a + F::kKpeOff + lane * F::kKRow + kpe_chunk_pos(2 * kc, lane, KF) * 16, t[0], t[1], t[2], t[3]);
    ldsm_x4(st_a + F::kKpeOff + lane * F::kKRow + kpe_chunk_pos(2 * kc + 1, lane, KF) * 16, u[0], u[1], u[2], u[3]);
#pragma unroll
    for (int n = 0; n < 2; ++n) {
      bk[n][0] = nh ? t[n + 2] : t[n];
      bk[n][1] = nh ? u[n + 2] : u[n];
    }
  } else if (F::kKpeInt4) {
    // warp w: k_pe group w = channels 8w .. 8w+7, in 32-channel chunk w / 4,
    // 16-channel half (w / 2) % 2; the MMA takes the half's 16 channels
    // (its A fragment is zero outside the group, as for INT8 k_pe)
    uint32_t t[4];
    ldsm_x4(st_a + F::kKpeOff + lane * F::kKRow + kpe_chunk_pos(w >> 2, lane, KF) * 16, t[0], t[1], t[2], t[3]);
    const __half2 zo = __floats2half2_rn(1032.f, 1032.f), zc = __floats2half2_rn(-72.f, -72.f);
    const bool hb = (w >> 1) & 1;
#pragma unroll
    for (int n = 0; n < 4; ++n) {
      uint32_t a0, a1, b0, b1;
      i4x8_to_f16(t[n], zo, zc, a0, a1, b0, b1);
      bk[n][0] = hb ? b0 : a0;
      bk[n][1] = hb ? b1 : a1;
    }
  } else {
    uint32_t t[4];
    ldsm_x4(st_a + F::kKpeOff + lane * F::kKRow + kpe_chunk_pos(w >> 1, lane, KF) * 16, t[0], t[1], t[2], t[3]);
#pragma unroll
    for (int n = 0; n < 4; ++n) i8x4_to_f16(t[n], bk[n][0], bk[n][1]);
  }

#pragma unroll
  for (int n = 0; n < 4; ++n)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[n][e] = 0.f;
  if (F::kLatBf16) {
#pragma unroll
    for (int g = 0; g < 4; ++g) {
#pragma unroll
      for (int n = 0; n < 4; ++n) mma_bf16(acc[n], q.hi[g], bq[g][n][0], bq[g][n][1], acc[n]);
#pragma unroll
      for (int n = 0; n < 4; ++n) mma_bf16(acc[n], q.lo[g], bq[g][n][0], bq[g][n][1], acc[n]);
    }
  } else if (F::kLatG8) {
    // two 8-channel scale groups per 16-channel step: one m16n8k8 MMA per
    // group (standard layout: A registers 0 / 1 and B register 0 carry
    // channels 0-7 of the step, A registers 2 / 3 and B register 1
    // channels 8-15) and one scale FMA per element; then each operand
    // register is scaled by its own group's scale for PV (fp16, one
    // rounding, as the P-side scaling of the other formats)
    const float zero4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int g = 0; g < 4; ++g) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int si = 2 * (4 * w + g) + hh;
        float d[4][4];
#pragma unroll
        for (int n = 0; n < 4; ++n) mma_f16_k8(d[n], q.hi[g][2 * hh], q.hi[g][2 * hh + 1], bq[g][n][hh], zero4);
#pragma unroll
        for (int n = 0; n < 4; ++n) mma_f16_k8(d[n], q.lo[g][2 * hh], q.lo[g][2 * hh + 1], bq[g][n][hh], d[n]);
#pragma unroll
        for (int n = 0; n < 4; ++n) {
          const float2 s2 = *reinterpret_cast<const float2*>(sc + si * kBlockTokens + 8 * n + 2 * j);
          const float sv = sc[si * kBlockTokens + 8 * n + r];
          scale_acc(acc[n], d[n], s2);
          bq[g][n][hh] = h2_bits(__hmul2(bits_h2(bq[g][n][hh]), __float2half2_rn(sv))) & mb[n];
        }
      }
    }
  } else {
    // the MMA steps of one scale group accumulate together (exact codes,
    // fp32 accumulator), then one FMA per element applies the scale
    const float zero4[4] = {0.f, 0.f, 0.f, 0.f};
    float d[4][4];
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const bool first = g % F::kSPG == 0, last = (g + 1) % F::kSPG == 0 || g == 3;
#pragma unroll
      for (int n = 0; n < 4; ++n) mma_f16(d[n], q.hi[g], bq[g][n][0], bq[g][n][1], first ? zero4 : d[n]);
#pragma unroll
      for (int n = 0; n < 4; ++n) mma_f16(d[n], q.lo[g], bq[g][n][0], bq[g][n][1], d[n]);
      if (last) {
        const int si = (4 * w + g) / F::kSPG;
#pragma unroll
        for (int n = 0; n < 4; ++n) {
          const float2 s2 = *reinterpret_cast<const float2*>(sc + si * kBlockTokens + 8 * n + 2 * j);
          scale_acc(acc[n], d[n], s2);
          const uint32_t sh = pack_f16(s2.x, s2.y) & mc[n];
#pragma unroll
          for (int g2 = 0; g2 < 4; ++g2)
            if (g2 <= g && g2 > g - F::kSPG) s2h[g2][n] = sh;
        }
      }
    }
  }
  if (F::kKpeBf16) {
    if (w >> 2) {
      mma_bf16(acc[2], q.ka, bk[0][0], bk[0][1], acc[2]);
      mma_bf16(acc[3], q.ka, bk[1][0], bk[1][1], acc[3]);
    } else {
      mma_bf16(acc[0], q.ka, bk[0][0], bk[0][1], acc[0]);
      mma_bf16(acc[1], q.ka, bk[1][0], bk[1][1], acc[1]);
    }
  } else {
    const float* ks = reinterpret_cast<const float*>(st + F::kKScaleOff);
    const float zero4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int n = 0; n < 4; ++n) {
      const float2 s2 = *reinterpret_cast<const float2*>(ks + w * kBlockTokens + 8 * n + 2 * j);
      float d[4];
      mma_f16(d, q.ka, bk[n][0], bk[n][1], zero4);
      scale_acc(acc[n], d, s2);
    }
  }
  if (F::kLatOut && 4 * w < kNOut) {
    // protected channels, slots 4w .. 4w+3 (rows [slot][32 tokens] of bf16):
    // QK^T adds q (bf16 hi + lo) x the stored values, one m16n8k8 step with
    // k = slot (B: slots 2j, 2j+1 of token 8n + r; zero for j >= 2 and for
    // slots past the 25th, whose rows do not exist); the P V operand (token
    // pairs of slot 4w + r, zero past the chunk's end) is kept for step C
    const uint16_t* ovs = reinterpret_cast<const uint16_t*>(st + F::kOutOff);
    const int s0 = 4 * w + 2 * j;
#pragma unroll
    for (int n = 0; n < 4; ++n) {
      uint32_t b = 0u;
      if (j < 2) {
        const uint32_t v0 = s0 < kNOut ? ovs[s0 * kBlockTokens + 8 * n + r] : 0u;
        const uint32_t v1 = s0 + 1 < kNOut ? ovs[(s0 + 1) * kBlockTokens + 8 * n + r] : 0u;
        b = v0 | (v1 << 16);
      }
      mma_bf16_k8(acc[n], q.oh[0], q.oh[1], b, acc[n]);
      mma_bf16_k8(acc[n], q.ol[0], q.ol[1], b, acc[n]);
    }
    const int sl = 4 * w + r;
#pragma unroll
    for (int ks2 = 0; ks2 < 2; ++ks2)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int tok = 16 * ks2 + 8 * e + 2 * j;
        uint32_t v = (r < 4 && sl < kNOut) ? *reinterpret_cast<const uint32_t*>(ovs + sl * kBlockTokens + tok) : 0u;
        v &= (tok < nv ? 0x0000FFFFu : 0u) | (tok + 1 < nv ? 0xFFFF0000u : 0u);
        ov[ks2][e] = v;
      }
  }
}

// Step C of one chunk for warp w: rescale o by the chunk's alpha and add
// P V with the operands bqv / scales s2v kept from its step A (and, with
// protected channels, their P V into oo with the operands ovv).  alpha_s:
// [2][16]; ptab: the P tiles [2 buf][kPTiles][16][kPStride].
template <int LF, int KF>
__device__ __forceinline__ void pv_chunk(float (&o)[4][2][4], float (&oo)[4], const float* alpha_s,
                                         const uint16_t* ptab, int buf, const uint32_t (&bqv)[4][4][2],
                                         const uint32_t (&s2v)[4][4], const uint32_t (&ovv)[2][2], int w, int lane) {
  using F = Fmt<LF, KF>;
  const int r = lane >> 2;
    {
    const float al0 = alpha_s[buf * kHT + r], al1 = alpha_s[buf * kHT + r + 8];
    if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
      if (F::kLatOut) {
        oo[0] *= al0;
        oo[1] *= al0;
        oo[2] *= al1;
        oo[3] *= al1;
      }
#pragma unroll
      for (int g = 0; g < 4; ++g)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float2 a = __fmul2_rn(make_float2(o[g][e][0], o[g][e][1]), make_float2(al0, al0));
          const float2 b = __fmul2_rn(make_float2(o[g][e][2], o[g][e][3]), make_float2(al1, al1));
          o[g][e][0] = a.x;
          o[g][e][1] = a.y;
          o[g][e][2] = b.x;
          o[g][e][3] = b.y;
        }
    }
  }
  uint32_t pa[2][2][4];      // [hi/lo][k step][reg]
  {
    const uint32_t pbase = smem_u32(ptab) + (F::kPTiles * buf) * kHT * kPStride * 2 +
                           ((lane & 7) + 8 * ((lane >> 3) & 1)) * kPStride * 2 + 8 * (lane >> 4) * 2;
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
      ldsm_x4(pbase + 32 * ks, pa[0][ks][0], pa[0][ks][1], pa[0][ks][2], pa[0][ks][3]);
      if (F::kLatBf16)
        ldsm_x4(pbase + kHT * kPStride * 2 + 32 * ks, pa[1][ks][0], pa[1][ks][1], pa[1][ks][2], pa[1][ks][3]);
    }
  }
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    uint32_t vt[4][2];
#pragma unroll
    for (int n = 0; n < 4; ++n) {
      vt[n][0] = movt(bqv[g][n][0]);
      vt[n][1] = movt(bqv[g][n][1]);
    }
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
      if (F::kLatBf16) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          mma_bf16(o[g][e], pa[0][ks], vt[2 * ks][e], vt[2 * ks + 1][e], o[g][e]);
          mma_bf16(o[g][e], pa[1][ks], vt[2 * ks][e], vt[2 * ks + 1][e], o[g][e]);
        }
      } else if (F::kLatG8) {
        // the operands already carry their 8-channel group's scale
#pragma unroll
        for (int e = 0; e < 2; ++e) mma_f16(o[g][e], pa[0][ks], vt[2 * ks][e], vt[2 * ks + 1][e], o[g][e]);
      } else {
        // A = P scaled per token (column) by the group's scale
        uint32_t ag[4];
        ag[0] = h2_bits(__hmul2(bits_h2(pa[0][ks][0]), bits_h2(s2v[g][2 * ks])));
        ag[1] = h2_bits(__hmul2(bits_h2(pa[0][ks][1]), bits_h2(s2v[g][2 * ks])));
        ag[2] = h2_bits(__hmul2(bits_h2(pa[0][ks][2]), bits_h2(s2v[g][2 * ks + 1])));
        ag[3] = h2_bits(__hmul2(bits_h2(pa[0][ks][3]), bits_h2(s2v[g][2 * ks + 1])));
#pragma unroll
        for (int e = 0; e < 2; ++e) mma_f16(o[g][e], ag, vt[2 * ks][e], vt[2 * ks + 1][e], o[g][e]);
      }
    }
  }
  if (F::kLatOut && 4 * w < kNOut) {
    // protected channels: oo [16 heads][slots 4w + 2j, +1] += P (bf16 hi + lo)
    // x values (m16n8k16, k = tokens, n = slot 4w + r; columns 4..7 are zero)
    const uint32_t pb = smem_u32(ptab) + (F::kPTiles * buf + 2) * kHT * kPStride * 2 +
                        ((lane & 7) + 8 * ((lane >> 3) & 1)) * kPStride * 2 + 8 * (lane >> 4) * 2;
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
      uint32_t ph[4], pl[4];
      ldsm_x4(pb + 32 * ks, ph[0], ph[1], ph[2], ph[3]);
      ldsm_x4(pb + kHT * kPStride * 2 + 32 * ks, pl[0], pl[1], pl[2], pl[3]);
      mma_bf16(oo, ph, ovv[ks][0], ovv[ks][1], oo);
      mma_bf16(oo, pl, ovv[ks][0], ovv[ks][1], oo);
    }
  }
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------
// Warps 0..7 compute QK^T (step A) and PV (step C) of their latent groups;
// warpgroup 2 (warps 8..11) runs the online softmax (step B) of every chunk
// and the loader.  Hand-offs go through mbarriers with bounded waits:
//   bx[i & 1]: the 8 compute warps have written chunk i's partial scores
//              (thread 0 also its valid-token count and score scale, warp 0
//              its tokens' bounds M_t into mbuf[i & 1]); the stage of chunk
//              i is free again;
//   bp[i & 1]: the 4 softmax warps have written chunk i's P and alpha (and
//              are done with mbuf[i & 1]);
//   qa: the compute warps have posted their query magnitudes.
// Each warp arrives once, from lane 0 after a __syncwarp that orders the
// whole warp's stores before the arrival.
// A compute warp therefore runs A(i), arrives on bx, waits for bp of chunk
// i - 1 and runs C(i - 1), while the softmax warpgroup works on chunk i - 1
// or i.  Registers move to the compute warps with setmaxnreg: the 384-thread
// block launches with 168 per thread (64,512), then 232 each for the 256
// compute threads and 40 for the softmax warpgroup.
constexpr int kWsThreads = kThreads + 128;
constexpr int kRegsLaunch = 168, kRegsCompute = 232, kRegsSoftmax = 40;
static_assert(kThreads * kRegsCompute + 128 * kRegsSoftmax == kWsThreads * kRegsLaunch &&
                  kWsThreads * kRegsLaunch <= 65536 && kWsThreads * (kRegsLaunch + 8) > 65536,
              "the warpgroups' register shares must add up to the block's launch allocation");
constexpr int kWsExtra = 5 * 8 + 4 * 4 + 64 * 4;   // bx[2], bp[2], qa; nvq[2], cwq[2]; mbuf[2][32]

__device__ __forceinline__ void ws_regs_dec() { asm volatile("setmaxnreg.dec.sync.aligned.u32 40;\n" ::: "memory"); }
__device__ __forceinline__ void ws_regs_inc() { asm volatile("setmaxnreg.inc.sync.aligned.u32 232;\n" ::: "memory"); }

template <int LF, int KF>
__global__ void __launch_bounds__(kWsThreads, 1) decode_mma_kernel(DecodeParams p) {
  using F = Fmt<LF, KF>;
  pdl_launch_dependents();
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* stages = smem;
  float2* xpart = reinterpret_cast<float2*>(smem + F::kStages * F::kBlock);   // [2][8 warps][16 rows][kXStride]
  uint16_t* ptab = reinterpret_cast<uint16_t*>(xpart + 2 * kCW * kHT * kXStride);  // [2 buf][kPTiles][16][kPStride]
  float* alpha_s = reinterpret_cast<float*>(ptab + 2 * F::kPTiles * kHT * kPStride);   // [2][16]
  float* amax_s = alpha_s + 2 * kHT;                                           // [8]
  float* mbuf = amax_s + kCW;                      // [2][32] token bounds M_t of chunks i & 1 (float4 reads)
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(mbuf + 64);
  uint64_t* bx = full_bar + F::kStages;                                        // [2]
  uint64_t* bp = bx + 2;                                                       // [2]
  uint64_t* qa = bp + 2;                                                       // [1]
  int32_t* meta = reinterpret_cast<int32_t*>(qa + 1);
  int32_t* nvq = meta + F::kStages;                                            // [2]
  float* cwq = reinterpret_cast<float*>(nvq + 2);                              // [2]
  int32_t* cum = reinterpret_cast<int32_t*>(cwq + 2);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // grid (H / 16, G): the head tiles of one split are neighbours in launch
  // order, so they run side by side and share the split's pages through L2
  const int x = blockIdx.y, G = gridDim.y, h0 = blockIdx.x * kHT;
  const bool lead = (blockIdx.x == 0 && blockIdx.y == 0);

  if (p.lens_after_wait) pdl_wait();     // the lengths come from the kernel just before
  if (warp == 0) {
    int carry = 0;
    for (int base = 0; base < p.B; base += 32) {
      const int b = base + lane;
      int v = 0;
      // a length out of range counts as 0; the combine, after its wait,
      // reports it (dev_err may be written by a kernel still in flight here)
      if (b < p.B) v = (checked_len(p, b, false) + kChunk - 1) / kChunk;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += t;
      }
      if (b < p.B) cum[b + 1] = carry + v;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
    if (lane == 0) cum[0] = 0;
  } else if (tid == 32) {
    for (int s = 0; s < F::kStages; ++s) mbar_init(smem_u32(&full_bar[s]), 1);
    for (int k = 0; k < 2; ++k) {
      mbar_init(smem_u32(&bx[k]), kCW);      // one arrival per compute warp
      mbar_init(smem_u32(&bp[k]), 4);        // one per softmax warp
    }
    mbar_init(smem_u32(qa), kCW);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncthreads();
  // Up to here only the sequence lengths were read, a call's input that no
  // kernel in flight may write (the API's rule): the chunk prefix sums thus
  // overlap the previous kernel's tail; the workspace, queries and cache wait
  // for it.  The prefill's per-row lengths were waited for above: only
  // griddepcontrol.wait makes the lengths kernel's stores visible.
  // The register split needs nothing from the previous kernel either: each
  // role resizes its allocation first, then waits (split_wait).
  auto split_wait = [&]() {
    pdl_wait();
    if (lead)
      for (int i = tid; i <= p.B; i += kWsThreads) p.ws.cum[i] = cum[i];
  };

  const int C = cum[p.B];
  const int Ge = G < C ? G : C;
  if (x >= Ge) {
    split_wait();
    return;
  }
  const int c_lo = (int)range_lo(C, x, Ge), c_hi = (int)range_lo(C, x + 1, Ge);

  if (warp >= kCW) {
    // ======================= softmax / loader warpgroup =======================
    ws_regs_dec();
    split_wait();
    const int t = tid - kThreads;              // 0..127: row hr, tokens 4 tq .. 4 tq + 3
    const int hr = t >> 3, tq = t & 7;
    int ld_c = c_lo, ld_b = 0, ld_len = 0, pl_page = -1, pl_t0 = 0;
    bool pl_ready = false;
    if (t == 0) {
      ld_b = seq_of_chunk(cum, p.B, c_lo);
      ld_len = checked_len(p, ld_b, false);
    }
    auto plan = [&]() {
      if (pl_ready || ld_c >= c_hi) return;
      while (cum[ld_b + 1] <= ld_c) ld_len = checked_len(p, ++ld_b, false);
      pl_t0 = (ld_c - cum[ld_b]) * kChunk;
      pl_page = p.block_table[(size_t)ld_b * p.bt_stride + (pl_t0 >> 6)];
      pl_ready = true;
    };
    auto commit = [&](int s) {
      plan();
      if (!pl_ready) return;
      int nv = ld_len - pl_t0 < kChunk ? ld_len - pl_t0 : kChunk;
      if (pl_page < 0 || pl_page >= p.num_pages) {
        set_err(p.dev_err, MLA_DEVERR_PAGE);
        nv = 0;
      }
      meta[s] = nv;
      const uint32_t fb = smem_u32(&full_bar[s]);
      if (nv > 0) {
        mbar_expect_tx(fb, F::kBlock);
        bulk_g2s(smem_u32(stages + s * F::kBlock),
                 p.pool + (int64_t)pl_page * p.L.page_bytes + ((pl_t0 >> 5) & 1) * p.L.block_bytes, F::kBlock, fb);
      } else {
        mbar_arrive(fb);
      }
      pl_ready = false;
      ++ld_c;
      plan();     // the next chunk's page id: its load has a whole iteration to land
    };
    if (t == 0)
      for (int s = 0; s < F::kStages; ++s) commit(s);

    float m_row = -INFINITY, l_row = 0.f, e2 = 0.f;
    int b = -1, s = 0;
    bool dead = false;
    // Flush of sequence bb's partial: m, l and, with a quantized latent,
    // e2 = sum_t (p_t M_t)^2 over the row (M_t the token's stored bound
    // on |c_hat_t|), the weight of the fp16 P V products.
    auto flush_ml = [&](int bb) {
      float e = e2;
      if (F::kRisk) {
#pragma unroll
        for (int off = 1; off < 8; off <<= 1) e += __shfl_xor_sync(0xffffffffu, e, off);
      }
      if (tq == 0) {
        const size_t slot = (size_t)x + bb;
        p.ws.m[slot * p.H + h0 + hr] = m_row;
        p.ws.l[slot * p.H + h0 + hr] = l_row;
        p.ws.e2[slot * p.H + h0 + hr] = e;
      }
    };
    for (int c = c_lo, i = 0; c < c_hi; ++c, ++i) {
      int nb = b < 0 ? seq_of_chunk(cum, p.B, c) : b;
      while (cum[nb + 1] <= c) ++nb;
      if (nb != b) {
        if (b >= 0) flush_ml(b);
        b = nb;
        m_row = -INFINITY;
        l_row = 0.f;
        e2 = 0.f;
      }
      if (t == 0) plan();
      if (!mbar_wait_warp(smem_u32(&bx[i & 1]), (uint32_t)((i >> 1) & 1), p.wait_ns)) {
        set_err(p.dev_err, MLA_DEVERR_TIMEOUT);
        dead = true;
        break;
      }
      float4 mb4 = make_float4(0.f, 0.f, 0.f, 0.f);
      if (F::kRisk) mb4 = *reinterpret_cast<const float4*>(mbuf + (i & 1) * 32 + 4 * tq);
      if (t == 0) commit(s);                   // every compute warp is past chunk i's stage
      const int buf = i & 1, nv = nvq[buf];
      const float cw = cwq[buf];
      // sum the 8 warps' partial scores of 4 tokens of row hr
      const float4* xp = reinterpret_cast<const float4*>(xpart + ((size_t)buf * kCW * kHT + hr) * kXStride) + tq;
      float2 s01 = make_float2(0.f, 0.f), s23 = make_float2(0.f, 0.f);
#pragma unroll
      for (int ww = 0; ww < kCW; ++ww) {
        const float4 v = xp[ww * kHT * kXStride / 2];
        s01 = __fadd2_rn(s01, make_float2(v.x, v.y));
        s23 = __fadd2_rn(s23, make_float2(v.z, v.w));
      }
      const float4 sm = make_float4(s01.x, s01.y, s23.x, s23.y);
      float xv[4] = {sm.x * cw, sm.y * cw, sm.z * cw, sm.w * cw};
#pragma unroll
      for (int k = 0; k < 4; ++k) xv[k] = 4 * tq + k < nv ? xv[k] : -INFINITY;
      float mx = fmaxf(fmaxf(xv[0], xv[1]), fmaxf(xv[2], xv[3]));
#pragma unroll
      for (int off = 1; off < 8; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float mn = fmaxf(m_row, mx);
      const float al = mn == -INFINITY ? 1.f : ex2(m_row - mn);
      const float sub = mn == -INFINITY ? 0.f : mn;
      float pv[4], ps = 0.f;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        pv[k] = ex2(xv[k] - sub);
        ps += pv[k];
      }
#pragma unroll
      for (int off = 1; off < 8; off <<= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
      l_row = l_row * al + ps;
      m_row = mn;
      if (F::kRisk) {
        const float a0 = pv[0] * mb4.x, a1 = pv[1] * mb4.y, a2 = pv[2] * mb4.z, a3 = pv[3] * mb4.w;
        e2 = fmaf(e2 * al, al, fmaf(a0, a0, fmaf(a1, a1, fmaf(a2, a2, a3 * a3))));
      }
      uint2* prow = reinterpret_cast<uint2*>(ptab + ((F::kPTiles * buf) * kHT + hr) * kPStride) + tq;
      if (F::kLatBf16) {
        uint32_t h0w, l0w, h1w, l1w;
        split_bf16(pv[0], pv[1], h0w, l0w);
        split_bf16(pv[2], pv[3], h1w, l1w);
        prow[0] = make_uint2(h0w, h1w);
        prow[kHT * kPStride / 4] = make_uint2(l0w, l1w);
      } else {
        prow[0] = make_uint2(pack_f16(pv[0], pv[1]), pack_f16(pv[2], pv[3]));
      }
      if (F::kLatOut) {                        // bf16 hi + lo of P for the protected channels
        uint32_t h0w, l0w, h1w, l1w;
        split_bf16(pv[0], pv[1], h0w, l0w);
        split_bf16(pv[2], pv[3], h1w, l1w);
        prow[2 * kHT * kPStride / 4] = make_uint2(h0w, h1w);
        prow[3 * kHT * kPStride / 4] = make_uint2(l0w, l1w);
      }
      if (tq == 0) alpha_s[buf * kHT + hr] = al;
      __syncwarp();                            // the warp's P and alpha stores, then one arrival
      if (lane == 0) mbar_arrive(smem_u32(&bp[buf]));
      if (++s == F::kStages) s = 0;
    }
    if (!dead && b >= 0) flush_ml(b);
    if (dead) {
      // gave up: empty partials (weight 0) for the sequence in hand and every
      // later one of the range, so that the combine reads finite values
      m_row = -INFINITY;
      l_row = 0.f;
      e2 = 0.f;
      for (int bb = b >= 0 ? b : seq_of_chunk(cum, p.B, c_lo); bb < p.B && cum[bb] < c_hi; ++bb)
        if (cum[bb] < cum[bb + 1]) flush_ml(bb);
    }
    if (t == 0) {
      // the loader leaves only once every bulk copy it issued has landed, so
      // that no copy writes into the shared memory of a block that has exited
      const int issued = ld_c - c_lo;
      for (int k = issued > F::kStages ? issued - F::kStages : 0; k < issued; ++k)
        if (!mbar_wait(smem_u32(&full_bar[k % F::kStages]), (uint32_t)((k / F::kStages) & 1), kDrainLimitNs)) {
          set_err(p.dev_err, MLA_DEVERR_TIMEOUT);
          break;
        }
    }
    return;
  }

  // ============================= compute warps =============================
  ws_regs_inc();
  split_wait();
  const int w = warp, r = lane >> 2, j = lane & 3;
  Query q;
  float cw = 0.f;
  float o[4][2][4];
  float oo[4] = {0.f, 0.f, 0.f, 0.f};     // protected channels (INT8_OUTLIER): rows r, r+8 x slots 4w+2j, +1
  ChunkRegs ra, rb;
  bool pending = false;
  int b = -1, s = 0, i = 0;
  uint32_t phase = 0, qphase = 0;
  bool dead = false;

  auto flush_o = [&](int bb) {
    const size_t slot = (size_t)x + bb;
    if (tid == 0 && blockIdx.x == 0) {
      if (c_lo <= cum[bb]) p.ws.span[2 * bb] = x;
      if (c_hi >= cum[bb + 1]) p.ws.span[2 * bb + 1] = x;
    }
    float* o0 = p.ws.o + (slot * p.H + h0 + r) * kDc;
    float* o1 = o0 + 8 * kDc;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const int base = 16 * (4 * w + g);
      if (F::kStdLayout) {
        *reinterpret_cast<float2*>(o0 + base + 2 * j) = make_float2(o[g][0][0], o[g][0][1]);
        *reinterpret_cast<float2*>(o0 + base + 8 + 2 * j) = make_float2(o[g][1][0], o[g][1][1]);
        *reinterpret_cast<float2*>(o1 + base + 2 * j) = make_float2(o[g][0][2], o[g][0][3]);
        *reinterpret_cast<float2*>(o1 + base + 8 + 2 * j) = make_float2(o[g][1][2], o[g][1][3]);
      } else {
        const float4 v0 = make_float4(o[g][0][0], o[g][0][1], o[g][1][0], o[g][1][1]);
        const float4 v1 = make_float4(o[g][0][2], o[g][0][3], o[g][1][2], o[g][1][3]);
        const int c0 = base + 4 * j;
        // protected channels are written below by their slot's owner
        const uint32_t pm = F::kLatOut ? (p.outl.mask[c0 >> 5] >> (c0 & 31)) & 0xFu : 0u;
        if (pm == 0u) {
          *reinterpret_cast<float4*>(o0 + c0) = v0;
          *reinterpret_cast<float4*>(o1 + c0) = v1;
        } else {
          const float a0[4] = {v0.x, v0.y, v0.z, v0.w}, a1[4] = {v1.x, v1.y, v1.z, v1.w};
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (!((pm >> e) & 1u)) {
              o0[c0 + e] = a0[e];
              o1[c0 + e] = a1[e];
            }
        }
      }
    }
    if (F::kLatOut && j < 2) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int sl = 4 * w + 2 * j + e;
        if (sl < kNOut) {
          const int ch = p.outl.ch[sl];
          o0[ch] = oo[e];
          o1[ch] = oo[2 + e];
        }
      }
    }
  };
  // C of the previous chunk: wait for its P, then accumulate
  auto finish_prev = [&](const ChunkRegs& prev) -> bool {
    if (!pending) return true;
    const int pi = i - 1;
    if (!mbar_wait_warp(smem_u32(&bp[pi & 1]), (uint32_t)((pi >> 1) & 1), p.wait_ns)) {
      set_err(p.dev_err, MLA_DEVERR_TIMEOUT);
      return false;
    }
    pv_chunk<LF, KF>(o, oo, alpha_s, ptab, pi & 1, prev.bq, prev.s2h, prev.ov, w, lane);
    pending = false;
    return true;
  };

  auto chunk_step = [&](int c, ChunkRegs& cur, ChunkRegs& prev) -> bool {
    int nb = b < 0 ? seq_of_chunk(cum, p.B, c) : b;
    while (cum[nb + 1] <= c) ++nb;
    if (nb != b) {
      if (!finish_prev(prev)) return false;
      if (b >= 0) flush_o(b);
      b = nb;
      QueryRaw raw;
      const float am = warp_max(load_query_raw<LF, KF>(p, b, h0, w, lane, raw));
      if (lane == 0) amax_s[w] = am;
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(qa));
      if (!mbar_wait_warp(smem_u32(qa), qphase, p.wait_ns)) {
        set_err(p.dev_err, MLA_DEVERR_TIMEOUT);
        return false;
      }
      qphase ^= 1u;
      float amx = 0.f;
#pragma unroll
      for (int k = 0; k < kCW; ++k) amx = fmaxf(amx, amax_s[k]);
      int ex = 0;
      if (!F::kLatBf16 && amx > 0.f && isfinite(amx)) {
        ex = 14 - ilogbf(amx);
        ex = ex < -100 ? -100 : (ex > 100 ? 100 : ex);
      }
      finish_query<LF, KF>(raw, __int_as_float((127 + ex) << 23), q);
      cw = p.scale_log2 * __int_as_float((127 - ex) << 23);
#pragma unroll
      for (int g = 0; g < 4; ++g)
#pragma unroll
        for (int e = 0; e < 2; ++e)
#pragma unroll
          for (int k = 0; k < 4; ++k) o[g][e][k] = 0.f;
#pragma unroll
      for (int k = 0; k < 4; ++k) oo[k] = 0.f;
    }
    if (!mbar_wait_warp(smem_u32(&full_bar[s]), phase, p.wait_ns)) {
      set_err(p.dev_err, MLA_DEVERR_TIMEOUT);
      return false;
    }
    const int nv = meta[s];
    float acc[4][4];
    qk_chunk<LF, KF>(stages + s * F::kBlock, nv, w, lane, q, cur.bq, cur.s2h, cur.ov, acc);
    {
      float2* xw = xpart + (((size_t)(i & 1) * kCW + w) * kHT + r) * kXStride + j;
#pragma unroll
      for (int n = 0; n < 4; ++n) {
        xw[4 * n] = make_float2(acc[n][0], acc[n][1]);
        xw[8 * kXStride + 4 * n] = make_float2(acc[n][2], acc[n][3]);
      }
    }
    if (w == 0) {                  // warp-uniform: every lane stores the same count and scale
      nvq[i & 1] = nv;
      cwq[i & 1] = cw;
      if (F::kRisk) {              // the tokens' stored bounds (0 past the chunk's end)
        const float* bnd = reinterpret_cast<const float*>(stages + s * F::kBlock + F::kBoundOff);
        mbuf[(i & 1) * 32 + lane] = lane < nv ? bnd[lane] : 0.f;
      }
    }
    __syncwarp();                              // the warp's partial-score stores, then one arrival
    if (lane == 0) mbar_arrive(smem_u32(&bx[i & 1]));
    if (!finish_prev(prev)) return false;
    pending = true;
    ++i;
    if (++s == F::kStages) {
      s = 0;
      phase ^= 1u;
    }
    return true;
  };

  bool last_in_a = false;
  for (int c = c_lo; c < c_hi; c += 2) {
    if (!chunk_step(c, ra, rb)) { dead = true; break; }
    last_in_a = true;
    if (c + 1 >= c_hi) break;
    if (!chunk_step(c + 1, rb, ra)) { dead = true; break; }
    last_in_a = false;
  }
  if (!dead) {
    const bool ok = last_in_a ? finish_prev(ra) : finish_prev(rb);
    if (ok && b >= 0) flush_o(b);
    dead = !ok;
  }
  if (dead) {
    // gave up: empty partials (o = 0) and the span entries for the sequence
    // in hand and every later one of the range
#pragma unroll
    for (int g = 0; g < 4; ++g)
#pragma unroll
      for (int e = 0; e < 2; ++e)
#pragma unroll
        for (int k = 0; k < 4; ++k) o[g][e][k] = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) oo[k] = 0.f;
    for (int bb = b >= 0 ? b : seq_of_chunk(cum, p.B, c_lo); bb < p.B && cum[bb] < c_hi; ++bb)
      if (cum[bb] < cum[bb + 1]) flush_o(bb);
  }
}

// Largest dynamic shared memory a block may opt into on the current device.
size_t smem_max() {
  static int cached[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && cached[dev]) return (size_t)cached[dev];
  int v = 0;
  cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (dev >= 0 && dev < 64) cached[dev] = v;
  return (size_t)v;
}

template <int LF, int KF>
mla_status launch_t(const DecodeParams& p, cudaStream_t stream) {
  using F = Fmt<LF, KF>;
  if (p.L.block_bytes != F::kBlock || p.H % kHT) return MLA_ERR_UNSUPPORTED;
  const size_t smem = F::kFixed + sizeof(int32_t) * (p.B + 1);
  static int configured[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    const mla_status st = cuda_status(cudaFuncSetAttribute(
        decode_mma_kernel<LF, KF>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_max()));
    if (st != MLA_OK) return st;
    if (dev >= 0 && dev < 64) configured[dev] = 1;
  }
  if (smem + kWsExtra > smem_max()) return MLA_ERR_UNSUPPORTED;
  return cuda_status(launch_pdl(decode_mma_kernel<LF, KF>, dim3(p.H / kHT, p.G), dim3(kWsThreads), smem + kWsExtra,
                                stream, p));
}

}  // namespace

mla_status launch_decode_mma(const DecodeParams& p, cudaStream_t stream) {
#define MLA_MMA_CASE(A, K) \
  if (p.latent_fmt == A && p.kpe_fmt == K) return launch_t<A, K>(p, stream);
  MLA_MMA_CASE(MLA_FMT_BF16, MLA_FMT_BF16)
  MLA_MMA_CASE(MLA_FMT_BF16, MLA_FMT_INT8_SYM)
  MLA_MMA_CASE(MLA_FMT_INT8_SYM, MLA_FMT_BF16)
  MLA_MMA_CASE(MLA_FMT_INT8_SYM, MLA_FMT_INT8_SYM)
  MLA_MMA_CASE(MLA_FMT_INT4_ASYM, MLA_FMT_BF16)
  MLA_MMA_CASE(MLA_FMT_INT4_ASYM, MLA_FMT_INT8_SYM)
  MLA_MMA_CASE(MLA_FMT_INT4_SYM, MLA_FMT_BF16)
  MLA_MMA_CASE(MLA_FMT_INT4_SYM, MLA_FMT_INT8_SYM)
  MLA_MMA_CASE(MLA_FMT_BF16, MLA_FMT_INT4_SYM)
  MLA_MMA_CASE(MLA_FMT_INT8_SYM, MLA_FMT_INT4_SYM)
  MLA_MMA_CASE(MLA_FMT_INT4_ASYM, MLA_FMT_INT4_SYM)
  MLA_MMA_CASE(MLA_FMT_INT4_SYM, MLA_FMT_INT4_SYM)
  MLA_MMA_CASE(MLA_FMT_INT8_G8, MLA_FMT_INT8_SYM)
  MLA_MMA_CASE(MLA_FMT_INT8_G32, MLA_FMT_INT8_SYM)
  MLA_MMA_CASE(MLA_FMT_INT8_G64, MLA_FMT_INT8_SYM)
  MLA_MMA_CASE(MLA_FMT_INT8_TOKEN, MLA_FMT_INT8_SYM)
  MLA_MMA_CASE(MLA_FMT_INT8_OUTLIER, MLA_FMT_BF16)
  MLA_MMA_CASE(MLA_FMT_INT8_OUTLIER, MLA_FMT_INT8_SYM)
#undef MLA_MMA_CASE
  return MLA_ERR_UNSUPPORTED;
}

}  // namespace mla
