// mla_decode_absorbed: split-K flash-decode of absorbed MLA attention over the
// paged latent cache, followed by the log-sum-exp combine.
//
// What is computed (English report "Absorbed MLA Cache Optimization on
// DeepSeek-V2-Lite — Technical Report" §2.1 get(): attention runs from the
// cached latent; juejin tutorial "步骤2" for K_i = C^KV W_i^upK, V_i = C^KV
// W_i^upV with the up-projections absorbed into q_lat and o_lat):
//   s[h,t] = (q_lat[h] . c_hat[t] + q_pe[h] . kpe_hat[t]) * softmax_scale
//   o_lat[h] = sum_t exp(s - max) c_hat[t] / sum_t exp(s - max)
//
// Work partition: the context of every sequence is cut into 32-token chunks;
// the C chunks of the whole batch are divided into G contiguous ranges, one
// per CTA along grid x (G = num SMs by default), so ragged batches stay
// balanced.  blockIdx.y selects a tile of 16 heads.  A CTA keeps the online
// softmax state (running max m, running sum l, unnormalised o) of the
// sequence it is in and writes it as a partial to slot (x + b) when the
// sequence or its range ends.  A combine kernel merges the partials of
// each sequence (combine_kernel, or combine_grouped_kernel for batches with
// few or very many partials per sequence); sequences shorter than 256
// tokens are recomputed exactly in fp32 there instead.  Scores are kept in
// the log2 domain (scaled by log2 e).
//
// This translation unit holds the combine kernels with the exact
// short-sequence path (fp32 CUDA cores, dequantized block in shared memory).
#include <cuda_fp16.h>
#include <math.h>

#include "mla_internal.cuh"

namespace mla {

namespace {

constexpr int kCS = kDc + 1;     // padded row stride of the latent chunk (floats)
constexpr int kKS = kDr + 1;     // padded row stride of the k_pe chunk

__device__ __forceinline__ int checked_len(const DecodeParams& p, int b, bool report) {
  int len = p.seq_lens[b];
  if (len < 0 || (int64_t)len > (int64_t)p.max_pages * kPage) {
    if (report) set_err(p.dev_err, MLA_DEVERR_SEQLEN);
    len = 0;
  }
  return len;
}

// Dequantizes tokens t0 .. t0 + 31 of sequence b (one 32-token block of a
// page) into s_c [32][kCS] and s_k [32][kKS], exactly as the oracle defines
// x_hat; tokens at or past len, or on a page id outside the pool (reported),
// read as 0.  s_valid, s_page: [32] scratch.  All NT threads of the block
// take part; the caller synchronizes before reading s_c / s_k.
template <int LF, int KF, int NT>
__device__ void dequant_chunk(const DecodeParams& p, int b, int t0, int len, float* s_c, float* s_k,
                              int32_t* s_valid, int32_t* s_page) {
  const int tid = threadIdx.x;
  const uint8_t* pool = p.pool;
  const int64_t pb = p.L.page_bytes;
  if (tid < kChunk) {
    const int t = t0 + tid;
    int valid = t < len;
    int page = 0;
    if (valid) {
      page = p.block_table[(size_t)b * p.bt_stride + (t >> 6)];
      if (page < 0 || page >= p.num_pages) {
        set_err(p.dev_err, MLA_DEVERR_PAGE);
        valid = 0;
      }
    }
    s_valid[tid] = valid;
    s_page[tid] = page;
  }
  __syncthreads();

  // ---- dequantize the chunk into shared memory (x_hat exactly as defined).
  // A chunk is one 32-token block of a page; t is the token in the block.
  const int64_t blk_off = (int64_t)((t0 >> 5) & 1) * p.L.block_bytes;
  if (LF == MLA_FMT_BF16) {
    for (int i = tid; i < kChunk * (kDc / 2); i += NT) {
      const int t = i / (kDc / 2), pr = i % (kDc / 2);
      float a = 0.f, bb = 0.f;
      if (s_valid[t]) {
        const uint32_t w = reinterpret_cast<const uint32_t*>(
            pool + s_page[t] * pb + blk_off + p.L.codes_off + (int64_t)t * p.L.codes_row)[
            latent_chunk_pos(pr >> 2, t) * 4 + (pr & 3)];
        a = bf16lo(w);
        bb = bf16hi(w);
      }
      s_c[t * kCS + 2 * pr] = a;
      s_c[t * kCS + 2 * pr + 1] = bb;
    }
  } else if (is_int8_latent(LF)) {
    for (int i = tid; i < kChunk * (kDc / 4); i += NT) {
      const int t = i / (kDc / 4), wi = i % (kDc / 4);
      float v[4] = {0.f, 0.f, 0.f, 0.f};
      // channel of byte j of word wi (8-channel groups store 2jj, 2jj+1,
      // 8+2jj, 8+2jj+1 in word jj of a 16-channel chunk)
      int ch[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        ch[j] = latent_group_size(LF) == 8 ? 16 * (wi >> 2) + 2 * (wi & 3) + (j & 1) + 8 * (j >> 1) : 4 * wi + j;
      if (s_valid[t]) {
        const uint8_t* blk = pool + s_page[t] * pb + blk_off;
        const uint32_t w = reinterpret_cast<const uint32_t*>(blk + p.L.codes_off + (int64_t)t * p.L.codes_row)[
            latent_chunk_pos(wi >> 2, t) * 4 + (wi & 3)];
        const float* sc = reinterpret_cast<const float*>(blk + p.L.scale_off);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          v[j] = __fmul_rn((float)(int8_t)(w >> (8 * j)), sc[(ch[j] / latent_group_size(LF)) * kBlockTokens + t]);
        if (LF == MLA_FMT_INT8_OUTLIER) {      // protected channels: the stored bf16 value
          const uint16_t* ov = reinterpret_cast<const uint16_t*>(blk + p.L.outlier_off);
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if ((p.outl.mask[ch[j] >> 5] >> (ch[j] & 31)) & 1u)
              for (int k = 0; k < kNOut; ++k)
                if (p.outl.ch[k] == ch[j]) v[j] = bf16f(ov[k * kBlockTokens + t]);
        }
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) s_c[t * kCS + ch[j]] = v[j];
    }
  } else {
    for (int i = tid; i < kChunk * (kDc / 8); i += NT) {
      const int t = i / (kDc / 8), pw = i % (kDc / 8);
      const int c = latent_chunk_pos(pw >> 2, t), j = pw & 3;   // logical chunk of this stored word
      float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      if (s_valid[t]) {
        const uint8_t* blk = pool + s_page[t] * pb + blk_off;
        const uint32_t w = reinterpret_cast<const uint32_t*>(blk + p.L.codes_off + (int64_t)t * p.L.codes_row)[pw];
        const float* sc = reinterpret_cast<const float*>(blk + p.L.scale_off);
        const float* zp = reinterpret_cast<const float*>(blk + p.L.zero_off);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int g = 2 * c + (int4_nibble_channel(j, k) >> 4);
          const float zero = LF == MLA_FMT_INT4_SYM ? 8.f : zp[g * kBlockTokens + t];
          v[k] = __fmul_rn(__fsub_rn((float)((w >> (4 * k)) & 15u), zero), sc[g * kBlockTokens + t]);
        }
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) s_c[t * kCS + 32 * c + int4_nibble_channel(j, k)] = v[k];
    }
  }
  if (KF == MLA_FMT_BF16) {
    for (int i = tid; i < kChunk * (kDr / 2); i += NT) {
      const int t = i / (kDr / 2), pr = i % (kDr / 2);
      float a = 0.f, bb = 0.f;
      if (s_valid[t]) {
        const uint32_t w = reinterpret_cast<const uint32_t*>(
            pool + s_page[t] * pb + blk_off + p.L.kpe_off + (int64_t)t * p.L.kpe_row)[
            kpe_chunk_pos(pr >> 2, t, KF) * 4 + (pr & 3)];
        a = bf16lo(w);
        bb = bf16hi(w);
      }
      s_k[t * kKS + 2 * pr] = a;
      s_k[t * kKS + 2 * pr + 1] = bb;
    }
  } else if (KF == MLA_FMT_INT4_SYM) {
    for (int i = tid; i < kChunk * (kDr / 8); i += NT) {
      const int t = i / (kDr / 8), pw = i % (kDr / 8);
      const int c = kpe_chunk_pos(pw >> 2, t, KF), j = pw & 3;   // logical chunk of this stored word
      float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      if (s_valid[t]) {
        const uint8_t* blk = pool + s_page[t] * pb + blk_off;
        const uint32_t w = reinterpret_cast<const uint32_t*>(blk + p.L.kpe_off + (int64_t)t * p.L.kpe_row)[pw];
        const float* sc = reinterpret_cast<const float*>(blk + p.L.kpe_scale_off);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int ch = 32 * c + int4_nibble_channel(j, k);
          v[k] = __fmul_rn(__fsub_rn((float)((w >> (4 * k)) & 15u), 8.f), sc[(ch >> 3) * kBlockTokens + t]);
        }
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) s_k[t * kKS + 32 * c + int4_nibble_channel(j, k)] = v[k];
    }
  } else {
    for (int i = tid; i < kChunk * (kDr / 4); i += NT) {
      const int t = i / (kDr / 4), wi = i % (kDr / 4);
      float v[4] = {0.f, 0.f, 0.f, 0.f};
      if (s_valid[t]) {
        const uint8_t* blk = pool + s_page[t] * pb + blk_off;
        const uint32_t w = reinterpret_cast<const uint32_t*>(blk + p.L.kpe_off + (int64_t)t * p.L.kpe_row)[
            kpe_chunk_pos(wi >> 2, t, KF) * 4 + (wi & 3)];
        const float s = reinterpret_cast<const float*>(blk + p.L.kpe_scale_off)[(wi >> 1) * kBlockTokens + t];
#pragma unroll
        for (int j = 0; j < 4; ++j) v[j] = __fmul_rn((float)(int8_t)(w >> (8 * j)), s);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) s_k[t * kKS + 4 * wi + j] = v[j];
    }
  }
}

// Formats whose split kernel records the weight of its fp16 P V products
// (every quantized latent; the bf16 path's P V is exact to ~2^-16).
template <int LF>
constexpr bool kRiskFmt = LF != MLA_FMT_BF16;

// combine_kernel: grid (B, H), block 1024: merge the partials of sequence b,
// head h (the grid for ~8 to ~32 slots per sequence).  CTAs
// span[2b] .. span[2b+1] wrote slots x + b.  The slots' maxima and sums are
// read in parallel (one slot per thread) and reduced (by warp 0 alone when
// there are at most 32 slots, else by the block); then each eighth of the
// block accumulates 4 channels per thread over every eighth slot (a long
// context spreads one sequence over every SM, so there can be ~150 slots)
// and the eighths are summed through shared memory.  Every slot in the span
// was written (o finite, weight 0 for an empty one), so the loads are
// unconditional; a thread's first partial rows load with the slot figures.
constexpr int kCombSlots = 1024;     // weights cached in shared memory
constexpr int kCombThreads = 1024;
constexpr int kCombParts = kCombThreads / (kDc / 4);
constexpr int kCombGroupHeads = 8;   // heads per block of the grouped grid

__device__ __forceinline__ float block_reduce(float v, bool is_max, float* red) {
#pragma unroll
  for (int off = 16; off; off >>= 1) {
    const float o = __shfl_xor_sync(0xffffffffu, v, off);
    v = is_max ? fmaxf(v, o) : v + o;
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  v = red[0];
#pragma unroll
  for (int k = 1; k < kCombThreads / 32; ++k) v = is_max ? fmaxf(v, red[k]) : v + red[k];
  return v;
}

// Rows recomputed exactly, in fp32, straight from the cache (exact_rows):
//  * sequences shorter than kExactLen tokens skip the split partials: over so
//    few tokens the split kernel's fp16 products P * s (fp16 P, fp16 group
//    scale) do not average out, and with a peaked softmax they would reach
//    the 2e-3 bound;
//  * rows whose split partials carry a large weight of fp16 products against
//    the merged output: sqrt(sum_t (w_t M_t)^2) > kRiskRatio * |o|_inf, with
//    w_t the normalised softmax weights and M_t a bound on max_c |c_hat_t[c]|
//    from token t's own scales (and zero-points).  The split kernel keeps
//    sum_t (p_t M_t)^2 per partial (relative to the partial's running
//    maximum) and the combine rescales and sums them.  This bounds the spread
//    of the fp16 roundings of the P V terms, sqrt(sum_t (w_t |c_hat_t|)^2),
//    from above.  Over natural data the ratio stays near 1 (the heavy
//    tokens' latents make up the output); it grows when heavy tokens'
//    latents cancel, where those roundings dominate the small result (the
//    fast path's error is a few 1e-4 times the ratio).
constexpr int kExactLen = 256;
constexpr float kRiskRatio = 4.f;
constexpr int kShortHeads = 8;             // heads per block of the short-sequence path
constexpr int kQS = kDc + kDr;             // a head's query row: q_lat, then q_pe
constexpr int kShortSmemBytes =
    (int)sizeof(float) * (kChunk * kCS + kChunk * kKS + kShortHeads * kQS + kChunk * kShortHeads + 3 * kShortHeads) +
    (int)sizeof(int32_t) * 2 * kChunk;

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int off = 16; off; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// Attention of sequence b, heads h0 .. h0 + 7, over its len tokens, in fp32,
// straight from the cache; rows j with bit j of `rows` set are written (o_lat
// and lse).  Per 32-token block: dequantize into shared memory once for the
// eight heads; four warps per head score eight tokens each (lanes over
// channels, log2 domain); warp j runs head j's online softmax over the block
// and overwrites the scores with the weights; then thread (c, half)
// accumulates channel c of heads 4 half .. 4 half + 3 over the block's
// tokens.  sm: kShortSmemBytes of shared memory.  Each combine kernel has a
// single call site (inlined: as a call it left spill code on the combine's
// common path, and a second inlined copy slowed that path down).
//
// exact_core is the computation over tokens t_begin .. len - 1 (t_begin a
// multiple of 32); with kPart it writes, instead of the normalised rows, the
// eight heads' partial state to part[8][kPartStride]: running maximum (log2
// domain), weight sum, then the 512 unnormalised channels.
constexpr int kPartStride = 2 + kDc;

template <int LF, int KF, bool kPart>
__device__ __forceinline__ void exact_core(const DecodeParams& p, int b, int h0, int t_begin, int len, uint32_t rows,
                                           float* sm, float* part) {
  float* s_c = sm;                                 // [32][kCS]
  float* s_k = s_c + kChunk * kCS;                 // [32][kKS]
  float* s_q = s_k + kChunk * kKS;                 // [8][kQS]
  float* s_w = s_q + kShortHeads * kQS;            // [32 tokens][8 heads] scores, then weights
  float* s_al = s_w + kChunk * kShortHeads;        // [8] the block's rescale factor per head
  float* s_ml = s_al + kShortHeads;                // [8][2] final running max and weight sum
  int32_t* s_valid = reinterpret_cast<int32_t*>(s_ml + 2 * kShortHeads);  // [32]
  int32_t* s_page = s_valid + kChunk;                                      // [32]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const size_t row0 = (size_t)b * p.H + h0;
  for (int i = tid; i < kShortHeads * kDc; i += kCombThreads) s_q[(i / kDc) * kQS + i % kDc] = p.q_lat[row0 * kDc + i];
  for (int i = tid; i < kShortHeads * kDr; i += kCombThreads)
    s_q[(i / kDr) * kQS + kDc + i % kDr] = bf16f(p.q_pe[row0 * kDr + i]);
  const int sh = warp >> 2, st0 = (warp & 3) * 8;  // scoring: head sh, tokens st0 .. st0 + 7
  const float* qrow = s_q + sh * kQS;
  const int c = tid & (kDc - 1), hb = (tid / kDc) * 4;
  float m = -INFINITY, l = 0.f;                    // warps 0..7: head `warp`'s running max and weight sum
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int t0 = t_begin; t0 < len; t0 += kChunk) {
    __syncthreads();                               // the previous block's readers are done; s_q in place
    dequant_chunk<LF, KF, kCombThreads>(p, b, t0, len, s_c, s_k, s_valid, s_page);
    __syncthreads();
    for (int u = 0; u < 8; u += 2) {
      const int ta = st0 + u;
      const float* ca = s_c + ta * kCS;
      const float* ka = s_k + ta * kKS;
      float a = 0.f, a2 = 0.f;
#pragma unroll 4
      for (int i = lane; i < kDc; i += 32) {
        const float q = qrow[i];
        a = fmaf(q, ca[i], a);
        a2 = fmaf(q, ca[kCS + i], a2);
      }
#pragma unroll
      for (int i = lane; i < kDr; i += 32) {
        const float q = qrow[kDc + i];
        a = fmaf(q, ka[i], a);
        a2 = fmaf(q, ka[kKS + i], a2);
      }
      a = warp_sum(a);
      a2 = warp_sum(a2);
      if (lane == 0) {
        s_w[ta * kShortHeads + sh] = (t0 + ta < len && s_valid[ta]) ? a * p.scale_log2 : -INFINITY;
        s_w[(ta + 1) * kShortHeads + sh] = (t0 + ta + 1 < len && s_valid[ta + 1]) ? a2 * p.scale_log2 : -INFINITY;
      }
    }
    __syncthreads();
    if (warp < kShortHeads) {
      const float sv = s_w[lane * kShortHeads + warp];
      const float mn = fmaxf(m, warp_max(sv));
      const float w = mn == -INFINITY ? 0.f : exp2f(sv - mn);
      const float al = mn == -INFINITY ? 1.f : exp2f(m - mn);
      s_w[lane * kShortHeads + warp] = w;
      if (lane == 0) s_al[warp] = al;
      l = fmaf(l, al, warp_sum(w));
      m = mn;
    }
    __syncthreads();
    const float4 al = *reinterpret_cast<const float4*>(s_al + hb);
    acc[0] *= al.x;
    acc[1] *= al.y;
    acc[2] *= al.z;
    acc[3] *= al.w;
#pragma unroll 8
    for (int t = 0; t < kChunk; ++t) {
      const float v = s_c[t * kCS + c];
      const float4 w = *reinterpret_cast<const float4*>(s_w + t * kShortHeads + hb);
      acc[0] = fmaf(w.x, v, acc[0]);
      acc[1] = fmaf(w.y, v, acc[1]);
      acc[2] = fmaf(w.z, v, acc[2]);
      acc[3] = fmaf(w.w, v, acc[3]);
    }
  }
  if (kPart) {
    if (warp < kShortHeads && lane == 0) {
      part[warp * kPartStride] = m;
      part[warp * kPartStride + 1] = l;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) part[(hb + j) * kPartStride + 2 + c] = acc[j];
    return;
  }
  if (warp < kShortHeads && lane == 0) {
    s_ml[2 * warp] = m;
    s_ml[2 * warp + 1] = l;
    if (p.lse && ((rows >> warp) & 1)) p.lse[row0 + warp] = l > 0.f ? (m + log2f(l)) * 0.69314718055994531f : -INFINITY;
  }
  __syncthreads();
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float lj = s_ml[2 * (hb + j) + 1];
    if ((rows >> (hb + j)) & 1) p.o_lat[(row0 + hb + j) * kDc + c] = lj > 0.f ? acc[j] / lj : 0.f;
  }
}

template <int LF, int KF>
__device__ __forceinline__ void exact_rows(const DecodeParams& p, int b, int h0, int len, uint32_t rows, float* sm) {
  exact_core<LF, KF, false>(p, b, h0, 0, len, rows, sm, nullptr);
}

// The output projection of rows b, h0 + j (bit j of `rows` set) that this
// block has just written to o_lat: o[b][h][v] = sum_c o_lat[b][h][c]
// W_UV[h][c][v] in fp32 (juejin tutorial "步骤2", V_i = C^KV W_i^upV, with
// W_UV[h] = W_i^upV).  Thread (v pair, 32-channel part) sums its part for
// two columns from bf16 pairs of W_UV (coalesced across the column pairs);
// the 16 parts are added through shared memory.  sm: 8 KB.  Every thread
// of the block takes part.
__device__ __forceinline__ void unabsorb_rows(const DecodeParams& p, int b, int h0, uint32_t rows, float* sm) {
  const int tid = threadIdx.x, vp = tid & 63, kp = tid >> 6;
  float2* red2 = reinterpret_cast<float2*>(sm);              // [16 parts][64 column pairs]
  for (int jh = 0; jh < kShortHeads; ++jh) {
    if (!((rows >> jh) & 1u)) continue;
    const int h = h0 + jh;
    const float* ol = p.o_lat + ((size_t)b * p.H + h) * kDc + 32 * kp;
    const uint32_t* w = reinterpret_cast<const uint32_t*>(p.w_uv + ((size_t)h * kDc + 32 * kp) * kDv) + vp;
    float a0 = 0.f, a1 = 0.f;
#pragma unroll 8
    for (int c = 0; c < 32; ++c) {
      const float x = ol[c];
      const uint32_t wv = __ldg(w + c * (kDv / 2));
      a0 = fmaf(x, bf16lo(wv), a0);
      a1 = fmaf(x, bf16hi(wv), a1);
    }
    red2[kp * 64 + vp] = make_float2(a0, a1);
    __syncthreads();
    if (tid < 64) {
      float2 sum = red2[tid];
#pragma unroll
      for (int k = 1; k < 16; ++k) {
        sum.x += red2[k * 64 + tid].x;
        sum.y += red2[k * 64 + tid].y;
      }
      *reinterpret_cast<float2*>(p.o + ((size_t)b * p.H + h) * kDv + 2 * tid) = sum;
    }
    __syncthreads();
  }
}

// The projection of one merged row (o_lat in shared memory, `row`) by
// W_UV[h]: the arithmetic of unabsorb_rows, with every weight load of a
// thread in flight at once and no re-read of the row from global memory.
__device__ __forceinline__ void unabsorb_row(const DecodeParams& p, int b, int h, const float* row, float* sm) {
  const int tid = threadIdx.x, vp = tid & 63, kp = tid >> 6;
  float2* red2 = reinterpret_cast<float2*>(sm);              // [16 parts][64 column pairs]
  const uint32_t* w = reinterpret_cast<const uint32_t*>(p.w_uv + ((size_t)h * kDc + 32 * kp) * kDv) + vp;
  uint32_t wv[32];
#pragma unroll
  for (int c = 0; c < 32; ++c) wv[c] = __ldg(w + c * (kDv / 2));
  float a0 = 0.f, a1 = 0.f;
#pragma unroll
  for (int c = 0; c < 32; ++c) {
    const float x = row[32 * kp + c];
    a0 = fmaf(x, bf16lo(wv[c]), a0);
    a1 = fmaf(x, bf16hi(wv[c]), a1);
  }
  red2[kp * 64 + vp] = make_float2(a0, a1);
  __syncthreads();
  if (tid < 64) {
    float2 sum = red2[tid];
#pragma unroll
    for (int k = 1; k < 16; ++k) {
      sum.x += red2[k * 64 + tid].x;
      sum.y += red2[k * 64 + tid].y;
    }
    *reinterpret_cast<float2*>(p.o + ((size_t)b * p.H + h) * kDv + 2 * tid) = sum;
  }
}

// For combine_kernel, before its wait: the chunk prefix sums at b and
// b + 1, their total, b's length, and the splits x0 .. x1 that wrote
// sequence b's slots, all derived from the call's lengths as the split kernel
// derives them.  The split kernel's partition gives split x the chunks
// [C x / Ge, C (x + 1) / Ge), Ge = min(G, C), so chunk c lies in split
// ceil((c + 1) Ge / C) - 1.  Run by warp 0; out: [c0, c1, C, len, x0, x1].
__device__ __forceinline__ void chunk_prefix(const DecodeParams& p, int b, int* out) {
  const int lane = threadIdx.x & 31;
  int carry = 0;
  for (int base = 0; base < p.B; base += 32) {
    const int bb = base + lane;
    const int len = bb < p.B ? checked_len(p, bb, false) : 0;
    int v = (len + kChunk - 1) / kChunk;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, v, off);
      if (lane >= off) v += t;
    }
    if (bb == b) {
      out[1] = carry + v;
      out[3] = len;
    }
    if (bb + 1 == b) out[0] = carry + v;
    carry += __shfl_sync(0xffffffffu, v, 31);
  }
  __syncwarp();
  if (lane == 0) {
    if (b == 0) out[0] = 0;
    out[2] = carry;
    const int c0 = out[0], c1 = out[1], C = carry, Ge = p.G < C ? p.G : C;
    if (c0 < c1) {                       // C > 0
      out[4] = (int)(((int64_t)(c0 + 1) * Ge + C - 1) / C) - 1;
      out[5] = (int)(((int64_t)c1 * Ge + C - 1) / C) - 1;
    }
  }
}

// Merge of sequence b, head h in a 1024-thread block (combine_kernel's
// grid) over the S slots from x0 on: writes o_lat and lse and returns true,
// or returns false (in every thread) when the row carries too much weight of
// fp16 P V products against its merged output and must be recomputed
// exactly.  The loads that do not wait for the maximum (every slot's figures,
// one per thread, and each thread's first kMergePre partial rows) are issued
// together: the merge is a few L2 round trips, not one per step.  (Three rows
// cover the ~20 slots of a 4K-token batch; the outlier format's combine has
// registers for two.)
template <int LF>
constexpr int kMergePre = LF == MLA_FMT_INT8_OUTLIER ? 2 : 3;
template <int LF>
__device__ __forceinline__ bool merge_head(const DecodeParams& p, int b, int h, int x0, int S, float* sw, float* red,
                                           float4 (*parts)[kDc / 4]) {
  const int tid = threadIdx.x;
  const int quad = tid & (kDc / 4 - 1), part = tid / (kDc / 4);
  float4* out = reinterpret_cast<float4*>(p.o_lat + ((size_t)b * p.H + h) * kDc) + quad;
  const float* mp = p.ws.m + (size_t)(x0 + b) * p.H + h;
  const float* lp = p.ws.l + (size_t)(x0 + b) * p.H + h;
  const float* ep = p.ws.e2 + (size_t)(x0 + b) * p.H + h;
  const float4* o4 = reinterpret_cast<const float4*>(p.ws.o + ((size_t)(x0 + b) * p.H + h) * kDc) + quad;
  float M, L, E2 = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (S == 1) {                          // one CTA held the whole sequence: normalise its partial
    if (!kRiskFmt<LF> && part > 0) return true;
    M = *mp;
    L = *lp;
    if (kRiskFmt<LF>) E2 = *ep;
    if (part == 0) acc = __ldcg(o4);
  } else {
    const size_t ostride = (size_t)p.H * (kDc / 4);
    float m0 = -INFINITY, l0 = 0.f, e0 = 0.f;
    if (tid < S) {
      m0 = mp[(size_t)tid * p.H];
      l0 = lp[(size_t)tid * p.H];
      if (kRiskFmt<LF>) e0 = ep[(size_t)tid * p.H];
    }
    float4 pre[kMergePre<LF>];
#pragma unroll
    for (int k = 0; k < kMergePre<LF>; ++k) {
      const int t = part + kCombParts * k;
      pre[k] = t < S ? __ldcg(o4 + (size_t)t * ostride) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (S <= 32) {
      // every slot's figures sit in warp 0: its shuffles give the block's
      // maximum and sums (the same trees as block_reduce, whose other warps
      // would add zeros), and one barrier publishes them with the weights
      if (tid < 32) {
        M = warp_max(m0);
        const float w = (M == -INFINITY || m0 == -INFINITY) ? 0.f : exp2f(m0 - M);
        sw[tid] = w;
        float lloc = 0.f, eloc = 0.f;
        if (w != 0.f) {
          lloc = fmaf(w, l0, 0.f);
          if (kRiskFmt<LF>) eloc = fmaf(w * w, e0, 0.f);
        }
        lloc = warp_sum(lloc);
        if (kRiskFmt<LF>) eloc = warp_sum(eloc);
        if (tid == 0) {                  // past the 32 weights: sw's last entries are free here
          sw[kCombSlots - 3] = M;
          sw[kCombSlots - 2] = lloc;
          sw[kCombSlots - 1] = eloc;
        }
      }
      __syncthreads();
      M = sw[kCombSlots - 3];
      L = sw[kCombSlots - 2];
      if (kRiskFmt<LF>) E2 = sw[kCombSlots - 1];
    } else {
      float mloc = m0;
      for (int t = tid + kCombThreads; t < S; t += kCombThreads) mloc = fmaxf(mloc, mp[(size_t)t * p.H]);
      M = block_reduce(mloc, true, red);
      float lloc = 0.f, eloc = 0.f;
      for (int t = tid; t < S; t += kCombThreads) {
        const float m = t == tid ? m0 : mp[(size_t)t * p.H];
        const float w = (M == -INFINITY || m == -INFINITY) ? 0.f : exp2f(m - M);
        if (t < kCombSlots) sw[t] = w;
        if (w != 0.f) {
          lloc = fmaf(w, t == tid ? l0 : lp[(size_t)t * p.H], lloc);
          if (kRiskFmt<LF>) eloc = fmaf(w * w, t == tid ? e0 : ep[(size_t)t * p.H], eloc);
        }
      }
      L = block_reduce(lloc, false, red);   // also orders the sw writes before the reads below
      if (kRiskFmt<LF>) E2 = block_reduce(eloc, false, red);
    }
#pragma unroll
    for (int k = 0; k < kMergePre<LF>; ++k) {   // slots part + 8 k < 24 <= kCombSlots: weights in sw
      const int t = part + kCombParts * k;
      if (t < S) {
        const float w = sw[t];
        acc.x = fmaf(w, pre[k].x, acc.x);
        acc.y = fmaf(w, pre[k].y, acc.y);
        acc.z = fmaf(w, pre[k].z, acc.z);
        acc.w = fmaf(w, pre[k].w, acc.w);
      }
    }
#pragma unroll 8
    for (int t = part + kCombParts * kMergePre<LF>; t < S; t += kCombParts) {
      float w;
      if (t < kCombSlots) {
        w = sw[t];
      } else {
        const float m = mp[(size_t)t * p.H];
        w = (M == -INFINITY || m == -INFINITY) ? 0.f : exp2f(m - M);
      }
      const float4 v = __ldcg(o4 + (size_t)t * ostride);
      acc.x = fmaf(w, v.x, acc.x);
      acc.y = fmaf(w, v.y, acc.y);
      acc.z = fmaf(w, v.z, acc.z);
      acc.w = fmaf(w, v.w, acc.w);
    }
    if (part > 0) {
      parts[part - 1][quad] = acc;
      acc = make_float4(0.f, 0.f, 0.f, 0.f);   // the row maximum below is taken over part 0's sums
    }
    __syncthreads();
    if (!kRiskFmt<LF> && part > 0) return true;
    if (part == 0) {
#pragma unroll
      for (int k = 0; k < kCombParts - 1; ++k) {
        const float4 a1 = parts[k][quad];
        acc.x += a1.x;
        acc.y += a1.y;
        acc.z += a1.z;
        acc.w += a1.w;
      }
    }
  }
  if (kRiskFmt<LF>) {                    // every thread takes part; parts > 0 hold 0
    const float amax = block_reduce(fmaxf(fmaxf(fabsf(acc.x), fabsf(acc.y)), fmaxf(fabsf(acc.z), fabsf(acc.w))),
                                    true, red);
    if (L > 0.f && sqrtf(E2) > kRiskRatio * amax) return false;
    if (part > 0) return true;
  }
  float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
  if (L > 0.f) {
    const float inv = 1.f / L;
    v = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    if (p.lse && tid == 0) p.lse[(size_t)b * p.H + h] = (M + log2f(L)) * 0.69314718055994531f;
  } else {
    if (p.lse && tid == 0) p.lse[(size_t)b * p.H + h] = -INFINITY;
  }
  *out = v;
  parts[0][quad] = v;                    // the row again, for the projection (part 0 read parts[] above)
  return true;
}

// One block per SM (64 registers a thread): at two per SM the 32-register
// limit spilled the merge and the exact path's live state, which cost more
// (4K INT8 call 26.6 against 19.7 us, step 0.908 against 0.772 ms) than the
// SM it leaves to the next kernel's early blocks.
template <int LF, int KF>
__global__ void __launch_bounds__(kCombThreads, 1) combine_kernel(DecodeParams p) {
  pdl_launch_dependents();
  const int b = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  extern __shared__ __align__(16) float short_smem[];
  __shared__ float sw[kCombSlots];
  __shared__ float red[kCombThreads / 32];
  __shared__ float4 parts[kCombParts - 1][kDc / 4];
  __shared__ int pre_c[6];
  // The lengths are a call input that no kernel in flight writes (except the
  // prefill's per-row lengths, which the kernel just before writes): the
  // sequence's chunk range and slot range come from them before the wait,
  // while the split kernel finishes.  This grid serves batches of at most
  // G / 8 sequences.
  const bool early = !p.lens_after_wait;
  if (early) {
    if (tid < 32) chunk_prefix(p, b, pre_c);
    __syncthreads();
  }
  pdl_wait();
  // a length out of range ran as 0 in the split kernel; it is reported here,
  // after the wait, so that no earlier kernel's write to dev_err can land later
  int len, c0, c1, x0, x1;
  if (early) {
    if (tid == 0) checked_len(p, b, true);
    c0 = pre_c[0];
    c1 = pre_c[1];
    len = pre_c[3];
    x0 = pre_c[4];
    x1 = pre_c[5];
  } else {
    // loaded together (the span entries are unused for an empty sequence,
    // whose entries nothing wrote)
    len = checked_len(p, b, tid == 0);
    c0 = p.ws.cum[b];
    c1 = p.ws.cum[b + 1];
    x0 = p.ws.span[2 * b];
    x1 = p.ws.span[2 * b + 1];
  }
  if (c0 == c1) {
    if (tid < kDc / 4) reinterpret_cast<float4*>(p.o_lat + ((size_t)b * p.H + h) * kDc)[tid] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (p.o && tid < kDv / 4) reinterpret_cast<float4*>(p.o + ((size_t)b * p.H + h) * kDv)[tid] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (p.lse && tid == 0) p.lse[(size_t)b * p.H + h] = -INFINITY;
    return;
  }
  // Rows recomputed exactly: the eight heads of a short sequence (by the
  // block of every eighth head), or this head when its merge asks for it
  // (computed with its seven neighbours, written alone).  One call site.
  // With the output projection requested, the block projects the rows it
  // wrote.
  const bool merged = len >= kExactLen && merge_head<LF>(p, b, h, x0, x1 - x0 + 1, sw, red, parts);
  if (merged || (len < kExactLen && h % kShortHeads != 0)) {
    if (merged && p.o) {
      __syncthreads();                      // the merged row in parts[0], before every thread reads it
      unabsorb_row(p, b, h, reinterpret_cast<const float*>(parts[0]), short_smem);
    }
    return;
  }
  const uint32_t rows = len < kExactLen ? 0xffu : 1u << (h % kShortHeads);
  exact_rows<LF, KF>(p, b, h - h % kShortHeads, len, rows, short_smem);
  if (p.o) {
    __syncthreads();
    unabsorb_rows(p, b, h - h % kShortHeads, rows, short_smem);
  }
}

// The same merge in two other grids, for the shapes where one block per
// (sequence, head) fits badly (chosen in launch_combine_t from the batch and
// the split count; G / B is the average number of slots per sequence):
//  * grid (B, H / 8), for many sequences with few slots each (G < 8 B): block
//    (b, g) merges heads 8 g .. 8 g + 7, 128 threads per head, each thread
//    summing every slot for its four channels; no block-wide reduction;
//  * grid (B, H, C), C = 2, 4 or 8, for few sequences with very many slots
//    (G >= 32 B) and a bf16 latent: block (b, h, z) merges channels
//    [512 z / C, 512 (z + 1) / C) with 8 C parts of ~19 slots each, after
//    the block-wide max and sum.
// Sequences shorter than kExactLen tokens go to exact_rows as in
// combine_kernel (in the sliced grid from the z = 0 block of every eighth
// head).  Its shared arrays live in the dynamic buffer, so this kernel adds
// no static shared memory to the exact path's.
template <int LF, int KF>
__global__ void __launch_bounds__(kCombThreads, 2) combine_grouped_kernel(DecodeParams p) {
  pdl_launch_dependents();
  pdl_wait();
  extern __shared__ __align__(16) float short_smem[];
  __shared__ float red[kCombThreads / 32];
  const int b = blockIdx.x, tid = threadIdx.x;
  const bool grouped = gridDim.y != (unsigned)p.H;
  // per-group grid: head h0 + tid / 128, channel quad tid % 128; per-head
  // grid: head blockIdx.y, the slice's quads split over 8 C parts
  const int h0 = grouped ? blockIdx.y * kCombGroupHeads : blockIdx.y;
  const int C = gridDim.z, z = blockIdx.z;
  const int qs_shift = 7 - (31 - __clz(C));          // quads per slice: 128 / C (C a power of two)
  const int ql = tid & ((1 << qs_shift) - 1);
  const int part = grouped ? 0 : tid >> qs_shift, nparts = kCombThreads >> qs_shift;
  const int h = grouped ? h0 + (tid >> 7) : h0;
  const int quad = grouped ? (tid & 127) : (z << qs_shift) + ql;
  const bool writes_lse = p.lse && (grouped ? (tid & 127) == 0 : (z == 0 && tid == 0));
  const size_t row = (size_t)b * p.H + h;
  const int32_t* cum = p.ws.cum;
  float4* out = reinterpret_cast<float4*>(p.o_lat + row * kDc) + quad;
  if (tid == 0) checked_len(p, b, true);            // reports, after the wait, as in combine_kernel
  if (cum[b] == cum[b + 1]) {
    if (part == 0) *out = make_float4(0.f, 0.f, 0.f, 0.f);
    if (writes_lse) p.lse[row] = -INFINITY;
    return;
  }
  const int len = checked_len(p, b, false);
  // The merge proper: writes the block's rows and returns true, or returns
  // false (in every thread; grouped grid, quantized latent) when one of its
  // eight heads carries too much weight of fp16 P V products against its
  // merged, unnormalised output, so that the eight are recomputed exactly.
  auto merge = [&]() -> bool {
  const int x0 = p.ws.span[2 * b], S = p.ws.span[2 * b + 1] - x0 + 1;
  const float* mp = p.ws.m + (size_t)(x0 + b) * p.H + h;
  const float* lp = p.ws.l + (size_t)(x0 + b) * p.H + h;
  const float* ep = p.ws.e2 + (size_t)(x0 + b) * p.H + h;
  const float4* o4 = reinterpret_cast<const float4*>(p.ws.o + ((size_t)(x0 + b) * p.H + h) * kDc) + quad;
  const size_t ostride = (size_t)p.H * (kDc / 4);
  // grouped grid, quantized latent: the block recomputes its eight heads
  // exactly when any of them carries too much weight of fp16 products
  // against its merged (unnormalised) output; every thread takes part
  auto risky = [&](const float4& un, float lsum, float e2sum) -> bool {
    float a = warp_max(fmaxf(fmaxf(fabsf(un.x), fabsf(un.y)), fmaxf(fabsf(un.z), fabsf(un.w))));
    if ((tid & 31) == 0) red[tid >> 5] = a;
    __syncthreads();
    const float* hr = red + 4 * (tid >> 7);
    a = fmaxf(fmaxf(hr[0], hr[1]), fmaxf(hr[2], hr[3]));
    return __syncthreads_or(lsum > 0.f && sqrtf(e2sum) > kRiskRatio * a) != 0;
  };
  if (S == 1) {                          // one CTA held the whole sequence: normalise its partial
    if (part > 0) return true;
    const float m = *mp, l = *lp;
    const float4 v = __ldcg(o4);
    if (kRiskFmt<LF> && grouped && risky(v, l, *ep)) return false;
    const float inv = l > 0.f ? 1.f / l : 0.f;
    *out = make_float4(v.x * inv, v.y * inv, v.z * inv, v.w * inv);
    if (writes_lse) p.lse[row] = l > 0.f ? (m + log2f(l)) * 0.69314718055994531f : -INFINITY;
    return true;
  }
  float M, L;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (grouped) {
    M = -INFINITY;
#pragma unroll 8
    for (int t = 0; t < S; ++t) M = fmaxf(M, mp[(size_t)t * p.H]);
    L = 0.f;
    float E2 = 0.f;
#pragma unroll 4
    for (int t = 0; t < S; ++t) {
      const float m = mp[(size_t)t * p.H], l = lp[(size_t)t * p.H];
      const float4 v = __ldcg(o4 + (size_t)t * ostride);
      const float w = (M == -INFINITY || m == -INFINITY) ? 0.f : exp2f(m - M);
      L = fmaf(w, l, L);
      if (kRiskFmt<LF> && w != 0.f) E2 = fmaf(w * w, ep[(size_t)t * p.H], E2);
      acc.x = fmaf(w, v.x, acc.x);
      acc.y = fmaf(w, v.y, acc.y);
      acc.z = fmaf(w, v.z, acc.z);
      acc.w = fmaf(w, v.w, acc.w);
    }
    if (kRiskFmt<LF> && risky(acc, L, E2)) return false;
  } else {
    float* sw = short_smem;                                        // [kCombSlots]
    float4* parts = reinterpret_cast<float4*>(short_smem + kCombSlots);   // [kCombThreads]
    float mloc = -INFINITY;
    for (int t = tid; t < S; t += kCombThreads) mloc = fmaxf(mloc, mp[(size_t)t * p.H]);
    M = block_reduce(mloc, true, red);
    float lloc = 0.f;
    for (int t = tid; t < S; t += kCombThreads) {
      const float m = mp[(size_t)t * p.H];
      const float w = (M == -INFINITY || m == -INFINITY) ? 0.f : exp2f(m - M);
      if (t < kCombSlots) sw[t] = w;
      if (w != 0.f) lloc = fmaf(w, lp[(size_t)t * p.H], lloc);
    }
    L = block_reduce(lloc, false, red);   // also orders the sw writes before the reads below
#pragma unroll 8
    for (int t = part; t < S; t += nparts) {
      float w;
      if (t < kCombSlots) {
        w = sw[t];
      } else {
        const float m = mp[(size_t)t * p.H];
        w = (M == -INFINITY || m == -INFINITY) ? 0.f : exp2f(m - M);
      }
      const float4 v = __ldcg(o4 + (size_t)t * ostride);
      acc.x = fmaf(w, v.x, acc.x);
      acc.y = fmaf(w, v.y, acc.y);
      acc.z = fmaf(w, v.z, acc.z);
      acc.w = fmaf(w, v.w, acc.w);
    }
    // parts 0..7 first fold in parts 8, 16, ... of their column, then part 0
    // adds parts 1..7
    parts[tid] = acc;
    __syncthreads();
    if (nparts > 8) {
      if (part < 8) {
        for (int k = part + 8; k < nparts; k += 8) {
          const float4 a1 = parts[(k << qs_shift) + ql];
          acc.x += a1.x;
          acc.y += a1.y;
          acc.z += a1.z;
          acc.w += a1.w;
        }
        parts[tid] = acc;
      }
      __syncthreads();
    }
    if (part > 0) return true;
#pragma unroll
    for (int k = 1; k < 8; ++k) {         // nparts >= 8
      const float4 a1 = parts[(k << qs_shift) + ql];
      acc.x += a1.x;
      acc.y += a1.y;
      acc.z += a1.z;
      acc.w += a1.w;
    }
  }
  if (L > 0.f) {
    const float inv = 1.f / L;
    *out = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    if (writes_lse) p.lse[row] = (M + log2f(L)) * 0.69314718055994531f;
  } else {
    *out = make_float4(0.f, 0.f, 0.f, 0.f);
    if (writes_lse) p.lse[row] = -INFINITY;
  }
  return true;
  };
  // Rows recomputed exactly (one call site): the eight heads of a short
  // sequence (in the sliced grid by the z = 0 block of every eighth head), or
  // the block's eight heads when its merge asks for it.
  const bool done = len < kExactLen ? !(grouped || (h0 % kShortHeads == 0 && z == 0)) : merge();
  if (done) return;
  exact_rows<LF, KF>(p, b, h0, len, 0xffu, short_smem);
}

// ---------------------------------------------------------------------------
// Support kernels of the tensor-core prefill (prefill_tc.cu).
//
// prefill_keys_kernel: grid (ceil(len / 128) * 4), block kKeyThreads.  Block
// x dequantizes tokens 32x .. 32x + 31 of the sequence (block-table row 0)
// as the oracle defines x_hat and writes each value as an fp16 pair
// (hi = rn(x), lo = rn(x - hi)) into the key tiles the tensor-core kernel
// copies from: tile kt = token / 128 holds, per 64-channel block kb (0..8:
// latent channels 64kb.., k_pe channels for kb = 8), a 128-token x 64-channel
// hi block and then the lo block, 16 KB each, rows 128 B with the 16-byte
// chunks of row r permuted by XOR with r mod 8 (the tensor core's 128-byte
// swizzle).  Tokens at or past len, or on a page outside the pool, are 0.
// mt[token] = the stored bound on |x_hat| (0 for bf16 latents, which keep no
// bound: their fp16 rounding is exact).  table (if not null): x_hat of
// tokens 0 .. kExactLen - 1 in fp32, [token][576].
constexpr int kKeyThreads = 256;
constexpr int kKeySmemBytes = (int)sizeof(float) * (kChunk * kCS + kChunk * kKS) + (int)sizeof(int32_t) * 2 * kChunk;
constexpr int kTcBlockBytes = 16384;

template <int LF, int KF>
__global__ void __launch_bounds__(kKeyThreads) prefill_keys_kernel(const DecodeParams p, int len, uint8_t* kws,
                                                                   float* mt, float* table) {
  extern __shared__ float key_smem[];
  float* s_c = key_smem;
  float* s_k = s_c + kChunk * kCS;
  int32_t* s_valid = reinterpret_cast<int32_t*>(s_k + kChunk * kKS);
  int32_t* s_page = s_valid + kChunk;
  pdl_launch_dependents();
  pdl_wait();
  const int t0 = blockIdx.x * kChunk;
  dequant_chunk<LF, KF, kKeyThreads>(p, 0, t0, len, s_c, s_k, s_valid, s_page);
  __syncthreads();
  const int tid = threadIdx.x;
  if (tid < kChunk) {
    float bound = 0.f;
    if (LF != MLA_FMT_BF16 && s_valid[tid]) {
      const uint8_t* blk = p.pool + s_page[tid] * p.L.page_bytes + (int64_t)((t0 >> 5) & 1) * p.L.block_bytes;
      bound = reinterpret_cast<const float*>(blk + p.L.bound_off)[tid];
    }
    mt[t0 + tid] = bound;
  }
  if (table && t0 < kExactLen) {       // x_hat of the first tokens for the short rows' exact recomputation
    for (int i = tid; i < kChunk * (kDc + kDr); i += kKeyThreads) {
      const int t = i / (kDc + kDr), c = i % (kDc + kDr);
      table[(size_t)(t0 + t) * (kDc + kDr) + c] = c < kDc ? s_c[t * kCS + c] : s_k[t * kKS + c - kDc];
    }
  }
  constexpr int kPieces = (kDc + kDr) / 8;         // 16-byte pieces of 8 channels per token
  for (int i = tid; i < kChunk * kPieces; i += kKeyThreads) {
    const int t = i / kPieces, c8 = i % kPieces;
    const float* src = c8 < kDc / 8 ? s_c + t * kCS + 8 * c8 : s_k + t * kKS + 8 * c8 - kDc;
    uint32_t hi[4], lo[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const __half2 h = __floats2half2_rn(src[2 * k], src[2 * k + 1]);
      const float2 hf = __half22float2(h);
      const __half2 r = __floats2half2_rn(src[2 * k] - hf.x, src[2 * k + 1] - hf.y);
      hi[k] = *reinterpret_cast<const uint32_t*>(&h);
      lo[k] = *reinterpret_cast<const uint32_t*>(&r);
    }
    const int tok = t0 + t, row = tok & 127, kb = c8 >> 3;
    uint8_t* dst = kws + ((int64_t)(tok >> 7) * 9 + kb) * 2 * kTcBlockBytes + row * 128 + (((c8 & 7) ^ (row & 7)) << 4);
    *reinterpret_cast<uint4*>(dst) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    *reinterpret_cast<uint4*>(dst + kTcBlockBytes) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
  }
}

// exact_fixup_kernel: block kCombThreads, a grid of at most two blocks per
// SM.  After the tensor-core prefill of B query rows (batch row b = query
// token, length p.seq_lens[b]), recomputes exactly in fp32 the heads h0 ..
// h0 + 7 of row b that need it: all of them when the row sees fewer than
// kExactLen tokens, else (quantized latents) those whose recorded check
// fails, risk[r] > kRiskRatio * max(omax[2r], omax[2r + 1]) with r = b H + h,
// the same criterion as the decode's combine (risk = sqrt(sum_t (w_t
// M_t)^2), omax = |o_lat|_inf of each 256-channel half).  Block x takes the
// (row, 8-head group) items x, x + G, x + 2G, .. (G = gridDim.x), 128 at a
// time: its threads test the 128 items' 8 heads at once, then the block
// recomputes the short items (unless skip_short: short_rows_kernel in
// prefill_tc.cu takes them) one after the other, and queues
// the long ones (up to kSplitCap per launch; past that it recomputes them
// itself) for exact_split_kernel, which spreads each over many blocks.  The
// stride spreads the short rows at the start of a chunk over every block.
constexpr int kFixupBatch = kCombThreads / kShortHeads;     // items tested per round: 128

template <int LF, int KF>
__global__ void __launch_bounds__(kCombThreads, 1) exact_fixup_kernel(const DecodeParams p, const float* risk,
                                                                      const float* omax, SplitQueue q,
                                                                      int skip_short) {
  extern __shared__ float short_smem[];
  __shared__ uint32_t s_bits[kFixupBatch];
  __shared__ int s_slot;
  pdl_launch_dependents();
  pdl_wait();
  const int groups = p.H / kShortHeads, items = p.B * groups;
  for (int first = blockIdx.x; first < items; first += gridDim.x * kFixupBatch) {
    __syncthreads();                               // the previous round's readers of s_bits are done
    const int it = first + gridDim.x * (threadIdx.x / kShortHeads);
    bool need = false;
    if (it < items) {
      const int b = it / groups, j = threadIdx.x % kShortHeads;
      const int len = checked_len(p, b, false);
      if (len < kExactLen) {
        need = !skip_short && len > 0;
      } else if (kRiskFmt<LF>) {
        const size_t r = (size_t)b * p.H + (it % groups) * kShortHeads + j;
        need = risk[r] > kRiskRatio * fmaxf(omax[2 * r], omax[2 * r + 1]);
      }
    }
    const uint32_t bal = __ballot_sync(0xffffffffu, need);
    if (threadIdx.x % kShortHeads == 0) s_bits[threadIdx.x / kShortHeads] = (bal >> (threadIdx.x & 31)) & 0xffu;
    __syncthreads();
    for (int i = 0; i < kFixupBatch; ++i) {
      const uint32_t rows = s_bits[i];
      if (rows == 0) continue;
      const int item = first + gridDim.x * i, b = item / groups, h0 = (item % groups) * kShortHeads;
      const int len = checked_len(p, b, false);
      if (len >= kExactLen) {          // a long row: queued for the split recomputation if there is room
        __syncthreads();
        if (threadIdx.x == 0) {
          const int slot = atomicAdd(q.count, 1);
          s_slot = slot;
          if (slot < kSplitCap) {
            q.items[4 * slot] = b;
            q.items[4 * slot + 1] = h0;
            q.items[4 * slot + 2] = (int)rows;
            q.items[4 * slot + 3] = len;
          }
        }
        __syncthreads();
        if (s_slot < kSplitCap) continue;
      }
      exact_rows<LF, KF>(p, b, h0, len, rows, short_smem);
    }
  }
}

// exact_split_kernel: block kCombThreads, a grid of at most two blocks per
// SM.  The long rows the fixup queued (q.items[0 .. min(*q.count, cap)))
// are recomputed exactly over kSplitParts contiguous token ranges each, one
// (item, range) per block at a time: the block writes the range's partial
// state, and the block that completes an item's last range (a counter per
// item) merges the partials into o_lat and lse (M = max m, L = sum 2^(m - M)
// l, o = sum 2^(m - M) o / L).  One block recomputing a 9K-token row alone
// took ~2.9 ms.
template <int LF, int KF>
__global__ void __launch_bounds__(kCombThreads, 1) exact_split_kernel(const DecodeParams p, SplitQueue q) {
  extern __shared__ float short_smem[];
  __shared__ int s_last;
  pdl_launch_dependents();
  pdl_wait();
  const int n = min(*q.count, kSplitCap);
  for (int unit = blockIdx.x; unit < n * kSplitParts; unit += gridDim.x) {
    const int item = unit / kSplitParts, part = unit % kSplitParts;
    const int b = q.items[4 * item], h0 = q.items[4 * item + 1], len = q.items[4 * item + 3];
    const uint32_t rows = (uint32_t)q.items[4 * item + 2];
    const int chunks = (len + kChunk - 1) / kChunk;
    const int c0 = chunks * part / kSplitParts, c1 = chunks * (part + 1) / kSplitParts;
    float* out = q.parts + ((size_t)item * kSplitParts + part) * kShortHeads * kPartStride;
    __syncthreads();
    exact_core<LF, KF, true>(p, b, h0, c0 * kChunk, min(c1 * kChunk, len), rows, short_smem, out);
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(q.done + item, 1) == kSplitParts - 1;
    __syncthreads();
    if (!s_last) continue;
    __threadfence();
    const int c = threadIdx.x & (kDc - 1), hb = (threadIdx.x / kDc) * 4;
    const float* base = q.parts + (size_t)item * kSplitParts * kShortHeads * kPartStride;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int h = hb + j;
      float M = -INFINITY;
      for (int r = 0; r < kSplitParts; ++r) M = fmaxf(M, __ldcg(base + (r * kShortHeads + h) * kPartStride));
      float L = 0.f, o = 0.f;
      for (int r = 0; r < kSplitParts; ++r) {
        const float* pr = base + (r * kShortHeads + h) * kPartStride;
        const float w = M == -INFINITY ? 0.f : exp2f(__ldcg(pr) - M);
        L = fmaf(w, __ldcg(pr + 1), L);
        o = fmaf(w, __ldcg(pr + 2 + c), o);
      }
      if ((rows >> h) & 1) {
        const size_t row = (size_t)b * p.H + h0 + h;
        p.o_lat[row * kDc + c] = L > 0.f ? o / L : 0.f;
        if (c == 0 && p.lse) p.lse[row] = L > 0.f ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
      }
    }
  }
}

}  // namespace

// The combine's grid for B sequences over G splits (G / B: the average
// number of partial slots per sequence): 0 = grouped (8 heads per block,
// G < 8 B), 1 = one block per (sequence, head), C > 1 = each head's channels
// sliced over C blocks (~19 slots or more per part; not for quantized
// latents, whose rows may need the exact path, which a slice cannot decide).
int combine_grid(int latent_fmt, int B, int G) {
  if (G < 8 * B) return 0;
  int c = 1;
  while (c < 8 && (int64_t)2 * c * 16 * B <= G) c *= 2;
  return latent_fmt == MLA_FMT_BF16 ? c : 1;
}

namespace {

// Launches the combine in the grid that suits the batch; *fused tells
// whether that grid also ran the requested output projection (the per-head
// grid does; the others leave it to out_unabsorb_kernel).
template <int LF, int KF>
mla_status launch_combine_t(const DecodeParams& p, cudaStream_t stream, bool* fused) {
  *fused = false;
  static int configured[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    const mla_status st = cuda_status(
        cudaFuncSetAttribute(combine_kernel<LF, KF>, cudaFuncAttributeMaxDynamicSharedMemorySize, kShortSmemBytes));
    if (st != MLA_OK) return st;
    if (dev >= 0 && dev < 64) configured[dev] = 1;
  }
  static int configured_g[64] = {0};
  if (dev < 0 || dev >= 64 || !configured_g[dev]) {
    const mla_status st = cuda_status(cudaFuncSetAttribute(
        combine_grouped_kernel<LF, KF>, cudaFuncAttributeMaxDynamicSharedMemorySize, kShortSmemBytes));
    if (st != MLA_OK) return st;
    if (dev >= 0 && dev < 64) configured_g[dev] = 1;
  }
  const int c = combine_grid(LF, p.B, p.G);
  if (c == 0)
    return cuda_status(launch_pdl(combine_grouped_kernel<LF, KF>, dim3(p.B, p.H / kCombGroupHeads, 1),
                                  dim3(kCombThreads), kShortSmemBytes, stream, p));
  if (c > 1)
    return cuda_status(launch_pdl(combine_grouped_kernel<LF, KF>, dim3(p.B, p.H, c), dim3(kCombThreads),
                                  kShortSmemBytes, stream, p));
  *fused = true;
  return cuda_status(
      launch_pdl(combine_kernel<LF, KF>, dim3(p.B, p.H), dim3(kCombThreads), kShortSmemBytes, stream, p));
}

mla_status launch_combine(const DecodeParams& p, cudaStream_t stream, bool* fused) {
#define MLA_COMBINE_CASE(A, K) \
  if (p.latent_fmt == A && p.kpe_fmt == K) return launch_combine_t<A, K>(p, stream, fused);
  MLA_COMBINE_CASE(MLA_FMT_BF16, MLA_FMT_BF16)
  MLA_COMBINE_CASE(MLA_FMT_BF16, MLA_FMT_INT8_SYM)
  MLA_COMBINE_CASE(MLA_FMT_INT8_SYM, MLA_FMT_BF16)
  MLA_COMBINE_CASE(MLA_FMT_INT8_SYM, MLA_FMT_INT8_SYM)
  MLA_COMBINE_CASE(MLA_FMT_INT4_ASYM, MLA_FMT_BF16)
  MLA_COMBINE_CASE(MLA_FMT_INT4_ASYM, MLA_FMT_INT8_SYM)
  MLA_COMBINE_CASE(MLA_FMT_INT4_SYM, MLA_FMT_BF16)
  MLA_COMBINE_CASE(MLA_FMT_INT4_SYM, MLA_FMT_INT8_SYM)
  MLA_COMBINE_CASE(MLA_FMT_BF16, MLA_FMT_INT4_SYM)
  MLA_COMBINE_CASE(MLA_FMT_INT8_SYM, MLA_FMT_INT4_SYM)
  MLA_COMBINE_CASE(MLA_FMT_INT4_ASYM, MLA_FMT_INT4_SYM)
  MLA_COMBINE_CASE(MLA_FMT_INT4_SYM, MLA_FMT_INT4_SYM)
  MLA_COMBINE_CASE(MLA_FMT_INT8_G8, MLA_FMT_INT8_SYM)
  MLA_COMBINE_CASE(MLA_FMT_INT8_G32, MLA_FMT_INT8_SYM)
  MLA_COMBINE_CASE(MLA_FMT_INT8_G64, MLA_FMT_INT8_SYM)
  MLA_COMBINE_CASE(MLA_FMT_INT8_TOKEN, MLA_FMT_INT8_SYM)
  MLA_COMBINE_CASE(MLA_FMT_INT8_OUTLIER, MLA_FMT_BF16)
  MLA_COMBINE_CASE(MLA_FMT_INT8_OUTLIER, MLA_FMT_INT8_SYM)
#undef MLA_COMBINE_CASE
  return MLA_ERR_UNSUPPORTED;
}

}  // namespace

mla_status launch_decode(const DecodeParams& p, cudaStream_t stream) {
  const mla_status st = launch_decode_mma(p, stream);
  if (st != MLA_OK) return st;
  bool fused = false;
  const mla_status sc = launch_combine(p, stream, &fused);
  if (sc != MLA_OK || !p.o || fused) return sc;
  return launch_out_unabsorb(p.o_lat, p.w_uv, p.o, p.B, p.H, stream);
}

namespace {

// Raises a kernel's dynamic shared-memory limit once per device.
template <typename K>
mla_status allow_smem(K kernel, int bytes, int* configured) {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && configured[dev]) return MLA_OK;
  const mla_status st = cuda_status(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes));
  if (st == MLA_OK && dev >= 0 && dev < 64) configured[dev] = 1;
  return st;
}

template <int LF, int KF>
mla_status launch_prefill_keys_t(const DecodeParams& p, int len, void* kws, float* mt, float* table,
                                 cudaStream_t stream) {
  static int configured[64] = {0};
  const mla_status st = allow_smem(prefill_keys_kernel<LF, KF>, kKeySmemBytes, configured);
  if (st != MLA_OK) return st;
  const int blocks = (len + 127) / 128 * 4;
  return cuda_status(launch_pdl(prefill_keys_kernel<LF, KF>, dim3(blocks), dim3(kKeyThreads), kKeySmemBytes, stream,
                                p, len, (uint8_t*)kws, mt, table));
}

template <int LF, int KF>
mla_status launch_exact_fixup_t(const DecodeParams& p, const float* risk, const float* omax, const SplitQueue& q,
                                int skip_short, cudaStream_t stream) {
  static int configured[64] = {0}, configured_s[64] = {0};
  mla_status st = allow_smem(exact_fixup_kernel<LF, KF>, kShortSmemBytes, configured);
  if (st != MLA_OK) return st;
  st = allow_smem(exact_split_kernel<LF, KF>, kShortSmemBytes, configured_s);
  if (st != MLA_OK) return st;
  const int items = p.B * (p.H / kShortHeads);
  const int sms = device_sm_count();
  const int cap = 2 * (sms > 0 ? sms : 1);
  st = cuda_status(launch_pdl(exact_fixup_kernel<LF, KF>, dim3(items < cap ? items : cap), dim3(kCombThreads),
                              kShortSmemBytes, stream, p, risk, omax, q, skip_short));
  if (st != MLA_OK) return st;
  return cuda_status(launch_pdl(exact_split_kernel<LF, KF>, dim3(cap), dim3(kCombThreads), kShortSmemBytes, stream,
                                p, q));
}

}  // namespace

#define MLA_FORMAT_PAIRS(X)                                                                                \
  X(MLA_FMT_BF16, MLA_FMT_BF16) X(MLA_FMT_BF16, MLA_FMT_INT8_SYM) X(MLA_FMT_INT8_SYM, MLA_FMT_BF16)         \
  X(MLA_FMT_INT8_SYM, MLA_FMT_INT8_SYM) X(MLA_FMT_INT4_ASYM, MLA_FMT_BF16)                                 \
  X(MLA_FMT_INT4_ASYM, MLA_FMT_INT8_SYM) X(MLA_FMT_INT4_SYM, MLA_FMT_BF16)                                 \
  X(MLA_FMT_INT4_SYM, MLA_FMT_INT8_SYM) X(MLA_FMT_BF16, MLA_FMT_INT4_SYM)                                  \
  X(MLA_FMT_INT8_SYM, MLA_FMT_INT4_SYM) X(MLA_FMT_INT4_ASYM, MLA_FMT_INT4_SYM)                             \
  X(MLA_FMT_INT4_SYM, MLA_FMT_INT4_SYM) X(MLA_FMT_INT8_G8, MLA_FMT_INT8_SYM)                               \
  X(MLA_FMT_INT8_G32, MLA_FMT_INT8_SYM) X(MLA_FMT_INT8_G64, MLA_FMT_INT8_SYM)                              \
  X(MLA_FMT_INT8_TOKEN, MLA_FMT_INT8_SYM) X(MLA_FMT_INT8_OUTLIER, MLA_FMT_BF16)                            \
  X(MLA_FMT_INT8_OUTLIER, MLA_FMT_INT8_SYM)

mla_status launch_prefill_keys(const DecodeParams& p, int len, void* kws, float* mt, float* table,
                               cudaStream_t stream) {
#define MLA_KEYS_CASE(A, K) \
  if (p.latent_fmt == A && p.kpe_fmt == K) return launch_prefill_keys_t<A, K>(p, len, kws, mt, table, stream);
  MLA_FORMAT_PAIRS(MLA_KEYS_CASE)
#undef MLA_KEYS_CASE
  return MLA_ERR_UNSUPPORTED;
}

mla_status launch_exact_fixup(const DecodeParams& p, const float* risk, const float* omax, const SplitQueue& q,
                              int skip_short, cudaStream_t stream) {
#define MLA_FIXUP_CASE(A, K) \
  if (p.latent_fmt == A && p.kpe_fmt == K) return launch_exact_fixup_t<A, K>(p, risk, omax, q, skip_short, stream);
  MLA_FORMAT_PAIRS(MLA_FIXUP_CASE)
#undef MLA_FIXUP_CASE
  return MLA_ERR_UNSUPPORTED;
}
#undef MLA_FORMAT_PAIRS

}  // namespace mla
