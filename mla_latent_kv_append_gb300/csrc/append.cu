// mla_cache_append: quantize-on-write of new tokens into the paged cache.
//
// English report "Absorbed MLA Cache Optimization on DeepSeek-V2-Lite —
// Technical Report" §2.1 (store() quantizes compressed_kv [seq, 512] and
// keeps k_pe [seq, 64]); Chinese report "DeepSeek-V2-Lite MLA 吸收式 KV 缓存优化"
// §3.2 (per-channel INT8 in 32 blocks, asymmetric INT4 in 32 blocks, k_pe
// INT8 in 8 blocks); juejin tutorial "量化压缩" (scale = absmax / 127).
//
// One warp per token.  Lane g owns latent group g (16 channels = 32 bytes of
// bf16 input), so a group's absmax / min / max needs no shuffles; lanes 0..7
// own the eight 8-channel k_pe groups.  The warp reads the token's 1152 input
// bytes in two coalesced sweeps and writes its code row (512 contiguous bytes
// for INT8) in the page's chunk order: 16-byte chunks swizzled by token, INT4
// nibbles of two groups interleaved per chunk (see mla_internal.cuh).  A
// quantized latent also gets its bound M_t (include/mla.h, mla_page_layout),
// the warp maximum of the groups' largest reachable |c_hat|.
//
// Bit-exactness: every step yields the IEEE fp32 round-to-nearest result of
// the plain definition's operation (x / s, max - min, ...), in the same order,
// followed by round-half-even to integer (rintf), so codes, scales,
// zero-points and bounds equal those of any correct fp32 implementation bit
// for bit.
// Denormals are kept (no flush-to-zero).  The per-element quotients x / s of
// a group share one divisor and use Markstein's FMA division (P. Markstein,
// "IA-64 and Elementary Functions", 2000): with y = RN(1/s), q0 = RN(x y) and
// one correction q1 = RN(q0 + RN(x - s q0) y), q1 is within an ulp of x / s,
// so the residual x - s q1 is exact in one FMA and q2 = RN(q1 + (x - s q1) y)
// is the correctly rounded quotient RN(x / s).  The theorem needs no
// overflow or underflow on the way, so a divisor outside [2^-100, 2^100]
// takes the plain IEEE division instead (quotients here are at most 127 for
// INT8 and 15 * 2^24 for INT4, so none overflows).
#include "mla_internal.cuh"

namespace mla {

namespace {

__device__ __forceinline__ void unpack16(const uint4& a, const uint4& b, float* x) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    x[2 * i] = bf16lo(w[i]);
    x[2 * i + 1] = bf16hi(w[i]);
  }
}

// RN(x[i] / s) for N values sharing the divisor s > 0 (see the header).
template <int N>
__device__ __forceinline__ void div_rn_shared(const float* x, float s, float* out) {
  if (s >= 0x1p-100f && s <= 0x1p100f) {
    const float y = __frcp_rn(s);
#pragma unroll
    for (int i = 0; i < N; ++i) {
      const float q0 = __fmul_rn(x[i], y);
      const float q1 = __fmaf_rn(__fmaf_rn(-q0, s, x[i]), y, q0);
      out[i] = __fmaf_rn(__fmaf_rn(-q1, s, x[i]), y, q1);
    }
  } else {
#pragma unroll
    for (int i = 0; i < N; ++i) out[i] = __fdiv_rn(x[i], s);
  }
}

template <int N>
__device__ __forceinline__ float absmax(const float* x) {
  float a = 0.f;
#pragma unroll
  for (int i = 0; i < N; ++i) a = fmaxf(a, fabsf(x[i]));
  return a;
}

// Symmetric quantization of N values with levels -QMAX .. QMAX (127 for
// INT8, 7 for INT4_SYM) given their group's absmax a (which may span more
// than these N values); returns the scale, writes the codes.
template <int N, int QMAX>
__device__ __forceinline__ float quant_sym_a(const float* x, float a, int8_t* q) {
  const float s = __fdiv_rn(a, (float)QMAX);
  float d[N];
  if (s > 0.f) div_rn_shared<N>(x, s, d);
#pragma unroll
  for (int i = 0; i < N; ++i) {
    const float r = s > 0.f ? fminf(fmaxf(rintf(d[i]), (float)-QMAX), (float)QMAX) : 0.f;
    q[i] = (int8_t)(int)r;
  }
  return s;
}

template <int N, int QMAX>
__device__ __forceinline__ float quant_sym(const float* x, int8_t* q) {
  return quant_sym_a<N, QMAX>(x, absmax<N>(x), q);
}

// Nibbles of one 16-channel half (or group) of a 4-bit chunk, placed in the
// chunk's four words: channels 4j, 4j+2, 4j+1, 4j+3 at nibbles 0, 1, 4, 5 of
// word j for the first half and 2, 3, 6, 7 for the second (half = 1), see
// int4_nibble_channel.  q[i] is the nibble value of channel i of the half.
__device__ __forceinline__ void int4_half_words(const uint8_t* q, int half, uint32_t* w) {
#pragma unroll
  for (int j = 0; j < 4; ++j)
    w[j] = ((uint32_t)q[4 * j] | ((uint32_t)q[4 * j + 2] << 4) | ((uint32_t)q[4 * j + 1] << 16) |
            ((uint32_t)q[4 * j + 3] << 20)) << (8 * half);
}

// Asymmetric INT4 of 16 values; returns scale, zero (fp32) and codes 0..15.
__device__ __forceinline__ void quant_asym4(const float* x, float& s_out, float& z_out, uint8_t* q) {
  float mn = x[0], mx = x[0];
#pragma unroll
  for (int i = 1; i < 16; ++i) {
    mn = fminf(mn, x[i]);
    mx = fmaxf(mx, x[i]);
  }
  float s = __fdiv_rn(__fsub_rn(mx, mn), 15.f);
  if (s == 0.f) s = fabsf(mn);
  float z = 0.f;
  float d[16];
  if (s > 0.f) {
    z = rintf(__fdiv_rn(-mn, s));
    div_rn_shared<16>(x, s, d);
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float r = s > 0.f ? fminf(fmaxf(__fadd_rn(rintf(d[i]), z), 0.f), 15.f) : 0.f;
    q[i] = (uint8_t)(int)r;
  }
  s_out = s;
  z_out = z;
}

template <int LF, int KF>
__global__ void __launch_bounds__(256) append_kernel(uint8_t* __restrict__ pool, PageLayout L, OutlierSet outl,
                                                     int64_t num_slots, const uint16_t* __restrict__ c_new,
                                                     const uint16_t* __restrict__ kpe_new,
                                                     const int32_t* __restrict__ slot, int n,
                                                     int32_t* dev_err) {
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  for (int i = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; i < n; i += warps) {
    const int32_t s = slot[i];
    if (s == -1) continue;
    if (s < 0 || (int64_t)s >= num_slots) {
      if (lane == 0) set_err(dev_err, MLA_DEVERR_SLOT);
      continue;
    }
    const int64_t page = s >> 6;
    const int t = s & 31;                       // token within its 32-token block
    uint8_t* blk = pool + page * L.page_bytes + ((s >> 5) & 1) * L.block_bytes;

    // ---- latent: lane g = group g (channels 16g .. 16g+15)
    const uint4* src = reinterpret_cast<const uint4*>(c_new + (size_t)i * kDc) + 2 * lane;
    const uint4 v0 = src[0], v1 = src[1];
    uint8_t* row = blk + L.codes_off + (int64_t)t * L.codes_row;
    if (LF == MLA_FMT_BF16) {
      reinterpret_cast<uint4*>(row)[latent_chunk_pos(2 * lane, t)] = v0;
      reinterpret_cast<uint4*>(row)[latent_chunk_pos(2 * lane + 1, t)] = v1;
    } else {
      float x[16];
      unpack16(v0, v1, x);
      float* scale = reinterpret_cast<float*>(blk + L.scale_off);
      float mb;      // this lane's share of the bound M_t (before the level factor)
      float mv = 0.f;  // INT8_OUTLIER: the largest protected magnitude of this lane's group
      if (LF == MLA_FMT_INT8_OUTLIER) {
        // protected channels of group `lane`: store their input bits in
        // their slot's row, then count them as 0 for the INT8 rule
        const uint32_t pm = (outl.mask[lane >> 1] >> (16 * (lane & 1))) & 0xFFFFu;
        if (pm) {
          const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
          uint16_t* ov = reinterpret_cast<uint16_t*>(blk + L.outlier_off);
          for (int k = 0; k < kNOut; ++k) {
            if ((outl.ch[k] >> 4) != lane) continue;
            const int ci = outl.ch[k] & 15;
            uint32_t bits = 0;
#pragma unroll
            for (int i = 0; i < 16; ++i)
              if (i == ci) bits = (w[i >> 1] >> (16 * (i & 1))) & 0xFFFFu;
            ov[k * kBlockTokens + t] = (uint16_t)bits;
            mv = fmaxf(mv, fabsf(__uint_as_float(bits << 16)));
          }
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if ((pm >> i) & 1u) x[i] = 0.f;
        }
      }
      if (is_int8_latent(LF)) {
        // lane = 16-channel chunk; a group of GS channels spans GS / 16
        // lanes (absmax by shuffles, every lane then derives the same
        // scale) or, for GS = 8, half a lane
        constexpr int GS = latent_group_size(LF);
        int8_t q[16];
        if constexpr (GS == 8) {
          const float s0 = quant_sym<8, 127>(x, q), s1 = quant_sym<8, 127>(x + 8, q + 8);
          scale[(2 * lane) * kBlockTokens + t] = s0;
          scale[(2 * lane + 1) * kBlockTokens + t] = s1;
          mb = fmaxf(s0, s1);
        } else {
          float a = absmax<16>(x);
#pragma unroll
          for (int o = 1; o < GS / 16; o <<= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
          const float sc = quant_sym_a<16, 127>(x, a, q);
          if (lane % (GS / 16) == 0) scale[(lane / (GS / 16)) * kBlockTokens + t] = sc;
          mb = sc;
        }
        // byte order of the chunk: channels in order, except for 8-channel
        // groups, where word j holds channels 2j, 2j+1, 8+2j, 8+2j+1
        uint32_t w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int c0 = GS == 8 ? 2 * j : 4 * j, c2 = GS == 8 ? 8 + 2 * j : 4 * j + 2;
          w[j] = (uint32_t)(uint8_t)q[c0] | ((uint32_t)(uint8_t)q[c0 + 1] << 8) |
                 ((uint32_t)(uint8_t)q[c2] << 16) | ((uint32_t)(uint8_t)q[c2 + 1] << 24);
        }
        reinterpret_cast<uint4*>(row)[latent_chunk_pos(lane, t)] = make_uint4(w[0], w[1], w[2], w[3]);
      } else {
        uint8_t q[16];
        if (LF == MLA_FMT_INT4_ASYM) {
          float sc, zp;
          quant_asym4(x, sc, zp, q);
          scale[lane * kBlockTokens + t] = sc;
          reinterpret_cast<float*>(blk + L.zero_off)[lane * kBlockTokens + t] = zp;
          // |q - z| <= max(|z|, |15 - z|) = |z - 7.5| + 7.5 over q in 0..15
          mb = __fmul_rn(sc, __fadd_rn(fabsf(__fsub_rn(zp, 7.5f)), 7.5f));
        } else {
          int8_t qs[16];
          mb = quant_sym<16, 7>(x, qs);
          scale[lane * kBlockTokens + t] = mb;
#pragma unroll
          for (int i = 0; i < 16; ++i) q[i] = (uint8_t)(qs[i] + 8);
        }
        // this lane's nibbles of the shared chunk (groups 2c and 2c+1), then
        // merge with the partner lane's
        uint32_t w[4];
        int4_half_words(q, lane & 1, w);
#pragma unroll
        for (int j = 0; j < 4; ++j) w[j] |= __shfl_xor_sync(0xffffffffu, w[j], 1);
        if ((lane & 1) == 0)
          reinterpret_cast<uint4*>(row)[latent_chunk_pos(lane >> 1, t)] = make_uint4(w[0], w[1], w[2], w[3]);
      }
      // the token's bound: the largest |c_hat| its codes can reach, the max
      // over groups of (levels a side) x s (asymmetric: s (|z - 7.5| + 7.5))
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, o));
        if (LF == MLA_FMT_INT8_OUTLIER) mv = fmaxf(mv, __shfl_xor_sync(0xffffffffu, mv, o));
      }
      if (lane == 0) {
        const float lv = is_int8_latent(LF) ? 127.f : (LF == MLA_FMT_INT4_SYM ? 7.f : 1.f);
        const float bd = LF == MLA_FMT_INT4_ASYM ? mb : __fmul_rn(lv, mb);
        reinterpret_cast<float*>(blk + L.bound_off)[t] = LF == MLA_FMT_INT8_OUTLIER ? fmaxf(bd, mv) : bd;
      }
    }

    // ---- k_pe: lanes 0..7, group = lane (channels 8g .. 8g+7).  For 4-bit
    // k_pe the eight lanes all take part in the shuffles (lanes 8.. idle).
    if (KF == MLA_FMT_INT4_SYM) {
      uint4 k = make_uint4(0u, 0u, 0u, 0u);
      if (lane < kNKG) k = reinterpret_cast<const uint4*>(kpe_new + (size_t)i * kDr)[lane];
      float x[8];
      const uint32_t kw[4] = {k.x, k.y, k.z, k.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        x[2 * j] = bf16lo(kw[j]);
        x[2 * j + 1] = bf16hi(kw[j]);
      }
      int8_t qs[8];
      const float sc = quant_sym<8, 7>(x, qs);
      // lane g: chunk g / 4, half (g / 2) % 2, channels 8 (g % 2) .. +7 of
      // the half; the half's channel i = 8 (g % 2) + i
      uint8_t q[16];
#pragma unroll
      for (int i2 = 0; i2 < 16; ++i2) q[i2] = 0;
      if (lane & 1) {
#pragma unroll
        for (int i2 = 0; i2 < 8; ++i2) q[8 + i2] = (uint8_t)(qs[i2] + 8);
      } else {
#pragma unroll
        for (int i2 = 0; i2 < 8; ++i2) q[i2] = (uint8_t)(qs[i2] + 8);
      }
      uint32_t w[4];
      int4_half_words(q, (lane >> 1) & 1, w);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        w[j] |= __shfl_xor_sync(0xffffffffu, w[j], 1);
        w[j] |= __shfl_xor_sync(0xffffffffu, w[j], 2);
      }
      if (lane < kNKG) {
        reinterpret_cast<float*>(blk + L.kpe_scale_off)[lane * kBlockTokens + t] = sc;
        if ((lane & 3) == 0) {
          uint8_t* krow = blk + L.kpe_off + (int64_t)t * L.kpe_row;
          reinterpret_cast<uint4*>(krow)[kpe_chunk_pos(lane >> 2, t, KF)] = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
    } else if (lane < kNKG) {
      const uint4 k = reinterpret_cast<const uint4*>(kpe_new + (size_t)i * kDr)[lane];
      uint8_t* krow = blk + L.kpe_off + (int64_t)t * L.kpe_row;
      if (KF == MLA_FMT_BF16) {
        reinterpret_cast<uint4*>(krow)[kpe_chunk_pos(lane, t, KF)] = k;
      } else {
        float x[8];
        const uint32_t w[4] = {k.x, k.y, k.z, k.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          x[2 * j] = bf16lo(w[j]);
          x[2 * j + 1] = bf16hi(w[j]);
        }
        int8_t q[8];
        reinterpret_cast<float*>(blk + L.kpe_scale_off)[lane * kBlockTokens + t] = quant_sym<8, 127>(x, q);
        const uint32_t lo = (uint32_t)(uint8_t)q[0] | ((uint32_t)(uint8_t)q[1] << 8) |
                            ((uint32_t)(uint8_t)q[2] << 16) | ((uint32_t)(uint8_t)q[3] << 24);
        const uint32_t hi = (uint32_t)(uint8_t)q[4] | ((uint32_t)(uint8_t)q[5] << 8) |
                            ((uint32_t)(uint8_t)q[6] << 16) | ((uint32_t)(uint8_t)q[7] << 24);
        *reinterpret_cast<uint2*>(krow + kpe_chunk_pos(lane >> 1, t, KF) * 16 + (lane & 1) * 8) =
            make_uint2(lo, hi);
      }
    }
  }
}

// Calibration of the INT8_OUTLIER protected set: one block, thread c takes
// latent channel c's max |x| over the n sample rows (row-major, so each row
// is one coalesced sweep), ranks it against the other 511 (larger maxima
// first, ties to the lower index) and, when it ranks below 25, writes c at
// its position among the selected channels in increasing order.
__global__ void __launch_bounds__(kDc) select_outliers_kernel(const uint16_t* __restrict__ c, int n,
                                                              int32_t* __restrict__ out) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ float amax[kDc];
  __shared__ int sel[kDc];
  const int ch = threadIdx.x;
  float m = 0.f;
#pragma unroll 8
  for (int i = 0; i < n; ++i) m = fmaxf(m, fabsf(bf16f(c[(size_t)i * kDc + ch])));
  amax[ch] = m;
  __syncthreads();
  int rank = 0;
  for (int k = 0; k < kDc; ++k) {
    const float v = amax[k];
    rank += (v > m || (v == m && k < ch)) ? 1 : 0;
  }
  sel[ch] = rank < kNOut ? 1 : 0;
  __syncthreads();
  if (sel[ch]) {
    int pos = 0;
    for (int k = 0; k < ch; ++k) pos += sel[k];
    out[pos] = ch;
  }
}

template <int LF, int KF>
mla_status launch_t(const mla_cache_layer* cache, const PageLayout& L, const OutlierSet& outl, const uint16_t* c_new,
                    const uint16_t* kpe_new, const int32_t* slot, int n, int32_t* dev_err,
                    cudaStream_t stream) {
  const int warps_per_block = 8;
  int sms = device_sm_count();
  int64_t want = ((int64_t)n + warps_per_block - 1) / warps_per_block;
  int64_t cap = (int64_t)(sms > 0 ? sms : 1) * 16;
  int grid = (int)(want < cap ? want : cap);
  return cuda_status(launch_pdl(append_kernel<LF, KF>, dim3(grid), dim3(32 * warps_per_block), 0, stream,
                                (uint8_t*)cache->pool, L, outl, (int64_t)cache->num_pages * kPage, c_new, kpe_new,
                                slot, n, dev_err));
}

}  // namespace

mla_status launch_select_outliers(const uint16_t* c_sample, int n, int32_t* out, cudaStream_t stream) {
  return cuda_status(launch_pdl(select_outliers_kernel, dim3(1), dim3(kDc), 0, stream, c_sample, n, out));
}

mla_status launch_append(const mla_cache_layer* cache, const PageLayout& L, const OutlierSet& outl,
                         const uint16_t* c_new, const uint16_t* kpe_new, const int32_t* slot, int n,
                         int32_t* dev_err, cudaStream_t stream) {
  const int lf = cache->latent_fmt, kf = cache->kpe_fmt;
#define MLA_APPEND_CASE(A, K) \
  if (lf == A && kf == K) return launch_t<A, K>(cache, L, outl, c_new, kpe_new, slot, n, dev_err, stream);
  MLA_APPEND_CASE(MLA_FMT_BF16, MLA_FMT_BF16)
  MLA_APPEND_CASE(MLA_FMT_BF16, MLA_FMT_INT8_SYM)
  MLA_APPEND_CASE(MLA_FMT_INT8_SYM, MLA_FMT_BF16)
  MLA_APPEND_CASE(MLA_FMT_INT8_SYM, MLA_FMT_INT8_SYM)
  MLA_APPEND_CASE(MLA_FMT_INT4_ASYM, MLA_FMT_BF16)
  MLA_APPEND_CASE(MLA_FMT_INT4_ASYM, MLA_FMT_INT8_SYM)
  MLA_APPEND_CASE(MLA_FMT_INT4_SYM, MLA_FMT_BF16)
  MLA_APPEND_CASE(MLA_FMT_INT4_SYM, MLA_FMT_INT8_SYM)
  MLA_APPEND_CASE(MLA_FMT_BF16, MLA_FMT_INT4_SYM)
  MLA_APPEND_CASE(MLA_FMT_INT8_SYM, MLA_FMT_INT4_SYM)
  MLA_APPEND_CASE(MLA_FMT_INT4_ASYM, MLA_FMT_INT4_SYM)
  MLA_APPEND_CASE(MLA_FMT_INT4_SYM, MLA_FMT_INT4_SYM)
  MLA_APPEND_CASE(MLA_FMT_INT8_G8, MLA_FMT_INT8_SYM)
  MLA_APPEND_CASE(MLA_FMT_INT8_G32, MLA_FMT_INT8_SYM)
  MLA_APPEND_CASE(MLA_FMT_INT8_G64, MLA_FMT_INT8_SYM)
  MLA_APPEND_CASE(MLA_FMT_INT8_TOKEN, MLA_FMT_INT8_SYM)
  MLA_APPEND_CASE(MLA_FMT_INT8_OUTLIER, MLA_FMT_BF16)
  MLA_APPEND_CASE(MLA_FMT_INT8_OUTLIER, MLA_FMT_INT8_SYM)
#undef MLA_APPEND_CASE
  return MLA_ERR_UNSUPPORTED;
}

}  // namespace mla
