// Tensor-core (tcgen05) causal attention of a prefill chunk.
//
// What is computed: for query row r = (token i, head h) of the chunk, at
// position qpos = ctx_before + i, the absorbed attention over the cached
// positions 0 .. qpos ("Absorbed MLA Cache Optimization on DeepSeek-V2-Lite
// — Technical Report" §2.1: attention straight from the cached latent; the
// juejin tutorial's FAQ on pairing MLA with FlashAttention-style tiling):
//   s[r,t] = (q_lat[r] . c_hat[t] + q_pe[r] . kpe_hat[t]) * softmax_scale
//   o_lat[r] = sum_t exp(s - max) c_hat[t] / sum_t exp(s - max)
// Every head of every query reads the same cached latent, so a tile of 128
// rows (any mix of tokens and heads) is a dense M = 128 contraction against
// the keys: this is where the tensor core pays.
//
// Data path (one launch per slice of query tokens):
//   * the key tiles: every cached token dequantized once (x_hat exactly as
//     the oracle defines it, prefill_keys_kernel in decode.cu) and stored as
//     an fp16 pair hi = rn(x), lo = rn(x - hi), pre-swizzled, so that a
//     128-token x 64-channel block is one contiguous 16 KB bulk copy;
//   * the query tiles (q_split_kernel below): the same split of q_lat and
//     q_pe, 128 rows x 64 channels per 16 KB block;
//   * prefill_tc_kernel: per CTA one 128-row tile and one 256-channel half
//     of o_lat (the fp32 accumulator of all 512 channels would fill the
//     512 TMEM columns alone).  Per 128-key tile:
//       S = Q_hi K_hi^T + Q_hi K_lo^T + Q_lo K_hi^T     (tcgen05.mma, f16 in,
//           f32 accumulate in TMEM; the split keeps the scores at ~1e-6
//           relative where one fp16 rounding of either side costs ~1e-2 on
//           latents with large outlier channels)
//       online softmax in the log2 domain, one row per thread of the
//       softmax warpgroup, P rounded to fp16 into shared memory
//       O_half += P V_half   (V = K_hi's latent channels, read MN-major)
//     The running maximum is raised only when a tile's maximum exceeds it by
//     more than 8 (P <= 256 in fp16); O is then rescaled in TMEM.
//   * rows that see fewer than 256 tokens, and rows of quantized latents
//     whose precision check fails (the decode's criterion: sqrt(sum_t (w_t
//     M_t)^2) > 4 |o_lat|_inf, M_t the token's stored bound), are recomputed
//     exactly in fp32 afterwards (exact_fixup_kernel in decode.cu).
//
// Warp roles (192 threads): warp 0 lane 0 issues the bulk copies, warp 1
// allocates TMEM and its lane 0 issues the MMAs, warps 2..5 run the softmax
// (warp w reads TMEM lanes 32 (w mod 4) ..) and the epilogue.
//
// TMEM (512 columns): S in columns 0..255 (Q_hi K_hi + Q_lo K_hi in 0..127,
// Q_hi K_lo in 128..255: the two Q_hi products are one N = 256 MMA), the O
// half in 256..511.  Shared memory (1024-aligned): a ring of three 64 KB
// slots, the 32 KB P tile, then the barriers.  The ring carries, per key
// tile j, nine QK items (Q_hi, Q_lo, K_hi, K_lo of one 64-channel block)
// and then the V item of tile j - 1 (the half's four 64-channel blocks of
// K_hi), in the order the MMAs consume them; three slots keep two 64 KB
// items in flight while the MMAs work on the third (with two stages the
// MMAs waited ~25 % of the time for data).
#include <cuda_fp16.h>
#include <math.h>

#include "mla_internal.cuh"

namespace mla {
namespace {

constexpr int kTcRows = 128;                    // query rows per tile (TMEM lanes)
constexpr int kTcKeys = 128;                    // keys per tile
constexpr int kTcKB = (kDc + kDr) / 64;         // 9 channel blocks of the contraction
constexpr int kBlk = kTcTileBytes / (2 * kTcKB);  // one 128 x 64 fp16 block: 16 KB
constexpr int kTileBytes = kTcTileBytes;        // hi + lo blocks of one 128-row tile
constexpr int kStageBytes = 4 * kBlk;           // a ring slot: one QK item or one V item
constexpr int kStages = 3;
constexpr int kPOff = kStages * kStageBytes;
constexpr int kBarOff = kPOff + 2 * kBlk;
constexpr int kTcSmem = kBarOff + 128 + 1024;   // barriers, TMEM address; 1024-byte alignment slack
constexpr int kTcThreads = 192;
constexpr float kRescaleSlack = 8.f;            // raise the running max only past this (log2 units)
constexpr uint64_t kDrainNs = 2000000000ull;    // bound on the final waits for this CTA's own copies / MMAs

// barrier indices (8 bytes each at kBarOff)
enum { kFull0 = 0, kEmpty0 = kStages, kSFull = 2 * kStages, kSRead, kPFull, kPVDone, kFin, kNumBars };


__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void bar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void bar_arrive(uint32_t bar) {
  asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.shared::cta.b64 st, [%0];\n}\n" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void bar_expect(uint32_t bar, uint32_t bytes) {
  asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}\n" ::"r"(bar),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool bar_test(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}
__device__ __forceinline__ uint64_t now_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Waits for the phase of `bar` with this parity.  Gives up (false) once
// limit_ns have passed or another role of the CTA has given up (*abort set).
__device__ __noinline__ bool bar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns, volatile int* abort) {
  if (bar_test(bar, parity)) return true;
  const uint64_t t0 = now_ns();
  for (;;) {
    if (bar_test(bar, parity)) return true;
    if (*abort || now_ns() - t0 >= limit_ns) return false;
  }
}

__device__ __forceinline__ void bulk_copy(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle (layout type 2,
// descriptor version 1).  K-major operands: rows of 64 fp16 channels, 8-row
// groups 1024 B apart (sbo); MN-major (the V operand): 64-channel blocks lbo
// apart, 8-key groups sbo apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor of kind::f16: f32 accumulator, f16 A and B, M = 128.
__host__ __device__ constexpr uint32_t f16_idesc(int n, bool b_mn_major) {
  return (1u << 4) | ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(kTcRows >> 4) << 24);
}

__device__ __forceinline__ void umma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(bar)
               : "memory");
}
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}

// q_split_kernel: query rows r < R (q_lat [R][512] fp32, q_pe [R][64] bf16)
// into row tiles of fp16 (hi, lo) blocks, swizzled like the key tiles; rows
// R .. 128 n_rt - 1 are zero.  One thread per 8 channels of a row.
__global__ void __launch_bounds__(256) q_split_kernel(const float* q_lat, const uint16_t* q_pe, int R, int n_rt,
                                                      uint8_t* qws) {
  pdl_launch_dependents();
  pdl_wait();
  constexpr int kPieces = (kDc + kDr) / 8;
  const int64_t total = (int64_t)n_rt * kTcRows * kPieces;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int row = (int)(i / kPieces), c8 = (int)(i % kPieces);
    float x[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (row < R) {
      if (c8 < kDc / 8) {
        const float4* src = reinterpret_cast<const float4*>(q_lat + (int64_t)row * kDc + 8 * c8);
        const float4 a = src[0], b = src[1];
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
        x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
      } else {
        const uint4 w = *reinterpret_cast<const uint4*>(q_pe + (int64_t)row * kDr + 8 * (c8 - kDc / 8));
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          x[2 * k] = bf16lo(ws[k]);
          x[2 * k + 1] = bf16hi(ws[k]);
        }
      }
    }
    uint32_t hi[4], lo[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const __half2 h = __floats2half2_rn(x[2 * k], x[2 * k + 1]);
      const float2 hf = __half22float2(h);
      const __half2 l = __floats2half2_rn(x[2 * k] - hf.x, x[2 * k + 1] - hf.y);
      hi[k] = *reinterpret_cast<const uint32_t*>(&h);
      lo[k] = *reinterpret_cast<const uint32_t*>(&l);
    }
    const int lr = row & (kTcRows - 1), kb = c8 >> 3;
    uint8_t* dst = qws + ((int64_t)(row / kTcRows) * kTcKB + kb) * 2 * kBlk + lr * 128 + (((c8 & 7) ^ (lr & 7)) << 4);
    *reinterpret_cast<uint4*>(dst) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    *reinterpret_cast<uint4*>(dst + kBlk) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
  }
}

// Bounded wait that ignores the abort flag: the final waits for this CTA's
// own bulk copies and MMAs before it frees shared memory and TMEM.
__device__ __noinline__ bool drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = now_ns();
  while (!bar_test(bar, parity))
    if (now_ns() - t0 >= kDrainNs) return false;
  return true;
}

// bar_wait by every lane of a warp, with a warp-uniform answer.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns, volatile int* abort) {
  return __all_sync(0xffffffffu, bar_wait(bar, parity, limit_ns, abort));
}

// 32 columns of this thread's TMEM lane into v (load and wait in one
// statement, so no use of v can be scheduled before the data is there).
__device__ __forceinline__ void tmem_load(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// v into 32 columns of this thread's TMEM lane, waiting for the store.
__device__ __forceinline__ void tmem_store(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n"
      "tcgen05.wait::st.sync.aligned;\n" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}

__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// prefill_tc_kernel: grid (2 n_rt), block kTcThreads, kTcSmem bytes of
// dynamic shared memory, one CTA per SM.  CTA x: row tile n_rt - 1 - x / 2
// (the longest prefixes first), o_lat channels 256 (x mod 2) .. + 255.
__global__ void __launch_bounds__(kTcThreads, 1) prefill_tc_kernel(const TcParams p) {
  extern __shared__ uint8_t tc_smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(tc_smem_raw) + 1023) & ~(uintptr_t)1023);
  const uint32_t sb = smem_addr(sm);
  const uint32_t bars = sb + kBarOff;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kBarOff + 8 * kNumBars);
  volatile int* abort = reinterpret_cast<volatile int*>(sm + kBarOff + 8 * kNumBars + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int half = blockIdx.x & 1;
  const int rt = p.n_rt - 1 - (int)(blockIdx.x >> 1);
  const int r0 = rt * kTcRows;
  const int rlast = min(r0 + kTcRows, p.R) - 1;
  const int J = (p.qpos0 + rlast / p.H + kTcKeys) / kTcKeys;   // key tiles the tile's last row reaches

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNumBars; ++i) bar_init(bars + 8 * i, i == kPFull || i == kSRead ? 128 : 1);
    *abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(smem_addr(tmem_slot)),
                 "r"(512));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  pdl_launch_dependents();
  pdl_wait();

  if (warp == 0) {
    // ---- loader: the ring items in the MMA order (QK items of tile j, then
    // the V item of tile j - 1)
    if (lane == 0) {
      const uint8_t* qt = p.qws + (int64_t)rt * kTileBytes;
      uint32_t it = 0;
      bool ok = true;
      for (int j = 0; j <= J && ok; ++j) {
        for (int kb = (j < J ? 0 : kTcKB); kb <= kTcKB && ok; ++kb) {
          if (kb == kTcKB && j == 0) break;            // no V item before the first tile's
          const uint32_t s = it % kStages;
          if (it >= kStages && !bar_wait(bars + 8 * (kEmpty0 + s), ((it / kStages) & 1) ^ 1, p.wait_ns, abort)) {
            ok = false;
            break;
          }
          const uint32_t dst = sb + s * kStageBytes, full = bars + 8 * (kFull0 + s);
          bar_expect(full, kStageBytes);
          if (kb < kTcKB) {
            const uint8_t* kt = p.kws + (int64_t)j * kTileBytes;
            bulk_copy(dst, qt + (int64_t)kb * 2 * kBlk, 2 * kBlk, full);              // Q_hi, Q_lo
            bulk_copy(dst + 2 * kBlk, kt + (int64_t)kb * 2 * kBlk, 2 * kBlk, full);   // K_hi, K_lo
          } else {
            const uint8_t* kt = p.kws + (int64_t)(j - 1) * kTileBytes;
            for (int c = 0; c < 4; ++c)                                             // V: K_hi of the half
              bulk_copy(dst + c * kBlk, kt + (int64_t)(4 * half + c) * 2 * kBlk, kBlk, full);
          }
          ++it;
        }
      }
      if (!ok) {
        set_err(p.dev_err, MLA_DEVERR_TIMEOUT);
        *abort = 1;
      }
      // the copies in flight land before the CTA exits
      for (uint32_t s = 0; s < kStages; ++s)
        if (it > s) drain_wait(bars + 8 * (kFull0 + s), ((it - 1 - s) / kStages) & 1);
    }
  } else if (warp == 1) {
    // ---- MMA issuer: QK(j) into S once the softmax has read S(j - 1), then
    // PV(j - 1) (which keeps the pipe busy while the softmax reads S(j)), one
    // ring item each
    if (lane == 0) {
      constexpr uint32_t kIdQK = f16_idesc(kTcKeys, false), kIdQK2 = f16_idesc(2 * kTcKeys, false),
                         kIdPV = f16_idesc(256, true);
      uint32_t it = 0;
      bool ok = true;
      for (int j = 0; j <= J && ok; ++j) {
        if (j < J) {
          if (j >= 1 && !bar_wait(bars + 8 * kSRead, (j - 1) & 1, p.wait_ns, abort)) {
            ok = false;
            break;
          }
          const uint32_t d = tbase;
          for (int kb = 0; kb < kTcKB; ++kb, ++it) {
            const uint32_t s = it % kStages;
            if (!bar_wait(bars + 8 * (kFull0 + s), (it / kStages) & 1, p.wait_ns, abort)) {
              ok = false;
              break;
            }
            tc_fence_after();
            // B = [K_hi; K_lo] as one 256-row operand (the lo block follows
            // the hi block): Q_hi is read once for both of its products
            const uint32_t a_hi = sb + s * kStageBytes, a_lo = a_hi + kBlk, b_hi = a_hi + 2 * kBlk;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint64_t ah = sw128_desc(a_hi + 32 * k, 16, 1024), al = sw128_desc(a_lo + 32 * k, 16, 1024);
              const uint64_t bh = sw128_desc(b_hi + 32 * k, 16, 1024);
              umma(d, ah, bh, kIdQK2, (kb | k) != 0);    // columns 0..127: Q_hi K_hi; 128..255: Q_hi K_lo
              umma(d, al, bh, kIdQK, 1u);               // columns 0..127: + Q_lo K_hi
            }
            umma_commit(bars + 8 * (kEmpty0 + s));
          }
          if (!ok) break;
          umma_commit(bars + 8 * kSFull);
        }
        if (j >= 1) {
          const uint32_t jp = (uint32_t)(j - 1), s = it % kStages;
          if (!bar_wait(bars + 8 * kPFull, jp & 1, p.wait_ns, abort) ||
              !bar_wait(bars + 8 * (kFull0 + s), (it / kStages) & 1, p.wait_ns, abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t v = sb + s * kStageBytes;
#pragma unroll
          for (int k = 0; k < kTcKeys / 16; ++k) {
            const uint64_t a = sw128_desc(sb + kPOff + (k >> 2) * kBlk + (k & 3) * 32, 16, 1024);
            const uint64_t b = sw128_desc(v + k * 2048, kBlk, 1024);
            umma(tbase + 256, a, b, kIdPV, (jp | (uint32_t)k) != 0);
          }
          umma_commit(bars + 8 * (kEmpty0 + s));
          umma_commit(bars + 8 * kPVDone);
          ++it;
        }
      }
      if (!ok) {
        set_err(p.dev_err, MLA_DEVERR_TIMEOUT);
        *abort = 1;
      }
      // every MMA issued completes before TMEM is freed
      umma_commit(bars + 8 * kFin);
      drain_wait(bars + 8 * kFin, 0);
    }
  } else {
    // ---- softmax warpgroup: row lr of the tile, TMEM lane lr
    const int q = warp & 3;
    const int lr = 32 * q + lane;
    const int row = r0 + lr;
    const bool live = row < p.R;
    const int qpos = p.qpos0 + (live ? row : rlast) / p.H;
    const uint32_t tl = tbase + ((uint32_t)(32 * q) << 16);
    uint8_t* prow = sm + kPOff + lr * 128;
    float m_run = -INFINITY, l = 0.f, e2 = 0.f;
    bool ok = true;
    for (int j = 0; j < J; ++j) {
      if (!warp_wait(bars + 8 * kSFull, j & 1, p.wait_ns, abort)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float x[kTcKeys];
#pragma unroll
      for (int c = 0; c < kTcKeys / 32; ++c) {
        float y[32];
        tmem_load(tl + (uint32_t)(32 * c), x + 32 * c);
        tmem_load(tl + (uint32_t)(kTcKeys + 32 * c), y);
#pragma unroll
        for (int i = 0; i < 32; ++i) x[32 * c + i] += y[i];
      }
      // S is in registers: QK(j + 1) may overwrite it
      tc_fence_before();
      bar_arrive(bars + 8 * kSRead);
      const int kpos0 = j * kTcKeys;
      float mx = -INFINITY;
      if (kpos0 + kTcKeys - 1 > qpos) {
#pragma unroll
        for (int c = 0; c < kTcKeys; ++c) {
          x[c] = kpos0 + c > qpos ? -INFINITY : x[c] * p.scale_log2;
          mx = fmaxf(mx, x[c]);
        }
      } else {
#pragma unroll
        for (int c = 0; c < kTcKeys; ++c) {
          x[c] *= p.scale_log2;
          mx = fmaxf(mx, x[c]);
        }
      }
      __syncwarp();
      const float m_new = fmaxf(m_run, mx);
      const bool raise = m_new > m_run + kRescaleSlack;
      const float m_use = raise ? m_new : m_run;
      const float alpha = raise ? exp2f(m_run - m_new) : 1.f;
      // P and O are free once PV(j - 1) has completed
      if (j >= 1 && !warp_wait(bars + 8 * kPVDone, (j - 1) & 1, p.wait_ns, abort)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (j >= 1 && __any_sync(0xffffffffu, raise)) {
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
          float o[32];
          tmem_load(tl + 256 + 32 * c, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= alpha;
          tmem_store(tl + 256 + 32 * c, o);
        }
      }
      float rs = 0.f, es = 0.f;
#pragma unroll
      for (int c8 = 0; c8 < kTcKeys / 8; ++c8) {
        float pv[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          pv[k] = exp2f(x[8 * c8 + k] - m_use);
          rs += pv[k];
        }
        if (p.risk) {
          const float4 ma = __ldg(reinterpret_cast<const float4*>(p.mt + kpos0 + 8 * c8));
          const float4 mb = __ldg(reinterpret_cast<const float4*>(p.mt + kpos0 + 8 * c8 + 4));
          const float mv[8] = {ma.x, ma.y, ma.z, ma.w, mb.x, mb.y, mb.z, mb.w};
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const float w = pv[k] * mv[k];
            es = fmaf(w, w, es);
          }
        }
        *reinterpret_cast<uint4*>(prow + (c8 >> 3) * kBlk + (((c8 & 7) ^ (lr & 7)) << 4)) =
            make_uint4(pack_half2(pv[0], pv[1]), pack_half2(pv[2], pv[3]), pack_half2(pv[4], pv[5]),
                       pack_half2(pv[6], pv[7]));
      }
      l = fmaf(l, alpha, rs);
      e2 = fmaf(e2, alpha * alpha, es);
      m_run = m_use;
      asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
      tc_fence_before();
      bar_arrive(bars + 8 * kPFull);
    }
    // ---- epilogue: O_half / l, the row's log-sum-exp and check figures
    if (ok && !warp_wait(bars + 8 * kPVDone, (J - 1) & 1, p.wait_ns, abort)) ok = false;
    if (ok) {
      tc_fence_after();
      const float inv = 1.f / l;
      float om = 0.f;
      float* orow = p.o_lat + (int64_t)(live ? row : 0) * kDc + 256 * half;
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {
        float o[32];
        __syncwarp();
        tmem_load(tl + 256 + 32 * c, o);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          o[i] *= inv;
          om = fmaxf(om, fabsf(o[i]));
        }
        if (live) {
#pragma unroll
          for (int v = 0; v < 8; ++v)
            reinterpret_cast<float4*>(orow + 32 * c)[v] = make_float4(o[4 * v], o[4 * v + 1], o[4 * v + 2], o[4 * v + 3]);
        }
      }
      if (live) {
        if (half == 0) {
          if (p.lse) p.lse[row] = (m_run + log2f(l)) * 0.69314718055994531f;
          if (p.risk) p.risk_out[row] = sqrtf(e2) / l;
        }
        p.omax[2 * row + half] = om;
      }
    } else {
      // given up: the row reads as attention over nothing (o_lat 0, lse
      // -inf, nothing for the fixup to check), finite like the decode's
      // empty partials
      set_err(p.dev_err, MLA_DEVERR_TIMEOUT);
      *abort = 1;
      if (live) {
        float* orow = p.o_lat + (int64_t)row * kDc + 256 * half;
        for (int v = 0; v < 64; ++v) reinterpret_cast<float4*>(orow)[v] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (half == 0) {
          if (p.lse) p.lse[row] = -INFINITY;
          p.risk_out[row] = 0.f;
        }
        p.omax[2 * row + half] = 0.f;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tbase), "r"(512));
  }
}

// short_rows_kernel: grid (ceil(n_short / 4), H / 8), block kSRThreads.
// The exact fp32 attention of the query rows that see fewer than 256
// positions (query tokens i < n_short of the slice, position qpos0 + i):
// the rule every prefill and decode path shares for short rows, where the
// fp16 roundings of P and V do not average out.  CTA (x, y) takes tokens
// 4x .. 4x + 3 and heads 8y .. 8y + 7 (32 rows); the positions' x_hat come
// from the fp32 table the key pass wrote ([256][576]), 32 at a time.  Warp w
// owns rows 2w, 2w + 1: lane k scores position k of the block for both
// (float4 loads, consecutive rows of the table tile: conflict-free with the
// padded stride), the warp runs the two rows' online softmax by shuffles
// (log2 domain), and lane L accumulates channels 4L + 128m (m = 0..3) of O
// for both rows, so a float4 load of a position's channels covers 512
// contiguous bytes.
constexpr int kSRThreads = 512;
constexpr int kSRTok = 4, kSRHeads = 8, kSRRows = kSRTok * kSRHeads, kSRKeys = 32;
constexpr int kSRStride = kDc + kDr + 4;        // padded row (floats): stride / 4 odd
constexpr int kSRSmem = (int)sizeof(float) * (kSRRows + kSRKeys) * kSRStride;
static_assert(kSRThreads / 32 * 2 == kSRRows, "a warp per row pair");

__global__ void __launch_bounds__(kSRThreads, 1) short_rows_kernel(const float* table, const float* q_lat,
                                                                   const uint16_t* q_pe, int H, int n_short,
                                                                   int qpos0, float scale_log2, float* o_lat,
                                                                   float* lse) {
  extern __shared__ float sr_smem[];
  float* sQ = sr_smem;                              // [32 rows][kSRStride]
  float* sX = sQ + kSRRows * kSRStride;             // [32 positions][kSRStride]
  pdl_launch_dependents();
  pdl_wait();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int i0 = blockIdx.x * kSRTok, h0 = blockIdx.y * kSRHeads;
  // row r = (token i0 + r / 8, head h0 + r % 8)
  for (int idx = tid; idx < kSRRows * (kDc + kDr); idx += kSRThreads) {
    const int r = idx / (kDc + kDr), c = idx % (kDc + kDr);
    const int i = min(i0 + r / kSRHeads, n_short - 1), h = h0 + r % kSRHeads;
    const size_t row = (size_t)i * H + h;
    sQ[r * kSRStride + c] = c < kDc ? q_lat[row * kDc + c] : bf16f(q_pe[row * kDr + c - kDc]);
  }
  const int maxlen = qpos0 + min(i0 + kSRTok, n_short);    // positions the CTA's longest row sees (< 256)
  const int r0 = 2 * warp;                                  // this warp's rows r0, r0 + 1
  const int len0 = qpos0 + min(i0 + r0 / kSRHeads, n_short - 1) + 1;
  const int len1 = qpos0 + min(i0 + (r0 + 1) / kSRHeads, n_short - 1) + 1;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float acc0[16], acc1[16];
#pragma unroll
  for (int v = 0; v < 16; ++v) acc0[v] = acc1[v] = 0.f;
  for (int t0 = 0; t0 < maxlen; t0 += kSRKeys) {
    __syncthreads();                                // the previous block's readers of sX are done
    for (int idx = tid; idx < kSRKeys * (kDc + kDr) / 4; idx += kSRThreads) {
      const int k = idx / ((kDc + kDr) / 4), c4 = 4 * (idx % ((kDc + kDr) / 4));
      *reinterpret_cast<float4*>(sX + k * kSRStride + c4) =
          *reinterpret_cast<const float4*>(table + (size_t)(t0 + k) * (kDc + kDr) + c4);
    }
    __syncthreads();
    // scores of position t0 + lane for rows r0, r0 + 1
    float a = 0.f, b = 0.f;
    const float* q0 = sQ + r0 * kSRStride;
    const float* xk = sX + lane * kSRStride;
#pragma unroll 4
    for (int c = 0; c < kDc + kDr; c += 4) {
      const float4 x = *reinterpret_cast<const float4*>(xk + c);
      const float4 u = *reinterpret_cast<const float4*>(q0 + c);
      const float4 w = *reinterpret_cast<const float4*>(q0 + kSRStride + c);
      a = fmaf(u.x, x.x, fmaf(u.y, x.y, fmaf(u.z, x.z, fmaf(u.w, x.w, a))));
      b = fmaf(w.x, x.x, fmaf(w.y, x.y, fmaf(w.z, x.z, fmaf(w.w, x.w, b))));
    }
    const int k = t0 + lane;
    a = k < len0 ? a * scale_log2 : -INFINITY;
    b = k < len1 ? b * scale_log2 : -INFINITY;
    float ma = a, mb = b;
#pragma unroll
    for (int off = 16; off; off >>= 1) {
      ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, off));
      mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, off));
    }
    const float n0 = fmaxf(m0, ma), n1 = fmaxf(m1, mb);      // position 0 is always visible: finite
    const float al0 = exp2f(m0 - n0), al1 = exp2f(m1 - n1);
    const float pa = exp2f(a - n0), pb = exp2f(b - n1);
    float sa = pa, sb = pb;
#pragma unroll
    for (int off = 16; off; off >>= 1) {
      sa += __shfl_xor_sync(0xffffffffu, sa, off);
      sb += __shfl_xor_sync(0xffffffffu, sb, off);
    }
    l0 = fmaf(l0, al0, sa);
    l1 = fmaf(l1, al1, sb);
    m0 = n0;
    m1 = n1;
#pragma unroll
    for (int v = 0; v < 16; ++v) {
      acc0[v] *= al0;
      acc1[v] *= al1;
    }
    // O += P X: position j's weights come from lane j by shuffle
    const int kend = min(kSRKeys, maxlen - t0);
    for (int j = 0; j < kend; ++j) {
      const float w0 = __shfl_sync(0xffffffffu, pa, j), w1 = __shfl_sync(0xffffffffu, pb, j);
      const float* xr = sX + j * kSRStride + 4 * lane;
#pragma unroll
      for (int mq = 0; mq < 4; ++mq) {
        const float4 x = *reinterpret_cast<const float4*>(xr + 128 * mq);
        acc0[4 * mq] = fmaf(w0, x.x, acc0[4 * mq]);
        acc0[4 * mq + 1] = fmaf(w0, x.y, acc0[4 * mq + 1]);
        acc0[4 * mq + 2] = fmaf(w0, x.z, acc0[4 * mq + 2]);
        acc0[4 * mq + 3] = fmaf(w0, x.w, acc0[4 * mq + 3]);
        acc1[4 * mq] = fmaf(w1, x.x, acc1[4 * mq]);
        acc1[4 * mq + 1] = fmaf(w1, x.y, acc1[4 * mq + 1]);
        acc1[4 * mq + 2] = fmaf(w1, x.z, acc1[4 * mq + 2]);
        acc1[4 * mq + 3] = fmaf(w1, x.w, acc1[4 * mq + 3]);
      }
    }
  }
  const int ia = i0 + r0 / kSRHeads, ib = i0 + (r0 + 1) / kSRHeads;
  const int ha = h0 + r0 % kSRHeads, hb = h0 + (r0 + 1) % kSRHeads;
  if (lane == 0 && lse) {
    if (ia < n_short) lse[(size_t)ia * H + ha] = (m0 + log2f(l0)) * 0.69314718055994531f;
    if (ib < n_short) lse[(size_t)ib * H + hb] = (m1 + log2f(l1)) * 0.69314718055994531f;
  }
  const float inv0 = 1.f / l0, inv1 = 1.f / l1;
#pragma unroll
  for (int mq = 0; mq < 4; ++mq) {
    if (ia < n_short)
      *reinterpret_cast<float4*>(o_lat + ((size_t)ia * H + ha) * kDc + 4 * lane + 128 * mq) =
          make_float4(acc0[4 * mq] * inv0, acc0[4 * mq + 1] * inv0, acc0[4 * mq + 2] * inv0,
                      acc0[4 * mq + 3] * inv0);
    if (ib < n_short)
      *reinterpret_cast<float4*>(o_lat + ((size_t)ib * H + hb) * kDc + 4 * lane + 128 * mq) =
          make_float4(acc1[4 * mq] * inv1, acc1[4 * mq + 1] * inv1, acc1[4 * mq + 2] * inv1,
                      acc1[4 * mq + 3] * inv1);
  }
}

// Raises the kernels' shared-memory limit once per device.
mla_status tc_configure() {
  static int configured[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && configured[dev]) return MLA_OK;
  const mla_status st =
      cuda_status(cudaFuncSetAttribute(prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem));
  if (st == MLA_OK && dev >= 0 && dev < 64) configured[dev] = 1;
  return st;
}

}  // namespace

mla_status launch_q_split(const float* q_lat, const uint16_t* q_pe, int R, int n_rt, uint8_t* qws,
                          cudaStream_t stream) {
  const int64_t pieces = (int64_t)n_rt * kTcRows * ((kDc + kDr) / 8);
  const int64_t blocks = (pieces + 255) / 256;
  const int grid = (int)(blocks < 8 * 152 ? blocks : 8 * 152);
  return cuda_status(launch_pdl(q_split_kernel, dim3(grid), dim3(256), 0, stream, q_lat, q_pe, R, n_rt, qws));
}

mla_status launch_short_rows(const float* table, const float* q_lat, const uint16_t* q_pe, int H, int n_short,
                             int qpos0, float scale_log2, float* o_lat, float* lse, cudaStream_t stream) {
  static int configured[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    const mla_status st =
        cuda_status(cudaFuncSetAttribute(short_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSRSmem));
    if (st != MLA_OK) return st;
    if (dev >= 0 && dev < 64) configured[dev] = 1;
  }
  return cuda_status(launch_pdl(short_rows_kernel, dim3((n_short + kSRTok - 1) / kSRTok, H / kSRHeads),
                                dim3(kSRThreads), kSRSmem, stream, table, q_lat, q_pe, H, n_short, qpos0,
                                scale_log2, o_lat, lse));
}

mla_status launch_prefill_tc(const TcParams& p, cudaStream_t stream) {
  const mla_status st = tc_configure();
  if (st != MLA_OK) return st;
  return cuda_status(launch_pdl(prefill_tc_kernel, dim3(2 * p.n_rt), dim3(kTcThreads), kTcSmem, stream, p));
}

}  // namespace mla
