// mla_q_absorb and mla_out_unabsorb: the two weight-absorption projections.
//
// juejin tutorial "DeepSeek的MLA技术：极致压缩KV Cache的创新方案", "步骤2":
// K_i = C^KV W_i^upK and V_i = C^KV W_i^upV.  Scores q.K_i = (q W_i^upK^T) . C^KV
// and outputs p V_i = (p C^KV) W_i^upV, so the per-head up-projections move
// onto the query (q_lat = q_nope @ W_UK[h], W_UK[h] = (W_i^upK)^T, [128, 512])
// and onto the attention output (o = o_lat @ W_UV[h], [512, 128]).
//
// Both are per-head GEMMs with M = batch (padded to 16), run on the tensor
// cores with mma.sync.m16n8k16 (bf16 in, fp32 accumulate).  The weight tile
// of a CTA is staged once in shared memory (rows padded so that ldmatrix is
// conflict-free) and read with ldmatrix.trans; the activations stream through
// 16-row tiles.  A decode batch's cost is reading the weights once (2 MiB per
// 16 heads each), so a CTA covers one head and one column tile; a prefill
// chunk's batch (512 rows or more) takes the *_big kernels, whose CTA keeps
// a head's whole weight and whose warps take whole row tiles.
//   absorb:   A = q_nope (bf16, exact), B = W_UK: products exact in fp32.
//   unabsorb: A = o_lat (fp32) split into three bf16 pieces (hi + mid + lo
//             carry all 24 significant bits), B = W_UV: three MMAs per step.
#include <cuda_bf16.h>

#include "mla_internal.cuh"

namespace mla {

namespace {

__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t* r) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;\n" : "=r"(r) : "f"(b), "f"(a));
  return r;
}
__device__ __forceinline__ float lo_f(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float hi_f(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

// fp32 pair -> three bf16 pairs whose sum reproduces the pair (24 bits)
__device__ __forceinline__ void split3(float a, float b, uint32_t& p0, uint32_t& p1, uint32_t& p2) {
  p0 = pack_bf16(a, b);
  const float ra = a - lo_f(p0), rb = b - hi_f(p0);
  p1 = pack_bf16(ra, rb);
  p2 = pack_bf16(ra - lo_f(p1), rb - hi_f(p1));
}

// ---------------------------------------------------------------------------
// q_absorb: grid (H, 512 / 64, batch splits), block 128.  Warp w computes columns
// n0 + 16w .. +15 of a 16-row tile; K = 128 in 8 k-steps.
// ---------------------------------------------------------------------------
constexpr int kAbN = 64;             // columns per CTA
constexpr int kAbWS = kAbN + 8;      // W tile row stride (bf16): 144 B
constexpr int kAbAS = kDn + 8;       // A tile row stride (bf16): 272 B

__global__ void __launch_bounds__(128) q_absorb_kernel(const uint16_t* __restrict__ q_nope,
                                                       const uint16_t* __restrict__ w_uk,
                                                       float* __restrict__ q_lat, int B, int H) {
  pdl_launch_dependents();
  __shared__ __align__(16) uint16_t ws[kDn * kAbWS];
  __shared__ __align__(16) uint16_t as[16 * kAbAS];
  const int h = blockIdx.x, n0 = blockIdx.y * kAbN;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, r = lane >> 2, j = lane & 3;
  // W_UK[h][k][n0 .. n0+63]: 128 rows x 8 chunks of 16 B.  No kernel of the
  // library writes the weights, so their fetch starts before the wait for
  // the previous kernel and overlaps its tail.
  const uint16_t* wsrc = w_uk + (size_t)h * kDn * kDc + n0;
  for (int i = tid; i < kDn * (kAbN / 8); i += 128) {
    const int k = i >> 3, c = i & 7;
    *reinterpret_cast<uint4*>(ws + k * kAbWS + 8 * c) = *reinterpret_cast<const uint4*>(wsrc + (size_t)k * kDc + 8 * c);
  }
  pdl_wait();
  const uint32_t a_base = smem_addr(as) + (((lane & 7) + 8 * ((lane >> 3) & 1)) * kAbAS + 8 * (lane >> 4)) * 2;
  const uint32_t b_base =
      smem_addr(ws) + (((lane & 7) + 8 * ((lane >> 3) & 1)) * kAbWS + 16 * warp + 8 * (lane >> 4)) * 2;
  const int tiles = (B + 15) / 16;
  const int t_lo = (int)((int64_t)tiles * blockIdx.z / gridDim.z);
  const int t_hi = (int)((int64_t)tiles * (blockIdx.z + 1) / gridDim.z);
  for (int b0 = 16 * t_lo; b0 < 16 * t_hi; b0 += 16) {
    __syncthreads();   // previous tile's readers are done (and the W tile is in place)
    for (int i = tid; i < 16 * (kDn / 8); i += 128) {
      const int m = i >> 4, c = i & 15;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (b0 + m < B) v = *reinterpret_cast<const uint4*>(q_nope + ((size_t)(b0 + m) * H + h) * kDn + 8 * c);
      *reinterpret_cast<uint4*>(as + m * kAbAS + 8 * c) = v;
    }
    __syncthreads();
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int ks = 0; ks < kDn / 16; ++ks) {
      uint32_t a[4], bf[4];
      ldsm_x4(a_base + 32 * ks, a);
      ldsm_x4_t(b_base + 16 * ks * kAbWS * 2, bf);
      mma_bf16(acc[0], a, bf[0], bf[1]);
      mma_bf16(acc[1], a, bf[2], bf[3]);
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int col = n0 + 16 * warp + 8 * nt + 2 * j;
      if (b0 + r < B)
        *reinterpret_cast<float2*>(q_lat + ((size_t)(b0 + r) * H + h) * kDc + col) = make_float2(acc[nt][0], acc[nt][1]);
      if (b0 + r + 8 < B)
        *reinterpret_cast<float2*>(q_lat + ((size_t)(b0 + r + 8) * H + h) * kDc + col) =
            make_float2(acc[nt][2], acc[nt][3]);
    }
  }
}

// ---------------------------------------------------------------------------
// out_unabsorb: grid (H, 128 / 16, batch splits), block 128.  Warp w takes K rows
// 128w .. 128w+127 for the CTA's 16 columns; all of the warp's A values are
// loaded up front (independent loads), and the 4 partial tiles are summed in
// shared memory.
// ---------------------------------------------------------------------------
constexpr int kUnN = 16;             // columns per CTA
constexpr int kUnWS = kUnN + 8;      // W tile row stride (bf16): 48 B, conflict-free ldmatrix

__global__ void __launch_bounds__(128) out_unabsorb_kernel(const float* __restrict__ o_lat,
                                                           const uint16_t* __restrict__ w_uv,
                                                           float* __restrict__ o, int B, int H) {
  pdl_launch_dependents();
  __shared__ __align__(16) uint16_t ws[kDc * kUnWS];
  __shared__ float part[4][16][kUnN];
  const int h = blockIdx.x, v0 = blockIdx.y * kUnN;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, r = lane >> 2, j = lane & 3;
  // the weight tile before the wait for the previous kernel (no kernel of
  // the library writes the weights): its fetch overlaps that kernel's tail
  const uint16_t* wsrc = w_uv + (size_t)h * kDc * kDv + v0;
  for (int i = tid; i < kDc * (kUnN / 8); i += 128) {
    const int k = i >> 1, c = i & 1;
    *reinterpret_cast<uint4*>(ws + k * kUnWS + 8 * c) = *reinterpret_cast<const uint4*>(wsrc + (size_t)k * kDv + 8 * c);
  }
  pdl_wait();
  const uint32_t b_base = smem_addr(ws) + (((lane & 7) + 8 * ((lane >> 3) & 1)) * kUnWS + 8 * (lane >> 4)) * 2;
  const int tiles = (B + 15) / 16;
  const int t_lo = (int)((int64_t)tiles * blockIdx.z / gridDim.z);
  const int t_hi = (int)((int64_t)tiles * (blockIdx.z + 1) / gridDim.z);
  for (int b0 = 16 * t_lo; b0 < 16 * t_hi; b0 += 16) {
    const float* a0p = o_lat + ((size_t)(b0 + r) * H + h) * kDc + 128 * warp;
    const float* a1p = o_lat + ((size_t)(b0 + r + 8) * H + h) * kDc + 128 * warp;
    const bool ok0 = b0 + r < B, ok1 = b0 + r + 8 < B;
    float2 xa[8][4];
    const float2 z = make_float2(0.f, 0.f);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      xa[ks][0] = ok0 ? *reinterpret_cast<const float2*>(a0p + 16 * ks + 2 * j) : z;
      xa[ks][1] = ok1 ? *reinterpret_cast<const float2*>(a1p + 16 * ks + 2 * j) : z;
      xa[ks][2] = ok0 ? *reinterpret_cast<const float2*>(a0p + 16 * ks + 8 + 2 * j) : z;
      xa[ks][3] = ok1 ? *reinterpret_cast<const float2*>(a1p + 16 * ks + 8 + 2 * j) : z;
    }
    __syncthreads();     // W tile in place; previous tile's partials consumed
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      uint32_t a[3][4];
#pragma unroll
      for (int e = 0; e < 4; ++e) split3(xa[ks][e].x, xa[ks][e].y, a[0][e], a[1][e], a[2][e]);
      uint32_t bf[4];
      ldsm_x4_t(b_base + (128 * warp + 16 * ks) * kUnWS * 2, bf);
#pragma unroll
      for (int part3 = 0; part3 < 3; ++part3) {
        mma_bf16(acc[0], a[part3], bf[0], bf[1]);
        mma_bf16(acc[1], a[part3], bf[2], bf[3]);
      }
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      part[warp][r][8 * nt + 2 * j] = acc[nt][0];
      part[warp][r][8 * nt + 2 * j + 1] = acc[nt][1];
      part[warp][r + 8][8 * nt + 2 * j] = acc[nt][2];
      part[warp][r + 8][8 * nt + 2 * j + 1] = acc[nt][3];
    }
    __syncthreads();
    for (int i = tid; i < 16 * kUnN; i += 128) {
      const int m = i / kUnN, c = i % kUnN;
      if (b0 + m < B)
        o[((size_t)(b0 + m) * H + h) * kDv + v0 + c] = (part[0][m][c] + part[1][m][c]) + (part[2][m][c] + part[3][m][c]);
    }
  }
}

// ---------------------------------------------------------------------------
// Batches of a prefill chunk (B >= kBigB): a CTA keeps the whole weight of
// one head in shared memory and its eight warps each take whole 16-row
// tiles (all output columns, the whole contraction), so every activation
// row is read and (unabsorb) split once; the small-batch kernels above read
// each weight tile once instead, which is what a decode batch is bound by.
// The work is H x U units (head-major; a unit is a 16-row tile, or for the
// absorb a tile's quarter of the 512 output columns).  Of G CTAs (about one
// per SM, big_grid), CTA c takes the contiguous units [H U c / G,
// H U (c + 1) / G) and warp w every eighth unit of each head in that range;
// the CTA loads a head's weight when its range enters the head.
// ---------------------------------------------------------------------------
constexpr int kBigB = 512;
constexpr int kBigThreads = 256;
constexpr int kBigAbWS = kDc + 8;                                  // W_UK row stride (bf16): 1040 B
constexpr int kBigUnWS = kDv + 8;                                  // W_UV row stride (bf16): 272 B
constexpr int kBigAbSmem = kDn * kBigAbWS * 2;                     // 133,120 B
constexpr int kBigUnSmem = kDc * kBigUnWS * 2;                     // 139,264 B

// q_lat tile: 16 rows x 128 columns (quarter cq of 512) per warp unit; the
// A fragments (bf16 pairs of q_nope) come straight from global memory.
__global__ void __launch_bounds__(kBigThreads, 1) q_absorb_big_kernel(const uint16_t* __restrict__ q_nope,
                                                                      const uint16_t* __restrict__ w_uk,
                                                                      float* __restrict__ q_lat, int B, int H) {
  extern __shared__ __align__(16) uint16_t big_ws[];
  pdl_launch_dependents();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, r = lane >> 2, j = lane & 3;
  const uint32_t b_base = smem_addr(big_ws) + (((lane & 7) + 8 * ((lane >> 3) & 1)) * kBigAbWS + 8 * (lane >> 4)) * 2;
  const int tiles = (B + 15) / 16;
  const int64_t per_head = 4 * (int64_t)tiles, total = per_head * H;
  const int64_t u_lo = total * blockIdx.x / gridDim.x, u_hi = total * (blockIdx.x + 1) / gridDim.x;
  bool waited = false;
  for (int h = (int)(u_lo / per_head); (int64_t)h * per_head < u_hi; ++h) {
    // the previous head's units are done with the weight before it is replaced
    if (waited) __syncthreads();
    const uint16_t* wsrc = w_uk + (size_t)h * kDn * kDc;
    for (int i = tid; i < kDn * (kDc / 8); i += kBigThreads) {
      const int k = i / (kDc / 8), c = i % (kDc / 8);
      *reinterpret_cast<uint4*>(big_ws + k * kBigAbWS + 8 * c) =
          *reinterpret_cast<const uint4*>(wsrc + (size_t)k * kDc + 8 * c);
    }
    __syncthreads();
    if (!waited) {
      pdl_wait();                                   // no kernel writes the weights: only q_nope waits
      waited = true;
    }
    const int64_t h0 = (int64_t)h * per_head;
    const int v_lo = (int)((u_lo > h0 ? u_lo : h0) - h0);
    const int v_hi = (int)((u_hi < h0 + per_head ? u_hi : h0 + per_head) - h0);
    for (int u = v_lo + warp; u < v_hi; u += kBigThreads / 32) {
      const int b0 = 16 * (u >> 2), cq = 128 * (u & 3);
      const bool ok0 = b0 + r < B, ok1 = b0 + r + 8 < B;
      const uint32_t* a0p = reinterpret_cast<const uint32_t*>(q_nope + ((size_t)(b0 + r) * H + h) * kDn) + j;
      const uint32_t* a1p = reinterpret_cast<const uint32_t*>(q_nope + ((size_t)(b0 + r + 8) * H + h) * kDn) + j;
      uint32_t a[8][4];
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        a[ks][0] = ok0 ? a0p[8 * ks] : 0u;
        a[ks][1] = ok1 ? a1p[8 * ks] : 0u;
        a[ks][2] = ok0 ? a0p[8 * ks + 4] : 0u;
        a[ks][3] = ok1 ? a1p[8 * ks + 4] : 0u;
      }
      float acc[16][4];
#pragma unroll
      for (int nt = 0; nt < 16; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
        for (int pr = 0; pr < 8; ++pr) {
          uint32_t bf[4];
          ldsm_x4_t(b_base + (16 * ks * kBigAbWS + cq + 16 * pr) * 2, bf);
          mma_bf16(acc[2 * pr], a[ks], bf[0], bf[1]);
          mma_bf16(acc[2 * pr + 1], a[ks], bf[2], bf[3]);
        }
      }
#pragma unroll
      for (int nt = 0; nt < 16; ++nt) {
        const int col = cq + 8 * nt + 2 * j;
        if (ok0)
          *reinterpret_cast<float2*>(q_lat + ((size_t)(b0 + r) * H + h) * kDc + col) =
              make_float2(acc[nt][0], acc[nt][1]);
        if (ok1)
          *reinterpret_cast<float2*>(q_lat + ((size_t)(b0 + r + 8) * H + h) * kDc + col) =
              make_float2(acc[nt][2], acc[nt][3]);
      }
    }
  }
  if (!waited) pdl_wait();
}

// o tile: 16 rows x all 128 columns per warp unit, K = 512 in 32 steps; the
// fp32 A fragments come from global memory one step ahead and are split
// into three bf16 pieces once.
__global__ void __launch_bounds__(kBigThreads, 1) out_unabsorb_big_kernel(const float* __restrict__ o_lat,
                                                                          const uint16_t* __restrict__ w_uv,
                                                                          float* __restrict__ o, int B, int H) {
  extern __shared__ __align__(16) uint16_t big_ws[];
  pdl_launch_dependents();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, r = lane >> 2, j = lane & 3;
  const uint32_t b_base = smem_addr(big_ws) + (((lane & 7) + 8 * ((lane >> 3) & 1)) * kBigUnWS + 8 * (lane >> 4)) * 2;
  const int64_t per_head = (B + 15) / 16, total = per_head * H;
  const int64_t u_lo = total * blockIdx.x / gridDim.x, u_hi = total * (blockIdx.x + 1) / gridDim.x;
  const float2 z = make_float2(0.f, 0.f);
  bool waited = false;
  for (int h = (int)(u_lo / per_head); (int64_t)h * per_head < u_hi; ++h) {
    if (waited) __syncthreads();
    const uint16_t* wsrc = w_uv + (size_t)h * kDc * kDv;
    for (int i = tid; i < kDc * (kDv / 8); i += kBigThreads) {
      const int k = i / (kDv / 8), c = i % (kDv / 8);
      *reinterpret_cast<uint4*>(big_ws + k * kBigUnWS + 8 * c) =
          *reinterpret_cast<const uint4*>(wsrc + (size_t)k * kDv + 8 * c);
    }
    __syncthreads();
    if (!waited) {
      pdl_wait();
      waited = true;
    }
    const int64_t h0 = (int64_t)h * per_head;
    const int t_lo = (int)((u_lo > h0 ? u_lo : h0) - h0);
    const int t_hi = (int)((u_hi < h0 + per_head ? u_hi : h0 + per_head) - h0);
    for (int t = t_lo + warp; t < t_hi; t += kBigThreads / 32) {
      const int b0 = 16 * t;
      const bool ok0 = b0 + r < B, ok1 = b0 + r + 8 < B;
      const float* a0p = o_lat + ((size_t)(b0 + r) * H + h) * kDc + 2 * j;
      const float* a1p = o_lat + ((size_t)(b0 + r + 8) * H + h) * kDc + 2 * j;
      float acc[16][4];
#pragma unroll
      for (int nt = 0; nt < 16; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
      float2 x[4];
      x[0] = ok0 ? *reinterpret_cast<const float2*>(a0p) : z;
      x[1] = ok1 ? *reinterpret_cast<const float2*>(a1p) : z;
      x[2] = ok0 ? *reinterpret_cast<const float2*>(a0p + 8) : z;
      x[3] = ok1 ? *reinterpret_cast<const float2*>(a1p + 8) : z;
#pragma unroll 1
      for (int ks = 0; ks < kDc / 16; ++ks) {
        uint32_t a[3][4];
#pragma unroll
        for (int e = 0; e < 4; ++e) split3(x[e].x, x[e].y, a[0][e], a[1][e], a[2][e]);
        if (ks + 1 < kDc / 16) {                    // the next step's fragments, in flight during this one
          const int o1 = 16 * (ks + 1);
          x[0] = ok0 ? *reinterpret_cast<const float2*>(a0p + o1) : z;
          x[1] = ok1 ? *reinterpret_cast<const float2*>(a1p + o1) : z;
          x[2] = ok0 ? *reinterpret_cast<const float2*>(a0p + o1 + 8) : z;
          x[3] = ok1 ? *reinterpret_cast<const float2*>(a1p + o1 + 8) : z;
        }
#pragma unroll
        for (int pr = 0; pr < 8; ++pr) {
          uint32_t bf[4];
          ldsm_x4_t(b_base + (16 * ks * kBigUnWS + 16 * pr) * 2, bf);
#pragma unroll
          for (int part3 = 0; part3 < 3; ++part3) {
            mma_bf16(acc[2 * pr], a[part3], bf[0], bf[1]);
            mma_bf16(acc[2 * pr + 1], a[part3], bf[2], bf[3]);
          }
        }
      }
#pragma unroll
      for (int nt = 0; nt < 16; ++nt) {
        const int col = 8 * nt + 2 * j;
        if (ok0)
          *reinterpret_cast<float2*>(o + ((size_t)(b0 + r) * H + h) * kDv + col) = make_float2(acc[nt][0], acc[nt][1]);
        if (ok1)
          *reinterpret_cast<float2*>(o + ((size_t)(b0 + r + 8) * H + h) * kDv + col) =
              make_float2(acc[nt][2], acc[nt][3]);
      }
    }
  }
  if (!waited) pdl_wait();
}

// CTAs of the large-batch kernels.  H * floor(SMs / H) CTAs split every head
// evenly (no CTA loads two weights); when that leaves more than a tenth of
// the SMs idle and each CTA still gets 64 units or more, one CTA per SM,
// whose ranges may cross a head boundary (a second weight load).
int big_grid(int64_t units, int H) {
  const int sms = device_sm_count() > 0 ? device_sm_count() : 152;
  const int64_t aligned = (int64_t)H * (sms / H);
  int64_t g = aligned;
  if (aligned == 0 || (10 * aligned < 9 * (int64_t)sms && units >= 64 * (int64_t)sms)) g = sms;
  return (int)(units < g ? (units > 0 ? units : 1) : g);
}

}  // namespace

// Large batches (a prefill chunk's queries) split their 16-row tiles over
// grid z, so that more CTAs stream them; each CTA still takes 8 or more
// tiles per weight tile it loads.
static int batch_splits(int B) {
  const int tiles = (B + 15) / 16, z = tiles / 8;
  return z < 1 ? 1 : (z > 32 ? 32 : z);
}

// Raises a kernel's dynamic shared-memory limit once per device.
template <typename K>
static mla_status allow_big_smem(K kernel, int bytes, int* configured) {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && configured[dev]) return MLA_OK;
  const mla_status st = cuda_status(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes));
  if (st == MLA_OK && dev >= 0 && dev < 64) configured[dev] = 1;
  return st;
}

mla_status launch_q_absorb(const uint16_t* q_nope, const uint16_t* w_uk, float* q_lat, int B, int H,
                           cudaStream_t stream) {
  if (B >= kBigB) {
    static int configured[64] = {0};
    const mla_status st = allow_big_smem(q_absorb_big_kernel, kBigAbSmem, configured);
    if (st != MLA_OK) return st;
    const dim3 grid(big_grid(4 * (int64_t)((B + 15) / 16) * H, H));
    return cuda_status(launch_pdl(q_absorb_big_kernel, grid, dim3(kBigThreads), kBigAbSmem, stream, q_nope, w_uk,
                                  q_lat, B, H));
  }
  return cuda_status(launch_pdl(q_absorb_kernel, dim3(H, kDc / kAbN, batch_splits(B)), dim3(128), 0, stream, q_nope,
                                w_uk, q_lat, B, H));
}

mla_status launch_out_unabsorb(const float* o_lat, const uint16_t* w_uv, float* o, int B, int H,
                               cudaStream_t stream) {
  if (B >= kBigB) {
    static int configured[64] = {0};
    const mla_status st = allow_big_smem(out_unabsorb_big_kernel, kBigUnSmem, configured);
    if (st != MLA_OK) return st;
    const dim3 grid(big_grid((int64_t)((B + 15) / 16) * H, H));
    return cuda_status(launch_pdl(out_unabsorb_big_kernel, grid, dim3(kBigThreads), kBigUnSmem, stream, o_lat, w_uv,
                                  o, B, H));
  }
  return cuda_status(launch_pdl(out_unabsorb_kernel, dim3(H, kDv / kUnN, batch_splits(B)), dim3(128), 0, stream, o_lat,
                                w_uv, o, B, H));
}

}  // namespace mla
