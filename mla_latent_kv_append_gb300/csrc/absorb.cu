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
// 16-row tiles.  Their cost is reading the weights once (2 MiB per 16 heads
// each), so a CTA covers one head and one column tile.
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

}  // namespace

// Large batches (a prefill chunk's queries) split their 16-row tiles over
// grid z, so that more CTAs stream them; each CTA still takes 8 or more
// tiles per weight tile it loads.
static int batch_splits(int B) {
  const int tiles = (B + 15) / 16, z = tiles / 8;
  return z < 1 ? 1 : (z > 32 ? 32 : z);
}

mla_status launch_q_absorb(const uint16_t* q_nope, const uint16_t* w_uk, float* q_lat, int B, int H,
                           cudaStream_t stream) {
  return cuda_status(launch_pdl(q_absorb_kernel, dim3(H, kDc / kAbN, batch_splits(B)), dim3(128), 0, stream, q_nope,
                                w_uk, q_lat, B, H));
}

mla_status launch_out_unabsorb(const float* o_lat, const uint16_t* w_uv, float* o, int B, int H,
                               cudaStream_t stream) {
  return cuda_status(launch_pdl(out_unabsorb_kernel, dim3(H, kDv / kUnN, batch_splits(B)), dim3(128), 0, stream, o_lat,
                                w_uv, o, B, H));
}

}  // namespace mla
