// mla_q_absorb and mla_out_unabsorb: the two weight-absorption projections.
//
// juejin tutorial "DeepSeek的MLA技术：极致压缩KV Cache的创新方案", "步骤2":
// K_i = C^KV W_i^upK and V_i = C^KV W_i^upV.  Scores q.K_i = (q W_i^upK^T) . C^KV
// and outputs p V_i = (p C^KV) W_i^upV, so the per-head up-projections move
// onto the query (q_lat = q_nope @ W_UK[h], W_UK[h] = (W_i^upK)^T, [128, 512])
// and onto the attention output (o = o_lat @ W_UV[h], [512, 128]).
//
// Both are small per-head GEMMs whose cost is reading the weights once
// (2 MiB per 16 heads each).  One CTA per (head, output tile); the weight
// tile is streamed with coalesced loads along the output dimension while the
// activations of up to 16 (absorb) or 8 (unabsorb) sequences sit in shared
// memory; fp32 accumulation of exact bf16 x bf16 / fp32 x bf16 products.
#include "mla_internal.cuh"

namespace mla {

namespace {

constexpr int kAbsBt = 16;   // sequences per pass (absorb)
constexpr int kUnBt = 8;     // sequences per pass (unabsorb)

// grid (H, 512 / 64); block 256 = 4 k-slices x 64 output columns
__global__ void __launch_bounds__(256) q_absorb_kernel(const uint16_t* __restrict__ q_nope,
                                                       const uint16_t* __restrict__ w_uk,
                                                       float* __restrict__ q_lat, int B, int H) {
  __shared__ float qn[kAbsBt][kDn];
  __shared__ float part[4][kAbsBt][64];
  const int h = blockIdx.x, n0 = blockIdx.y * 64;
  const int tid = threadIdx.x, ks = tid >> 6, nl = tid & 63;
  const uint16_t* w = w_uk + (size_t)h * kDn * kDc + n0 + nl;
  for (int b0 = 0; b0 < B; b0 += kAbsBt) {
    for (int idx = tid; idx < kAbsBt * kDn; idx += 256) {
      const int j = idx / kDn, k = idx % kDn;
      qn[j][k] = (b0 + j < B) ? bf16f(q_nope[((size_t)(b0 + j) * H + h) * kDn + k]) : 0.f;
    }
    __syncthreads();
    float acc[kAbsBt];
#pragma unroll
    for (int j = 0; j < kAbsBt; ++j) acc[j] = 0.f;
    for (int k = ks * 32; k < ks * 32 + 32; ++k) {
      const float wv = bf16f(w[(size_t)k * kDc]);
#pragma unroll
      for (int j = 0; j < kAbsBt; ++j) acc[j] = fmaf(qn[j][k], wv, acc[j]);
    }
#pragma unroll
    for (int j = 0; j < kAbsBt; ++j) part[ks][j][nl] = acc[j];
    __syncthreads();
    for (int idx = tid; idx < kAbsBt * 64; idx += 256) {
      const int j = idx >> 6, c = idx & 63;
      if (b0 + j < B)
        q_lat[((size_t)(b0 + j) * H + h) * kDc + n0 + c] =
            (part[0][j][c] + part[1][j][c]) + (part[2][j][c] + part[3][j][c]);
    }
    __syncthreads();
  }
}

// grid (H, 128 / 32); block 256 = 8 c-slices x 32 output columns
__global__ void __launch_bounds__(256) out_unabsorb_kernel(const float* __restrict__ o_lat,
                                                           const uint16_t* __restrict__ w_uv,
                                                           float* __restrict__ o, int B, int H) {
  __shared__ float ol[kUnBt][kDc];
  __shared__ float part[8][kUnBt][32];
  const int h = blockIdx.x, v0 = blockIdx.y * 32;
  const int tid = threadIdx.x, cs = tid >> 5, vl = tid & 31;
  const uint16_t* w = w_uv + (size_t)h * kDc * kDv + v0 + vl;
  for (int b0 = 0; b0 < B; b0 += kUnBt) {
    for (int idx = tid; idx < kUnBt * kDc; idx += 256) {
      const int j = idx / kDc, c = idx % kDc;
      ol[j][c] = (b0 + j < B) ? o_lat[((size_t)(b0 + j) * H + h) * kDc + c] : 0.f;
    }
    __syncthreads();
    float acc[kUnBt];
#pragma unroll
    for (int j = 0; j < kUnBt; ++j) acc[j] = 0.f;
    for (int c = cs * 64; c < cs * 64 + 64; ++c) {
      const float wv = bf16f(w[(size_t)c * kDv]);
#pragma unroll
      for (int j = 0; j < kUnBt; ++j) acc[j] = fmaf(ol[j][c], wv, acc[j]);
    }
#pragma unroll
    for (int j = 0; j < kUnBt; ++j) part[cs][j][vl] = acc[j];
    __syncthreads();
    if (tid < kUnBt * 32) {
      const int j = tid >> 5, v = tid & 31;
      float s = 0.f;
#pragma unroll
      for (int r = 0; r < 8; ++r) s += part[r][j][v];
      if (b0 + j < B) o[((size_t)(b0 + j) * H + h) * kDv + v0 + v] = s;
    }
    __syncthreads();
  }
}

}  // namespace

mla_status launch_q_absorb(const uint16_t* q_nope, const uint16_t* w_uk, float* q_lat, int B, int H,
                           cudaStream_t stream) {
  q_absorb_kernel<<<dim3(H, kDc / 64), 256, 0, stream>>>(q_nope, w_uk, q_lat, B, H);
  return launch_status();
}

mla_status launch_out_unabsorb(const float* o_lat, const uint16_t* w_uv, float* o, int B, int H,
                               cudaStream_t stream) {
  out_unabsorb_kernel<<<dim3(H, kDv / 32), 256, 0, stream>>>(o_lat, w_uv, o, B, H);
  return launch_status();
}

}  // namespace mla
