// mla_lse_merge: attention over the union of disjoint context parts from the
// parts' own results.  For one (sequence, head) with parts r = 0..R-1, each
// part's result is o_r = sum_{t in r} e^{s_t} c_t / sum_{t in r} e^{s_t} and
// lse_r = ln sum_{t in r} e^{s_t}.  The softmax over the union (English
// report "Absorbed MLA Cache Optimization on DeepSeek-V2-Lite — Technical
// Report" §2.1 attention from the latent) is then exactly
//   M = max_r lse_r,  w_r = e^{lse_r - M},
//   o = sum_r w_r o_r / sum_r w_r,   lse = M + ln sum_r w_r.
// This is the exchange step of a context-sharded decode: every rank decodes
// its own pages and the gathered (o_lat, lse) pairs are merged here.
#include <math.h>

#include "mla_internal.cuh"

namespace mla {

namespace {

constexpr int kMergeThreads = 128;              // 4 channels each

__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  v = red[0];
#pragma unroll
  for (int w = 1; w < kMergeThreads / 32; ++w) v = fmaxf(v, red[w]);
  return v;
}

__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  v = 0.f;
#pragma unroll
  for (int w = 0; w < kMergeThreads / 32; ++w) v += red[w];
  return v;
}

// grid (B, H), block 128
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const float* __restrict__ o_parts,
                                                              const float* __restrict__ lse_parts, int R, int B,
                                                              int H, float* __restrict__ o_lat,
                                                              float* __restrict__ lse) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ float wts[kMaxMergeParts];
  __shared__ float red[kMergeThreads / 32];
  const int b = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  const size_t row = (size_t)b * H + h, stride = (size_t)B * H;
  float m = -INFINITY;
  for (int r = tid; r < R; r += kMergeThreads) m = fmaxf(m, lse_parts[r * stride + row]);
  m = block_max(m, red);
  float4* out = reinterpret_cast<float4*>(o_lat + row * kDc) + tid;
  if (m == -INFINITY) {                         // every part empty
    *out = make_float4(0.f, 0.f, 0.f, 0.f);
    if (lse && tid == 0) lse[row] = -INFINITY;
    return;
  }
  float l = 0.f;
  for (int r = tid; r < R; r += kMergeThreads) {
    const float v = lse_parts[r * stride + row];
    const float w = v == -INFINITY ? 0.f : expf(v - m);
    wts[r] = w;
    l += w;
  }
  l = block_sum(l, red);                        // also orders the wts writes before the reads below
  // an empty part (weight 0) may hold any values, even non-finite ones:
  // its loads are skipped by a select, not a branch, so that up to eight
  // loads are in flight at a time
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  const float4* src = reinterpret_cast<const float4*>(o_parts + row * kDc) + tid;
#pragma unroll 8
  for (int r = 0; r < R; ++r) {
    const float w = wts[r];
    float4 v = __ldcg(src + r * stride * (kDc / 4));
    if (w == 0.f) v = make_float4(0.f, 0.f, 0.f, 0.f);
    acc.x = fmaf(w, v.x, acc.x);
    acc.y = fmaf(w, v.y, acc.y);
    acc.z = fmaf(w, v.z, acc.z);
    acc.w = fmaf(w, v.w, acc.w);
  }
  const float inv = 1.f / l;
  *out = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  if (lse && tid == 0) lse[row] = m + logf(l);
}

}  // namespace

mla_status launch_lse_merge(const float* o_parts, const float* lse_parts, int R, int B, int H, float* o_lat,
                            float* lse, cudaStream_t stream) {
  return cuda_status(launch_pdl(merge_kernel, dim3(B, H), dim3(kMergeThreads), 0, stream, o_parts, lse_parts, R, B,
                                H, o_lat, lse));
}

}  // namespace mla
