// Device twin of synth/__init__.py: the same counter-based generator
// (splitmix64 finaliser, Irwin-Hall n = 4 normal), the same fp32 operation
// order and round-to-nearest-even bf16 narrowing, so that every value equals
// the host generator's bit for bit.  Used to fill large caches quickly; holds
// no arithmetic of the attention method.  All pointers are device pointers.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

constexpr uint64_t kGolden = 0x9E3779B97F4A7C15ull;

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ float normal_at(uint64_t key, uint64_t idx, float ns) {
  const uint64_t h = mix64(key + idx * kGolden);
  const uint32_t s = (uint32_t)(h & 0xFFFF) + (uint32_t)((h >> 16) & 0xFFFF) + (uint32_t)((h >> 32) & 0xFFFF) +
                     (uint32_t)(h >> 48);
  return __fmul_rn((float)((int32_t)s - 131070), ns);
}

__device__ __forceinline__ uint16_t bf16_bits(float v) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

__device__ __forceinline__ uint64_t token_index(uint64_t b, uint64_t t, uint64_t ch) {
  return (((b << 22) | t) << 10) | ch;
}

__global__ void latent_kernel(uint64_t key, int b, int t0, int n_tok, const float* __restrict__ mu,
                              const float* __restrict__ sigma, float ns, uint32_t* __restrict__ out) {
  const int64_t total = (int64_t)n_tok * 256;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int t = (int)(i >> 8), pr = (int)(i & 255), ch = 2 * pr;
    const uint64_t base = token_index(b, (uint64_t)(t0 + t), 0);
    const float z0 = normal_at(key, base | ch, ns), z1 = normal_at(key, base | (ch + 1), ns);
    const float v0 = __fadd_rn(mu[ch], __fmul_rn(sigma[ch], z0));
    const float v1 = __fadd_rn(mu[ch + 1], __fmul_rn(sigma[ch + 1], z1));
    out[i] = (uint32_t)bf16_bits(v0) | ((uint32_t)bf16_bits(v1) << 16);
  }
}

__global__ void kpe_kernel(uint64_t key, int b, int t0, int n_tok, const float* __restrict__ cos_tab,
                           const float* __restrict__ sin_tab, float ns, uint16_t* __restrict__ out) {
  const int64_t total = (int64_t)n_tok * 32;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int t = (int)(i >> 5), k = (int)(i & 31);
    const int64_t pos = (int64_t)t0 + t;
    const uint64_t base = token_index(b, (uint64_t)pos, 0);
    const float z1 = normal_at(key, base | k, ns), z2 = normal_at(key, base | (k + 32), ns);
    const float c = cos_tab[pos * 32 + k], s = sin_tab[pos * 32 + k];
    const float lo = __fsub_rn(__fmul_rn(z1, c), __fmul_rn(z2, s));
    const float hi = __fadd_rn(__fmul_rn(z1, s), __fmul_rn(z2, c));
    out[(int64_t)t * 64 + k] = bf16_bits(lo);
    out[(int64_t)t * 64 + k + 32] = bf16_bits(hi);
  }
}

__global__ void normal3_kernel(uint64_t key, int d0, int d1, int d2, float mul, float ns, uint16_t* __restrict__ out) {
  const int64_t total = (int64_t)d0 * d1 * d2;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t i2 = i % d2, i1 = (i / d2) % d1, i0 = i / ((int64_t)d1 * d2);
    const uint64_t idx = ((((uint64_t)i0 << 10) | (uint64_t)i1) << 10) | (uint64_t)i2;
    out[i] = bf16_bits(__fmul_rn(normal_at(key, idx, ns), mul));
  }
}

int grid_for(int64_t n) {
  int64_t g = (n + 255) / 256;
  return (int)(g < 152 * 64 ? (g > 0 ? g : 1) : 152 * 64);
}

}  // namespace

extern "C" {

int synth_latent_bf16(uint64_t key, int32_t b, int32_t t0, int32_t n_tok, const float* mu, const float* sigma,
                      float normal_scale, uint16_t* out, void* stream) {
  if (n_tok <= 0) return 0;
  latent_kernel<<<grid_for((int64_t)n_tok * 256), 256, 0, (cudaStream_t)stream>>>(
      key, b, t0, n_tok, mu, sigma, normal_scale, reinterpret_cast<uint32_t*>(out));
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

int synth_kpe_bf16(uint64_t key, int32_t b, int32_t t0, int32_t n_tok, const float* cos_tab, const float* sin_tab,
                   float normal_scale, uint16_t* out, void* stream) {
  if (n_tok <= 0) return 0;
  kpe_kernel<<<grid_for((int64_t)n_tok * 32), 256, 0, (cudaStream_t)stream>>>(key, b, t0, n_tok, cos_tab, sin_tab,
                                                                              normal_scale, out);
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

int synth_normal3_bf16(uint64_t key, int32_t d0, int32_t d1, int32_t d2, float mul, float normal_scale,
                       uint16_t* out, void* stream) {
  if ((int64_t)d0 * d1 * d2 <= 0) return 0;
  normal3_kernel<<<grid_for((int64_t)d0 * d1 * d2), 256, 0, (cudaStream_t)stream>>>(key, d0, d1, d2, mul,
                                                                                   normal_scale, out);
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

}  // extern "C"
