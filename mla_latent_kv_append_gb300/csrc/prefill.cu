// mla_prefill_absorbed: causal absorbed attention of a prefill chunk.
//
// Query i of the chunk sits at position ctx_before + i of its sequence and
// attends to the cached positions 0 .. ctx_before + i (the chunk's own
// tokens, appended before the call, included).  In absorbed form each query
// row is exactly a decode query over a prefix of one sequence ("Absorbed MLA
// Cache Optimization on DeepSeek-V2-Lite — Technical Report" §2.1: attention
// straight from the cached latent), so the chunk runs through the decode
// kernels: the queries become the batch, every batch row shares the
// sequence's block-table row (row stride 0), and row i's length is
// ctx_before + i + 1.  The split-K partition then balances the triangle of
// (query, key) pairs over the SMs by 32-token chunks, and the log-sum-exp
// combine writes normalised rows.  Queries go in slices of kSlice so the
// split-K workspace stays bounded for long chunks.
#include <math.h>

#include "mla_internal.cuh"

namespace mla {
namespace {

constexpr int kSlice = 2048;

// len[i] = base + i + 1 for the slice's rows
__global__ void causal_lengths_kernel(int32_t* len, int n, int base) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) len[i] = base + i + 1;
}

int64_t lengths_bytes() { return align256((int64_t)kSlice * 4); }

int prefill_grid() {
  const int sms = device_sm_count();
  return sms > 0 ? sms : 1;
}

bool aligned_to(const void* p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" {

size_t mla_prefill_workspace_bytes(int32_t n, int32_t heads) {
  if (n < 0 || heads < 16 || heads > 128 || heads % 16) return 0;
  const int s = n < kSlice ? (n > 0 ? n : 1) : kSlice;
  return (size_t)(lengths_bytes() + workspace_bytes(s, heads, prefill_grid()));
}

mla_status mla_prefill_absorbed(const mla_cache_layer* cache, const float* q_lat, const uint16_t* q_pe,
                                const int32_t* block_table, int32_t max_pages, int32_t ctx_before, int32_t n,
                                int32_t heads, float softmax_scale, void* workspace, size_t workspace_bytes_,
                                float* o_lat, float* lse, int32_t* dev_err, mla_stream_t stream) {
  PageLayout L;
  OutlierSet outl;
  if (!cache_check(cache, &L, &outl)) return MLA_ERR_INVALID_ARG;
  if (n < 0 || ctx_before < 0 || heads < 16 || heads > 128 || heads % 16) return MLA_ERR_INVALID_ARG;
  if (n == 0) return MLA_OK;
  if (max_pages <= 0 || (int64_t)max_pages * kPage > (int64_t)INT32_MAX) return MLA_ERR_INVALID_ARG;
  if ((int64_t)ctx_before + n > (int64_t)max_pages * kPage) return MLA_ERR_INVALID_ARG;
  // every 32-token chunk of a slice gets a 32-bit index
  if ((int64_t)(n < kSlice ? n : kSlice) * max_pages * (kPage / kChunk) > (int64_t)INT32_MAX)
    return MLA_ERR_INVALID_ARG;
  if (!q_lat || !q_pe || !block_table || !workspace || !o_lat) return MLA_ERR_INVALID_ARG;
  if (!aligned_to(q_lat, 16) || !aligned_to(q_pe, 16) || !aligned_to(block_table, 4) ||
      !aligned_to(workspace, 256) || !aligned_to(o_lat, 16) || (lse && !aligned_to(lse, 4)) ||
      (dev_err && !aligned_to(dev_err, 4)))
    return MLA_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.f) || !isfinite(softmax_scale)) return MLA_ERR_INVALID_ARG;
  if (workspace_bytes_ < mla_prefill_workspace_bytes(n, heads)) return MLA_ERR_INVALID_ARG;

  const cudaStream_t st = (cudaStream_t)stream;
  const int G = prefill_grid();
  int32_t* lens = (int32_t*)workspace;
  void* split_ws = (char*)workspace + lengths_bytes();
  for (int i0 = 0; i0 < n; i0 += kSlice) {
    const int s = n - i0 < kSlice ? n - i0 : kSlice;
    // a plain launch: it starts after the previous slice's combine has
    // finished with the lengths and the split-K workspace.  Its stores are
    // visible to the decode kernel only once that kernel has waited on it
    // (lens_after_wait)
    causal_lengths_kernel<<<(s + 255) / 256, 256, 0, st>>>(lens, s, ctx_before + i0);
    const mla_status ls = launch_status();
    if (ls != MLA_OK) return ls;
    DecodeParams p;
    p.pool = (const uint8_t*)cache->pool;
    p.L = L;
    p.latent_fmt = cache->latent_fmt;
    p.kpe_fmt = cache->kpe_fmt;
    p.num_pages = cache->num_pages;
    p.q_lat = q_lat + (size_t)i0 * heads * kDc;
    p.q_pe = q_pe + (size_t)i0 * heads * kDr;
    p.block_table = block_table;
    p.max_pages = max_pages;
    p.bt_stride = 0;
    p.seq_lens = lens;
    p.lens_after_wait = 1;
    p.B = s;
    p.H = heads;
    p.G = G;
    p.scale_log2 = softmax_scale * 1.4426950408889634f;
    p.outl = outl;
    p.wait_ns = wait_limit_ns();
    p.ws = carve_workspace(split_ws, s, heads, G);
    p.o_lat = o_lat + (size_t)i0 * heads * kDc;
    p.lse = lse ? lse + (size_t)i0 * heads : nullptr;
    p.w_uv = nullptr;
    p.o = nullptr;
    p.dev_err = dev_err;
    const mla_status ds = launch_decode(p, st);
    if (ds != MLA_OK) return ds;
  }
  return MLA_OK;
}

}  // extern "C"
