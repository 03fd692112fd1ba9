// Host side of the C ABI declared in include/mla.h: argument checks, layout
// arithmetic and dispatch to the kernel launchers.  Nothing here allocates.
#include <math.h>

#include <atomic>

#include "mla_internal.cuh"

namespace mla {

int device_sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) cached[dev] = n;
  return n;
}

static std::atomic<int64_t> g_wait_limit_ns{10000000000ll};

uint64_t wait_limit_ns() { return (uint64_t)g_wait_limit_ns.load(std::memory_order_relaxed); }

static thread_local const char* g_last_cuda_error = "no error";

mla_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return MLA_OK;
  g_last_cuda_error = cudaGetErrorString(e);
  return MLA_ERR_CUDA;
}

mla_status launch_status() { return cuda_status(cudaGetLastError()); }

static bool aligned(const void* p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }

static bool heads_ok(int H) { return H >= 16 && H <= 128 && H % 16 == 0; }

bool cache_check(const mla_cache_layer* c, PageLayout* L, OutlierSet* o) {
  if (!c || c->num_pages <= 0 || c->reserved != 0 || !c->pool) return false;
  if (!aligned(c->pool, 256)) return false;
  if (!compute_layout(c->latent_fmt, c->kpe_fmt, L)) return false;
  for (int k = 0; k < kOutSlots; ++k) o->ch[k] = -1;
  for (int k = 0; k < kDc / 32; ++k) o->mask[k] = 0u;
  if (c->latent_fmt != MLA_FMT_INT8_OUTLIER) return c->outlier_channels == nullptr;
  if (!c->outlier_channels) return false;
  for (int k = 0; k < kNOut; ++k) {
    const int32_t ch = c->outlier_channels[k];
    if (ch < 0 || ch >= kDc || (k > 0 && ch <= c->outlier_channels[k - 1])) return false;
    o->ch[k] = (int16_t)ch;
    o->mask[ch >> 5] |= 1u << (ch & 31);
  }
  return true;
}

// Context splits of a decode call: the caller's count, else one CTA per SM
// over all head tiles (the H / 16 CTAs of a split run side by side and read
// the split's pages once between them, through L2).
static int decode_grid(int num_splits, int heads) {
  if (num_splits > 0) return num_splits;
  const int sms = device_sm_count();
  const int g = sms / (heads / 16);
  return g > 0 ? g : 1;
}

}  // namespace mla

using namespace mla;

extern "C" {

int32_t mla_abi_version(void) { return 107; }

const char* mla_last_cuda_error(void) { return g_last_cuda_error; }

int64_t mla_set_wait_limit_ns(int64_t ns) {
  if (ns < 0) return -1;
  return g_wait_limit_ns.exchange(ns);
}

const char* mla_status_string(mla_status s) {
  switch (s) {
    case MLA_OK: return "ok";
    case MLA_ERR_INVALID_ARG: return "invalid argument";
    case MLA_ERR_UNSUPPORTED: return "unsupported shape or format";
    case MLA_ERR_CUDA: return "CUDA launch error";
    case MLA_ERR_DEVICE_BOUNDS: return "device-side bounds error";
  }
  return "unknown status";
}

mla_status mla_cache_page_layout(const mla_cache_layer* cache, mla_page_layout* out) {
  if (!cache || !out) return MLA_ERR_INVALID_ARG;
  PageLayout L;
  if (!compute_layout(cache->latent_fmt, cache->kpe_fmt, &L)) return MLA_ERR_INVALID_ARG;
  out->page_bytes = L.page_bytes;
  out->block_bytes = L.block_bytes;
  out->codes_off = L.codes_off;
  out->codes_row_bytes = L.codes_row;
  out->scale_off = L.scale_off;
  out->zero_off = L.zero_off;
  out->kpe_off = L.kpe_off;
  out->kpe_row_bytes = L.kpe_row;
  out->kpe_scale_off = L.kpe_scale_off;
  out->bound_off = L.bound_off;
  out->outlier_off = L.outlier_off;
  return MLA_OK;
}

size_t mla_cache_pool_bytes(const mla_cache_layer* cache) {
  if (!cache || cache->num_pages <= 0) return 0;
  PageLayout L;
  if (!compute_layout(cache->latent_fmt, cache->kpe_fmt, &L)) return 0;
  return (size_t)L.page_bytes * (size_t)cache->num_pages;
}

mla_status mla_cache_append(const mla_cache_layer* cache, const uint16_t* c_new,
                            const uint16_t* kpe_new, const int32_t* slot, int32_t n,
                            int32_t* dev_err, mla_stream_t stream) {
  PageLayout L;
  OutlierSet outl;
  if (!cache_check(cache, &L, &outl) || n < 0) return MLA_ERR_INVALID_ARG;
  if (n == 0) return MLA_OK;
  if (!c_new || !kpe_new || !slot) return MLA_ERR_INVALID_ARG;
  if (!aligned(c_new, 16) || !aligned(kpe_new, 16) || !aligned(slot, 4)) return MLA_ERR_INVALID_ARG;
  if (dev_err && !aligned(dev_err, 4)) return MLA_ERR_INVALID_ARG;
  return launch_append(cache, L, outl, c_new, kpe_new, slot, n, dev_err, (cudaStream_t)stream);
}

mla_status mla_select_outlier_channels(const uint16_t* c_sample, int32_t n, int32_t* channels_out,
                                       mla_stream_t stream) {
  if (n < 1 || !c_sample || !channels_out || !aligned(c_sample, 16) || !aligned(channels_out, 4))
    return MLA_ERR_INVALID_ARG;
  return launch_select_outliers(c_sample, n, channels_out, (cudaStream_t)stream);
}

mla_status mla_q_absorb(const uint16_t* q_nope, const uint16_t* w_uk, float* q_lat, int32_t batch,
                        int32_t heads, mla_stream_t stream) {
  if (batch < 0 || !heads_ok(heads)) return MLA_ERR_INVALID_ARG;
  if (batch == 0) return MLA_OK;
  if (!q_nope || !w_uk || !q_lat) return MLA_ERR_INVALID_ARG;
  if (!aligned(q_nope, 16) || !aligned(w_uk, 16) || !aligned(q_lat, 16)) return MLA_ERR_INVALID_ARG;
  return launch_q_absorb(q_nope, w_uk, q_lat, batch, heads, (cudaStream_t)stream);
}

mla_status mla_out_unabsorb(const float* o_lat, const uint16_t* w_uv, float* o, int32_t batch,
                            int32_t heads, mla_stream_t stream) {
  if (batch < 0 || !heads_ok(heads)) return MLA_ERR_INVALID_ARG;
  if (batch == 0) return MLA_OK;
  if (!o_lat || !w_uv || !o) return MLA_ERR_INVALID_ARG;
  if (!aligned(o_lat, 16) || !aligned(w_uv, 16) || !aligned(o, 16)) return MLA_ERR_INVALID_ARG;
  return launch_out_unabsorb(o_lat, w_uv, o, batch, heads, (cudaStream_t)stream);
}

mla_status mla_lse_merge(const float* o_parts, const float* lse_parts, int32_t parts, int32_t batch,
                         int32_t heads, float* o_lat, float* lse, mla_stream_t stream) {
  if (parts < 1 || parts > kMaxMergeParts || batch < 0 || batch > kMaxBatch || !heads_ok(heads))
    return MLA_ERR_INVALID_ARG;
  if (batch == 0) return MLA_OK;
  if (!o_parts || !lse_parts || !o_lat) return MLA_ERR_INVALID_ARG;
  if (!aligned(o_parts, 16) || !aligned(lse_parts, 4) || !aligned(o_lat, 16) || (lse && !aligned(lse, 4)))
    return MLA_ERR_INVALID_ARG;
  const char* a = (const char*)o_parts;
  const char* e = a + (size_t)parts * batch * heads * kDc * sizeof(float);
  const char* o = (const char*)o_lat;
  if (o < e && a < o + (size_t)batch * heads * kDc * sizeof(float)) return MLA_ERR_INVALID_ARG;
  return launch_lse_merge(o_parts, lse_parts, parts, batch, heads, o_lat, lse, (cudaStream_t)stream);
}

size_t mla_decode_workspace_bytes(int32_t batch, int32_t heads, int32_t num_splits) {
  if (batch < 0 || batch > kMaxBatch || !heads_ok(heads) || num_splits < 0 || num_splits > kMaxSplits) return 0;
  return (size_t)workspace_bytes(batch, heads, decode_grid(num_splits, heads));
}

static mla_status decode_call(const mla_cache_layer* cache, const float* q_lat,
                               const uint16_t* q_pe, const int32_t* block_table,
                               int32_t max_pages, const int32_t* seq_lens, int32_t batch,
                               int32_t heads, float softmax_scale, int32_t num_splits,
                               void* workspace, size_t workspace_bytes_, float* o_lat,
                               float* lse, const uint16_t* w_uv, float* o, int32_t* dev_err,
                               mla_stream_t stream) {
  PageLayout L;
  OutlierSet outl;
  if (!cache_check(cache, &L, &outl)) return MLA_ERR_INVALID_ARG;
  if (batch < 0 || batch > kMaxBatch || !heads_ok(heads) || num_splits < 0 || num_splits > kMaxSplits)
    return MLA_ERR_INVALID_ARG;
  if (batch == 0) return MLA_OK;
  if (max_pages <= 0 || (int64_t)max_pages * kPage > (int64_t)INT32_MAX) return MLA_ERR_INVALID_ARG;
  // every 32-token chunk of the batch gets a 32-bit index
  if ((int64_t)batch * max_pages * (kPage / kChunk) > (int64_t)INT32_MAX) return MLA_ERR_INVALID_ARG;
  if (!q_lat || !q_pe || !block_table || !seq_lens || !workspace || !o_lat) return MLA_ERR_INVALID_ARG;
  if (!aligned(q_lat, 16) || !aligned(q_pe, 16) || !aligned(block_table, 4) || !aligned(seq_lens, 4) ||
      !aligned(workspace, 256) || !aligned(o_lat, 16) || (lse && !aligned(lse, 4)) ||
      (dev_err && !aligned(dev_err, 4)))
    return MLA_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.f) || !isfinite(softmax_scale)) return MLA_ERR_INVALID_ARG;
  if ((w_uv == nullptr) != (o == nullptr) || (w_uv && (!aligned(w_uv, 16) || !aligned(o, 16))))
    return MLA_ERR_INVALID_ARG;
  int G = decode_grid(num_splits, heads);
  if ((int64_t)workspace_bytes_ < workspace_bytes(batch, heads, G)) return MLA_ERR_INVALID_ARG;
  DecodeParams p;
  p.pool = (const uint8_t*)cache->pool;
  p.L = L;
  p.latent_fmt = cache->latent_fmt;
  p.kpe_fmt = cache->kpe_fmt;
  p.num_pages = cache->num_pages;
  p.q_lat = q_lat;
  p.q_pe = q_pe;
  p.block_table = block_table;
  p.max_pages = max_pages;
  p.bt_stride = max_pages;
  p.lens_after_wait = 0;
  p.seq_lens = seq_lens;
  p.B = batch;
  p.H = heads;
  p.G = G;
  p.scale_log2 = softmax_scale * 1.4426950408889634f;
  p.outl = outl;
  p.wait_ns = wait_limit_ns();
  p.ws = carve_workspace(workspace, batch, heads, G);
  p.o_lat = o_lat;
  p.lse = lse;
  p.w_uv = w_uv;
  p.o = o;
  p.dev_err = dev_err;
  return launch_decode(p, (cudaStream_t)stream);
}

mla_status mla_decode_absorbed(const mla_cache_layer* cache, const float* q_lat,
                               const uint16_t* q_pe, const int32_t* block_table,
                               int32_t max_pages, const int32_t* seq_lens, int32_t batch,
                               int32_t heads, float softmax_scale, int32_t num_splits,
                               void* workspace, size_t workspace_bytes_, float* o_lat,
                               float* lse, int32_t* dev_err, mla_stream_t stream) {
  return decode_call(cache, q_lat, q_pe, block_table, max_pages, seq_lens, batch, heads, softmax_scale, num_splits,
                     workspace, workspace_bytes_, o_lat, lse, nullptr, nullptr, dev_err, stream);
}

int32_t mla_decode_kernel_count(const mla_cache_layer* cache, int32_t batch, int32_t heads, int32_t num_splits,
                                int32_t with_unabsorb) {
  if (!cache || batch < 0 || batch > kMaxBatch || !heads_ok(heads) || num_splits < 0 || num_splits > kMaxSplits)
    return -1;
  PageLayout L;
  if (!compute_layout(cache->latent_fmt, cache->kpe_fmt, &L)) return -1;
  if (batch == 0) return 0;
  const int fused = combine_grid(cache->latent_fmt, batch, decode_grid(num_splits, heads)) == 1;
  return 2 + (with_unabsorb && !fused ? 1 : 0);
}

mla_status mla_decode_absorbed_unabsorb(const mla_cache_layer* cache, const float* q_lat,
                                        const uint16_t* q_pe, const int32_t* block_table,
                                        int32_t max_pages, const int32_t* seq_lens, int32_t batch,
                                        int32_t heads, float softmax_scale, int32_t num_splits,
                                        void* workspace, size_t workspace_bytes_, float* o_lat,
                                        float* lse, const uint16_t* w_uv, float* o, int32_t* dev_err,
                                        mla_stream_t stream) {
  if (!w_uv || !o) return MLA_ERR_INVALID_ARG;
  return decode_call(cache, q_lat, q_pe, block_table, max_pages, seq_lens, batch, heads, softmax_scale, num_splits,
                     workspace, workspace_bytes_, o_lat, lse, w_uv, o, dev_err, stream);
}

}  // extern "C"
