// mla_decode_absorbed_noalloc: the decode call for callers that cannot
// allocate device memory.
//
// Some callers of a decode kernel have device pointers for their inputs and
// outputs but no way to obtain scratch memory: a plugin inside an inference
// engine that is handed only its I/O buffers, code that runs while a CUDA
// graph is being captured (a cudaMalloc there is not capturable), or a
// serving loop that forbids allocation after start-up because cudaMalloc can
// synchronize the device and fragment a carefully budgeted memory pool.  For
// them this entry point uses a fixed scratch array compiled into the library
// instead of a caller-provided workspace; it allocates nothing.
//
// The array lives in every device's copy of the module from the moment the
// library is loaded until the process exits.  Every call shares it, so two
// calls that overlap on the GPU (different streams, or different host
// threads) race on it.  Nothing in it has to start at zero: every byte a call
// reads was written earlier by the same call.
#include <mutex>

#include "mla_internal.cuh"

namespace {

__device__ __align__(256) uint8_t g_decode_scratch[MLA_NOALLOC_SCRATCH_BYTES];

std::mutex g_scratch_mutex;
void* g_scratch_ptr[64] = {nullptr};

// Device address of the scratch array on the current device, looked up once
// per device (with that device current) and cached.
mla_status scratch_for_current_device(void** out) {
  int dev = 0;
  if (mla::cuda_status(cudaGetDevice(&dev)) != MLA_OK) return MLA_ERR_CUDA;
  if (dev < 0 || dev >= 64) return MLA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (mla::cuda_status(cudaGetSymbolAddress(&p, g_decode_scratch)) != MLA_OK) return MLA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return MLA_OK;
}

}  // namespace

extern "C" mla_status mla_decode_absorbed_noalloc(const mla_cache_layer* cache, const float* q_lat,
                                                  const uint16_t* q_pe, const int32_t* block_table,
                                                  int32_t max_pages, const int32_t* seq_lens, int32_t batch,
                                                  int32_t heads, float softmax_scale, int32_t num_splits,
                                                  float* o_lat, float* lse, int32_t* dev_err,
                                                  mla_stream_t stream) {
  if (batch == 0) return MLA_OK;
  const size_t need = mla_decode_workspace_bytes(batch, heads, num_splits);
  if (need == 0 || need > (size_t)MLA_NOALLOC_SCRATCH_BYTES) return MLA_ERR_INVALID_ARG;
  void* scratch = nullptr;
  const mla_status st = scratch_for_current_device(&scratch);
  if (st != MLA_OK) return st;
  return mla_decode_absorbed(cache, q_lat, q_pe, block_table, max_pages, seq_lens, batch, heads, softmax_scale,
                             num_splits, scratch, (size_t)MLA_NOALLOC_SCRATCH_BYTES, o_lat, lse, dev_err, stream);
}
