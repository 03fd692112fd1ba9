// mla_prefill_absorbed: causal absorbed attention of a prefill chunk.
//
// Query i of the chunk sits at position ctx_before + i of its sequence and
// attends to the cached positions 0 .. ctx_before + i (the chunk's own
// tokens, appended before the call, included).  In absorbed form each query
// row is exactly a decode query over a prefix of one sequence ("Absorbed MLA
// Cache Optimization on DeepSeek-V2-Lite — Technical Report" §2.1: attention
// straight from the cached latent).  Two implementations:
//
//  * tensor cores (prefill_tc.cu): every cached token dequantized once into
//    fp16 (hi, lo) key tiles, the queries split the same way, and a tcgen05
//    kernel over 128-row x 128-key tiles; rows that see fewer than 256
//    tokens, or fail the precision check, are recomputed exactly afterwards.
//    Used when the chunk has enough rows to fill the GPU and the prefix fits
//    the key tiles (kTcMaxKeys tokens).
//  * the decode kernels: the queries become the batch, every batch row
//    shares the sequence's block-table row (row stride 0), and row i's
//    length is ctx_before + i + 1.  The split-K partition then balances the
//    triangle of (query, key) pairs over the SMs by 32-token chunks, and the
//    log-sum-exp combine writes normalised rows.
//
// Queries go in slices (kSlice / kTcSlice tokens) so the workspace stays
// bounded for long chunks.
#include <math.h>

#include <atomic>

#include "mla_internal.cuh"

namespace mla {
namespace {

constexpr int kSlice = 2048;

// len[i] = base + i + 1 for the slice's rows; zero[0 .. nzero) = 0 (the
// tensor-core path's queue counters)
__global__ void causal_lengths_kernel(int32_t* len, int n, int base, int32_t* zero, int nzero) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) len[i] = base + i + 1;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < nzero; i += gridDim.x * blockDim.x) zero[i] = 0;
}

int64_t lengths_bytes() { return align256((int64_t)kSlice * 4); }

int prefill_grid() {
  const int sms = device_sm_count();
  return sms > 0 ? sms : 1;
}

bool aligned_to(const void* p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }

// ---- tensor-core path
constexpr int kTcSlice = 4096;           // query tokens per launch (1024: +4 % time; 8192: no gain)
constexpr int kTcMaxKeys = 65536;        // positions the key tiles hold (151 MB)
// The automatic choice (measured on GB300 against the decode kernels, INT8,
// 16 and 64 heads, 0 to 8192 positions before the chunk): the tensor cores
// from 8192 rows (n x H) on, or from 2048 rows once the chunk's prefixes
// reach 4096 positions; never when every row sees at most 256 positions
// (they are all recomputed exactly).
constexpr int64_t kTcMinRows = 8192;
constexpr int64_t kTcMinRowsLong = 2048;
constexpr int kTcLongKeys = 4096;
constexpr int kTcExactLen = 256;

std::atomic<int> g_prefill_path{MLA_PREFILL_AUTO};

struct TcWorkspace {
  uint8_t* kws;
  uint8_t* qws;
  float* mt;
  int32_t* lens;
  float* risk;
  float* omax;
  SplitQueue queue;
  float* table;          // x_hat of positions 0 .. 255, fp32 [256][576]
};

int64_t tc_row_tiles(int64_t rows) { return (rows + 127) / 128; }

int64_t tc_workspace_bytes(int n, int heads, TcWorkspace* w, void* base) {
  const int64_t s = n < kTcSlice ? (n > 0 ? n : 1) : kTcSlice;
  const int64_t rows = s * heads;
  const int64_t sizes[8] = {(int64_t)(kTcMaxKeys / 128) * kTcTileBytes, tc_row_tiles(rows) * kTcTileBytes,
                            align256((int64_t)kTcMaxKeys * 4), align256(s * 4), align256(rows * 4),
                            align256(rows * 8), split_queue_bytes(), (int64_t)kTcExactLen * (kDc + kDr) * 4};
  int64_t off = 0;
  char* b = (char*)base;
  void* ptrs[8];
  for (int i = 0; i < 8; ++i) {
    ptrs[i] = b ? b + off : nullptr;
    off += sizes[i];
  }
  if (w) {
    w->kws = (uint8_t*)ptrs[0];
    w->qws = (uint8_t*)ptrs[1];
    w->mt = (float*)ptrs[2];
    w->lens = (int32_t*)ptrs[3];
    w->risk = (float*)ptrs[4];
    w->omax = (float*)ptrs[5];
    w->queue = carve_split_queue(ptrs[6] ? ptrs[6] : (void*)nullptr);
    w->table = (float*)ptrs[7];
  }
  return off;
}

int64_t decode_path_bytes(int n, int heads) {
  const int s = n < kSlice ? (n > 0 ? n : 1) : kSlice;
  return lengths_bytes() + workspace_bytes(s, heads, prefill_grid());
}

// The path a call takes: 1 = decode kernels, 2 = tensor cores.  ctx_before
// < 0: the choice made without knowing it (the workspace size).
int choose_path(int ctx_before, int n, int heads) {
  const int forced = g_prefill_path.load(std::memory_order_relaxed);
  if (forced != MLA_PREFILL_AUTO) return forced;
  const int64_t rows = (int64_t)n * heads;
  if (rows < kTcMinRowsLong) return MLA_PREFILL_DECODE_KERNELS;
  if (ctx_before < 0) return MLA_PREFILL_TENSOR_CORES;      // the workspace covers either path
  const int64_t keys = (int64_t)ctx_before + n;
  if (keys <= kTcExactLen || keys > kTcMaxKeys) return MLA_PREFILL_DECODE_KERNELS;
  return rows >= kTcMinRows || keys >= kTcLongKeys ? MLA_PREFILL_TENSOR_CORES : MLA_PREFILL_DECODE_KERNELS;
}

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" {

size_t mla_prefill_workspace_bytes(int32_t n, int32_t heads) {
  if (n < 0 || heads < 16 || heads > 128 || heads % 16) return 0;
  const int64_t dec = decode_path_bytes(n, heads);
  if (choose_path(-1, n, heads) != MLA_PREFILL_TENSOR_CORES) return (size_t)dec;
  const int64_t tc = tc_workspace_bytes(n, heads, nullptr, nullptr);
  return (size_t)(tc > dec ? tc : dec);
}

int32_t mla_prefill_path_taken(int32_t ctx_before, int32_t n, int32_t heads) {
  if (n < 0 || ctx_before < 0 || heads < 16 || heads > 128 || heads % 16) return -1;
  return choose_path(ctx_before, n, heads);
}

int32_t mla_set_prefill_path(int32_t path) {
  if (path != MLA_PREFILL_AUTO && path != MLA_PREFILL_DECODE_KERNELS && path != MLA_PREFILL_TENSOR_CORES) return -1;
  return g_prefill_path.exchange(path);
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
  if (!q_lat || !q_pe || !block_table || !workspace || !o_lat) return MLA_ERR_INVALID_ARG;
  if (!aligned_to(q_lat, 16) || !aligned_to(q_pe, 16) || !aligned_to(block_table, 4) ||
      !aligned_to(workspace, 256) || !aligned_to(o_lat, 16) || (lse && !aligned_to(lse, 4)) ||
      (dev_err && !aligned_to(dev_err, 4)))
    return MLA_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.f) || !isfinite(softmax_scale)) return MLA_ERR_INVALID_ARG;
  const int path = choose_path(ctx_before, n, heads);
  const cudaStream_t st = (cudaStream_t)stream;
  if (path == MLA_PREFILL_TENSOR_CORES) {
    if ((int64_t)ctx_before + n > kTcMaxKeys) return MLA_ERR_UNSUPPORTED;
    TcWorkspace w;
    if ((int64_t)workspace_bytes_ < tc_workspace_bytes(n, heads, &w, workspace)) return MLA_ERR_INVALID_ARG;
    DecodeParams p;
    p.pool = (const uint8_t*)cache->pool;
    p.L = L;
    p.latent_fmt = cache->latent_fmt;
    p.kpe_fmt = cache->kpe_fmt;
    p.num_pages = cache->num_pages;
    p.block_table = block_table;
    p.max_pages = max_pages;
    p.bt_stride = 0;
    p.seq_lens = w.lens;
    p.lens_after_wait = 1;
    p.H = heads;
    p.G = 0;
    p.scale_log2 = softmax_scale * 1.4426950408889634f;
    p.outl = outl;
    p.wait_ns = wait_limit_ns();
    p.ws = Workspace{};
    p.w_uv = nullptr;
    p.o = nullptr;
    p.dev_err = dev_err;
    const int keys = ctx_before + n;
    // the short rows' table is needed only when some query sees < 256 positions
    float* table = ctx_before + 1 < kTcExactLen ? w.table : nullptr;
    mla_status ks = launch_prefill_keys(p, keys, w.kws, w.mt, table, st);
    if (ks != MLA_OK) return ks;
    for (int i0 = 0; i0 < n; i0 += kTcSlice) {
      const int s = n - i0 < kTcSlice ? n - i0 : kTcSlice;
      const int R = s * heads;
      const int n_rt = (int)tc_row_tiles(R);
      // the fixup's per-row lengths; a plain launch, after the previous
      // slice's fixup has finished with them
      causal_lengths_kernel<<<(s + 255) / 256, 256, 0, st>>>(w.lens, s, ctx_before + i0, w.queue.count,
                                                             1 + kSplitCap);
      const mla_status ls = launch_status();
      if (ls != MLA_OK) return ls;
      const float* ql = q_lat + (size_t)i0 * heads * kDc;
      const uint16_t* qp = q_pe + (size_t)i0 * heads * kDr;
      float* ol = o_lat + (size_t)i0 * heads * kDc;
      float* lo = lse ? lse + (size_t)i0 * heads : nullptr;
      ks = launch_q_split(ql, qp, R, n_rt, w.qws, st);
      if (ks != MLA_OK) return ks;
      TcParams t;
      t.qws = w.qws;
      t.kws = w.kws;
      t.mt = w.mt;
      t.R = R;
      t.H = heads;
      t.qpos0 = ctx_before + i0;
      t.n_rt = n_rt;
      t.scale_log2 = p.scale_log2;
      t.risk = cache->latent_fmt != MLA_FMT_BF16;
      t.o_lat = ol;
      t.lse = lo;
      t.risk_out = w.risk;
      t.omax = w.omax;
      t.dev_err = dev_err;
      t.wait_ns = p.wait_ns;
      ks = launch_prefill_tc(t, st);
      if (ks != MLA_OK) return ks;
      DecodeParams f = p;
      f.q_lat = ql;
      f.q_pe = qp;
      f.B = s;
      f.o_lat = ol;
      f.lse = lo;
      ks = launch_exact_fixup(f, w.risk, w.omax, w.queue, table != nullptr, st);
      if (ks != MLA_OK) return ks;
      // the slice's rows below 256 positions: exact, from the x_hat table
      const int n_short = table ? (kTcExactLen - 1 - (ctx_before + i0) < s ? kTcExactLen - 1 - (ctx_before + i0) : s)
                                : 0;
      if (n_short > 0) {
        ks = launch_short_rows(table, ql, qp, heads, n_short, ctx_before + i0, p.scale_log2, ol, lo, st);
        if (ks != MLA_OK) return ks;
      }
    }
    return MLA_OK;
  }
  // every 32-token chunk of a slice gets a 32-bit index
  if ((int64_t)(n < kSlice ? n : kSlice) * max_pages * (kPage / kChunk) > (int64_t)INT32_MAX)
    return MLA_ERR_INVALID_ARG;
  if ((int64_t)workspace_bytes_ < decode_path_bytes(n, heads)) return MLA_ERR_INVALID_ARG;

  const int G = prefill_grid();
  int32_t* lens = (int32_t*)workspace;
  void* split_ws = (char*)workspace + lengths_bytes();
  for (int i0 = 0; i0 < n; i0 += kSlice) {
    const int s = n - i0 < kSlice ? n - i0 : kSlice;
    // a plain launch: it starts after the previous slice's combine has
    // finished with the lengths and the split-K workspace.  Its stores are
    // visible to the decode kernel only once that kernel has waited on it
    // (lens_after_wait)
    causal_lengths_kernel<<<(s + 255) / 256, 256, 0, st>>>(lens, s, ctx_before + i0, nullptr, 0);
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
