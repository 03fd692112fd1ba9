"""Absorbed MLA decode over a quantized paged latent KV cache, for GB300.

Thin Python binding over the C ABI in ``include/mla.h`` (``libmla_gb300.so``,
built in-tree by ``mla_latent_kv_append_gb300.build``).  The functions here
only marshal arguments - torch tensors supply device memory and the current
CUDA stream - and every step of the computation runs in the library's CUDA
kernels.  Importing this package without the built library raises; there is
no CPU fallback.

Names follow the C ABI:

    mla_cache_append(cache, c_new, kpe_new, slot, dev_err=None)
    mla_q_absorb(q_nope, w_uk, q_lat)
    mla_decode_absorbed(cache, q_lat, q_pe, block_table, seq_lens, workspace,
                        o_lat, lse=None, dev_err=None, softmax_scale=None,
                        num_splits=0)
    mla_out_unabsorb(o_lat, w_uv, o)

plus ``CacheLayer`` (one layer's pool, formats and, for the outlier-protected
format, its protected channels), ``mla_select_outlier_channels`` (their
calibration), ``mla_cache_page_layout``,
``mla_cache_pool_bytes``, ``mla_decode_workspace_bytes``,
``mla_decode_absorbed_unabsorb`` (the decode and the output projection in
one call), ``mla_decode_absorbed_noalloc`` (the decode for callers that cannot allocate),
``mla_prefill_absorbed`` / ``mla_prefill_workspace_bytes`` (causal attention
of a prefill chunk; ``mla_set_prefill_path`` / ``mla_prefill_path_taken``
choose and report its implementation: tcgen05 tensor cores or the decode
kernels) and ``mla_lse_merge`` (merges per-part results of a context-sharded decode;
the host side of that exchange is in ``sharded``).
"""

import ctypes
import math
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmla_gb300.so")

FMT_BF16, FMT_INT8_SYM, FMT_INT4_ASYM, FMT_INT4_SYM = 0, 1, 2, 3
FMT_INT8_G8, FMT_INT8_G32, FMT_INT8_G64, FMT_INT8_TOKEN = 4, 5, 6, 7    # INT8 latent, other block counts
FMT_INT8_OUTLIER = 8        # INT8 latent with OUTLIER_CHANNELS protected bf16 channels

PREFILL_AUTO = 0            # mla_set_prefill_path: tensor cores for large chunks, else decode kernels
PREFILL_DECODE_KERNELS = 1
PREFILL_TENSOR_CORES = 2
OUTLIER_CHANNELS = 25
DEVERR_SLOT, DEVERR_PAGE, DEVERR_SEQLEN, DEVERR_TIMEOUT = 1, 2, 4, 8
KV_LORA_RANK, ROPE_DIM, QK_NOPE_DIM, V_DIM, PAGE_TOKENS = 512, 64, 128, 128, 64
DEFAULT_SOFTMAX_SCALE = 1.0 / math.sqrt(QK_NOPE_DIM + ROPE_DIM)

STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "CUDA error", 4: "device bounds error"}


class MlaError(RuntimeError):
    def __init__(self, fn, status, detail=""):
        super().__init__("%s failed: %s (status %d)%s" % (fn, STATUS.get(status, "?"), status,
                                                         ": " + detail if detail else ""))
        self.status = status


class _CacheLayer(ctypes.Structure):
    _fields_ = [("num_pages", ctypes.c_int32), ("latent_fmt", ctypes.c_int32), ("kpe_fmt", ctypes.c_int32),
                ("reserved", ctypes.c_int32), ("pool", ctypes.c_void_p),
                ("outlier_channels", ctypes.POINTER(ctypes.c_int32))]


class PageLayout(ctypes.Structure):
    _fields_ = [("page_bytes", ctypes.c_int64), ("block_bytes", ctypes.c_int64), ("codes_off", ctypes.c_int64),
                ("codes_row_bytes", ctypes.c_int64),
                ("scale_off", ctypes.c_int64), ("zero_off", ctypes.c_int64), ("kpe_off", ctypes.c_int64),
                ("kpe_row_bytes", ctypes.c_int64), ("kpe_scale_off", ctypes.c_int64),
                ("bound_off", ctypes.c_int64), ("outlier_off", ctypes.c_int64)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError("libmla_gb300.so is not built: run `python mla_latent_kv_append_gb300/build.py` "
                          "(or __graft_entry__.build()) on a machine with nvcc")
    lib = ctypes.CDLL(LIB_PATH)
    P, I32, SZ, F32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t, ctypes.c_float
    CP = ctypes.POINTER(_CacheLayer)
    sig = {
        "mla_abi_version": (I32, []),
        "mla_status_string": (ctypes.c_char_p, [I32]),
        "mla_last_cuda_error": (ctypes.c_char_p, []),
        "mla_cache_page_layout": (I32, [CP, ctypes.POINTER(PageLayout)]),
        "mla_cache_pool_bytes": (SZ, [CP]),
        "mla_cache_append": (I32, [CP, P, P, P, I32, P, P]),
        "mla_q_absorb": (I32, [P, P, P, I32, I32, P]),
        "mla_decode_workspace_bytes": (SZ, [I32, I32, I32]),
        "mla_decode_absorbed": (I32, [CP, P, P, P, I32, P, I32, I32, F32, I32, P, SZ, P, P, P, P]),
        "mla_decode_absorbed_unabsorb": (I32, [CP, P, P, P, I32, P, I32, I32, F32, I32, P, SZ, P, P, P, P, P, P]),
        "mla_decode_kernel_count": (I32, [CP, I32, I32, I32, I32]),
        "mla_out_unabsorb": (I32, [P, P, P, I32, I32, P]),
        "mla_decode_absorbed_noalloc": (I32, [CP, P, P, P, I32, P, I32, I32, F32, I32, P, P, P, P]),
        "mla_lse_merge": (I32, [P, P, I32, I32, I32, P, P, P]),
        "mla_prefill_workspace_bytes": (SZ, [I32, I32]),
        "mla_prefill_absorbed": (I32, [CP, P, P, P, I32, I32, I32, I32, F32, P, SZ, P, P, P, P]),
        "mla_set_wait_limit_ns": (ctypes.c_int64, [ctypes.c_int64]),
        "mla_set_prefill_path": (I32, [I32]),
        "mla_prefill_path_taken": (I32, [I32, I32, I32]),
        "mla_select_outlier_channels": (I32, [P, I32, P, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(fn, status):
    if status != 0:
        detail = lib.mla_last_cuda_error().decode() if status == 3 else ""
        raise MlaError(fn, status, detail)


def _need(t, dtype, shape, name):
    if t.dtype != dtype or tuple(t.shape) != tuple(shape) or not t.is_contiguous() or not t.is_cuda:
        raise ValueError("%s: expected contiguous CUDA %s %s, got %s %s" % (name, dtype, tuple(shape), t.dtype,
                                                                            tuple(t.shape)))


class CacheLayer:
    """One layer's paged latent cache: a caller-owned pool tensor plus formats
    (and, for FMT_INT8_OUTLIER, the layer's OUTLIER_CHANNELS protected
    channels: a sequence of increasing ints in [0, 512))."""

    def __init__(self, num_pages, latent_fmt, kpe_fmt, device="cuda", pool=None, outlier_channels=None):
        self.num_pages, self.latent_fmt, self.kpe_fmt = int(num_pages), int(latent_fmt), int(kpe_fmt)
        self.outlier_channels = None
        if outlier_channels is not None:
            ch = [int(c) for c in outlier_channels]
            self.outlier_channels = (ctypes.c_int32 * len(ch))(*ch)
        nbytes = mla_cache_pool_bytes(self.num_pages, self.latent_fmt, self.kpe_fmt)
        if nbytes == 0:
            raise ValueError("invalid cache descriptor")
        if pool is None:
            pool = torch.zeros(nbytes, dtype=torch.uint8, device=device)
        if pool.numel() < nbytes or pool.dtype != torch.uint8 or pool.data_ptr() % 256:
            raise ValueError("pool must be a uint8 tensor of >= %d bytes, 256-byte aligned" % nbytes)
        self.pool = pool
        self.layout = mla_cache_page_layout(self.latent_fmt, self.kpe_fmt)

    def c_struct(self):
        oc = None if self.outlier_channels is None else ctypes.cast(self.outlier_channels,
                                                                      ctypes.POINTER(ctypes.c_int32))
        return _CacheLayer(self.num_pages, self.latent_fmt, self.kpe_fmt, 0, self.pool.data_ptr(), oc)


def mla_cache_page_layout(latent_fmt, kpe_fmt):
    out = PageLayout()
    c = _CacheLayer(1, latent_fmt, kpe_fmt, 0, None)
    _check("mla_cache_page_layout", lib.mla_cache_page_layout(ctypes.byref(c), ctypes.byref(out)))
    return out


def mla_cache_pool_bytes(num_pages, latent_fmt, kpe_fmt):
    c = _CacheLayer(num_pages, latent_fmt, kpe_fmt, 0, None)
    return int(lib.mla_cache_pool_bytes(ctypes.byref(c)))


def mla_select_outlier_channels(c_sample, out=None, stream=None):
    """Protected channels of FMT_INT8_OUTLIER from a calibration sample
    (bf16 [n, 512] on the GPU): the OUTLIER_CHANNELS channels with the
    largest max |x|, increasing; returns the int32 device tensor."""
    n = c_sample.shape[0]
    _need(c_sample, torch.bfloat16, (n, KV_LORA_RANK), "c_sample")
    if out is None:
        out = torch.empty(OUTLIER_CHANNELS, dtype=torch.int32, device=c_sample.device)
    _need(out, torch.int32, (OUTLIER_CHANNELS,), "out")
    _check("mla_select_outlier_channels", lib.mla_select_outlier_channels(_ptr(c_sample), n, _ptr(out),
                                                                          _stream(stream)))
    return out


def mla_decode_workspace_bytes(batch, heads, num_splits=0):
    return int(lib.mla_decode_workspace_bytes(batch, heads, num_splits))


def mla_cache_append(cache, c_new, kpe_new, slot, dev_err=None, stream=None):
    n = slot.numel()
    _need(c_new, torch.bfloat16, (n, KV_LORA_RANK), "c_new")
    _need(kpe_new, torch.bfloat16, (n, ROPE_DIM), "kpe_new")
    _need(slot, torch.int32, (n,), "slot")
    cs = cache.c_struct()
    _check("mla_cache_append", lib.mla_cache_append(ctypes.byref(cs), _ptr(c_new), _ptr(kpe_new), _ptr(slot), n,
                                                    _ptr(dev_err), _stream(stream)))


def mla_q_absorb(q_nope, w_uk, q_lat, stream=None):
    B, H = q_nope.shape[0], q_nope.shape[1]
    _need(q_nope, torch.bfloat16, (B, H, QK_NOPE_DIM), "q_nope")
    _need(w_uk, torch.bfloat16, (H, QK_NOPE_DIM, KV_LORA_RANK), "w_uk")
    _need(q_lat, torch.float32, (B, H, KV_LORA_RANK), "q_lat")
    _check("mla_q_absorb", lib.mla_q_absorb(_ptr(q_nope), _ptr(w_uk), _ptr(q_lat), B, H, _stream(stream)))


def mla_out_unabsorb(o_lat, w_uv, o, stream=None):
    B, H = o_lat.shape[0], o_lat.shape[1]
    _need(o_lat, torch.float32, (B, H, KV_LORA_RANK), "o_lat")
    _need(w_uv, torch.bfloat16, (H, KV_LORA_RANK, V_DIM), "w_uv")
    _need(o, torch.float32, (B, H, V_DIM), "o")
    _check("mla_out_unabsorb", lib.mla_out_unabsorb(_ptr(o_lat), _ptr(w_uv), _ptr(o), B, H, _stream(stream)))


def mla_decode_absorbed(cache, q_lat, q_pe, block_table, seq_lens, workspace, o_lat, lse=None, dev_err=None,
                        softmax_scale=None, num_splits=0, stream=None):
    B, H = q_lat.shape[0], q_lat.shape[1]
    _need(q_lat, torch.float32, (B, H, KV_LORA_RANK), "q_lat")
    _need(q_pe, torch.bfloat16, (B, H, ROPE_DIM), "q_pe")
    _need(block_table, torch.int32, (B, block_table.shape[1]), "block_table")
    _need(seq_lens, torch.int32, (B,), "seq_lens")
    _need(o_lat, torch.float32, (B, H, KV_LORA_RANK), "o_lat")
    if lse is not None:
        _need(lse, torch.float32, (B, H), "lse")
    scale = DEFAULT_SOFTMAX_SCALE if softmax_scale is None else float(softmax_scale)
    cs = cache.c_struct()
    _check("mla_decode_absorbed", lib.mla_decode_absorbed(
        ctypes.byref(cs), _ptr(q_lat), _ptr(q_pe), _ptr(block_table), block_table.shape[1], _ptr(seq_lens), B, H,
        scale, int(num_splits), _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(o_lat),
        _ptr(lse), _ptr(dev_err), _stream(stream)))


def mla_decode_kernel_count(cache, batch, heads, num_splits=0, with_unabsorb=False):
    cs = cache.c_struct()
    return int(lib.mla_decode_kernel_count(ctypes.byref(cs), batch, heads, num_splits, 1 if with_unabsorb else 0))


def mla_decode_absorbed_unabsorb(cache, q_lat, q_pe, block_table, seq_lens, workspace, o_lat, w_uv, o, lse=None,
                                 dev_err=None, softmax_scale=None, num_splits=0, stream=None):
    """mla_decode_absorbed then mla_out_unabsorb on its o_lat, in one call
    (the projection fused into the combine where its grid allows)."""
    B, H = q_lat.shape[0], q_lat.shape[1]
    _need(q_lat, torch.float32, (B, H, KV_LORA_RANK), "q_lat")
    _need(q_pe, torch.bfloat16, (B, H, ROPE_DIM), "q_pe")
    _need(block_table, torch.int32, (B, block_table.shape[1]), "block_table")
    _need(seq_lens, torch.int32, (B,), "seq_lens")
    _need(o_lat, torch.float32, (B, H, KV_LORA_RANK), "o_lat")
    _need(w_uv, torch.bfloat16, (H, KV_LORA_RANK, V_DIM), "w_uv")
    _need(o, torch.float32, (B, H, V_DIM), "o")
    if lse is not None:
        _need(lse, torch.float32, (B, H), "lse")
    scale = DEFAULT_SOFTMAX_SCALE if softmax_scale is None else float(softmax_scale)
    cs = cache.c_struct()
    _check("mla_decode_absorbed_unabsorb", lib.mla_decode_absorbed_unabsorb(
        ctypes.byref(cs), _ptr(q_lat), _ptr(q_pe), _ptr(block_table), block_table.shape[1], _ptr(seq_lens), B, H,
        scale, int(num_splits), _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(o_lat),
        _ptr(lse), _ptr(w_uv), _ptr(o), _ptr(dev_err), _stream(stream)))


def mla_decode_absorbed_noalloc(cache, q_lat, q_pe, block_table, seq_lens, o_lat, lse=None, dev_err=None,
                                softmax_scale=None, num_splits=0, stream=None):
    """mla_decode_absorbed without a workspace argument: for callers that
    cannot allocate device memory (see include/mla.h).  Concurrent calls on
    different streams share the library's scratch array and race."""
    B, H = q_lat.shape[0], q_lat.shape[1]
    _need(q_lat, torch.float32, (B, H, KV_LORA_RANK), "q_lat")
    _need(q_pe, torch.bfloat16, (B, H, ROPE_DIM), "q_pe")
    _need(block_table, torch.int32, (B, block_table.shape[1]), "block_table")
    _need(seq_lens, torch.int32, (B,), "seq_lens")
    _need(o_lat, torch.float32, (B, H, KV_LORA_RANK), "o_lat")
    if lse is not None:
        _need(lse, torch.float32, (B, H), "lse")
    scale = DEFAULT_SOFTMAX_SCALE if softmax_scale is None else float(softmax_scale)
    cs = cache.c_struct()
    _check("mla_decode_absorbed_noalloc", lib.mla_decode_absorbed_noalloc(
        ctypes.byref(cs), _ptr(q_lat), _ptr(q_pe), _ptr(block_table), block_table.shape[1], _ptr(seq_lens), B, H,
        scale, int(num_splits), _ptr(o_lat), _ptr(lse), _ptr(dev_err), _stream(stream)))


def mla_prefill_workspace_bytes(n, heads):
    return int(lib.mla_prefill_workspace_bytes(int(n), int(heads)))


def mla_prefill_absorbed(cache, q_lat, q_pe, block_table, ctx_before, workspace, o_lat, lse=None, dev_err=None,
                         softmax_scale=None, stream=None):
    """Causal attention of n just-appended query tokens of one sequence:
    query i (position ctx_before + i) attends to positions 0 .. ctx_before + i.
    block_table is the sequence's int32 page list [max_pages]."""
    n, H = q_lat.shape[0], q_lat.shape[1]
    _need(q_lat, torch.float32, (n, H, KV_LORA_RANK), "q_lat")
    _need(q_pe, torch.bfloat16, (n, H, ROPE_DIM), "q_pe")
    _need(block_table, torch.int32, (block_table.shape[0],), "block_table")
    _need(o_lat, torch.float32, (n, H, KV_LORA_RANK), "o_lat")
    if lse is not None:
        _need(lse, torch.float32, (n, H), "lse")
    scale = DEFAULT_SOFTMAX_SCALE if softmax_scale is None else float(softmax_scale)
    cs = cache.c_struct()
    _check("mla_prefill_absorbed", lib.mla_prefill_absorbed(
        ctypes.byref(cs), _ptr(q_lat), _ptr(q_pe), _ptr(block_table), block_table.shape[0], int(ctx_before), n, H,
        scale, _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(o_lat), _ptr(lse),
        _ptr(dev_err), _stream(stream)))


def mla_lse_merge(o_parts, lse_parts, o_lat, lse=None, stream=None):
    """Merge R per-part results (o_lat, lse) of the same sequences over
    disjoint context parts into the result over their union."""
    R, B, H = o_parts.shape[0], o_parts.shape[1], o_parts.shape[2]
    _need(o_parts, torch.float32, (R, B, H, KV_LORA_RANK), "o_parts")
    _need(lse_parts, torch.float32, (R, B, H), "lse_parts")
    _need(o_lat, torch.float32, (B, H, KV_LORA_RANK), "o_lat")
    if lse is not None:
        _need(lse, torch.float32, (B, H), "lse")
    _check("mla_lse_merge", lib.mla_lse_merge(_ptr(o_parts), _ptr(lse_parts), R, B, H, _ptr(o_lat), _ptr(lse),
                                              _stream(stream)))


def mla_set_prefill_path(path):
    """Select the prefill implementation for later calls (PREFILL_AUTO,
    PREFILL_DECODE_KERNELS or PREFILL_TENSOR_CORES); returns the previous one."""
    prev = int(lib.mla_set_prefill_path(int(path)))
    if prev < 0:
        raise ValueError("unknown prefill path %r" % (path,))
    return prev


def mla_prefill_path_taken(ctx_before, n, heads):
    """PREFILL_DECODE_KERNELS or PREFILL_TENSOR_CORES: the implementation a
    prefill call with these sizes takes under the current setting."""
    return int(lib.mla_prefill_path_taken(int(ctx_before), int(n), int(heads)))


def mla_set_wait_limit_ns(ns):
    """Bound (ns) on every wait inside the decode kernels launched afterwards;
    returns the previous bound.  A test and diagnostic hook (default 10 s)."""
    prev = int(lib.mla_set_wait_limit_ns(int(ns)))
    if prev < 0:
        raise ValueError("wait limit must be >= 0")
    return prev


def abi_version():
    return int(lib.mla_abi_version())
