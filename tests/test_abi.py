"""The C ABI without a GPU: the library loads, exports every function that
include/mla.h declares, computes layouts and sizes, and rejects bad arguments
on the host before any launch (no kernel runs in these tests)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mla.h")


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    try:
        __graft_entry__.build()
    except RuntimeError as e:  # pragma: no cover - needs nvcc
        pytest.skip("cannot build: %s" % e)
    import mla_latent_kv_append_gb300 as mla
    return mla


def declared_functions():
    src = open(HEADER, encoding="utf-8").read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 9
    raw = ctypes.CDLL(lib.LIB_PATH)
    for n in names:
        assert hasattr(raw, n), n
    assert lib.abi_version() == 107


def test_layouts_match_the_accounting(lib):
    from oracle import accounting as acc
    pairs = [(lf, kf) for lf in (0, 1, 2, 3) for kf in (0, 1, 3)] + [(lf, 1) for lf in (4, 5, 6, 7)]
    for lf, kf in pairs:
        L = lib.mla_cache_page_layout(lf, kf)
        # the pages' bytes with metadata, plus the 4-byte bound of a quantized latent
        assert L.page_bytes == 64 * (acc.layer_bytes(lf, kf, metadata=True) + (4 if lf != 0 else 0))
        for off in (L.codes_off, L.scale_off, L.zero_off, L.kpe_off, L.kpe_scale_off, L.bound_off):
            assert off == -1 or off % 128 == 0
        assert (L.zero_off == -1) == (lf != 2)
        assert (L.bound_off == -1) == (lf == 0)
        assert L.bound_off == -1 or L.bound_off + 32 * 4 == L.block_bytes
    for lf in (4, 5, 6, 7):                           # other block counts: INT8 k_pe only
        for kf in (0, 3):
            with pytest.raises(lib.MlaError):
                lib.mla_cache_page_layout(lf, kf)
    assert lib.mla_cache_pool_bytes(10, 1, 1) == 10 * 64 * 740
    assert lib.mla_cache_pool_bytes(10, 2, 3) == 10 * 64 * 580   # the 7.6 KB-per-token scheme, with metadata
    assert lib.mla_cache_pool_bytes(0, 1, 1) == 0
    assert lib.mla_cache_pool_bytes(4, 9, 1) == 0
    assert lib.mla_cache_pool_bytes(4, 1, 2) == 0     # asymmetric INT4 k_pe is not a cache format


def test_workspace_size(lib):
    # explicit split count: no device query needed
    G, B, H = 10, 3, 16
    slots = G + B
    align = lambda x: (x + 255) // 256 * 256
    # chunk prefix sums, spans, then per slot and head: max, sum, the weight
    # of the fp16 P V products, and the 512-wide unnormalised output
    expect = align((B + 1) * 4) + align(2 * B * 4) + 3 * align(slots * H * 4) + slots * H * 512 * 4
    assert lib.mla_decode_workspace_bytes(B, H, G) == expect
    assert lib.mla_decode_workspace_bytes(B, 24, G) == 0
    assert lib.mla_decode_workspace_bytes(5000, 16, G) == 0
    assert lib.mla_decode_workspace_bytes(B, H, 65536) == 0        # more splits than the grid allows


def test_invalid_arguments_rejected_on_host(lib):
    raw = lib.lib
    fake = ctypes.c_void_p(0x10000)          # never dereferenced: checks fail first
    cs = lib._CacheLayer(4, 1, 1, 0, 0x100000)
    # n < 0
    assert raw.mla_cache_append(ctypes.byref(cs), fake, fake, fake, -1, None, None) == 1
    # misaligned c_new
    assert raw.mla_cache_append(ctypes.byref(cs), ctypes.c_void_p(0x10002), fake, fake, 4, None, None) == 1
    # bad pool alignment
    bad = lib._CacheLayer(4, 1, 1, 0, 0x100010)
    assert raw.mla_cache_append(ctypes.byref(bad), fake, fake, fake, 4, None, None) == 1
    # heads not a multiple of 16
    assert raw.mla_q_absorb(fake, fake, fake, 2, 24, None) == 1
    assert raw.mla_out_unabsorb(fake, fake, fake, 2, 8, None) == 1
    # n == 0 / batch == 0 are no-ops that launch nothing
    assert raw.mla_cache_append(ctypes.byref(cs), None, None, None, 0, None, None) == 0
    assert raw.mla_q_absorb(None, None, None, 0, 16, None) == 0
    # decode: workspace too small, bad softmax scale, batch too large
    args = lambda ws_bytes, scale, B: (ctypes.byref(cs), fake, fake, fake, 4, fake, B, 16, scale, 3,
                                       ctypes.c_void_p(0x200000), ws_bytes, fake, None, None, None)
    assert raw.mla_decode_absorbed(*args(16, 0.07, 2)) == 1
    assert raw.mla_decode_absorbed(*args(1 << 30, 0.0, 2)) == 1
    assert raw.mla_decode_absorbed(*args(1 << 30, 0.07, 5000)) == 1
    assert raw.mla_decode_absorbed(*args(1 << 30, 0.07, 0)) == 0
    # the decode with the output projection: both of w_uv and o, 16-byte aligned
    fused = lambda w, o: (ctypes.byref(cs), fake, fake, fake, 4, fake, 2, 16, 0.07, 3, ctypes.c_void_p(0x200000),
                          1 << 30, fake, None, w, o, None, None)
    assert raw.mla_decode_absorbed_unabsorb(*fused(None, fake)) == 1
    assert raw.mla_decode_absorbed_unabsorb(*fused(fake, None)) == 1
    assert raw.mla_decode_absorbed_unabsorb(*fused(ctypes.c_void_p(0x10008), fake)) == 1
    # decode: the batch's chunk capacity B * max_pages * 2 must stay below 2^31
    big = (ctypes.byref(cs), fake, fake, fake, 1 << 18, fake, 4096, 16, 0.07, 3, ctypes.c_void_p(0x200000), 1 << 40,
           fake, None, None, None)
    assert raw.mla_decode_absorbed(*big) == 1
    # merge: part count out of range, output overlapping the parts
    a16 = ctypes.c_void_p(0x10000)
    assert raw.mla_lse_merge(a16, a16, 0, 2, 16, ctypes.c_void_p(0x900000), None, None) == 1
    assert raw.mla_lse_merge(a16, a16, 5000, 2, 16, ctypes.c_void_p(0x900000), None, None) == 1
    assert raw.mla_lse_merge(a16, a16, 2, 2, 16, ctypes.c_void_p(0x10000 + 4096), None, None) == 1
    assert raw.mla_lse_merge(a16, a16, 2, 0, 16, a16, None, None) == 0
    # prefill: n < 0, ctx_before < 0, bad heads, chunk past the block table,
    # workspace too small, bad softmax scale, misaligned q_lat; n == 0 is a no-op
    ws = ctypes.c_void_p(0x200000)
    pre = lambda q, bt_pages, ctx, n, H, scale, ws_bytes: (ctypes.byref(cs), q, fake, fake, bt_pages, ctx, n, H, scale,
                                                           ws, ws_bytes, fake, None, None, None)
    assert raw.mla_prefill_absorbed(*pre(fake, 4, 0, -1, 16, 0.07, 1 << 40)) == 1
    assert raw.mla_prefill_absorbed(*pre(fake, 4, -1, 8, 16, 0.07, 1 << 40)) == 1
    assert raw.mla_prefill_absorbed(*pre(fake, 4, 0, 8, 24, 0.07, 1 << 40)) == 1
    assert raw.mla_prefill_absorbed(*pre(fake, 4, 250, 7, 16, 0.07, 1 << 40)) == 1     # 257 > 4 pages * 64
    assert raw.mla_prefill_absorbed(*pre(fake, 4, 0, 8, 16, 0.07, 64)) == 1
    assert raw.mla_prefill_absorbed(*pre(fake, 4, 0, 8, 16, float("nan"), 1 << 40)) == 1
    assert raw.mla_prefill_absorbed(*pre(ctypes.c_void_p(0x10004), 4, 0, 8, 16, 0.07, 1 << 40)) == 1
    assert raw.mla_prefill_absorbed(*pre(None, 4, 0, 0, 16, 0.07, 0)) == 0
    assert raw.mla_prefill_workspace_bytes(-1, 16) == 0
    assert raw.mla_prefill_workspace_bytes(8, 24) == 0
    assert raw.mla_prefill_workspace_bytes(100, 16) <= raw.mla_prefill_workspace_bytes(5000, 16)
    assert raw.mla_prefill_workspace_bytes(5000, 16) == raw.mla_prefill_workspace_bytes(50000, 16)
    assert raw.mla_status_string(4) == b"device-side bounds error"


def test_prefill_path_hook(lib):
    """The prefill path setting: set, read back, reject an unknown value,
    and the workspace size it implies (the tensor-core path adds the key
    tiles of 65536 positions and the query tiles of a 4096-token slice, 288
    KB per 128 rows, to per-row check figures)."""
    prev = lib.mla_set_prefill_path(lib.PREFILL_DECODE_KERNELS)
    try:
        dec = lib.mla_prefill_workspace_bytes(8192, 64)
        assert lib.mla_set_prefill_path(lib.PREFILL_TENSOR_CORES) == lib.PREFILL_DECODE_KERNELS
        tile = 9 * 2 * 16384
        rows = 4096 * 64
        # the queue of long rows for the split exact recomputation: counters,
        # 64 items, 64 x 32 ranges x 8 heads x (2 + 512) floats
        queue = 512 + 1024 + 64 * 32 * 8 * 514 * 4 + 256 * 576 * 4    # + x_hat of the first 256 positions
        tc = 512 * tile + rows // 128 * tile + 65536 * 4 + 4096 * 4 + rows * 4 + rows * 8 + queue
        assert lib.mla_prefill_workspace_bytes(8192, 64) == max(tc, dec)
        # a 100-token chunk at 16 heads: one 1600-row slice, 13 row tiles
        tc_small = 512 * tile + 13 * tile + 65536 * 4 + 512 + 6400 + 12800 + queue
        assert lib.mla_prefill_workspace_bytes(100, 16) == max(tc_small, lib.mla_prefill_workspace_bytes(1, 16))
        assert lib.mla_prefill_path_taken(10**6, 8192, 64) == lib.PREFILL_TENSOR_CORES
        assert lib.mla_set_prefill_path(lib.PREFILL_AUTO) == lib.PREFILL_TENSOR_CORES
        assert lib.mla_prefill_path_taken(0, 8192, 64) == lib.PREFILL_TENSOR_CORES
        assert lib.mla_prefill_path_taken(65536 - 8191, 8192, 64) == lib.PREFILL_DECODE_KERNELS
        assert lib.mla_prefill_path_taken(0, 200, 64) == lib.PREFILL_DECODE_KERNELS      # every row < 256 tokens
        assert lib.mla_prefill_path_taken(300, 100, 16) == lib.PREFILL_DECODE_KERNELS    # 1600 rows
        assert lib.mla_prefill_path_taken(8192, 128, 16) == lib.PREFILL_TENSOR_CORES     # 2048 rows, long prefixes
        assert lib.mla_prefill_path_taken(1024, 128, 16) == lib.PREFILL_DECODE_KERNELS   # 2048 rows, short prefixes
        assert lib.mla_prefill_path_taken(0, 512, 16) == lib.PREFILL_TENSOR_CORES        # 8192 rows
        assert lib.mla_prefill_path_taken(0, 8192, 24) == -1
        # automatic: the tensor-core size only from 2048 rows on
        assert lib.mla_prefill_workspace_bytes(100, 16) < tc_small
        assert lib.mla_prefill_workspace_bytes(8192, 64) == max(tc, dec)
        with pytest.raises(ValueError):
            lib.mla_set_prefill_path(7)
    finally:
        lib.mla_set_prefill_path(prev)
    assert prev == lib.PREFILL_AUTO


def test_wait_limit_hook(lib):
    """The wait-limit hook only sets a host-side value: set, read back,
    reject a negative limit, restore."""
    prev = lib.mla_set_wait_limit_ns(12345)
    try:
        assert lib.mla_set_wait_limit_ns(777) == 12345
        with pytest.raises(ValueError):
            lib.mla_set_wait_limit_ns(-1)
        assert lib.mla_set_wait_limit_ns(777) == 777
    finally:
        lib.mla_set_wait_limit_ns(prev)
    assert prev == 10 ** 10


def test_outlier_format_descriptor_rules(lib):
    """INT8_OUTLIER layouts, and the host checks of the protected set: present,
    25 strictly increasing channels in [0, 512), absent for other formats."""
    from oracle import accounting as acc
    for kf in (0, 1):
        L = lib.mla_cache_page_layout(8, kf)
        # the pages' 690 B (+64 for INT8 k_pe) and scales, the bound, 2 B of padding
        assert L.page_bytes == 64 * (acc.layer_bytes(8, kf, metadata=True) + 4 + 2)
        assert L.outlier_off == L.scale_off + 32 * 32 * 4 and L.outlier_off % 128 == 0
        assert L.kpe_off == L.outlier_off + 1664
    assert lib.mla_cache_pool_bytes(2, 8, 3) == 0                 # 4-bit k_pe is not offered with it
    assert lib.mla_cache_page_layout(1, 1).outlier_off == -1
    raw = lib.lib
    fake = ctypes.c_void_p(0x10000)
    good = list(range(0, 500, 20))
    assert len(good) == 25

    def call(fmt, channels):
        arr = None if channels is None else (ctypes.c_int32 * len(channels))(*channels)
        cs = lib._CacheLayer(4, fmt, 0, 0, 0x100000,
                             None if arr is None else ctypes.cast(arr, ctypes.POINTER(ctypes.c_int32)))
        return raw.mla_cache_append(ctypes.byref(cs), fake, fake, fake, 0, None, None)   # n = 0: no launch
    assert call(8, good) == 0
    assert call(8, None) == 1
    assert call(8, [good[1]] + [good[0]] + good[2:]) == 1       # not increasing
    assert call(8, good[:24] + [good[23]]) == 1                  # repeated
    assert call(8, good[:24] + [512]) == 1                       # out of range
    assert call(8, [-1] + good[1:]) == 1
    assert call(1, good) == 1                                    # other formats take none
    assert call(1, None) == 0
    assert raw.mla_select_outlier_channels(fake, 0, fake, None) == 1
    assert raw.mla_select_outlier_channels(ctypes.c_void_p(0x10002), 4, fake, None) == 1


def test_decode_kernel_count(lib):
    """Kernels per decode call: split kernel + combine, plus the unabsorb
    kernel unless the combine's per-head grid projects the rows itself."""
    cnt = lambda lf, B, H, G, u: lib.lib.mla_decode_kernel_count(
        ctypes.byref(lib._CacheLayer(4, lf, 1 if lf else 0, 0, 0x100000)), B, H, G, u)
    assert cnt(1, 8, 16, 152, 0) == 2
    assert cnt(1, 8, 16, 152, 1) == 2        # ~19 splits per sequence: per-head grid, fused
    assert cnt(1, 32, 16, 152, 1) == 3       # grouped grid: separate unabsorb
    assert cnt(0, 1, 16, 152, 1) == 3        # bf16, one long sequence: channel-sliced grid
    assert cnt(1, 1, 16, 152, 1) == 2        # quantized: per-head grid (the exact path needs whole rows)
    assert cnt(1, 0, 16, 152, 1) == 0
    assert cnt(1, 8, 24, 152, 1) == -1
    assert cnt(9, 8, 16, 152, 1) == -1
