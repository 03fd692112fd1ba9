"""GPU-resident synthetic decode workloads (tests, bench, smoke check).

A workload is L layers of paged latent caches for a batch of sequences with
given context lengths, plus per-layer weights and decode queries, all drawn
from the seeded generator.  The first T-1 tokens of every sequence are written
into the caches by the library's own quantize-on-write call; the decode step
appends token T-1 and attends over all T.  Physical pages are a seeded
permutation, so block tables are scattered as in a real pool.

A workload may also carry a prefill: P tokens of one further sequence
(index B, positions 0..P-1) that every step appends to every layer before the
decode step, into spare pages of the same pools (the mixed serving step:
prefill quantize-on-write plus batched decode).

The outlier-protected format's protected channels (per layer) come from the
library's calibration call over the rows ``synth.calibration_latent_bf16``
gives on the host (the first synth.CALIBRATION_TOKENS latent rows of
sequence 0), from which the oracle makes its own selection.

Host twins of every tensor come from ``synth`` (NumPy) for the oracle.
"""

import numpy as np
import torch

import synth
import synth.device as sd
import mla_latent_kv_append_gb300 as mla


class Workload:
    def __init__(self, layers, heads, seq_lens, latent_fmt, kpe_fmt, seed, device="cuda", fill=True,
                 fill_chunk=65536, prefill=0):
        self.L, self.H = int(layers), int(heads)
        self.seq_lens = [int(t) for t in seq_lens]
        self.B = len(self.seq_lens)
        self.latent_fmt, self.kpe_fmt, self.seed, self.device = latent_fmt, kpe_fmt, seed, device
        pages = [(t + 63) // 64 for t in self.seq_lens]
        self.max_pages = max(1, max(pages) if pages else 1)
        self.num_pages = max(1, sum(pages))
        self.prefill = int(prefill)
        self.prefill_pages = (self.prefill + 63) // 64
        perm = synth.page_permutation(seed, self.num_pages)
        bt = np.full((self.B, self.max_pages), -1, np.int32)
        k = 0
        for b, n in enumerate(pages):
            bt[b, :n] = perm[k:k + n]
            k += n
        self.block_table_host = bt
        self.block_table = torch.from_numpy(bt).to(device)
        self.seq_lens_dev = torch.tensor(self.seq_lens, dtype=torch.int32, device=device)
        self.outliers = [None] * self.L
        if latent_fmt == mla.FMT_INT8_OUTLIER:
            for l in range(self.L):
                sample = torch.empty((synth.CALIBRATION_TOKENS, synth.D_C), dtype=torch.bfloat16, device=device)
                sd.latent_into(sample, seed, l, 0, 0, sd.LayerStats(seed, l, device))
                self.outliers[l] = mla.mla_select_outlier_channels(sample).cpu().tolist()
        self.caches = [mla.CacheLayer(self.num_pages + self.prefill_pages, latent_fmt, kpe_fmt, device=device,
                                      outlier_channels=self.outliers[l])
                       for l in range(self.L)]
        self.rope = sd.RopeTables(max(1, self.prefill, max(self.seq_lens) if self.seq_lens else 1), device)
        self.w_uk = [sd.w_uk(seed, l, self.H, device) for l in range(self.L)]
        self.w_uv = [sd.w_uv(seed, l, self.H, device) for l in range(self.L)]
        self.q_nope = [sd.q_nope(seed, l, self.B, self.H, device) for l in range(self.L)]
        self.q_pe = [sd.q_pe(seed, l, self.B, self.H, device) for l in range(self.L)]
        # the decode step's new token per sequence (position T-1; skipped for T == 0)
        self.slot_new = torch.tensor([self.slot_of(b, t - 1) if t > 0 else -1 for b, t in enumerate(self.seq_lens)],
                                     dtype=torch.int32, device=device)
        self.c_new, self.kpe_new = [], []
        for l in range(self.L):
            st = sd.LayerStats(seed, l, device)
            c = torch.zeros((self.B, synth.D_C), dtype=torch.bfloat16, device=device)
            kk = torch.zeros((self.B, synth.D_R), dtype=torch.bfloat16, device=device)
            for b, t in enumerate(self.seq_lens):
                if t > 0:
                    sd.latent_into(c[b:b + 1], seed, l, b, t - 1, st, kind=synth.KIND_NEW_LATENT)
                    sd.kpe_into(kk[b:b + 1], seed, l, b, t - 1, self.rope, kind=synth.KIND_NEW_KPE)
            self.c_new.append(c)
            self.kpe_new.append(kk)
        # prefill: sequence B's P tokens, in a seeded order of the spare pages
        self.c_pre, self.kpe_pre, self.slot_pre_host = [], [], None
        if self.prefill:
            spare = self.num_pages + synth.page_permutation(seed + 1, self.prefill_pages).astype(np.int64)
            t = np.arange(self.prefill)
            self.slot_pre_host = (spare[t // 64] * 64 + t % 64).astype(np.int32)
            self.slot_pre = torch.from_numpy(self.slot_pre_host).to(device)
            # the sequence's page list, and its chunk queries (prefill attention)
            self.prefill_block_table = torch.from_numpy(spare.astype(np.int32)).to(device)
            self.q_nope_pre = [sd.prefill_q_nope(seed, l, self.prefill, self.H, device) for l in range(self.L)]
            self.q_pe_pre = [sd.prefill_q_pe(seed, l, self.prefill, self.H, device) for l in range(self.L)]
            for l in range(self.L):
                st = sd.LayerStats(seed, l, device)
                c = torch.empty((self.prefill, synth.D_C), dtype=torch.bfloat16, device=device)
                kk = torch.empty((self.prefill, synth.D_R), dtype=torch.bfloat16, device=device)
                sd.latent_into(c, seed, l, self.B, 0, st)
                sd.kpe_into(kk, seed, l, self.B, 0, self.rope)
                self.c_pre.append(c)
                self.kpe_pre.append(kk)
        self._pack_step_inputs()
        if fill:
            self.fill(fill_chunk)

    def _pack_step_inputs(self):
        """Place every per-step input (new tokens, queries, prefill tokens of
        all layers) in one device buffer, so that a host copy of a step's
        inputs is a single transfer; the per-layer tensors become views."""
        groups = [self.c_new, self.kpe_new, self.q_nope, self.q_pe, self.c_pre, self.kpe_pre]
        total = 0
        for lst in groups:
            for t in lst:
                total = (total + 255) // 256 * 256 + t.numel() * t.element_size()
        self.step_inputs = torch.empty(max(1, total), dtype=torch.uint8, device=self.device)
        off = 0
        for lst in groups:
            for i, t in enumerate(lst):
                off = (off + 255) // 256 * 256
                n = t.numel() * t.element_size()
                v = self.step_inputs[off:off + n].view(t.dtype).view(t.shape)
                v.copy_(t)
                lst[i] = v
                off += n

    def slot_of(self, b, t):
        return int(self.block_table_host[b, t // 64]) * 64 + t % 64

    def slots(self, b, t0, t1):
        t = np.arange(t0, t1)
        return (self.block_table_host[b, t // 64].astype(np.int64) * 64 + t % 64).astype(np.int32)

    def fill(self, chunk=65536):
        """Write the T-1 context tokens of every sequence into every layer."""
        dev = self.device
        for l in range(self.L):
            st = sd.LayerStats(self.seed, l, dev)
            for b, T in enumerate(self.seq_lens):
                for t0 in range(0, max(0, T - 1), chunk):
                    t1 = min(T - 1, t0 + chunk)
                    n = t1 - t0
                    c = torch.empty((n, synth.D_C), dtype=torch.bfloat16, device=dev)
                    k = torch.empty((n, synth.D_R), dtype=torch.bfloat16, device=dev)
                    sd.latent_into(c, self.seed, l, b, t0, st)
                    sd.kpe_into(k, self.seed, l, b, t0, self.rope)
                    slot = torch.from_numpy(self.slots(b, t0, t1)).to(dev)
                    mla.mla_cache_append(self.caches[l], c, k, slot)

    # ---- host twins for the oracle -------------------------------------------------
    def host_sequence(self, layer, b):
        """bf16 bits of all T tokens of sequence b (context + appended token)."""
        T = self.seq_lens[b]
        cos, sin = synth.rope_tables(max(1, T))
        return synth.sequence_bf16(self.seed, layer, b, T, cos, sin, stats=synth.channel_stats(self.seed, layer))

    def host_calibration_sample(self, layer):
        """bf16 bits of the rows the protected channels are calibrated on."""
        return synth.calibration_latent_bf16(self.seed, layer)

    def host_prefill(self, layer):
        """bf16 bits of the prefill tokens (sequence B, positions 0..P-1)."""
        cos, sin = synth.rope_tables(max(1, self.prefill))
        stats = synth.channel_stats(self.seed, layer)
        return (synth.latent_bf16(self.seed, layer, self.B, 0, self.prefill, stats=stats),
                synth.kpe_bf16(self.seed, layer, self.B, 0, self.prefill, cos, sin))

    def host_query(self, layer):
        return (synth.q_nope_bf16(self.seed, layer, self.B, self.H), synth.q_pe_bf16(self.seed, layer, self.B, self.H),
                synth.w_uk_bf16(self.seed, layer, self.H), synth.w_uv_bf16(self.seed, layer, self.H))


class DecodeStep:
    """Buffers and the per-layer call sequence of one decode step:
    [prefill append ->] append -> absorb -> decode (+ combine + unabsorb, one
    call), for every layer.  The appends and the absorb of a layer depend only on
    the layer's inputs, so the appends run on a side stream beside the
    absorb and the decode waits for both."""

    def __init__(self, wl, num_splits=0, with_lse=True):
        dev = wl.device
        self.wl, self.num_splits = wl, num_splits
        self.q_lat = torch.empty((wl.B, wl.H, synth.D_C), dtype=torch.float32, device=dev)
        self.o_lat = torch.empty((wl.B, wl.H, synth.D_C), dtype=torch.float32, device=dev)
        self.lse = torch.empty((wl.L, wl.B, wl.H), dtype=torch.float32, device=dev) if with_lse else None
        self.o = torch.empty((wl.L, wl.B, wl.H, synth.D_V), dtype=torch.float32, device=dev)
        nbytes = mla.mla_decode_workspace_bytes(wl.B, wl.H, num_splits)
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        self.dev_err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.side = torch.cuda.Stream(device=dev)

    def run(self, keep_o_lat=None):
        wl = self.wl
        main = torch.cuda.current_stream(self.q_lat.device)
        for l in range(wl.L):
            self.side.wait_stream(main)
            with torch.cuda.stream(self.side):
                if wl.prefill:
                    mla.mla_cache_append(wl.caches[l], wl.c_pre[l], wl.kpe_pre[l], wl.slot_pre, self.dev_err)
                mla.mla_cache_append(wl.caches[l], wl.c_new[l], wl.kpe_new[l], wl.slot_new, self.dev_err)
            mla.mla_q_absorb(wl.q_nope[l], wl.w_uk[l], self.q_lat)
            main.wait_stream(self.side)
            mla.mla_decode_absorbed_unabsorb(wl.caches[l], self.q_lat, wl.q_pe[l], wl.block_table, wl.seq_lens_dev,
                                             self.workspace, self.o_lat, wl.w_uv[l], self.o[l],
                                             lse=None if self.lse is None else self.lse[l], dev_err=self.dev_err,
                                             num_splits=self.num_splits)
            if keep_o_lat is not None:
                keep_o_lat[l].copy_(self.o_lat)
        return self.o


class PrefillStep:
    """Causal attention of the workload's prefill chunk (sequence B, positions
    0 .. P-1) in every layer: absorb the P queries, mla_prefill_absorbed over
    the chunk's own pages (nothing cached before it), unabsorb.  The chunk's
    tokens must already be in the cache (a DecodeStep run appends them)."""

    def __init__(self, wl):
        dev = wl.device
        P, H = wl.prefill, wl.H
        self.wl = wl
        self.q_lat = torch.empty((P, H, synth.D_C), dtype=torch.float32, device=dev)
        self.o_lat = torch.empty((P, H, synth.D_C), dtype=torch.float32, device=dev)
        self.lse = torch.empty((wl.L, P, H), dtype=torch.float32, device=dev)
        self.o = torch.empty((wl.L, P, H, synth.D_V), dtype=torch.float32, device=dev)
        self.workspace = torch.empty(mla.mla_prefill_workspace_bytes(P, H), dtype=torch.uint8, device=dev)
        self.dev_err = torch.zeros(1, dtype=torch.int32, device=dev)

    def run(self, keep_o_lat=None):
        wl = self.wl
        for l in range(wl.L):
            mla.mla_q_absorb(wl.q_nope_pre[l], wl.w_uk[l], self.q_lat)
            mla.mla_prefill_absorbed(wl.caches[l], self.q_lat, wl.q_pe_pre[l], wl.prefill_block_table, 0,
                                     self.workspace, self.o_lat, self.lse[l], self.dev_err)
            if keep_o_lat is not None:
                keep_o_lat[l].copy_(self.o_lat)
            mla.mla_out_unabsorb(self.o_lat, wl.w_uv[l], self.o[l])
        return self.o
