"""Benchmark: absorbed MLA decode over a quantized paged latent cache.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference] [--aux]

A step is one decode step of the whole model: for every layer, append the new
token of every sequence (quantize-on-write), absorb the query, run the
split-K decode + log-sum-exp combine, and un-absorb the output.  The step is
captured in a CUDA graph and timed with CUDA events on its stream after W
warm-up replays; the per-step working set (the whole cache) is larger than
L2, so no flush is needed between steps.  Inputs are synthetic and seeded
(DeepSeek-V2-Lite shapes, random-init weights); caches are resident in HBM
before the timed region.  Prints one JSON line on rank 0.

--impl reference times the CPU oracle (NumPy, fp64 attention) on the same
workload: each step is a bounded sample (one sequence through all layers,
layers spread over the host cores).

--aux times, instead of the step, the two calls that are not part of it:
the merge of a context-sharded decode (mla_lse_merge) and the outlier
format's calibration (mla_select_outlier_channels); one JSON line of GB/s
against the measured HBM peak.
"""

import argparse
import hashlib
import re
import json
import math
import multiprocessing as mp
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

# name -> (layers, heads, seq_lens spec, latent fmt, kpe fmt, description)
CONFIGS = {
    "v2lite_int8": dict(layers=27, heads=16, batch=8, ctx=4096, latent="int8", kpe="int8",
                        desc="DeepSeek-V2-Lite shapes, 27 layers, 16 heads, batch 8, context 4096, "
                             "INT8 latent (32 groups) + INT8 k_pe, 64-token pages"),
    "v2lite_int4_32k": dict(layers=27, heads=16, batch=32, ctx=32768, latent="int4", kpe="int8",
                            desc="V2-Lite shapes, batch 32, context 32768, asymmetric INT4 latent + INT8 k_pe"),
    "v2lite_int8_32k": dict(layers=27, heads=16, batch=32, ctx=32768, latent="int8", kpe="int8",
                            desc="V2-Lite shapes, batch 32, context 32768, INT8 latent (32 groups) + INT8 k_pe"),
    "v2lite_int4_kpe4_32k": dict(layers=27, heads=16, batch=32, ctx=32768, latent="int4", kpe="int4sym",
                                 desc="V2-Lite shapes, batch 32, context 32768, asymmetric INT4 latent + "
                                      "symmetric INT4 k_pe (the 7.6 KB-per-token scheme; 580 B per token-layer "
                                      "with scales, zero-points and the bound)"),
    "v2lite_int4sym_32k": dict(layers=27, heads=16, batch=32, ctx=32768, latent="int4sym", kpe="int8",
                               desc="V2-Lite shapes, batch 32, context 32768, symmetric INT4 latent + INT8 k_pe"),
    # the English report's block-count sweep (8 / 32 / 64 blocks) and the
    # per-token row, on the V2-Lite INT8 workload
    "v2lite_int8_8blocks": dict(layers=27, heads=16, batch=8, ctx=4096, latent="int8g64", kpe="int8",
                                desc="V2-Lite INT8 workload with 8 blocks of 64 latent channels"),
    "v2lite_int8_16blocks": dict(layers=27, heads=16, batch=8, ctx=4096, latent="int8g32", kpe="int8",
                                 desc="V2-Lite INT8 workload with 16 blocks of 32 latent channels"),
    "v2lite_int8_64blocks": dict(layers=27, heads=16, batch=8, ctx=4096, latent="int8g8", kpe="int8",
                                 desc="V2-Lite INT8 workload with 64 blocks of 8 latent channels"),
    "v2lite_int8_per_token": dict(layers=27, heads=16, batch=8, ctx=4096, latent="int8tok", kpe="int8",
                                  desc="V2-Lite INT8 workload with one scale per token (per-token INT8)"),
    # the English report's §4.3 row C (outlier-protected mixed precision) on
    # the V2-Lite INT8 workload: 25 protected bf16 channels per layer, bf16 k_pe
    "v2lite_int8_outlier": dict(layers=27, heads=16, batch=8, ctx=4096, latent="int8out", kpe="bf16",
                                desc="DeepSeek-V2-Lite shapes, batch 8, context 4096, INT8 latent with 25 "
                                     "protected bf16 channels (calibrated per layer) + bf16 k_pe"),
    "long_int4_1m": dict(layers=27, heads=16, batch=1, ctx=1048576, latent="int4", kpe="int8",
                         desc="V2-Lite shapes, batch 1, context 1,048,576, asymmetric INT4 latent + INT8 k_pe"),
    "long_bf16_256k": dict(layers=27, heads=16, batch=1, ctx=262144, latent="bf16", kpe="bf16",
                           desc="V2-Lite shapes, batch 1, context 262,144, bf16 latent + bf16 k_pe"),
    "mixed_h64_int8": dict(layers=1, heads=64, batch=64, ctx="loguniform", latent="int8", kpe="int8", prefill=8192,
                           desc="mixed serving step: prefill append of 8192 tokens + decode of batch 64 with "
                                "context log-uniform in [1K, 64K], 64 heads, INT8 latent + k_pe"),
    "mixed_h64_int4": dict(layers=1, heads=64, batch=64, ctx="loguniform", latent="int4", kpe="int8", prefill=8192,
                           desc="mixed serving step: prefill append of 8192 tokens + decode of batch 64 with "
                                "context log-uniform in [1K, 64K], 64 heads, INT4 latent + INT8 k_pe"),
    "mixed_h64_bf16": dict(layers=1, heads=64, batch=64, ctx="loguniform", latent="bf16", kpe="bf16", prefill=8192,
                           desc="mixed serving step: prefill append of 8192 tokens + decode of batch 64 with "
                                "context log-uniform in [1K, 64K], 64 heads, bf16 latent + k_pe"),
    "tiny": dict(layers=1, heads=16, batch=1, ctx=256, latent="int8", kpe="int8",
                 desc="1 layer, 16 heads, batch 1, context 256"),
}
FMT = {"bf16": 0, "int8": 1, "int4": 2, "int4sym": 3, "int8g8": 4, "int8g32": 5, "int8g64": 6, "int8tok": 7,
       "int8out": 8}
def _beta(latent, kpe):
    """Stored bytes per token and layer (codes + fp32 scales / zero-points +
    the fp32 bound of a quantized latent), as laid out in include/mla.h:
    32 latent groups of 16, 8 k_pe groups of 8."""
    # int8out: 512 codes + 25 protected bf16 values, their field padded to 52 B a token
    code = {"bf16": 1024, "int4": 256, "int4sym": 256, "int8out": 512 + 52}.get(latent, 512)
    groups = {"int8g8": 64, "int8g32": 16, "int8g64": 8, "int8tok": 1}.get(latent, 32)
    meta = {"bf16": 0, "int4": 8 * groups + 4}.get(latent, 4 * groups + 4)
    kcode = {"bf16": 128, "int8": 64, "int4sym": 32}[kpe]
    kmeta = 0 if kpe == "bf16" else 32
    return code + meta + kcode + kmeta


BETA = {(a, b): _beta(a, b) for a in ("bf16", "int8", "int4", "int4sym") for b in ("bf16", "int8", "int4sym")}
BETA.update({(a, "int8"): _beta(a, "int8") for a in ("int8g8", "int8g32", "int8g64", "int8tok")})
BETA.update({("int8out", b): _beta("int8out", b) for b in ("bf16", "int8")})
METRIC = "decode tokens/s & achieved HBM GB/s (% of GB300 peak) for absorbed MLA decode"
SEED = 0x4D4C41
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def seq_lens_for(cfg, seed):
    if cfg["ctx"] == "loguniform":
        import synth
        return [int(t) for t in synth.log_uniform_lengths(seed, cfg["batch"], 1024, 65536)]
    return [int(cfg["ctx"])] * cfg["batch"]


def hbm_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def tensor_peak():
    """Dense 16-bit tensor peak (TFLOP/s) for a kernel timed alone: the burst
    cuBLAS figure of MEASURED_PEAKS.json (fp16 and bf16 run at one rate)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


def prefill_flops(P, H, ctx_before=0):
    """Useful absorbed-attention flops of a P-token chunk: each of the
    sum_i (ctx_before + i + 1) (query, key) pairs per head costs a 576-wide
    score dot product and a 512-wide P V update (2 flops per multiply-add)."""
    pairs = P * ctx_before + P * (P + 1) // 2
    return pairs * H * 2 * (576 + 512)


def code_text(src):
    """Source text without comments and whitespace: what the compiler sees."""
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    return re.sub(r"\s+", "", src)


def decode_source_hash():
    """Hash of the decode path's code (comments and whitespace ignored)."""
    h = hashlib.sha256()
    for name in ("decode.cu", "decode_mma.cu", "mla_internal.cuh"):
        p = os.path.join(ROOT, "mla_latent_kv_append_gb300", "csrc", name)
        if os.path.exists(p):
            h.update(code_text(open(p, encoding="utf-8").read()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(config_name):
    """DRAM bytes per decode launch from the committed ncu summary, if it was
    taken on the current decode source; else None."""
    p = os.path.join(ROOT, "profiles", "decode_traffic.json")
    try:
        with open(p) as f:
            rec = json.load(f)
        e = rec.get(config_name)
        if e and e.get("source_hash") == decode_source_hash():
            return e.get("bytes_per_launch")
    except Exception:
        pass
    return None


# ----------------------------------------------------------------------------------
# clocks sampled during the timed region
# ----------------------------------------------------------------------------------
class Clocks:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            # the timed region starts once the sampler is running (first line written)
            t0 = time.time()
            while time.time() - t0 < 5 and os.path.getsize(self.path) == 0 and self.proc.poll() is None:
                time.sleep(0.05)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------------
# the oracle on the host (cpu_baseline and --impl reference)
# ----------------------------------------------------------------------------------
def _oracle_worker(conn, cfg, seq_lens, tasks, seed):
    os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
    import numpy as np
    import synth
    from oracle import attention as A
    from oracle import quant as Q
    lf, kf = FMT[cfg["latent"]], FMT[cfg["kpe"]]
    H, B = cfg["heads"], len(seq_lens)
    P = cfg.get("prefill", 0)
    state = []
    for (l, b) in tasks:                     # untimed: the cache as the step finds it
        T = seq_lens[b]
        cos, sin = synth.rope_tables(max(1, T))
        c_bits, k_bits = synth.sequence_bf16(seed, l, b, T, cos, sin)
        c, k = synth.bf16_to_f32(c_bits), synth.bf16_to_f32(k_bits)
        outl = None                          # the layer's protected channels (outlier format)
        if lf == Q.FMT_INT8_OUTLIER:
            outl = Q.select_outlier_channels(synth.bf16_to_f32(synth.calibration_latent_bf16(seed, l)))
        stored = Q.quantize_token_rows(c[:T - 1], k[:T - 1], lf, kf, outliers=outl)
        q = [synth.bf16_to_f32(a) for a in (synth.q_nope_bf16(seed, l, B, H)[b:b + 1],
                                             synth.q_pe_bf16(seed, l, B, H)[b:b + 1],
                                             synth.w_uk_bf16(seed, l, H), synth.w_uv_bf16(seed, l, H))]
        pre = None
        if P:                                # the prefill tokens this layer appends every step
            pcos, psin = synth.rope_tables(P)
            st = synth.channel_stats(seed, l)
            pre = (synth.bf16_to_f32(synth.latent_bf16(seed, l, B, 0, P, stats=st)),
                   synth.bf16_to_f32(synth.kpe_bf16(seed, l, B, 0, P, pcos, psin)))
        state.append((stored, c[T - 1:], k[T - 1:], q, pre, outl))
    conn.send("ready")
    while True:
        msg = conn.recv()
        if msg == "stop":
            break
        t0 = time.perf_counter()
        for stored, c_new, k_new, (qn, qp, wuk, wuv), pre, outl in state:
            if pre is not None:
                Q.quantize_token_rows(pre[0], pre[1], lf, kf, outliers=outl)      # prefill append
            new = Q.quantize_token_rows(c_new, k_new, lf, kf, outliers=outl)    # append the new token
            c_hat = np.concatenate([_dequant_latent(Q, stored, lf, outl), new["c_hat"]])
            kpe_hat = np.concatenate([_dequant_kpe(Q, stored, kf), new["kpe_hat"]])
            A.absorbed_decode_full(qn[0], qp[0], wuk, wuv, c_hat, kpe_hat)
        conn.send(time.perf_counter() - t0)


def _dequant_latent(Q, stored, lf, outl=None):
    if lf == 1:
        return Q.dequantize_sym_int8(stored["c_codes"], stored["c_scale"], 16)
    if lf == Q.FMT_INT8_OUTLIER:
        return Q.dequantize_int8_outlier(stored["c_codes"], stored["c_scale"], stored["c_outlier"], outl, 16)
    if lf == 2:
        return Q.dequantize_asym_int4(stored["c_codes"], stored["c_scale"], stored["c_zero"], 16)
    if lf == 3:
        return Q.dequantize_sym_int4(stored["c_codes"], stored["c_scale"], 16)
    return stored["c_hat"]                      # bf16 cache: the values themselves


def _dequant_kpe(Q, stored, kf):
    if kf == 1:
        return Q.dequantize_sym_int8(stored["kpe_codes"], stored["kpe_scale"], 8)
    if kf == 3:
        return Q.dequantize_sym_int4(stored["kpe_codes"], stored["kpe_scale"], 8)
    return stored["kpe_hat"]


class OracleRunner:
    """Worker processes (spawned, one BLAS thread each) that together run the
    oracle's decode step for one sequence through all layers."""

    def __init__(self, cfg, seq_lens, seed, workers=None):
        n = workers or min(os.cpu_count() or 1, cfg["layers"], 16)
        self.n = n
        tasks = [[] for _ in range(n)]
        for l in range(cfg["layers"]):
            tasks[l % n].append((l, 0))
        ctx = mp.get_context("spawn")
        self.procs, self.conns = [], []
        for w in range(n):
            a, b = ctx.Pipe()
            p = ctx.Process(target=_oracle_worker, args=(b, cfg, seq_lens, tasks[w], seed), daemon=True)
            p.start()
            self.procs.append(p)
            self.conns.append(a)
        for c in self.conns:
            assert c.recv() == "ready"

    def step(self):
        t0 = time.perf_counter()
        for c in self.conns:
            c.send("go")
        for c in self.conns:
            c.recv()
        return time.perf_counter() - t0

    def close(self):
        for c in self.conns:
            c.send("stop")
        for p in self.procs:
            p.join(timeout=10)


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo), or None."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu model")):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return None


def cpu_baseline(cfg, seq_lens, min_seconds=8.0, steps=None, warmup=1):
    r = OracleRunner(cfg, seq_lens, SEED)
    for _ in range(warmup):
        r.step()
    times = []
    t_start = time.perf_counter()
    while True:
        times.append(r.step())
        if steps is not None and len(times) >= steps:
            break
        if steps is None and time.perf_counter() - t_start >= min_seconds and len(times) >= 2:
            break
    r.close()
    total = sum(times)
    return {"value": len(times) / total, "unit": "tokens/s", "cores": r.n, "kind": "oracle",
            "workers": r.n, "host_cores": os.cpu_count(), "cpu_model": cpu_model(),
            "sample": "sequence 0 through all %d layers per step (context %d)%s, layers spread over %d "
                      "spawned single-BLAS-thread processes; %d steps, %.1f s" % (
                          cfg["layers"], seq_lens[0],
                          (" plus the %d-token prefill append" % cfg["prefill"]) if cfg.get("prefill") else "",
                          r.n, len(times), total),
            "ms_per_step": 1000 * total / len(times), "steps": len(times)}


# ----------------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------------
def run_ours(args, cfg, rank, world, local_rank):
    import torch
    import mla_latent_kv_append_gb300 as mla
    from synth.workload import DecodeStep, PrefillStep, Workload

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    seed = SEED + rank
    seq_lens = seq_lens_for(cfg, seed)
    layers = args.layers or cfg["layers"]
    t_setup = time.time()
    wl = Workload(layers, cfg["heads"], seq_lens, FMT[cfg["latent"]], FMT[cfg["kpe"]], seed, device=dev,
                  prefill=cfg.get("prefill", 0))
    step = DecodeStep(wl, num_splits=args.num_splits)
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        step.run()                                    # eager once (configures kernels)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step.run()
    torch.cuda.synchronize()
    setup_s = time.time() - t_setup

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            graph.replay()
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    clocks = Clocks(local_rank)
    clocks.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(args.steps):
            graph.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = e0.elapsed_time(e1) / args.steps
    if world > 1:
        import torch.distributed as dist
        t = torch.tensor([ms], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    err_word = int(step.dev_err.item())

    # ---- the decode call (split-K kernel + combine) timed alone: a CUDA graph
    # of the L per-layer decode calls (each reads its own layer's cache, so
    # the sequence is not L2-resident), replayed on the same stream
    dgraph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(dgraph, stream=stream):
        for l in range(wl.L):
            mla.mla_decode_absorbed(wl.caches[l], step.q_lat, wl.q_pe[l], wl.block_table, wl.seq_lens_dev,
                                    step.workspace, step.o_lat, step.lse[l], step.dev_err,
                                    num_splits=args.num_splits)
    reps = max(3, min(50, args.steps))
    with torch.cuda.stream(stream):
        dgraph.replay()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            dgraph.replay()
        b.record(stream)
    torch.cuda.synchronize()
    dec_ms = a.elapsed_time(b) / (reps * wl.L)

    # ---- the prefill append (mixed serving step) timed alone: one graph of R
    # appends, each from its own input copy into its own pages of a scratch
    # pool, so that the R x (inputs + pages) working set exceeds L2
    pre = None
    if wl.prefill:
        import numpy as np
        R, P, pp = 16, wl.prefill, wl.prefill_pages
        tcache = mla.CacheLayer(R * pp, wl.latent_fmt, wl.kpe_fmt, device=dev)
        t = np.arange(P)
        sets = [(wl.c_pre[0].clone(), wl.kpe_pre[0].clone(),
                 torch.from_numpy(((t // 64 + r * pp) * 64 + t % 64).astype(np.int32)).to(dev)) for r in range(R)]
        pgraph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(pgraph, stream=stream):
            for c_in, k_in, sl in sets:
                mla.mla_cache_append(tcache, c_in, k_in, sl, step.dev_err)
        with torch.cuda.stream(stream):
            pgraph.replay()
            a.record(stream)
            for _ in range(reps):
                pgraph.replay()
            b.record(stream)
        torch.cuda.synchronize()
        pre_ms = a.elapsed_time(b) / (reps * R)
        del sets, tcache
        beta_w = BETA[(cfg["latent"], cfg["kpe"])]
        pre_bytes = wl.prefill * ((512 + 64) * 2 + 4 + beta_w)     # bf16 rows + slot in, cache bytes out
        peak0, _ = hbm_peak()
        pre = {"bound": "hbm", "tokens": wl.prefill, "bytes_per_launch": pre_bytes, "launch_ms": pre_ms,
               "achieved": pre_bytes / (pre_ms * 1e-3) / 1e9, "peak": peak0, "unit": "GB/s",
               "frac": pre_bytes / (pre_ms * 1e-3) / 1e9 / peak0}

    # ---- the prefill chunk's causal attention (mixed serving step): absorb
    # the P queries, mla_prefill_absorbed over the chunk, unabsorb; the
    # attention call is also timed alone.  Its cache pages (a few MB) stay in
    # L2: this part is bound by the tensor pipe, not by HBM.
    pattn = None
    if wl.prefill:
        pstep = PrefillStep(wl)
        with torch.cuda.stream(stream):
            pstep.run()
        torch.cuda.synchronize()
        fgraph, agraph = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(fgraph, stream=stream):
            pstep.run()
        with torch.cuda.graph(agraph, stream=stream):
            mla.mla_prefill_absorbed(wl.caches[0], pstep.q_lat, wl.q_pe_pre[0], wl.prefill_block_table, 0,
                                     pstep.workspace, pstep.o_lat, pstep.lse[0], pstep.dev_err)
        preps = 3
        with torch.cuda.stream(stream):
            fgraph.replay()
            a.record(stream)
            for _ in range(preps):
                fgraph.replay()
            b.record(stream)
        torch.cuda.synchronize()
        full_ms = a.elapsed_time(b) / (preps * wl.L)
        with torch.cuda.stream(stream):
            a.record(stream)
            for _ in range(preps):
                agraph.replay()
            b.record(stream)
        torch.cuda.synchronize()
        attn_ms = a.elapsed_time(b) / preps
        path = mla.mla_prefill_path_taken(0, wl.prefill, wl.H)
        # the other implementation of the same call, for comparison
        other = mla.PREFILL_DECODE_KERNELS if path == mla.PREFILL_TENSOR_CORES else mla.PREFILL_TENSOR_CORES
        prev_path = mla.mla_set_prefill_path(other)
        ows = torch.empty(mla.mla_prefill_workspace_bytes(wl.prefill, wl.H), dtype=torch.uint8, device="cuda")
        ograph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(ograph, stream=stream):
            mla.mla_prefill_absorbed(wl.caches[0], pstep.q_lat, wl.q_pe_pre[0], wl.prefill_block_table, 0,
                                     ows, pstep.o_lat, pstep.lse[0], pstep.dev_err)
        mla.mla_set_prefill_path(prev_path)
        with torch.cuda.stream(stream):
            ograph.replay()
            a.record(stream)
            for _ in range(preps):
                ograph.replay()
            b.record(stream)
        torch.cuda.synchronize()
        other_ms = a.elapsed_time(b) / preps
        del ograph, ows
        flops = prefill_flops(wl.prefill, wl.H)
        tpk, tpk_kind = tensor_peak()
        achieved_t = flops / (attn_ms * 1e-3) / 1e12
        pattn = {"bound": "tensor", "tokens": wl.prefill, "heads": wl.H, "flops_per_launch": flops,
                 "launch_ms": attn_ms, "achieved": achieved_t, "peak": tpk, "unit": "TFLOP/s",
                 "frac": achieved_t / tpk, "peak_source": "%s bf16_tflops (MEASURED_PEAKS.json)" % tpk_kind,
                 "ms_with_absorb_unabsorb": full_ms, "device_error_word": int(pstep.dev_err.item()),
                 "kernel": ("mla_prefill_absorbed (tcgen05 tensor-core path: key tiles, query split, "
                            "128x128 tiles, exact fixup)" if path == mla.PREFILL_TENSOR_CORES else
                            "mla_prefill_absorbed (split-K decode kernels over the causal prefixes + combine)"),
                 ("decode_kernels_ms" if other == mla.PREFILL_DECODE_KERNELS else "tensor_cores_ms"): other_ms}
        del pstep, fgraph, agraph
        torch.cuda.empty_cache()

    # ---- end to end through the public API with host buffers
    # every step's inputs of all layers live in one device buffer
    # (wl.step_inputs): one pinned host buffer, one copy in, one copy out
    host_in = torch.empty(wl.step_inputs.shape, dtype=torch.uint8, pin_memory=True).copy_(wl.step_inputs.cpu())
    host_out = torch.empty(step.o.shape, dtype=step.o.dtype, pin_memory=True)
    h2d = host_in.numel()
    d2h = host_out.numel() * host_out.element_size()
    e2e_steps = max(3, min(args.steps, 50))
    done = torch.cuda.Event()
    torch.cuda.synchronize()
    barrier()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for _ in range(e2e_steps):
            wl.step_inputs.copy_(host_in, non_blocking=True)
            graph.replay()
            host_out.copy_(step.o, non_blocking=True)
            done.record(stream)
            done.synchronize()
    e2e_s = (time.perf_counter() - t0) / e2e_steps
    if world > 1:
        import torch.distributed as dist
        t = torch.tensor([e2e_s], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        e2e_s = float(t.item())

    tokens_per_step = wl.B * world
    beta = BETA[(cfg["latent"], cfg["kpe"])]
    cache_bytes_launch = sum(seq_lens) * beta
    peak, peak_kind = hbm_peak()
    achieved = cache_bytes_launch / (dec_ms * 1e-3) / 1e9
    weight_bytes = 2 * cfg["heads"] * 128 * 512 * 2
    step_bytes = layers * (cache_bytes_launch + weight_bytes)
    out = {
        "metric": METRIC,
        "value": tokens_per_step / (ms * 1e-3),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16" if cfg["latent"] != "bf16" else "bf16",
        "data": "synthetic (seeded; DeepSeek-V2-Lite shapes, random-init weights)",
        "config": {"workload": args.config, "description": cfg["desc"],
                   "arithmetic": "f16 MMA on exact integer codes, f32 accumulate" if cfg["latent"] != "bf16"
                   else "bf16 MMA, f32 accumulate",
                   "layers": layers, "heads": cfg["heads"],
                   "batch_per_gpu": wl.B, "context": (seq_lens[0] if len(set(seq_lens)) == 1 else
                                                      "log-uniform, mean %d" % (sum(seq_lens) // len(seq_lens))),
                   "latent_fmt": cfg["latent"], "kpe_fmt": cfg["kpe"], "page_tokens": 64,
                   "num_splits": args.num_splits or "auto",
                   "l2": "no flush: each step reads %.0f MB of cache, > 129 MB L2" % (step_bytes / 1e6),
                   "parallelism": "replicas by sequence (dp%d)" % world, "cuda_graph": True},
        "cache_gbs": achieved,
        "step_gbs": step_bytes / (ms * 1e-3) / 1e9,
        "hbm_frac_of_peak": achieved / peak,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": ncu_traffic(args.config),
                     "kernel": "mla_decode_absorbed (split-K decode + LSE combine)",
                     "bytes_per_launch": cache_bytes_launch, "launch_ms": dec_ms,
                     "peak_source": "%s hbm_gbs (MEASURED_PEAKS.json)" % peak_kind if peak_kind == "measured"
                     else "fallback 6.8 TB/s"},
        "e2e": {"value": tokens_per_step / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        # per layer: append (and the prefill's append), absorb, then the
        # decode call's kernels (the unabsorb is fused into the combine for
        # some batch shapes)
        "gpu_launches": args.steps * layers * ((3 if wl.prefill else 2) + mla.mla_decode_kernel_count(
            wl.caches[0], wl.B, wl.H, args.num_splits, with_unabsorb=True)),
        "device_error_word": err_word,
        "clocks": clk,
        "prefill_append": pre,
        "prefill_attention": pattn,
        "setup_s": round(setup_s, 1),
    }
    return out, seq_lens


def aux_kernels(steps):
    """The two calls off the decode step: the merge of a context-sharded
    decode (mla_lse_merge, one launch per layer and step on the gathered
    parts) and the outlier format's calibration (mla_select_outlier_channels,
    once per layer).  Each is timed alone, warm, with CUDA events on its
    stream over `steps` calls; achieved = algorithmic bytes / call time (the
    small cases stay in L2 between calls; the largest merge does not)."""
    import torch
    import synth
    import mla_latent_kv_append_gb300 as mla
    dev = torch.device("cuda")
    clocks = Clocks(torch.cuda.current_device())
    clocks.start()
    stream = torch.cuda.Stream()
    peak, peak_kind = hbm_peak()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def timed(fn):
        with torch.cuda.stream(stream):
            for _ in range(3):
                fn()
            a.record(stream)
            for _ in range(steps):
                fn()
            b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / steps

    out = {"merge": [], "select_outliers": []}
    g = torch.Generator(device=dev)
    g.manual_seed(SEED)
    for desc, (R, B, H) in [("V2-Lite INT4 32K batch, one layer, 8 context shards", (8, 32, 16)),
                            ("one long sequence, one layer, 8 context shards", (8, 1, 16)),
                            ("4096 sequences x 16 heads, 8 shards (> L2)", (8, 4096, 16))]:
        o_parts = torch.randn((R, B, H, mla.KV_LORA_RANK), generator=g, device=dev)
        lse_parts = torch.randn((R, B, H), generator=g, device=dev) * 4
        o_lat = torch.empty((B, H, mla.KV_LORA_RANK), device=dev)
        lse = torch.empty((B, H), device=dev)
        ms = timed(lambda: mla.mla_lse_merge(o_parts, lse_parts, o_lat, lse, stream=stream))
        nbytes = (R + 1) * B * H * (4 * mla.KV_LORA_RANK + 4)
        gbs = nbytes / (ms * 1e-3) / 1e9
        out["merge"].append({"workload": desc, "parts": R, "batch": B, "heads": H, "bytes_per_launch": nbytes,
                             "launch_us": ms * 1e3, "achieved": gbs, "frac": gbs / peak})
        del o_parts, lse_parts, o_lat, lse
    for n in (synth.CALIBRATION_TOKENS, 65536):
        sample = (torch.randn((n, mla.KV_LORA_RANK), generator=g, device=dev) * 3).to(torch.bfloat16)
        chans = torch.empty(mla.OUTLIER_CHANNELS, dtype=torch.int32, device=dev)
        ms = timed(lambda: mla.mla_select_outlier_channels(sample, chans, stream=stream))
        nbytes = n * 2 * mla.KV_LORA_RANK + 4 * mla.OUTLIER_CHANNELS
        gbs = nbytes / (ms * 1e-3) / 1e9
        out["select_outliers"].append({"tokens": n, "bytes_per_launch": nbytes, "launch_us": ms * 1e3,
                                       "achieved": gbs, "frac": gbs / peak,
                                       "note": "one CTA by design (a calibration call, off the step)"})
    return {"aux": "calls off the decode step", "unit": "GB/s", "peak": peak,
            "peak_source": "%s hbm_gbs (MEASURED_PEAKS.json)" % peak_kind, "steps": steps,
            "clocks": clocks.stop(), **out}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="v2lite_int4_32k", choices=sorted(CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--layers", type=int, default=0, help="override the layer count (testing only)")
    ap.add_argument("--num-splits", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--aux", action="store_true",
                    help="time the merge and calibration calls (one JSON line) instead of the step")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    cfg = CONFIGS[args.config]

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return 0
        seq_lens = seq_lens_for(cfg, SEED)
        if args.layers:
            cfg = dict(cfg, layers=args.layers)
        steps = max(1, args.steps)
        cb = cpu_baseline(cfg, seq_lens, steps=steps, warmup=max(1, min(args.warmup, 3)))
        value = cb["value"] * world
        line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
                "steps": steps, "warmup": args.warmup, "ms_per_step": cb["ms_per_step"], "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic (seeded; DeepSeek-V2-Lite shapes, random-init weights)",
                "config": {"workload": args.config, "description": cfg["desc"],
                           "arithmetic": "f64 attention / fp32 quantization"},
                "cpu_baseline": cb, "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                                            "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return 0

    if args.aux:
        if rank == 0:
            import torch
            torch.cuda.set_device(local_rank)
            print(json.dumps(aux_kernels(max(1, args.steps))))
        return 0
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    out, seq_lens = run_ours(args, cfg, rank, world, local_rank)
    if rank == 0:
        if not args.no_cpu_baseline and world == 1:
            c = dict(cfg, layers=args.layers or cfg["layers"])
            out["cpu_baseline"] = cpu_baseline(c, seq_lens)
        print(json.dumps(out))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
