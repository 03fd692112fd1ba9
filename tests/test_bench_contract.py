"""The benchmark's host side on CPU: every preset's algorithmic bytes per
token equal the library's page layout, and the reference arm (the CPU
oracle) prints one JSON line with the fields the bench contract names."""

import json
import os
import subprocess
import sys

import bench
import mla_latent_kv_append_gb300 as mla

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_preset_bytes_match_the_page_layout():
    for name, cfg in bench.CONFIGS.items():
        lf, kf = bench.FMT[cfg["latent"]], bench.FMT[cfg["kpe"]]
        assert mla.mla_cache_page_layout(lf, kf).page_bytes == 64 * bench.BETA[(cfg["latent"], cfg["kpe"])], name


def test_reference_arm_prints_the_contract_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "tiny",
                          "--steps", "2", "--warmup", "1"], capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["value"] > 0 and d["config"]["workload"] == "tiny"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]


def test_prefill_flop_count():
    """Useful flops of a prefill chunk: (query, key) pairs of the causal
    triangle (plus ctx_before keys per query) x heads x 2 x (576 + 512)."""
    import bench
    assert bench.prefill_flops(1, 1) == 2 * 1088
    assert bench.prefill_flops(2, 1) == 3 * 2 * 1088
    assert bench.prefill_flops(2, 4, ctx_before=1) == 5 * 4 * 2 * 1088
    assert bench.prefill_flops(8192, 64) == 8192 * 8193 // 2 * 64 * 2176


def test_traffic_record_follows_the_code_not_its_comments():
    """The committed ncu traffic is tied to a hash of the decode path's code:
    comments and whitespace do not change it, any code token does."""
    a = "int f(int x) {  // doubles\n  return 2 * x; /* plain */ }\n"
    b = "int f(int x)\n{\n    return 2*x;   // twice, reworded\n}\n"
    c = "int f(int x) { return 3 * x; }\n"
    assert bench.code_text(a) == bench.code_text(b)
    assert bench.code_text(a) != bench.code_text(c)
    rec = json.load(open(os.path.join(bench.ROOT, "profiles", "decode_traffic.json")))
    for name, e in rec.items():
        if name.startswith("_"):
            continue
        assert e["bytes_per_launch"] > 0
        if e["source_hash"] == bench.decode_source_hash():
            assert bench.ncu_traffic(name) == e["bytes_per_launch"]
        else:
            assert bench.ncu_traffic(name) is None
