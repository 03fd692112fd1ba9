"""Build the CUDA shared libraries in-tree with nvcc (sm_103a only).

    python mla_latent_kv_append_gb300/build.py          # library + synth generator

Translation units compile in parallel, then link into
``mla_latent_kv_append_gb300/libmla_gb300.so`` and ``synth/libmla_synth.so``.
A target is rebuilt only when one of its sources or headers is newer.
"""

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
BUILD = os.path.join(ROOT, "_build")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "-Xptxas", "-v" if os.environ.get("MLA_PTXAS_VERBOSE") else "-O3",
         "--expt-relaxed-constexpr"]

LIB = os.path.join(PKG, "libmla_gb300.so")
SYNTH_LIB = os.path.join(ROOT, "synth", "libmla_synth.so")


def nvcc():
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src, obj, deps):
    if not _stale(obj, [src] + deps):
        return obj, ""
    tmp = obj + ".tmp%d" % os.getpid()
    cmd = [nvcc()] + ARCH + FLAGS + ["-c", src, "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, r.stdout, r.stderr))
    os.replace(tmp, obj)        # an interrupted compile leaves no object that looks current
    return obj, r.stdout + r.stderr


def _link(objs, out):
    tmp = out + ".tmp%d" % os.getpid()
    cmd = [nvcc()] + ARCH + ["-shared", "-Xcompiler", "-fPIC", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed for %s:\n%s\n%s" % (out, r.stdout, r.stderr))
    os.replace(tmp, out)        # readers see the old library or the new one, never a partial file


def build_target(srcs, headers, out, tag, verbose=False):
    os.makedirs(BUILD, exist_ok=True)
    objs = [os.path.join(BUILD, "%s_%s.o" % (tag, os.path.splitext(os.path.basename(s))[0])) for s in srcs]
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        logs = list(ex.map(lambda so: _compile(so[0], so[1], headers), zip(srcs, objs)))
    if verbose:
        for _, log in logs:
            if log.strip():
                print(log)
    if _stale(out, objs):
        _link(objs, out)
    return out


def build(verbose=False):
    csrc = os.path.join(PKG, "csrc")
    srcs = sorted(glob.glob(os.path.join(csrc, "*.cu")))
    headers = sorted(glob.glob(os.path.join(csrc, "*.cuh"))) + [os.path.join(ROOT, "include", "mla.h")]
    synth_src = [os.path.join(ROOT, "synth", "synth_gen.cu")]
    with cf.ThreadPoolExecutor(max_workers=2) as ex:
        f1 = ex.submit(build_target, srcs, headers, LIB, "mla", verbose)
        f2 = ex.submit(build_target, synth_src, [], SYNTH_LIB, "synth", verbose)
        return f1.result(), f2.result()


if __name__ == "__main__":
    for p in build(verbose="-v" in sys.argv):
        print(p)
