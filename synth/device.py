"""Device twin of the host generator (libmla_synth.so, built from synth_gen.cu).

Fills torch CUDA tensors with exactly the values synth/__init__.py produces on
the host, for workloads too large to generate in NumPy.
"""

import ctypes
import os

import numpy as np
import torch

import synth

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmla_synth.so")

_lib = None


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError("libmla_synth.so is not built (run mla_latent_kv_append_gb300.build)")
        L = ctypes.CDLL(LIB_PATH)
        U64, I32, F32, P = ctypes.c_uint64, ctypes.c_int32, ctypes.c_float, ctypes.c_void_p
        L.synth_latent_bf16.argtypes = [U64, I32, I32, I32, P, P, F32, P, P]
        L.synth_kpe_bf16.argtypes = [U64, I32, I32, I32, P, P, F32, P, P]
        L.synth_normal3_bf16.argtypes = [U64, I32, I32, I32, F32, F32, P, P]
        for f in (L.synth_latent_bf16, L.synth_kpe_bf16, L.synth_normal3_bf16):
            f.restype = ctypes.c_int
        _lib = L
    return _lib


def _s():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _ok(rc):
    if rc != 0:
        raise RuntimeError("synth kernel launch failed (%d)" % rc)


class LayerStats:
    """Per-layer channel statistics uploaded once."""

    def __init__(self, seed, layer, device="cuda"):
        mu, sigma = synth.channel_stats(seed, layer)
        self.mu = torch.from_numpy(mu).to(device)
        self.sigma = torch.from_numpy(sigma).to(device)


class RopeTables:
    def __init__(self, n_pos, device="cuda"):
        cos, sin = synth.rope_tables(n_pos)
        self.n_pos = n_pos
        self.cos = torch.from_numpy(cos).to(device)
        self.sin = torch.from_numpy(sin).to(device)


def latent_into(out, seed, layer, b, t0, stats, kind=synth.KIND_LATENT):
    """out: bf16 CUDA tensor [n, 512] <- latent rows t0..t0+n-1 of sequence b."""
    n = out.shape[0]
    key = synth.stream_key(seed, layer, kind)
    _ok(lib().synth_latent_bf16(key, b, t0, n, stats.mu.data_ptr(), stats.sigma.data_ptr(),
                                float(synth.NORMAL_SCALE), out.data_ptr(), _s()))


def kpe_into(out, seed, layer, b, t0, rope, kind=synth.KIND_KPE):
    n = out.shape[0]
    if t0 + n > rope.n_pos:
        raise ValueError("rope table too short")
    key = synth.stream_key(seed, layer, kind)
    _ok(lib().synth_kpe_bf16(key, b, t0, n, rope.cos.data_ptr(), rope.sin.data_ptr(), float(synth.NORMAL_SCALE),
                             out.data_ptr(), _s()))


def normal3_into(out, seed, layer, kind, mul):
    d0, d1, d2 = out.shape
    key = synth.stream_key(seed, layer, kind)
    _ok(lib().synth_normal3_bf16(key, d0, d1, d2, float(np.float32(mul)), float(synth.NORMAL_SCALE),
                                 out.data_ptr(), _s()))


def q_nope(seed, layer, B, H, device="cuda"):
    t = torch.empty((B, H, synth.D_NOPE), dtype=torch.bfloat16, device=device)
    normal3_into(t, seed, layer, synth.KIND_QNOPE, synth.UNIT_SCALE)
    return t


def q_pe(seed, layer, B, H, device="cuda"):
    t = torch.empty((B, H, synth.D_R), dtype=torch.bfloat16, device=device)
    normal3_into(t, seed, layer, synth.KIND_QPE, synth.UNIT_SCALE)
    return t


def prefill_q_nope(seed, layer, n, H, device="cuda"):
    t = torch.empty((n, H, synth.D_NOPE), dtype=torch.bfloat16, device=device)
    normal3_into(t, seed, layer, synth.KIND_PRE_QNOPE, synth.UNIT_SCALE)
    return t


def prefill_q_pe(seed, layer, n, H, device="cuda"):
    t = torch.empty((n, H, synth.D_R), dtype=torch.bfloat16, device=device)
    normal3_into(t, seed, layer, synth.KIND_PRE_QPE, synth.UNIT_SCALE)
    return t


def w_uk(seed, layer, H, device="cuda"):
    t = torch.empty((H, synth.D_NOPE, synth.D_C), dtype=torch.bfloat16, device=device)
    normal3_into(t, seed, layer, synth.KIND_WUK, synth.WEIGHT_SCALE)
    return t


def w_uv(seed, layer, H, device="cuda"):
    t = torch.empty((H, synth.D_C, synth.D_V), dtype=torch.bfloat16, device=device)
    normal3_into(t, seed, layer, synth.KIND_WUV, synth.WEIGHT_SCALE)
    return t
