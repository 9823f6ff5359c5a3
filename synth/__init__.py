"""Seeded synthetic inputs for the W4A4 MXFP4 MoE layer (shared by oracle and CUDA path).

Holds no arithmetic of the layer itself: it only draws the random tensors the
layer consumes.  Workloads follow the DeepSeek-V4-Flash expert layer that the
pages "[deepseek-v4] Bump sgl-deep-gemm for packed FP4xFP4 mega-MoE (W4A4)"
(Appendix, measured data) describe: hidden 4096, inter 2048, 256 experts,
top-6, plus one tiny shape for exhaustive checks.

Recipes (seed 0 everywhere unless a caller says otherwise):
  x        bf16 bits of fp32(N(0,1)); the large-prefill case multiplies
           round(0.001*T*H) distinct positions by 50 before rounding.
  routing  k distinct experts per token, uniform (partial Fisher-Yates) or
           Zipf s=1.1 by popularity rank e+1 (sequential draws without
           replacement); weights = softmax of k N(0,1) draws, fp32.
  weights  fp32 N(0, 1/sqrt(K)) per expert, K = H for the gate/up projection
           [2I, H] (gate rows first, then up rows), K = I for the down
           projection [H, I].
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mxsynth.c")
_LIB = os.path.join(_HERE, "libmxsynth.so")


def build(force: bool = False) -> str:
    """Compile libmxsynth.so next to its source (plain C, portable flags)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=gnu11", "-fPIC", "-shared", "-ffp-contract=off", "-pthread",
             _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        l = ctypes.CDLL(build())
        u64, i64, i32, dbl = ctypes.c_uint64, ctypes.c_int64, ctypes.c_int32, ctypes.c_double
        vp = ctypes.c_void_p
        l.synth_normal_f32.argtypes = [u64, u64, u64, u64, dbl, vp, ctypes.c_int]
        l.synth_normal_bf16.argtypes = [u64, u64, u64, u64, dbl, vp, ctypes.c_int]
        l.synth_hidden_bf16.argtypes = [u64, i64, i64, i64, dbl, vp, ctypes.c_int]
        l.synth_hidden_bf16.restype = ctypes.c_int
        l.synth_routing_uniform.argtypes = [u64, i64, i32, i32, vp, vp]
        l.synth_routing_uniform.restype = ctypes.c_int
        l.synth_routing_zipf.argtypes = [u64, i64, i32, i32, dbl, vp, vp]
        l.synth_routing_zipf.restype = ctypes.c_int
        l.synth_expert_weights_f32.argtypes = [u64, i32, i32, i64, i64, i64, dbl, vp, ctypes.c_int]
        _lib = l
    return _lib


def _threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    I: int
    E: int
    k: int
    routing: str = "uniform"   # or "zipf"
    zipf_s: float = 1.1
    outlier_frac: float = 0.0
    outlier_mult: float = 50.0

    @property
    def n_outliers(self) -> int:
        return int(round(self.outlier_frac * self.T * self.H))


# The five workloads: a tiny exhaustive case and four DeepSeek-V4-Flash layers.
WORKLOADS = {
    "tiny": Workload("tiny", T=16, H=256, I=128, E=8, k=2),
    "decode_T64": Workload("decode_T64", T=64, H=4096, I=2048, E=256, k=6),
    "layer_T512": Workload("layer_T512", T=512, H=4096, I=2048, E=256, k=6),
    "prefill_T4096": Workload("prefill_T4096", T=4096, H=4096, I=2048, E=256, k=6),
    "prefill_T16384_zipf": Workload("prefill_T16384_zipf", T=16384, H=4096, I=2048, E=256, k=6,
                                    routing="zipf", outlier_frac=0.001),
}


def _ptr(a: np.ndarray) -> int:
    assert a.flags.c_contiguous
    return a.ctypes.data


def hidden_bf16(w: Workload, seed: int = 0) -> np.ndarray:
    """x [T, H] as uint16 bf16 bits."""
    out = np.empty((w.T, w.H), dtype=np.uint16)
    rc = lib().synth_hidden_bf16(seed, w.T, w.H, w.n_outliers, w.outlier_mult, _ptr(out), _threads())
    if rc != 0:
        raise RuntimeError(f"synth_hidden_bf16 failed ({rc})")
    return out


def routing(w: Workload, seed: int = 0):
    """(topk_ids int32 [T, k], topk_weights float32 [T, k])."""
    ids = np.empty((w.T, w.k), dtype=np.int32)
    wt = np.empty((w.T, w.k), dtype=np.float32)
    if w.routing == "uniform":
        rc = lib().synth_routing_uniform(seed, w.T, w.k, w.E, _ptr(ids), _ptr(wt))
    elif w.routing == "zipf":
        rc = lib().synth_routing_zipf(seed, w.T, w.k, w.E, w.zipf_s, _ptr(ids), _ptr(wt))
    else:
        raise ValueError(w.routing)
    if rc != 0:
        raise RuntimeError(f"routing generation failed ({rc})")
    return ids, wt


def expert_w1_f32(w: Workload, expert: int, seed: int = 0, first_row: int = 0,
                  num_rows: int | None = None, out: np.ndarray | None = None) -> np.ndarray:
    """Gate/up weights of one expert, fp32 [2I, H] (rows 0..I-1 gate, I..2I-1 up)."""
    rows = 2 * w.I if num_rows is None else num_rows
    if out is None:
        out = np.empty((rows, w.H), dtype=np.float32)
    lib().synth_expert_weights_f32(seed, 1, expert, w.H, first_row, rows, 1.0 / np.sqrt(w.H),
                                   _ptr(out), _threads())
    return out


def expert_w2_f32(w: Workload, expert: int, seed: int = 0, first_row: int = 0,
                  num_rows: int | None = None, out: np.ndarray | None = None) -> np.ndarray:
    """Down-projection weights of one expert, fp32 [H, I]."""
    rows = w.H if num_rows is None else num_rows
    if out is None:
        out = np.empty((rows, w.I), dtype=np.float32)
    lib().synth_expert_weights_f32(seed, 2, expert, w.I, first_row, rows, 1.0 / np.sqrt(w.I),
                                   _ptr(out), _threads())
    return out


def normals_f32(seed: int, stream: int, count: int, sigma: float = 1.0, first: int = 0) -> np.ndarray:
    """Raw N(0, sigma) fp32 draws of a named stream (for tests that need plain data)."""
    out = np.empty(count, dtype=np.float32)
    lib().synth_normal_f32(seed, stream, first, count, sigma, _ptr(out), _threads())
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32 (a bit shift, not arithmetic)."""
    return (bits.astype(np.uint32) << 16).view(np.float32)
