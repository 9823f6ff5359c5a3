"""Python access to the CPU oracle (test infrastructure only).

Only tests, the smoke check and the benchmark's CPU-baseline leg import this
package.  The CUDA library never links or calls it.  The arithmetic lives in
mxmoe_oracle.cpp; this module only compiles it and marshals numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mxmoe_oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")


def build(force: bool = False) -> str:
    """Compile liboracle.so (plain C++17, asserts on, no fast-math, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-ffp-contract=off", "-pthread",
             _SRC, "-o", tmp])
        os.replace(tmp, _LIB)
    return _LIB


class Shape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("H", ctypes.c_int64), ("I", ctypes.c_int64),
                ("E", ctypes.c_int64), ("k", ctypes.c_int64)]


_lib = None


def lib():
    global _lib
    if _lib is None:
        l = ctypes.CDLL(build())
        vp, i64, ci = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        l.oracle_e2m1_value.argtypes = [ci]
        l.oracle_e2m1_value.restype = ctypes.c_double
        l.oracle_mx_exponent.argtypes = [ctypes.c_double]
        l.oracle_mx_exponent.restype = ci
        l.oracle_e2m1_encode.argtypes = [ctypes.c_double]
        l.oracle_e2m1_encode.restype = ci
        l.oracle_quantize_f32.argtypes = [vp, i64, i64, vp, vp, ci]
        l.oracle_quantize_bf16.argtypes = [vp, i64, i64, vp, vp, ci]
        l.oracle_dequantize.argtypes = [vp, vp, i64, i64, vp]
        l.oracle_bf16_round.argtypes = [ctypes.c_double]
        l.oracle_bf16_round.restype = ctypes.c_uint16
        l.oracle_interleave_source_row.argtypes = [i64, i64]
        l.oracle_interleave_source_row.restype = i64
        l.oracle_scale_block_offset.argtypes = [i64, i64, i64]
        l.oracle_scale_block_offset.restype = i64
        l.oracle_bucket.argtypes = [vp, i64, i64, i64, vp, vp, vp, vp]
        l.oracle_bucket.restype = i64
        l.oracle_moe.argtypes = [ctypes.POINTER(Shape)] + [vp] * 15 + [ci]
        l.oracle_moe.restype = i64
        l.oracle_moe_down.argtypes = [ctypes.POINTER(Shape)] + [vp] * 8 + [ci]
        l.oracle_e4m3_value.argtypes = [ci]
        l.oracle_e4m3_value.restype = ctypes.c_double
        l.oracle_mxfp8_exponent.argtypes = [ctypes.c_double]
        l.oracle_mxfp8_exponent.restype = ci
        l.oracle_e4m3_encode.argtypes = [ctypes.c_double]
        l.oracle_e4m3_encode.restype = ci
        l.oracle_mxfp8_quantize_bf16.argtypes = [vp, i64, i64, vp, vp, ci]
        l.oracle_mxfp8_quantize_f32.argtypes = [vp, i64, i64, vp, vp, ci]
        l.oracle_mxfp8_dequantize.argtypes = [vp, vp, i64, i64, vp]
        l.oracle_interleave_source_row_gran8.argtypes = [i64, i64]
        l.oracle_interleave_source_row_gran8.restype = i64
        l.oracle_moe_w4a8.argtypes = [ctypes.POINTER(Shape)] + [vp] * 15 + [ci]
        l.oracle_moe_w4a8.restype = i64
        l.oracle_moe_w4a8_down.argtypes = [ctypes.POINTER(Shape)] + [vp] * 8 + [ci]
        l.oracle_nvfp4_quantize_f32.argtypes = [vp, i64, i64, vp, vp, ci]
        l.oracle_nvfp4_quantize_bf16.argtypes = [vp, i64, i64, vp, vp, ci]
        l.oracle_nvfp4_dequantize.argtypes = [vp, vp, i64, i64, vp]
        l.oracle_moe_nvf4.argtypes = [ctypes.POINTER(Shape)] + [vp] * 15 + [ci]
        l.oracle_moe_nvf4.restype = i64
        _lib = l
    return _lib


def threads() -> int:
    return max(1, min(64, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity")
                      else (os.cpu_count() or 1)))


def _p(a):
    if a is None:
        return None
    assert isinstance(a, np.ndarray) and a.flags.c_contiguous, "need C-contiguous numpy array"
    return a.ctypes.data


def e2m1_value(code: int) -> float:
    return lib().oracle_e2m1_value(int(code))


def mx_exponent(amax: float) -> int:
    return lib().oracle_mx_exponent(float(amax))


def e2m1_encode(q: float) -> int:
    return lib().oracle_e2m1_encode(float(q))


def bf16_round(v: float) -> int:
    return int(lib().oracle_bf16_round(float(v)))


def quantize_f32(x: np.ndarray, nthreads: int | None = None):
    x = np.ascontiguousarray(x, dtype=np.float32)
    rows, K = x.shape
    codes = np.empty((rows, K // 2), np.uint8)
    sf = np.empty((rows, K // 32), np.uint8)
    lib().oracle_quantize_f32(_p(x), rows, K, _p(codes), _p(sf), nthreads or threads())
    return codes, sf


def quantize_bf16(bits: np.ndarray, nthreads: int | None = None):
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    rows, K = bits.shape
    codes = np.empty((rows, K // 2), np.uint8)
    sf = np.empty((rows, K // 32), np.uint8)
    lib().oracle_quantize_bf16(_p(bits), rows, K, _p(codes), _p(sf), nthreads or threads())
    return codes, sf


def dequantize(codes: np.ndarray, sf: np.ndarray) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    sf = np.ascontiguousarray(sf, dtype=np.uint8)
    rows, half = codes.shape
    out = np.empty((rows, half * 2), np.float64)
    lib().oracle_dequantize(_p(codes), _p(sf), rows, half * 2, _p(out))
    return out


def e4m3_value(code: int) -> float:
    return float(lib().oracle_e4m3_value(int(code)))


def mxfp8_exponent(amax: float) -> int:
    return int(lib().oracle_mxfp8_exponent(float(amax)))


def e4m3_encode(q: float) -> int:
    return int(lib().oracle_e4m3_encode(float(q)))


def mxfp8_quantize_bf16(bits: np.ndarray, nthreads: int | None = None):
    """bf16 bits [rows, K] -> (E4M3 codes [rows, K] uint8, scale bytes [rows, K/32] uint8)."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    rows, K = bits.shape
    q = np.zeros((rows, K), np.uint8)
    sf = np.zeros((rows, K // 32), np.uint8)
    lib().oracle_mxfp8_quantize_bf16(_p(bits), rows, K, _p(q), _p(sf), nthreads or threads())
    return q, sf


def mxfp8_packed_scales(sf: np.ndarray) -> np.ndarray:
    """Scale bytes [rows, K/32] -> packed int32 [rows, K/128] (groups 4j..4j+3 in bytes 0..3)."""
    rows, kc = sf.shape
    assert kc % 4 == 0
    b = sf.astype(np.uint32).reshape(rows, kc // 4, 4)
    return (b[..., 0] | (b[..., 1] << 8) | (b[..., 2] << 16) | (b[..., 3] << 24)).astype(np.uint32)


def mxfp8_quantize_f32(x: np.ndarray, nthreads: int | None = None):
    """fp32 [rows, K] -> (E4M3 codes [rows, K] uint8, scale bytes [rows, K/32] uint8)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    rows, K = x.shape
    q = np.zeros((rows, K), np.uint8)
    sf = np.zeros((rows, K // 32), np.uint8)
    lib().oracle_mxfp8_quantize_f32(_p(x), rows, K, _p(q), _p(sf), nthreads or threads())
    return q, sf


def mxfp8_dequantize(q: np.ndarray, sf: np.ndarray) -> np.ndarray:
    q = np.ascontiguousarray(q, np.uint8)
    sf = np.ascontiguousarray(sf, np.uint8)
    rows, K = q.shape
    out = np.zeros((rows, K), np.float64)
    lib().oracle_mxfp8_dequantize(_p(q), _p(sf), rows, K, _p(out))
    return out


def interleave_source_rows(I: int, gran: int = 16) -> np.ndarray:
    """src[r] = canonical row of the first weight that lands at prepared row r: gran=16
    (even/odd, MXFP4 activations) or gran=8 (contiguous, FP8 activations)."""
    fn = {16: lib().oracle_interleave_source_row, 8: lib().oracle_interleave_source_row_gran8}[gran]
    return np.array([fn(r, I) for r in range(2 * I)], np.int64)


def scale_block_offset(r: int, s: int, Kc: int) -> int:
    return int(lib().oracle_scale_block_offset(r, s, Kc))


def scale_block_layout(sf: np.ndarray) -> np.ndarray:
    """Canonical scales [rows, Kc] -> bytes of the 128x4 block layout (rows padded to 128, pad = 0)."""
    rows, Kc = sf.shape
    assert Kc % 4 == 0
    nb = (rows + 127) // 128
    out = np.zeros(nb * 128 * Kc, np.uint8)
    l = lib()
    for r in range(rows):
        for s in range(Kc):
            out[l.oracle_scale_block_offset(r, s, Kc)] = sf[r, s]
    return out


def bucket(ids: np.ndarray, E: int):
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    T, k = ids.shape
    counts = np.zeros(E, np.int64)
    offsets = np.zeros(E + 1, np.int64)
    st = np.full(T * k, -1, np.int32)
    sj = np.full(T * k, -1, np.int32)
    bad = lib().oracle_bucket(_p(ids), T, k, E, _p(counts), _p(offsets), _p(st), _p(sj))
    n = int(offsets[-1])
    return counts, offsets, st[:n], sj[:n], int(bad)


def moe(x_bf16, ids, tw, w1_codes, w1_sf, w2_codes, w2_sf, *, want_intermediates: bool = False,
        want_y: bool = False, nthreads: int | None = None) -> dict:
    """Run the whole layer.  Weights are canonical MXFP4 arrays:
    w1_codes [E, 2I, H/2], w1_sf [E, 2I, H/32], w2_codes [E, H, I/2], w2_sf [E, H, I/32]."""
    x_bf16 = np.ascontiguousarray(x_bf16, np.uint16)
    ids = np.ascontiguousarray(ids, np.int32)
    tw = np.ascontiguousarray(tw, np.float32)
    T, H = x_bf16.shape
    k = ids.shape[1]
    E, twoI, _ = w1_codes.shape
    I = twoI // 2
    A = T * k
    arrs = [np.ascontiguousarray(a, np.uint8) for a in (w1_codes, w1_sf, w2_codes, w2_sf)]
    assert arrs[0].shape == (E, 2 * I, H // 2) and arrs[1].shape == (E, 2 * I, H // 32)
    assert arrs[2].shape == (E, H, I // 2) and arrs[3].shape == (E, H, I // 32)
    res = {
        "out_f64": np.zeros((T, H), np.float64),
        "out_bf16": np.zeros((T, H), np.uint16),
        "x_codes": np.zeros((T, H // 2), np.uint8),
        "x_sf": np.zeros((T, H // 32), np.uint8),
    }
    if want_intermediates:
        res["gate_up"] = np.zeros((A, 2 * I), np.float64)
        res["h_codes"] = np.zeros((A, I // 2), np.uint8)
        res["h_sf"] = np.zeros((A, I // 32), np.uint8)
    if want_y:
        res["y"] = np.zeros((A, H), np.float64)
    shape = Shape(T, H, I, E, k)
    bad = lib().oracle_moe(ctypes.byref(shape), _p(x_bf16), _p(ids), _p(tw), *[_p(a) for a in arrs],
                           _p(res["out_f64"]), _p(res["out_bf16"]), _p(res["x_codes"]), _p(res["x_sf"]),
                           _p(res.get("gate_up")), _p(res.get("h_codes")), _p(res.get("h_sf")),
                           _p(res.get("y")), nthreads or threads())
    res["invalid_ids"] = int(bad)
    return res


def moe_w4a8(x_bf16, ids, tw, w1_codes, w1_sf, w2_codes, w2_sf, *, want_intermediates: bool = False,
             want_y: bool = False, nthreads: int | None = None) -> dict:
    """The fp8xfp4 (W4A8) layer on the same canonical MXFP4 weights as moe(); the
    quantised activations are E4M3 codes, one byte each: x_codes [T, H], h_codes [A, I]."""
    x_bf16 = np.ascontiguousarray(x_bf16, np.uint16)
    ids = np.ascontiguousarray(ids, np.int32)
    tw = np.ascontiguousarray(tw, np.float32)
    T, H = x_bf16.shape
    k = ids.shape[1]
    E, twoI, _ = w1_codes.shape
    I = twoI // 2
    A = T * k
    arrs = [np.ascontiguousarray(a, np.uint8) for a in (w1_codes, w1_sf, w2_codes, w2_sf)]
    assert arrs[0].shape == (E, 2 * I, H // 2) and arrs[1].shape == (E, 2 * I, H // 32)
    assert arrs[2].shape == (E, H, I // 2) and arrs[3].shape == (E, H, I // 32)
    res = {
        "out_f64": np.zeros((T, H), np.float64),
        "out_bf16": np.zeros((T, H), np.uint16),
        "x_codes": np.zeros((T, H), np.uint8),
        "x_sf": np.zeros((T, H // 32), np.uint8),
    }
    if want_intermediates:
        res["gate_up"] = np.zeros((A, 2 * I), np.float64)
        res["h_codes"] = np.zeros((A, I), np.uint8)
        res["h_sf"] = np.zeros((A, I // 32), np.uint8)
    if want_y:
        res["y"] = np.zeros((A, H), np.float64)
    shape = Shape(T, H, I, E, k)
    bad = lib().oracle_moe_w4a8(ctypes.byref(shape), _p(x_bf16), _p(ids), _p(tw),
                                *[_p(a) for a in arrs], _p(res["out_f64"]), _p(res["out_bf16"]),
                                _p(res["x_codes"]), _p(res["x_sf"]), _p(res.get("gate_up")),
                                _p(res.get("h_codes")), _p(res.get("h_sf")), _p(res.get("y")),
                                nthreads or threads())
    res["invalid_ids"] = int(bad)
    return res


def moe_w4a8_down(ids, tw, w2_codes, w2_sf, h_codes, h_sf, H: int,
                  nthreads: int | None = None) -> dict:
    """W4A8 down projection + combine from given MXFP8 intermediate codes [A, I] and
    scales [A, I/32]."""
    ids = np.ascontiguousarray(ids, np.int32)
    tw = np.ascontiguousarray(tw, np.float32)
    T, k = ids.shape
    E = w2_codes.shape[0]
    I = w2_codes.shape[2] * 2
    out_f64 = np.zeros((T, H), np.float64)
    out_bf16 = np.zeros((T, H), np.uint16)
    shape = Shape(T, H, I, E, k)
    arrs = [np.ascontiguousarray(a, np.uint8) for a in (w2_codes, w2_sf, h_codes, h_sf)]
    lib().oracle_moe_w4a8_down(ctypes.byref(shape), _p(ids), _p(tw), *[_p(a) for a in arrs],
                               _p(out_f64), _p(out_bf16), nthreads or threads())
    return {"out_f64": out_f64, "out_bf16": out_bf16}


def nvfp4_quantize_f32(x: np.ndarray, nthreads: int | None = None):
    """fp32 [rows, K] -> (packed E2M1 codes [rows, K/2], E4M3 scale bytes [rows, K/16])."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    rows, K = x.shape
    codes = np.zeros((rows, K // 2), np.uint8)
    sf = np.zeros((rows, K // 16), np.uint8)
    lib().oracle_nvfp4_quantize_f32(_p(x), rows, K, _p(codes), _p(sf), nthreads or threads())
    return codes, sf


def nvfp4_quantize_bf16(bits: np.ndarray, nthreads: int | None = None):
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    rows, K = bits.shape
    codes = np.zeros((rows, K // 2), np.uint8)
    sf = np.zeros((rows, K // 16), np.uint8)
    lib().oracle_nvfp4_quantize_bf16(_p(bits), rows, K, _p(codes), _p(sf), nthreads or threads())
    return codes, sf


def nvfp4_dequantize(codes: np.ndarray, sf: np.ndarray) -> np.ndarray:
    codes = np.ascontiguousarray(codes, np.uint8)
    sf = np.ascontiguousarray(sf, np.uint8)
    rows, half = codes.shape
    out = np.zeros((rows, 2 * half), np.float64)
    lib().oracle_nvfp4_dequantize(_p(codes), _p(sf), rows, 2 * half, _p(out))
    return out


def moe_nvf4(x_bf16, ids, tw, w1_codes, w1_sf, w2_codes, w2_sf, *, want_intermediates: bool = False,
             want_y: bool = False, nthreads: int | None = None) -> dict:
    """The NVFP4 layer: canonical NVFP4 weights w1_codes [E, 2I, H/2], w1_sf [E, 2I, H/16],
    w2_codes [E, H, I/2], w2_sf [E, H, I/16] (E4M3 scale bytes, one per 16 elements)."""
    x_bf16 = np.ascontiguousarray(x_bf16, np.uint16)
    ids = np.ascontiguousarray(ids, np.int32)
    tw = np.ascontiguousarray(tw, np.float32)
    T, H = x_bf16.shape
    k = ids.shape[1]
    E, twoI, _ = w1_codes.shape
    I = twoI // 2
    A = T * k
    arrs = [np.ascontiguousarray(a, np.uint8) for a in (w1_codes, w1_sf, w2_codes, w2_sf)]
    assert arrs[0].shape == (E, 2 * I, H // 2) and arrs[1].shape == (E, 2 * I, H // 16)
    assert arrs[2].shape == (E, H, I // 2) and arrs[3].shape == (E, H, I // 16)
    res = {
        "out_f64": np.zeros((T, H), np.float64),
        "out_bf16": np.zeros((T, H), np.uint16),
        "x_codes": np.zeros((T, H // 2), np.uint8),
        "x_sf": np.zeros((T, H // 16), np.uint8),
    }
    if want_intermediates:
        res["gate_up"] = np.zeros((A, 2 * I), np.float64)
        res["h_codes"] = np.zeros((A, I // 2), np.uint8)
        res["h_sf"] = np.zeros((A, I // 16), np.uint8)
    if want_y:
        res["y"] = np.zeros((A, H), np.float64)
    shape = Shape(T, H, I, E, k)
    bad = lib().oracle_moe_nvf4(ctypes.byref(shape), _p(x_bf16), _p(ids), _p(tw),
                                *[_p(a) for a in arrs], _p(res["out_f64"]), _p(res["out_bf16"]),
                                _p(res["x_codes"]), _p(res["x_sf"]), _p(res.get("gate_up")),
                                _p(res.get("h_codes")), _p(res.get("h_sf")), _p(res.get("y")),
                                nthreads or threads())
    res["invalid_ids"] = int(bad)
    return res


def moe_down(ids, tw, w2_codes, w2_sf, h_codes, h_sf, H: int, nthreads: int | None = None) -> dict:
    """Down projection + combine from given intermediate codes [A, I/2] and scales [A, I/32]."""
    ids = np.ascontiguousarray(ids, np.int32)
    tw = np.ascontiguousarray(tw, np.float32)
    T, k = ids.shape
    E = w2_codes.shape[0]
    I = w2_codes.shape[2] * 2
    out_f64 = np.zeros((T, H), np.float64)
    out_bf16 = np.zeros((T, H), np.uint16)
    shape = Shape(T, H, I, E, k)
    arrs = [np.ascontiguousarray(a, np.uint8) for a in (w2_codes, w2_sf, h_codes, h_sf)]
    lib().oracle_moe_down(ctypes.byref(shape), _p(ids), _p(tw), *[_p(a) for a in arrs],
                          _p(out_f64), _p(out_bf16), nthreads or threads())
    return {"out_f64": out_f64, "out_bf16": out_bf16}


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
