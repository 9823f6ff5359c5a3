"""Python binding of libmxmoe, a GB300 (sm_103a) W4A4 MXFP4 mixture-of-experts layer.

Argument marshalling only: every step of the layer runs in the CUDA kernels of
libmxmoe.so, whose C ABI is include/mxmoe.h.  Function names match the C entry
points.  Device buffers are torch tensors (or raw integer addresses); PyTorch is
used for device memory and streams only.  There is no CPU fallback: if the
library is missing, importing the functions raises.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch  # loads the CUDA runtime libmxmoe links against

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmxmoe.so")

MOE_MMA_MXF4xMXF4 = 1
MOE_MMA_FP8xFP4 = 2
MOE_MMA_NVF4xNVF4 = 3
MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_WORKSPACE_TOO_SMALL = 3
MOE_ERR_WORKSPACE_MISMATCH = 4
MOE_ERR_CUDA = 5
MOE_ERR_ROUTING = 6
MOE_ERR_TIMEOUT = 7


class MoeDims(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("inter", ctypes.c_int32),
                ("num_experts", ctypes.c_int32), ("topk", ctypes.c_int32),
                ("max_tokens", ctypes.c_int32), ("mma_type", ctypes.c_int32)]

    def __repr__(self):
        return (f"MoeDims(hidden={self.hidden}, inter={self.inter}, num_experts={self.num_experts}, "
                f"topk={self.topk}, max_tokens={self.max_tokens}, mma_type={self.mma_type})")


def make_dims(hidden: int, inter: int, num_experts: int, topk: int, max_tokens: int,
              mma_type: int = MOE_MMA_MXF4xMXF4) -> MoeDims:
    return MoeDims(hidden, inter, num_experts, topk, max_tokens, mma_type)


class MoeError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{status_string(status)}: {message}")
        self.status = status


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libmxmoe.so (built by __graft_entry__.build() / build.py)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        l = ctypes.CDLL(LIB_PATH)
        D = ctypes.POINTER(MoeDims)
        vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        sigs = {
            "moe_last_error": ([], ctypes.c_char_p),
            "moe_status_string": ([i32], ctypes.c_char_p),
            "moe_validate_dims": ([D], i32),
            "moe_prepared_weights_size": ([D], sz),
            "moe_workspace_size": ([D], sz),
            "moe_workspace_init": ([D, vp, sz, vp], i32),
            "moe_quantize_mxfp4": ([vp, i64, i32, vp, vp, vp], i32),
            "moe_quantize_nvfp4": ([vp, i64, i32, vp, vp, vp], i32),
            "moe_prepare_weights": ([D, vp, vp, vp, vp, vp, sz, vp], i32),
            "moe_pre_dispatch": ([D, vp, vp, vp, i32, vp, sz, vp], i32),
            "moe_forward": ([D, vp, vp, sz, vp, i32, vp], i32),
            "moe_run_host": ([D, vp, vp, sz, vp, vp, vp, vp, i32, vp], i32),
            "moe_check": ([vp, vp], i32),
            "moe_read_dispatch": ([D, vp, i32, vp, vp, vp, vp, vp], i32),
            "moe_read_intermediate": ([D, vp, i32, vp, vp], i32),
            "moe_debug_gate_up": ([D, vp, vp, sz, vp, i32, vp], i32),
            "moe_profile_enable": ([i32], i32),
            "moe_profile_read": ([ctypes.POINTER(ctypes.c_char_p), vp, vp, i32], i32),
            "moe_profile_reset": ([], None),
            "moe_device_sm_count": ([], i32),
            "moe_bucket_noalloc": ([D, vp, vp, i32, vp, vp, vp], i32),
            "moe_debug_wait_probe": ([vp, i64, vp], i32),
            "moe_fp4_mma_probe": ([vp, i32, i32, i32, i64, vp], i32),
            "moe_fp4_mma_probe_pair": ([vp, i32, i32, i64, vp], i32),
            "moe_mxfp8_scale_bytes": ([i64, i64, i32], ctypes.c_size_t),
            "moe_workspace_set_dispatch": ([vp, i32], i32),
            "moe_workspace_set_tiles": ([vp, i32], i32),
            "moe_mxfp8_quantize": ([vp, i64, i64, vp, vp, i32, i64, vp], i32),
        }
        for name, (args, res) in sigs.items():
            f = getattr(l, name)
            f.argtypes = args
            f.restype = res
        _lib = l
    return _lib


def moe_status_string(status: int) -> str:
    return lib().moe_status_string(int(status)).decode()


status_string = moe_status_string


def moe_last_error() -> str:
    return lib().moe_last_error().decode()


def _check(status: int) -> int:
    if status != MOE_OK:
        raise MoeError(status, moe_last_error())
    return status


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, torch.Tensor):
        return t.data_ptr()
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    return int(t)


def _nbytes(t) -> int:
    if isinstance(t, torch.Tensor):
        return t.numel() * t.element_size()
    if isinstance(t, np.ndarray):
        return t.nbytes
    raise TypeError("need a tensor or array to know its size")


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


# ---------------------------------------------------------------------------
# Entry points (same names as the C ABI)

def moe_validate_dims(dims: MoeDims) -> None:
    _check(lib().moe_validate_dims(ctypes.byref(dims)))


def moe_prepared_weights_size(dims: MoeDims) -> int:
    return int(lib().moe_prepared_weights_size(ctypes.byref(dims)))


def moe_workspace_size(dims: MoeDims) -> int:
    return int(lib().moe_workspace_size(ctypes.byref(dims)))


def moe_workspace_init(dims: MoeDims, ws, stream=None) -> None:
    _check(lib().moe_workspace_init(ctypes.byref(dims), _ptr(ws), _nbytes(ws), _stream(stream)))


def moe_quantize_mxfp4(src, codes, scales, stream=None) -> None:
    rows, K = src.shape
    _check(lib().moe_quantize_mxfp4(_ptr(src), rows, K, _ptr(codes), _ptr(scales), _stream(stream)))


def moe_quantize_nvfp4(src, codes, scales, stream=None) -> None:
    rows, K = src.shape
    _check(lib().moe_quantize_nvfp4(_ptr(src), rows, K, _ptr(codes), _ptr(scales), _stream(stream)))


def sf_group(dims: MoeDims) -> int:
    """Elements per scale: 16 for nvf4xnvf4, 32 otherwise."""
    return 16 if dims.mma_type == MOE_MMA_NVF4xNVF4 else 32


def moe_prepare_weights(dims: MoeDims, w1_codes, w1_scales, w2_codes, w2_scales, prepared,
                        stream=None) -> None:
    _check(lib().moe_prepare_weights(ctypes.byref(dims), _ptr(w1_codes), _ptr(w1_scales),
                                     _ptr(w2_codes), _ptr(w2_scales), _ptr(prepared),
                                     _nbytes(prepared), _stream(stream)))


def moe_pre_dispatch(dims: MoeDims, x, topk_ids, topk_weights, num_tokens: int, ws,
                     stream=None) -> None:
    _check(lib().moe_pre_dispatch(ctypes.byref(dims), _ptr(x), _ptr(topk_ids), _ptr(topk_weights),
                                  int(num_tokens), _ptr(ws), _nbytes(ws), _stream(stream)))


def moe_forward(dims: MoeDims, prepared, ws, out, num_tokens: int, stream=None) -> None:
    _check(lib().moe_forward(ctypes.byref(dims), _ptr(prepared), _ptr(ws), _nbytes(ws), _ptr(out),
                             int(num_tokens), _stream(stream)))


def moe_run_host(dims: MoeDims, prepared, ws, x_host, topk_ids_host, topk_weights_host, out_host,
                 num_tokens: int, stream=None) -> None:
    _check(lib().moe_run_host(ctypes.byref(dims), _ptr(prepared), _ptr(ws), _nbytes(ws),
                              _ptr(x_host), _ptr(topk_ids_host), _ptr(topk_weights_host),
                              _ptr(out_host), int(num_tokens), _stream(stream)))


def moe_check(ws, stream=None) -> None:
    _check(lib().moe_check(_ptr(ws), _stream(stream)))


def _act_row_bytes(dims: MoeDims, K: int) -> int:
    """Bytes of a quantised activation row: E4M3 (fp8xfp4) or packed E2M1."""
    return K if dims.mma_type == MOE_MMA_FP8xFP4 else K // 2


def moe_read_dispatch(dims: MoeDims, ws, num_tokens: int) -> dict:
    T, k, H, E = int(num_tokens), dims.topk, dims.hidden, dims.num_experts
    out = {
        "counts": np.zeros(E, np.int32),
        "assign_slot": np.zeros(T * k, np.int32),
        "x_codes": np.zeros((T * k, _act_row_bytes(dims, H)), np.uint8),
        "x_scales": np.zeros((T * k, H // sf_group(dims)), np.uint8),
        "slot_token": np.zeros(T * k, np.int32),
    }
    _check(lib().moe_read_dispatch(ctypes.byref(dims), _ptr(ws), T, *[_ptr(out[n]) for n in
                                   ("counts", "assign_slot", "x_codes", "x_scales", "slot_token")]))
    return out


def moe_read_intermediate(dims: MoeDims, ws, num_tokens: int) -> dict:
    T, k, I = int(num_tokens), dims.topk, dims.inter
    out = {"h_codes": np.zeros((T * k, _act_row_bytes(dims, I)), np.uint8),
           "h_scales": np.zeros((T * k, I // sf_group(dims)), np.uint8)}
    _check(lib().moe_read_intermediate(ctypes.byref(dims), _ptr(ws), T, _ptr(out["h_codes"]),
                                       _ptr(out["h_scales"])))
    return out


def moe_debug_gate_up(dims: MoeDims, prepared, ws, gate_up, num_tokens: int, stream=None) -> None:
    _check(lib().moe_debug_gate_up(ctypes.byref(dims), _ptr(prepared), _ptr(ws), _nbytes(ws),
                                   _ptr(gate_up), int(num_tokens), _stream(stream)))


def moe_debug_wait_probe(ws, limit_ns: int, stream=None) -> None:
    _check(lib().moe_debug_wait_probe(_ptr(ws), int(limit_ns), _stream(stream)))


MOE_DISPATCH_BUCKETED = 0
MOE_DISPATCH_PULL = 1
MOE_TILES_AUTO = 0
MOE_TILES_WIDE = 1
MOE_TILES_NARROW = 2
MOE_TILES_MEDIUM = 3
MOE_TILES_PAIR = 4


def moe_workspace_set_dispatch(ws, mode: int) -> None:
    """Bucketed token copies (TMA) or per-token rows gathered by the layer kernel."""
    _check(lib().moe_workspace_set_dispatch(_ptr(ws), int(mode)))


def moe_workspace_set_tiles(ws, mode: int) -> None:
    """Token tiles of 128 rows (wide), 64 (medium), 32 (narrow) or chosen per dispatch (auto)."""
    _check(lib().moe_workspace_set_tiles(_ptr(ws), int(mode)))


MOE_SF_PACKED = 0
MOE_SF_128X4 = 1


def moe_mxfp8_scale_bytes(rows_cap: int, K: int, layout: int) -> int:
    return int(lib().moe_mxfp8_scale_bytes(int(rows_cap), int(K), int(layout)))


def moe_mxfp8_quantize(x, rows: int, K: int, q, sf, layout: int, rows_cap: int | None = None,
                       stream=None) -> None:
    """bf16 rows -> E4M3 values and UE8M0 scales (packed int32 or the 4-D 128x4 layout)."""
    _check(lib().moe_mxfp8_quantize(_ptr(x), int(rows), int(K), _ptr(q), _ptr(sf), int(layout),
                                    int(rows if rows_cap is None else rows_cap), _stream(stream)))


def moe_fp4_mma_probe(ws, n: int, blocks_per_sm: int, blocks: int, mma_count: int,
                      stream=None) -> None:
    _check(lib().moe_fp4_mma_probe(_ptr(ws), int(n), int(blocks_per_sm), int(blocks),
                                   int(mma_count), _stream(stream)))


def moe_fp4_mma_probe_pair(ws, n: int, pairs: int, mma_count: int, stream=None) -> None:
    """The probe's M=256 form across SM pairs (tcgen05 cta_group::2)."""
    _check(lib().moe_fp4_mma_probe_pair(_ptr(ws), int(n), int(pairs), int(mma_count),
                                        _stream(stream)))


def moe_profile_enable(on: bool) -> None:
    _check(lib().moe_profile_enable(1 if on else 0))


def moe_profile_read(max_kernels: int = 32) -> dict:
    names = (ctypes.c_char_p * max_kernels)()
    ms = np.zeros(max_kernels, np.float32)
    n_launch = np.zeros(max_kernels, np.int32)
    n = lib().moe_profile_read(names, _ptr(ms), _ptr(n_launch), max_kernels)
    return {names[i].decode(): (float(ms[i]), int(n_launch[i])) for i in range(n)}


def moe_profile_reset() -> None:
    lib().moe_profile_reset()


def moe_device_sm_count() -> int:
    return int(lib().moe_device_sm_count())


def moe_bucket_noalloc(dims: MoeDims, topk_ids, topk_weights, num_tokens: int, counts,
                       assign_slot, stream=None) -> None:
    """Bucketing with the library's own static scratch; allocates nothing on the device."""
    _check(lib().moe_bucket_noalloc(ctypes.byref(dims), _ptr(topk_ids), _ptr(topk_weights),
                                    int(num_tokens), _ptr(counts), _ptr(assign_slot),
                                    _stream(stream)))
