"""Host-side checks of the C ABI (no GPU needed, no compute call): the library
loads, exports every entry point declared in include/mxmoe.h, and its host-only
argument checks and sizing behave as documented."""
from __future__ import annotations

import os
import re
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mxmoe.h")


@pytest.fixture(scope="module")
def mx():
    from block_scaled_fp4_pre_gb300 import build

    build.build()
    import block_scaled_fp4_pre_gb300 as m

    m.lib()
    return m


def declared_functions():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"MXMOE_API[^;(]*?\b(moe_\w+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("moe_prepare_weights", "moe_pre_dispatch", "moe_forward",
                     "moe_workspace_size", "moe_prepared_weights_size", "moe_check",
                     "moe_last_error"):
        assert required in names


def test_library_exports_every_declared_symbol(mx):
    out = subprocess.run(["nm", "-D", "--defined-only", mx.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r" T (moe_\w+)$", out, flags=re.M))
    assert set(declared_functions()) <= exported
    for name in declared_functions():
        assert hasattr(mx.lib(), name)


def test_header_compiles_as_c():
    r = subprocess.run(["gcc", "-std=c99", "-fsyntax-only", "-Wall", "-Werror", "-x", "c", "-"],
                       input=f'#include "{HEADER}"\nint main(void){{return 0;}}\n',
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_dims_validation(mx):
    ok = mx.make_dims(4096, 2048, 256, 6, 512)
    mx.moe_validate_dims(ok)
    w4a8 = mx.make_dims(4096, 2048, 256, 6, 512, mma_type=mx.MOE_MMA_FP8xFP4)
    mx.moe_validate_dims(w4a8)
    # same weights; the E4M3 activation rows take twice the bytes of packed E2M1 rows
    assert mx.moe_prepared_weights_size(w4a8) == mx.moe_prepared_weights_size(ok)
    assert mx.moe_workspace_size(w4a8) > mx.moe_workspace_size(ok)
    nv = mx.make_dims(4096, 2048, 256, 6, 512, mma_type=mx.MOE_MMA_NVF4xNVF4)
    mx.moe_validate_dims(nv)
    # NVFP4: the same codes, twice the scale bytes (one per 16 elements)
    E, H, I = 256, 4096, 2048
    scales4 = E * 2 * I * H // 32 + E * H * I // 32
    assert mx.moe_prepared_weights_size(nv) - mx.moe_prepared_weights_size(ok) == scales4
    bad = [
        (mx.make_dims(4096, 2048, 256, 6, 512, mma_type=4), mx.MOE_ERR_UNSUPPORTED),
        (mx.make_dims(4096, 2048, 256, 6, 512, mma_type=0), mx.MOE_ERR_UNSUPPORTED),
        (mx.make_dims(4000, 2048, 256, 6, 512), mx.MOE_ERR_INVALID_ARG),
        (mx.make_dims(128, 2048, 256, 6, 512), mx.MOE_ERR_INVALID_ARG),
        (mx.make_dims(4096, 2000, 256, 6, 512), mx.MOE_ERR_INVALID_ARG),
        (mx.make_dims(4096, 2048, 0, 1, 512), mx.MOE_ERR_INVALID_ARG),
        (mx.make_dims(4096, 2048, 4, 6, 512), mx.MOE_ERR_INVALID_ARG),
        (mx.make_dims(4096, 2048, 256, 0, 512), mx.MOE_ERR_INVALID_ARG),
        (mx.make_dims(4096, 2048, 256, 6, 0), mx.MOE_ERR_INVALID_ARG),
        (mx.make_dims(4096, 2048, 2048, 6, 512), mx.MOE_ERR_INVALID_ARG),
    ]
    for d, want in bad:
        with pytest.raises(mx.MoeError) as ei:
            mx.moe_validate_dims(d)
        assert ei.value.status == want, d
        assert mx.moe_workspace_size(d) == 0 and mx.moe_prepared_weights_size(d) == 0
        assert mx.moe_last_error()


def test_prepared_size_is_canonical_mxfp4_bytes(mx):
    d = mx.make_dims(4096, 2048, 256, 6, 512)
    # gate/up [E, 2I, H] + down [E, H, I] at 4 bits plus one byte per 32 elements
    assert mx.moe_prepared_weights_size(d) == 256 * (2 * 2048 * 4096 + 4096 * 2048) * 17 // 32
    assert mx.moe_prepared_weights_size(d) == 3_422_552_064


def test_prepared_size_pads_a_short_last_k_block(mx):
    """Codes are stored in k-block tiles of 256 elements (128 for fp8xfp4); a K that
    ends in half a k-block is padded to a whole one, scales are not."""
    def align(v):
        return (v + 1023) // 1024 * 1024

    H, I, E = 384, 384, 2
    w1c, w2c = E * 2 * I * 2 * 128, E * H * 2 * 128     # two k-blocks of 128 bytes a row
    w1s, w2s = E * 2 * I * H // 32, E * H * I // 32
    want = align(align(align(align(w1c) + w1s) + w2c) + w2s)
    assert mx.moe_prepared_weights_size(mx.make_dims(H, I, E, 2, 64)) == want
    # fp8xfp4 k-blocks are 128 elements: 384 is three whole ones, no padding
    want8 = align(align(align(align(E * 2 * I * H // 2) + w1s) + E * H * I // 2) + w2s)
    assert mx.moe_prepared_weights_size(mx.make_dims(H, I, E, 2, 64, mx.MOE_MMA_FP8xFP4)) == want8


def test_untile_codes_follows_the_byte_formula():
    """The tests' untiling against the per-byte position of the k-block tile layout:
    byte j of row R at ((R // 128 * nkb + j // kb) * 128 + R % 128) * kb + j % kb."""
    from tests.helpers import untile_codes
    rng = np.random.default_rng(3)
    for rows, K, kb in ((256, 384, 128), (128, 256, 64), (384, 128, 128)):
        nkb = -(-K // (2 * kb))
        codes = rng.integers(0, 256, size=(rows, K // 2), dtype=np.uint8)
        flat = np.zeros(rows * nkb * kb, np.uint8)
        for R in range(rows):
            for j in range(K // 2):
                flat[((R // 128 * nkb + j // kb) * 128 + R % 128) * kb + j % kb] = codes[R, j]
        assert np.array_equal(untile_codes(flat, rows, K, kb), codes)


def test_workspace_size_grows_with_capacity(mx):
    a = mx.moe_workspace_size(mx.make_dims(4096, 2048, 256, 6, 512))
    b = mx.moe_workspace_size(mx.make_dims(4096, 2048, 256, 6, 16384))
    assert 0 < a < b
    assert b < 2 * 2 ** 30   # well under the device memory


def test_hot_calls_reject_uninitialised_workspace_without_touching_the_gpu(mx):
    d = mx.make_dims(256, 128, 8, 2, 16)
    fake = 256 * 1024   # never dereferenced: the host check fails first
    lib = mx.lib()
    import ctypes

    rc = lib.moe_pre_dispatch(ctypes.byref(d), 16, 16, 16, 4, fake, 1 << 30, None)
    assert rc == mx.MOE_ERR_WORKSPACE_MISMATCH
    rc = lib.moe_forward(ctypes.byref(d), 256, fake, 1 << 30, 16, 4, None)
    assert rc == mx.MOE_ERR_WORKSPACE_MISMATCH
    rc = lib.moe_pre_dispatch(ctypes.byref(d), 16, 16, 16, 17, fake, 1 << 30, None)
    assert rc == mx.MOE_ERR_INVALID_ARG           # num_tokens > max_tokens
    rc = lib.moe_pre_dispatch(ctypes.byref(d), 16, 16, 16, 4, fake, 10, None)
    assert rc == mx.MOE_ERR_WORKSPACE_TOO_SMALL
    rc = lib.moe_pre_dispatch(ctypes.byref(d), 16, 16, 16, 4, fake + 8, 1 << 30, None)
    assert rc == mx.MOE_ERR_INVALID_ARG           # misaligned workspace
    rc = lib.moe_quantize_mxfp4(16, 4, 48, 16, 16, None)
    assert rc == mx.MOE_ERR_INVALID_ARG           # K not a multiple of 32
    assert lib.moe_status_string(mx.MOE_ERR_ROUTING) == b"MOE_ERR_ROUTING"


def test_binding_has_the_c_names(mx):
    for name in declared_functions():
        assert hasattr(mx, name), name


def test_mxfp8_producer_and_dispatch_mode_host_checks(mx):
    """Sizing of the MXFP8 scale buffers and the argument checks of the producer and of
    the dispatch-mode setter, all decided on the host before any CUDA call."""
    lib = mx.lib()
    # 4-D layout: rows padded to whole 128-row blocks, 512 bytes per block per 128 of K
    assert mx.moe_mxfp8_scale_bytes(1, 256, mx.MOE_SF_128X4) == 1 * 2 * 512
    assert mx.moe_mxfp8_scale_bytes(129, 256, mx.MOE_SF_128X4) == 2 * 2 * 512
    # packed: one int32 per row per 128 of K
    assert mx.moe_mxfp8_scale_bytes(129, 256, mx.MOE_SF_PACKED) == 129 * 2 * 4
    assert mx.moe_mxfp8_scale_bytes(10, 100, mx.MOE_SF_PACKED) == 0     # K % 128 != 0
    assert mx.moe_mxfp8_scale_bytes(10, 256, 9) == 0                     # unknown layout
    fake = 1 << 20   # 16-byte aligned, never dereferenced: the host checks fail first
    bad = [
        (fake, 4, 100, fake, fake, 0, 4),        # K not a multiple of 128
        (fake, 5, 128, fake, fake, 0, 4),        # rows > rows_cap
        (fake, -1, 128, fake, fake, 0, 4),       # negative rows
        (fake, 4, 128, fake, fake, 7, 4),        # unknown layout
        (fake + 1, 4, 128, fake, fake, 0, 4),    # misaligned input
        (fake, 4, 128, fake, fake + 8, 1, 4),    # misaligned scales
        # the limits: K past 65535 * 128 (one grid row of blocks per 128 columns) and
        # rows_cap past 2^23, both refused before any launch
        (fake, 4, 65536 * 128, fake, fake, 0, 4),
        (fake, 4, 128, fake, fake, 0, (1 << 23) + 1),
    ]
    for args in bad:
        assert lib.moe_mxfp8_quantize(*args, None) == mx.MOE_ERR_INVALID_ARG, args
    assert lib.moe_workspace_set_dispatch(fake, 5) == mx.MOE_ERR_INVALID_ARG
    assert lib.moe_workspace_set_dispatch(None, 1) == mx.MOE_ERR_INVALID_ARG
    assert lib.moe_workspace_set_dispatch(fake, 1) == mx.MOE_ERR_WORKSPACE_MISMATCH


def test_tile_mode_and_nvfp4_quantiser_host_checks(mx):
    """The tile-mode setter and the NVFP4 weight quantiser reject bad arguments on the
    host, before any CUDA call."""
    lib = mx.lib()
    fake = 1 << 20
    assert lib.moe_workspace_set_tiles(fake, 9) == mx.MOE_ERR_INVALID_ARG
    assert lib.moe_workspace_set_tiles(None, mx.MOE_TILES_NARROW) == mx.MOE_ERR_INVALID_ARG
    assert lib.moe_workspace_set_tiles(fake, mx.MOE_TILES_MEDIUM) == mx.MOE_ERR_WORKSPACE_MISMATCH
    for rows, K, src in ((4, 24, fake), (-1, 32, fake), (4, 32, fake + 4)):
        assert lib.moe_quantize_nvfp4(src, rows, K, fake, fake, None) == mx.MOE_ERR_INVALID_ARG
    assert lib.moe_quantize_nvfp4(fake, 0, 32, fake, fake, None) == mx.MOE_OK   # no rows: no-op
    # the three mma types' workspaces: E4M3 rows take more room, NVFP4 scales twice
    # the bytes of MXFP4's; all accept the same dims otherwise
    sizes = [mx.moe_workspace_size(mx.make_dims(4096, 2048, 256, 6, 512, m))
             for m in (mx.MOE_MMA_MXF4xMXF4, mx.MOE_MMA_FP8xFP4, mx.MOE_MMA_NVF4xNVF4)]
    assert all(v > 0 for v in sizes)
    assert sizes[1] > sizes[0] and sizes[2] > sizes[0]


def test_bucket_noalloc_reads_only_experts_topk_and_mma_type(mx):
    """moe_bucket_noalloc checks only the dims fields bucketing uses; with zero tokens
    it returns before any CUDA call, so these checks run on the host."""
    lib = mx.lib()
    fake = 1 << 20
    # hidden, inter and max_tokens unused: zero values pass
    d = mx.make_dims(0, 0, 32, 4, 0)
    assert lib.moe_bucket_noalloc(d, fake, fake, 0, fake, fake, None) == mx.MOE_OK
    assert lib.moe_bucket_noalloc(mx.make_dims(0, 0, 4, 8, 0), fake, fake, 0, fake, fake,
                                  None) == mx.MOE_ERR_INVALID_ARG     # topk > experts
    assert lib.moe_bucket_noalloc(mx.make_dims(0, 0, 0, 1, 0), fake, fake, 0, fake, fake,
                                  None) == mx.MOE_ERR_INVALID_ARG     # no experts
    assert lib.moe_bucket_noalloc(mx.make_dims(0, 0, 32, 4, 0, 9), fake, fake, 0, fake, fake,
                                  None) == mx.MOE_ERR_UNSUPPORTED     # unknown mma_type
    assert lib.moe_bucket_noalloc(None, fake, fake, 0, fake, fake, None) == mx.MOE_ERR_INVALID_ARG
