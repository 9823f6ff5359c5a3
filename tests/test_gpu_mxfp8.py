"""MXFP8 producer (moe_mxfp8_quantize) against the CPU oracle, through the C ABI.

SGLang PR #48424, section "DeepGEMM producers write FlashInfer's 128x4 scale layout":
the producer's FP8 data and its scales in either layout must be bitwise what the
definition gives, at the row counts the page checks (1, 129, 1000, 4100, 16384),
with NaN-filled padding before the call, padded rows' scales zero after it, and the
live rows' scales a prefix of a buffer sized for more rows.  Integer and byte
outputs: bit-exact.
"""
from __future__ import annotations

import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import block_scaled_fp4_pre_gb300 as mx  # noqa: E402
import oracle  # noqa: E402

pytestmark = pytest.mark.gpu


def _rows_bf16(rows: int, K: int, seed: int) -> np.ndarray:
    """bf16 bits of N(0,1) rows with per-row magnitudes over eight decades, a few
    outliers, an all-zero group, ties of the E4M3 grid and signed zeros."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((rows, K)) * 10.0 ** rng.uniform(-4, 4, (rows, 1))
    if rows > 3:
        x[1, 64:96] = 0.0
        x[2, :32] = [448.0, 0.5 * (2.0 ** -9)] + [2.0 ** -7 * 1.0625] * 30   # tie on the grid
        x[3, ::97] *= 1e3
        x[0, 5] = -0.0
    t = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _run(bits: np.ndarray, layout: int, rows_cap: int):
    rows, K = bits.shape
    dev = torch.device("cuda")
    x = torch.from_numpy(bits.view(np.int16)).to(dev)
    q = torch.full((max(rows, 1), K), 0xFF, dtype=torch.uint8, device=dev)
    nsf = mx.moe_mxfp8_scale_bytes(rows_cap, K, layout)
    sf = torch.full((nsf,), 0xFF, dtype=torch.uint8, device=dev)    # NaN-filled padding
    mx.moe_mxfp8_quantize(x, rows, K, q, sf, layout, rows_cap)
    torch.cuda.synchronize()
    return q.cpu().numpy()[:rows], sf.cpu().numpy()


def _expected_scales(sf_rows: np.ndarray, layout: int, rows_cap: int) -> np.ndarray:
    rows, kc = sf_rows.shape
    if layout == mx.MOE_SF_PACKED:
        out = np.zeros((rows_cap, kc), np.uint8)
        out[:rows] = sf_rows
        return out.reshape(-1)
    full = np.zeros((rows_cap, kc), np.uint8)
    full[:rows] = sf_rows
    return oracle.scale_block_layout(full)      # R9 byte order, rows padded to 128


@pytest.mark.parametrize("rows", [1, 129, 1000, 4100])
@pytest.mark.parametrize("layout", [0, 1])
def test_bit_exact_against_oracle(rows, layout):
    K = 1024
    bits = _rows_bf16(rows, K, seed=rows)
    q_ref, sf_ref = oracle.mxfp8_quantize_bf16(bits)
    q, sf = _run(bits, layout, rows)
    assert np.array_equal(q, q_ref)
    assert np.array_equal(sf, _expected_scales(sf_ref, layout, rows))
    if layout == mx.MOE_SF_PACKED:
        assert np.array_equal(sf.view(np.uint32).reshape(rows, K // 128),
                              oracle.mxfp8_packed_scales(sf_ref))


def test_sixteen_thousand_rows_both_layouts():
    bits = _rows_bf16(16384, 256, seed=5)
    q_ref, sf_ref = oracle.mxfp8_quantize_bf16(bits)
    for layout in (0, 1):
        q, sf = _run(bits, layout, 16384)
        assert np.array_equal(q, q_ref)
        assert np.array_equal(sf, _expected_scales(sf_ref, layout, 16384))


@pytest.mark.parametrize("layout", [0, 1])
def test_live_rows_are_a_prefix_of_a_larger_buffer(layout):
    """The same 300 rows written into buffers sized for 300 and for 1000 rows: the
    first gives the second's prefix, and everything after the live rows is zero."""
    K = 512
    bits = _rows_bf16(300, K, seed=7)
    _, sf_small = _run(bits, layout, 300)
    _, sf_big = _run(bits, layout, 1000)
    assert sf_big.size == mx.moe_mxfp8_scale_bytes(1000, K, layout)
    assert np.array_equal(sf_big[:sf_small.size], sf_small)
    assert not sf_big[sf_small.size:].any()


def test_zero_rows_only_clears_the_padding():
    dev = torch.device("cuda")
    sf = torch.full((mx.moe_mxfp8_scale_bytes(256, 256, 1),), 0xFF, dtype=torch.uint8, device=dev)
    mx.moe_mxfp8_quantize(None, 0, 256, None, sf, 1, 256)
    torch.cuda.synchronize()
    assert not sf.cpu().numpy().any()


def test_argument_errors():
    dev = torch.device("cuda")
    buf = torch.zeros(1 << 16, dtype=torch.uint8, device=dev)
    bad = [
        (buf, 4, 100, buf, buf, 0, 4),        # K not a multiple of 128
        (buf, 5, 128, buf, buf, 0, 4),        # rows > rows_cap
        (buf, 4, 128, buf, buf, 7, 4),        # unknown layout
        (buf[1:], 4, 128, buf, buf, 0, 4),    # misaligned x
        (buf, 4, 128, buf, buf[8:], 1, 4),    # misaligned scales
    ]
    for args in bad:
        with pytest.raises(mx.MoeError) as ei:
            mx.moe_mxfp8_quantize(*args)
        assert ei.value.status == mx.MOE_ERR_INVALID_ARG
