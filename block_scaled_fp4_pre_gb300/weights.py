"""Loading fp32 expert weights into the layer's prepared MXFP4 (or NVFP4) blob on the device.

The fp32 rows of each expert come from a caller-supplied function (a checkpoint
reader, or the seeded generator in tests and the benchmark).  They are staged
through pinned host memory, quantised on the GPU by moe_quantize_mxfp4 into
canonical MXFP4 tensors, and then turned into the kernel layout by
moe_prepare_weights.  Host generation of expert e+1 overlaps the copy and
quantisation of expert e (two staging buffers).
"""
from __future__ import annotations

from typing import Callable

import numpy as np
import torch

from . import (MOE_MMA_NVF4xNVF4, MoeDims, moe_prepare_weights, moe_prepared_weights_size,
               moe_quantize_mxfp4, moe_quantize_nvfp4, sf_group)


def canonical_empty(dims: MoeDims, device) -> dict:
    E, H, I = dims.num_experts, dims.hidden, dims.inter
    g = sf_group(dims)       # MXFP4: one scale per 32; NVFP4: per 16
    u8 = torch.uint8
    return {
        "w1_codes": torch.empty((E, 2 * I, H // 2), dtype=u8, device=device),
        "w1_scales": torch.empty((E, 2 * I, H // g), dtype=u8, device=device),
        "w2_codes": torch.empty((E, H, I // 2), dtype=u8, device=device),
        "w2_scales": torch.empty((E, H, I // g), dtype=u8, device=device),
    }


def quantize_experts(dims: MoeDims, fill_w1: Callable[[int, np.ndarray], None],
                     fill_w2: Callable[[int, np.ndarray], None], device,
                     stream: torch.cuda.Stream | None = None) -> dict:
    """Canonical MXFP4 weights of all experts on `device`.

    fill_w1(e, out) writes expert e's gate/up weight, fp32 [2I, H] (gate rows first),
    into the numpy array `out`; fill_w2(e, out) writes the down weight, fp32 [H, I]."""
    E, H, I = dims.num_experts, dims.hidden, dims.inter
    can = canonical_empty(dims, device)
    quantize = moe_quantize_nvfp4 if dims.mma_type == MOE_MMA_NVF4xNVF4 else moe_quantize_mxfp4
    stream = stream or torch.cuda.current_stream(device)
    n1, n2 = 2 * I * H, H * I
    host = [torch.empty(n1 + n2, dtype=torch.float32, pin_memory=True) for _ in range(2)]
    dev = [torch.empty(n1 + n2, dtype=torch.float32, device=device) for _ in range(2)]
    done = [None, None]
    with torch.cuda.stream(stream):
        for e in range(E):
            b = e & 1
            if done[b] is not None:
                done[b].synchronize()          # staging buffer b is free again
            hv = host[b].numpy()
            fill_w1(e, hv[:n1].reshape(2 * I, H))
            fill_w2(e, hv[n1:].reshape(H, I))
            dev[b].copy_(host[b], non_blocking=True)
            quantize(dev[b][:n1].view(2 * I, H), can["w1_codes"][e], can["w1_scales"][e], stream)
            quantize(dev[b][n1:].view(H, I), can["w2_codes"][e], can["w2_scales"][e], stream)
            ev = torch.cuda.Event()
            ev.record(stream)
            done[b] = ev
    stream.synchronize()
    return can


def prepare(dims: MoeDims, canonical: dict, device, stream=None) -> torch.Tensor:
    """The prepared blob (interleaved gate/up rows, 128x4 scale blocks) from canonical MXFP4."""
    prepared = torch.empty(moe_prepared_weights_size(dims), dtype=torch.uint8, device=device)
    moe_prepare_weights(dims, canonical["w1_codes"], canonical["w1_scales"], canonical["w2_codes"],
                        canonical["w2_scales"], prepared, stream)
    return prepared
