"""Upload a workload's synthetic inputs to the GPU.

Routed experts are drawn on the host in checkpoint layout, a block of experts at
a time, copied to the device and relaid into the packed table by the library's
own ``k3moe_pack_mxfp4``; nothing here computes any part of the layer.
"""
from __future__ import annotations

import numpy as np

from . import (EXPERT_TENSORS, Workload, make_bias, make_experts_block, make_router,
               make_shared, make_x)


def to_device_u16(a: np.ndarray, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device)


def to_device(a: np.ndarray, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def build_layer(w: Workload, T_max: int | None = None, device="cuda", block: int = 32,
                experts: range | None = None):
    """A MoELayer holding workload w's weights on `device` (all experts packed,
    unless `experts` restricts which are drawn; the rest stay uninitialised)."""
    import torch
    from sparse_moe_expert_k3moe_gb300 import MoELayer, k3moe_config

    cfg = k3moe_config(**w.config_kwargs())
    layer = MoELayer(cfg, T_max if T_max is not None else w.T, device)
    layer.w_router = to_device_u16(make_router(w), device)
    bias = make_bias(w)
    layer.bias = to_device(bias, device) if bias is not None else None
    if w.S:
        sh = make_shared(w)
        layer.sh_w1 = to_device_u16(sh["w1"], device)
        layer.sh_w3 = to_device_u16(sh["w3"], device)
        layer.sh_w2 = to_device_u16(sh["w2"], device)
    rng = experts if experts is not None else range(w.E)
    lo, hi = rng.start, rng.stop
    for e0 in range(lo, hi, block):
        n = min(block, hi - e0)
        blk = make_experts_block(w, e0, n)
        dev = {k: to_device(blk[k], device) for k in EXPERT_TENSORS}
        layer.pack_experts(e0, n, *(dev[k] for k in EXPERT_TENSORS))
        del dev
    torch.cuda.synchronize(layer.device)
    return layer


def device_x(w: Workload, device="cuda"):
    return to_device_u16(make_x(w), device)
