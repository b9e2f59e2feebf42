"""Upload a workload's synthetic inputs to the GPU.

Routed experts are drawn on the host in checkpoint layout, a block of experts at
a time, copied to the device and relaid into the packed table by the library's
own ``k3moe_pack_mxfp4``; nothing here computes any part of the layer.
"""
from __future__ import annotations

import numpy as np

from . import (EXPERT_TENSORS, Workload, make_bias, make_experts_block, make_full,
               make_full_router, make_router, make_shared, make_x)


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


def build_block(w: Workload, T_max: int | None = None, device="cuda", block: int = 32):
    """A MoEBlock holding full-width workload w's tensors on `device`, every routed
    expert packed by the library."""
    import torch
    from sparse_moe_expert_k3moe_gb300 import MoEBlock, k3moe_config, k3moe_full_dims

    cfg = k3moe_config(**w.config_kwargs())
    blk = MoEBlock(cfg, k3moe_full_dims(w.hidden, w.latent_norm, w.rms_eps),
                   T_max if T_max is not None else w.T, device)
    full = make_full(w)
    blk.w_router = to_device_u16(make_full_router(w), device)
    bias = make_bias(w)
    blk.bias = to_device(bias, device) if bias is not None else None
    blk.w_down = to_device_u16(full["down"], device)
    blk.w_up = to_device_u16(full["up"], device)
    blk.gain = to_device(full["gain"], device)
    if w.S:
        blk.sh_w1, blk.sh_w3, blk.sh_w2 = (to_device_u16(full[m], device) for m in ("sh1", "sh3", "sh2"))
    for e0 in range(0, w.E, block):
        n = min(block, w.E - e0)
        eb = make_experts_block(w, e0, n)
        dev = {k: to_device(eb[k], device) for k in EXPERT_TENSORS}
        blk.pack_experts(e0, n, *(dev[k] for k in EXPERT_TENSORS))
        del dev
    torch.cuda.synchronize(blk.device)
    return blk
