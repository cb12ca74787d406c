"""Upload host (numpy) layer tensors to the GPU as the binding's weight containers.

bf16 tensors arrive as uint16 bit patterns and MXFP4 tensors as uint8, in the
layouts of include/moe.h; this only copies bytes (no conversion of values).
"""
from __future__ import annotations

from typing import Optional

import numpy as np
import torch

from . import Experts, Router, Shared


def bf16_tensor(a: Optional[np.ndarray], device="cuda", pin: bool = False) -> Optional[torch.Tensor]:
    """uint16 bf16 bit patterns -> torch.bfloat16 tensor on `device` (bytes unchanged)."""
    if a is None:
        return None
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    if device == "cpu":
        return t.pin_memory() if pin else t.clone()
    return t.to(device)


def u8_tensor(a: Optional[np.ndarray], device="cuda") -> Optional[torch.Tensor]:
    if a is None:
        return None
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def to_numpy_bf16(t: torch.Tensor) -> np.ndarray:
    """torch.bfloat16 -> uint16 bit patterns on the host."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def upload(layer, device="cuda"):
    """(x, Router, Experts, Shared | None) for an object with the layer's host arrays."""
    x = bf16_tensor(layer.x, device)
    router = Router(bf16_tensor(layer.router_w, device), bf16_tensor(layer.router_b, device),
                    bf16_tensor(getattr(layer, "norm_w", None), device))
    if getattr(layer, "gu_blocks", None) is not None:
        experts = Experts(gate_up=u8_tensor(layer.gu_blocks, device),
                          gate_up_scales=u8_tensor(layer.gu_scales, device),
                          gate_up_bias=bf16_tensor(layer.gu_bias, device),
                          down=u8_tensor(layer.dn_blocks, device),
                          down_scales=u8_tensor(layer.dn_scales, device),
                          down_bias=bf16_tensor(layer.dn_bias, device))
    elif getattr(layer, "gate_up", None) is not None:
        experts = Experts(gate_up=bf16_tensor(layer.gate_up, device),
                          gate_up_bias=bf16_tensor(getattr(layer, "gu_bias", None), device),
                          down=bf16_tensor(layer.down, device),
                          down_bias=bf16_tensor(getattr(layer, "dn_bias", None), device))
    else:
        experts = Experts(gate=bf16_tensor(layer.gate, device), up=bf16_tensor(layer.up, device),
                          down=bf16_tensor(layer.down, device),
                          down_bias=bf16_tensor(getattr(layer, "dn_bias", None), device))
    shared = None
    if getattr(layer, "sh_gate", None) is not None:
        shared = Shared(bf16_tensor(layer.sh_gate, device), bf16_tensor(layer.sh_up, device),
                        bf16_tensor(layer.sh_down, device), bf16_tensor(layer.sh_gate_inp, device))
    return x, router, experts, shared
