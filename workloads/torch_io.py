"""Move generated input bytes into torch tensors (no arithmetic on the values)."""

from __future__ import annotations

import numpy as np
import torch


def bf16_tensor(bits: np.ndarray, device="cuda", pin=False) -> torch.Tensor:
    """uint16 bf16 bit patterns -> torch.bfloat16 tensor with the same bits."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    if device == "cpu":
        return t.pin_memory() if pin else t
    return t.to(device)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """torch.bfloat16 tensor -> uint16 bit patterns (host copy)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def layer_tensors(inp, device="cuda", pin=False) -> dict:
    """The five input tensors of one layer (workloads.LayerInputs) as bf16 tensors."""
    return {name: bf16_tensor(getattr(inp, name), device, pin) for name in ("k_old", "v_old", "k_new", "v_new", "q")}
