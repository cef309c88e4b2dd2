"""Moving synthetic host arrays to and from device tensors (marshalling only).

BF16-exact float32 numpy arrays become torch.bfloat16 device tensors by their
16-bit words, so the device holds exactly the values the oracle widens.
"""
from __future__ import annotations

import numpy as np
import torch

from .synth import bf16_bits


def bf16_to_device(x, device="cuda"):
    bits = np.ascontiguousarray(bf16_bits(x)).view(np.int16)
    return torch.from_numpy(bits).to(device).view(torch.bfloat16)


def i32_to_device(x, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.int32)).to(device)


def slabs_to_device(slabs, device="cuda"):
    raw = np.ascontiguousarray(slabs).view(np.uint8)
    return torch.from_numpy(raw.copy()).to(device)


def bf16_tensor_to_f32(t) -> np.ndarray:
    """Exact float32 values of a BF16 device tensor."""
    return t.float().cpu().numpy()
