"""Shared test helpers: conversions between torch tensors and the oracle's
numpy inputs (bf16/fp16 as raw uint16 bits).  No arithmetic of the method."""
import numpy as np
import torch

import oracle

DT = {torch.float32: oracle.F32, torch.bfloat16: oracle.BF16, torch.float16: oracle.F16,
      torch.int8: oracle.I8}


def to_np(x: torch.Tensor) -> np.ndarray:
    x = x.detach().cpu().contiguous()
    if x.dtype in (torch.bfloat16, torch.float16):
        return x.view(torch.int16).numpy().view(np.uint16)
    return x.numpy()


def odt(x: torch.Tensor) -> int:
    return DT[x.dtype]


def from_bits(a: np.ndarray, dtype) -> torch.Tensor:
    """uint16 bit pattern -> bf16/fp16 tensor (or pass-through for fp32)."""
    if dtype in (torch.bfloat16, torch.float16):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(dtype)
    return torch.from_numpy(np.ascontiguousarray(a))
