"""Shared helpers for the tests: moving bf16 bit arrays between numpy (the
oracle's representation) and torch device tensors (the library's)."""
import numpy as np
import torch


def to_dev(a: np.ndarray, dtype=torch.bfloat16, device="cuda"):
    a = np.ascontiguousarray(a)
    if dtype == torch.bfloat16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(a).to(device)


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> uint16 bit patterns on the host."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().numpy()
