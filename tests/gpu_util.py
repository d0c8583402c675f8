"""Helpers for GPU tests: moving BF16 bit patterns between numpy and torch."""
import numpy as np
import torch


def to_dev(a: np.ndarray, device="cuda") -> torch.Tensor:
    """numpy uint16 BF16 bits -> contiguous torch.bfloat16 on the device."""
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16))
    return t.view(torch.bfloat16).to(device).contiguous()


def to_host(t: torch.Tensor) -> np.ndarray:
    """torch.bfloat16 -> numpy uint16 BF16 bits."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def empty_out(B: int, N: int, device="cuda") -> torch.Tensor:
    """Output buffer pre-filled with a NaN pattern, so unwritten entries show."""
    return torch.full((B, N), float("nan"), dtype=torch.bfloat16, device=device)
