"""Helpers shared by the GPU parity tests (device transfer of synth arrays)."""
import numpy as np
import torch

DEV = "cuda:0"


def to_dev(a: np.ndarray, bf16: bool = False) -> torch.Tensor:
    """numpy -> cuda tensor; uint16 arrays holding bf16 bits become bfloat16."""
    if bf16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(DEV).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def u8(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy()


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def guarded(shape, dtype, fill, guard=4096):
    """An output view followed by a guard band; returns (view, buffer, n)."""
    n = int(np.prod(shape))
    buf = torch.full((n + guard,), fill, dtype=dtype, device=DEV)
    return buf[:n].view(shape), buf, n


def guard_intact(buf, n, fill):
    return bool(torch.all(buf[n:] == fill).item())
