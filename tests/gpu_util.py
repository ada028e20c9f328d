"""Helpers for GPU tests: device buffers through torch (plumbing only)."""
import numpy as np
import torch


def cuda(a, dtype):
    return torch.from_numpy(np.ascontiguousarray(a)).to(device="cuda", dtype=dtype)


def bf16_values(a) -> np.ndarray:
    """float32 array -> the float32 values of its bf16 rounding (torch RNE)."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16).float().numpy()


def host(t) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def stream() -> int:
    return torch.cuda.current_stream().cuda_stream


def sync():
    torch.cuda.synchronize()
