"""Helpers for the GPU tests: move the generator's numpy bytes to the device
unchanged (bf16 as raw bits reinterpreted, never re-rounded)."""
import numpy as np
import torch


def dev(a, dtype=None):
    """numpy -> CUDA tensor with identical bytes.  uint16 arrays are bf16 bits."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    t = torch.from_numpy(a).cuda()
    return t if dtype is None else t.to(dtype)


def host(t):
    """CUDA tensor -> numpy; bf16 comes back as uint16 bits."""
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def bf16_to_f64(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
