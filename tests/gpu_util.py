"""Host <-> device helpers shared by the GPU tests (plumbing only)."""
from __future__ import annotations

import numpy as np
import torch

DEV = torch.device("cuda:0")


def d(a, dtype=None):
    """numpy -> CUDA tensor; uint16 arrays become bfloat16 unless dtype given."""
    a = np.ascontiguousarray(a)
    t = torch.from_numpy(a)
    if a.dtype == np.uint16:
        t = t.view(torch.int16).view(torch.bfloat16)
    if dtype is not None:
        t = t.view(dtype)
    return t.to(DEV)


def h(t):
    """CUDA tensor -> numpy; bfloat16 becomes uint16 bit patterns."""
    t = t.detach()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def status_word():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


def bf16_ulp_distance(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Distance in units of the last place between bf16 bit patterns, on the
    ordered-integer line (+0 and -0 are 0 apart)."""
    def ordered(x):
        x = x.astype(np.int32)
        return np.where(x & 0x8000, 0x8000 - (x & 0x7FFF), 0x8000 + x)
    return np.abs(ordered(a) - ordered(b))


def gprobs_bound(rows_f, gy_f, o_gp):
    """Bound on |fp32 reduction - fp64 sum| for g_probs[t,k] = sum_h r_h g_h:
    (H-1) * 2^-24 * sum_h |r_h g_h| + 2^-24 * |exact| (any summation order)."""
    H = rows_f.shape[-1]
    absdot = np.sum(np.abs(rows_f.astype(np.float64) * gy_f.astype(np.float64)), axis=-1)
    return (H - 1) * 2.0**-24 * absdot + 2.0**-24 * np.abs(o_gp) + 1e-30
