"""Seeded synthetic inputs for the Q8_0 decode-projection workloads.

This module only draws numbers: it holds none of the path's arithmetic
(no quantizer, no norm, no dot), so both the library's tests/benchmark and
the CPU oracle can take their inputs from it.

Recipe (the workloads described for the Q8_0 GEMV):
  * weight levels: int8 uniform on [-127, 127] (-128 never drawn);
  * block scales: f16 of |N(0, 0.02)| + 1e-4, one per 32 weights of a row,
    rounded to nearest-even binary16 and handed over as uint16 bit patterns;
  * activations: f32 N(0, 1); with ``outliers`` each element is independently
    multiplied by 20 with probability 0.01;
  * RMSNorm gain: f32 N(1, 0.1).

Host arrays come from numpy's PCG64 generator; the large device-resident
weights of the benchmark come from a seeded ``torch.Generator`` on the device
with the same distributions (different values: only sampled rows of those are
ever compared, after copying them back).
"""
from __future__ import annotations

import numpy as np

SEED_BASE = 0x51A70000


def rng(seed: int) -> np.random.Generator:
    return np.random.default_rng(seed)


def q8_matrix(N: int, K: int, seed: int):
    """(wq int8 [N, K], ws uint16 f16-bits [N, K/32]) on the host."""
    assert K % 32 == 0
    r = rng(seed)
    wq = r.integers(-127, 128, size=(N, K), dtype=np.int8)
    sc = np.abs(r.normal(0.0, 0.02, size=(N, K // 32))) + 1e-4
    ws = sc.astype(np.float16).view(np.uint16)
    return wq, ws


def activation(M: int, K: int, seed: int, outliers: bool = False) -> np.ndarray:
    r = rng(seed)
    x = r.standard_normal(size=(M, K), dtype=np.float32)
    if outliers:
        mask = r.random(size=(M, K)) < 0.01
        x[mask] *= np.float32(20.0)
    return x


def norm_gain(K: int, seed: int) -> np.ndarray:
    r = rng(seed)
    return (1.0 + 0.1 * r.standard_normal(size=K)).astype(np.float32)


# ---- device-side generation for the multi-GB benchmark matrices -------------

def q8_matrix_torch(N: int, K: int, seed: int, device, chunk_rows: int = 8192):
    """(wq int8 [N, K], ws int16 holding f16 bits [N, K/32]) generated on
    ``device`` with a seeded torch generator, in row chunks."""
    import torch

    assert K % 32 == 0
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    wq = torch.empty((N, K), dtype=torch.int8, device=device)
    ws = torch.empty((N, K // 32), dtype=torch.float16, device=device)
    for r0 in range(0, N, chunk_rows):
        r1 = min(N, r0 + chunk_rows)
        wq[r0:r1] = torch.randint(-127, 128, (r1 - r0, K), generator=g, device=device,
                                  dtype=torch.int16).to(torch.int8)
        s = torch.randn((r1 - r0, K // 32), generator=g, device=device, dtype=torch.float32)
        ws[r0:r1] = (s.mul_(0.02).abs_().add_(1e-4)).to(torch.float16)
    return wq, ws.view(torch.int16)


def activation_torch(M: int, K: int, seed: int, device, outliers: bool = False):
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(seed)
    x = torch.randn((M, K), generator=g, device=device, dtype=torch.float32)
    if outliers:
        mask = torch.rand((M, K), generator=g, device=device) < 0.01
        x = torch.where(mask, x * 20.0, x)
    return x


def norm_gain_torch(K: int, seed: int, device):
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return 1.0 + 0.1 * torch.randn((K,), generator=g, device=device, dtype=torch.float32)
