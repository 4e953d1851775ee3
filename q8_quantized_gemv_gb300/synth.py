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


# ---- the GGUF block formats other than Q8_0 ----------------------------------------
# Per format: (values a block, bytes a block, byte offsets of its f16 scale
# fields, byte offset of an E8M0 exponent byte or None).  Only where the
# scale fields sit, to draw valid blocks: every other byte of a block (levels,
# packed sub-scales, high bits) is uniform random; the f16 fields are
# |N(0, 0.02)| + 1e-4 as for Q8_0, the E8M0 exponents 118..128 (scales
# 2^-10 .. 1), so the products stay finite.
BLK_LAYOUT = {
    "q4_0": (32, 18, (0,), None), "q4_1": (32, 20, (0, 2), None), "q5_0": (32, 22, (0,), None),
    "q5_1": (32, 24, (0, 2), None), "iq4_nl": (32, 18, (0,), None), "mxfp4": (32, 17, (), 0),
    "q2_k": (256, 84, (80, 82), None), "q3_k": (256, 110, (108,), None), "q4_k": (256, 144, (0, 2), None),
    "q5_k": (256, 176, (0, 2), None), "q6_k": (256, 210, (208,), None), "iq4_xs": (256, 136, (0,), None),
}


def blk_matrix(fmt: str, N: int, K: int, seed: int) -> np.ndarray:
    """A block-format matrix: uint8 [N, K / values * bytes] (host)."""
    qk, nbytes, f16_at, e8_at = BLK_LAYOUT[fmt]
    assert K % qk == 0
    r = rng(seed)
    nblk = N * (K // qk)
    blocks = r.integers(0, 256, size=(nblk, nbytes), dtype=np.uint8)
    for off in f16_at:
        s = (np.abs(r.standard_normal(nblk)) * 0.02 + 1e-4).astype(np.float16)
        blocks[:, off:off + 2] = s.view(np.uint8).reshape(nblk, 2)
    if e8_at is not None:
        blocks[:, e8_at] = r.integers(118, 129, size=nblk, dtype=np.uint8)
    return blocks.reshape(N, (K // qk) * nbytes)


def blk_matrix_torch(fmt: str, N: int, K: int, seed: int, device, chunk_rows: int = 4096):
    """blk_matrix's distributions on ``device`` (seeded torch generator, rows
    in chunks): uint8 [N, row bytes]."""
    import torch

    qk, nbytes, f16_at, e8_at = BLK_LAYOUT[fmt]
    assert K % qk == 0
    nb = K // qk
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    w = torch.empty((N, nb * nbytes), dtype=torch.uint8, device=device)
    for r0 in range(0, N, chunk_rows):
        r1 = min(N, r0 + chunk_rows)
        blk = torch.randint(0, 256, ((r1 - r0) * nb, nbytes), generator=g, device=device, dtype=torch.int16)
        blk = blk.to(torch.uint8)
        for off in f16_at:
            s = torch.randn(((r1 - r0) * nb,), generator=g, device=device).mul_(0.02).abs_().add_(1e-4)
            blk[:, off:off + 2] = s.to(torch.float16).view(torch.uint8).view(-1, 2)
        if e8_at is not None:
            blk[:, e8_at] = torch.randint(118, 129, ((r1 - r0) * nb,), generator=g, device=device,
                                          dtype=torch.int16).to(torch.uint8)
        w[r0:r1] = blk.view(r1 - r0, nb * nbytes)
    return w
