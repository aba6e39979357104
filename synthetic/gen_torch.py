"""Device-side seeded draws for workloads too large to generate on the host in time.

Same shapes, distributions and keys as ``gen.py`` (uniform b_max-bit codes, sorted fp16
N(0, sigma) centroid tables, bf16 N(0, 0.02) shared weights), drawn with torch's CUDA
generator seeded from the same (seed, tag, layer, expert, u, b) keys.  The values differ
from the numpy draws; a test that compares against the oracle copies these arrays to the
host and hands them to the oracle.
"""
from __future__ import annotations

import numpy as np
import torch

from .gen import TAG_IDX, TAG_LUT, TAG_SHARED, LayerShape, block_shape


def _seed(*key: int) -> int:
    ss = np.random.SeedSequence([int(k) & 0xFFFFFFFF for k in key])
    return int(ss.generate_state(1, np.uint64)[0] & np.uint64((1 << 63) - 1))


def gen_block_torch(shape: LayerShape, seed: int, layer: int, expert: int, u: int, device="cuda"):
    """(idx uint8 [N][K], lut int16 view of fp16: LUTs of every supported b concatenated)."""
    N, K = block_shape(shape, u)
    g = torch.Generator(device=device)
    g.manual_seed(_seed(seed, TAG_IDX, layer, expert, u))
    idx = torch.randint(0, 1 << shape.bmax, (N, K), generator=g, device=device, dtype=torch.uint8)
    parts = []
    for b in shape.bits:
        g.manual_seed(_seed(seed, TAG_LUT, layer, expert, u, b))
        v = (torch.randn((N, 1 << b), generator=g, device=device) * shape.sigma_lut).half()
        v = torch.sort(v, dim=1).values
        parts.append(v.view(torch.int16).reshape(-1))
    return idx, torch.cat(parts)


def gen_shared_torch(shape: LayerShape, seed: int, layer: int, device="cuda"):
    """Shared-expert weights as int16 views of bf16: wgu [2Is][H], wd [H][Is]."""
    g = torch.Generator(device=device)
    g.manual_seed(_seed(seed, TAG_SHARED, layer))
    wgu = (torch.randn((2 * shape.Is, shape.H), generator=g, device=device) * 0.02).bfloat16()
    wd = (torch.randn((shape.H, shape.Is), generator=g, device=device) * 0.02).bfloat16()
    return wgu.view(torch.int16), wd.view(torch.int16)


def split_luts(lut: np.ndarray, N: int, bits):
    """Host view of a concatenated LUT array as dict b -> uint16 [N][2^b]."""
    out, off = {}, 0
    lut = np.asarray(lut).view(np.uint16)
    for b in bits:
        n = N * (1 << b)
        out[b] = lut[off:off + n].reshape(N, 1 << b)
        off += n
    return out
