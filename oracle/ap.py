"""Any-Precision bit-plane codes, centroid lookup and resident bytes (oracle; test infrastructure).

PagedWeight, Sec. 2.2: a quantised tensor keeps shared bit-planes; a subset of planes
gives a lower effective bitwidth, and a per-bitwidth lookup table (LUT) holds the
centroids.  Sec. 3.1, Eq. 3: the bytes released by b -> b' are M^b - M^{b'}, where M^b
counts the planes and the LUTs resident at b.

Readings where the pages are silent:
* plane 0 holds the most significant bit, so a b-bit code is the top b planes;
* inside a plane, rows are uint32 words, bit j of word w is column 32*w + j, and each
  row is padded with zero bits to a multiple of 128 columns (16 bytes);
* the LUT for bitwidth b is 2^b fp16 centroids per output row;
* page p is plane p plus LUT_{p+1} (when p+1 is a supported bitwidth), so at bitwidth
  q the resident bytes are planes 0..q-1 and the LUTs of every supported c <= q.
"""
from __future__ import annotations

import numpy as np


def kpad(K: int) -> int:
    """Columns per plane row after padding to a multiple of 128 bits."""
    return 128 * ((K + 127) // 128)


def plane_bytes(N: int, K: int) -> int:
    """Bytes of one bit-plane of an N x K block (P in the resident-bytes formula)."""
    return N * kpad(K) // 8


def pack_planes(idx: np.ndarray, bmax: int) -> np.ndarray:
    """Split b_max-bit codes into b_max bit-planes, most significant plane first.

    Returns uint32 [bmax][N][kpad(K)/32]; plane p carries bit (bmax-1-p) of every code.
    """
    idx = np.asarray(idx)
    N, K = idx.shape
    Kp = kpad(K)
    codes = np.zeros((N, Kp), dtype=np.uint32)
    codes[:, :K] = idx
    out = np.zeros((bmax, N, Kp // 32), dtype=np.uint32)
    weights = (np.uint32(1) << np.arange(32, dtype=np.uint32))
    for p in range(bmax):
        bits = (codes >> np.uint32(bmax - 1 - p)) & np.uint32(1)
        out[p] = (bits.reshape(N, Kp // 32, 32) * weights).sum(axis=2, dtype=np.uint64).astype(np.uint32)
    return out


def unpack_indices(planes: np.ndarray, b: int, K: int) -> np.ndarray:
    """b-bit codes from the top b planes only: idx_b = sum_{p<b} bit_p * 2^(b-1-p)."""
    nplanes, N, W = planes.shape
    if b > nplanes:
        raise ValueError("not enough planes")
    acc = np.zeros((N, W * 32), dtype=np.uint32)
    shifts = np.arange(32, dtype=np.uint32)
    for p in range(b):
        bits = (planes[p][:, :, None] >> shifts) & np.uint32(1)
        acc += bits.reshape(N, W * 32) << np.uint32(b - 1 - p)
    return acc[:, :K].astype(np.uint8)


def fp16_bits_to_f64(lut_bits: np.ndarray) -> np.ndarray:
    return np.asarray(lut_bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def dequant(idx_b: np.ndarray, lut_b_bits: np.ndarray) -> np.ndarray:
    """W^(b)[n][k] = LUT_b[n][idx_b[n][k]] as float64."""
    lut = fp16_bits_to_f64(lut_b_bits)
    rows = np.arange(idx_b.shape[0])[:, None]
    return lut[rows, idx_b.astype(np.int64)]


def dequant_fp16_bits(idx_b: np.ndarray, lut_b_bits: np.ndarray) -> np.ndarray:
    """The same lookup returning the raw fp16 bits (for bit-exact comparisons)."""
    rows = np.arange(idx_b.shape[0])[:, None]
    return np.asarray(lut_b_bits, dtype=np.uint16)[rows, idx_b.astype(np.int64)]


def block_bytes(N: int, K: int, bits, b: int) -> int:
    """M^b: planes 0..b-1 plus LUT_c (2^c fp16 per row) for every supported c <= b."""
    return b * plane_bytes(N, K) + sum(N * (1 << c) * 2 for c in bits if c <= b)


def delta_bytes(N: int, K: int, bits, b: int, b2: int) -> int:
    """Eq. 3: bytes released by lowering a block from b to b2 < b."""
    if not b2 < b:
        raise ValueError("Eq. 3 needs b' < b")
    return block_bytes(N, K, bits, b) - block_bytes(N, K, bits, b2)


def read_bytes(N: int, K: int, b: int) -> int:
    """Bytes a forward pass must read for one block at bitwidth b: b planes plus LUT_b."""
    return b * plane_bytes(N, K) + N * (1 << b) * 2
