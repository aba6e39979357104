"""Pins of the oracle's bit-plane, lookup and bytes functions (CPU only)."""
import numpy as np
import pytest

from conftest import load_golden
from oracle import ap


def test_planes_hand_example():
    g = load_golden("planes_hand.json")
    idx = np.array(g["idx"], dtype=np.uint8)
    planes = ap.pack_planes(idx, g["bmax"])
    assert planes.shape == (g["bmax"], 1, g["words_per_row"])
    assert [int(planes[p, 0, 0]) for p in range(g["bmax"])] == g["plane_word0"]
    assert not planes[:, :, 1:].any()  # pad columns are zero bits
    assert ap.unpack_indices(planes, 2, 3).tolist() == g["idx_top2"]
    assert ap.unpack_indices(planes, 1, 3).tolist() == g["idx_top1"]
    assert ap.unpack_indices(planes, 3, 3).tolist() == g["idx"]


def _brute_bits(code, bmax, b):
    """Top-b code from the bmax-bit code, one bit at a time with Python ints."""
    v = 0
    for p in range(b):
        bit = (int(code) >> (bmax - 1 - p)) & 1
        v = v * 2 + bit
    return v


@pytest.mark.parametrize("bmax,K", [(6, 5), (6, 128), (8, 131), (8, 300), (4, 64)])
def test_unpack_brute_force(bmax, K):
    rng = np.random.default_rng(bmax * 1000 + K)
    idx = rng.integers(0, 1 << bmax, size=(3, K), dtype=np.uint8)
    planes = ap.pack_planes(idx, bmax)
    assert planes.shape[2] * 32 == ap.kpad(K)
    for b in range(1, bmax + 1):
        got = ap.unpack_indices(planes, b, K)
        for n in range(3):
            for k in range(K):
                assert got[n, k] == _brute_bits(idx[n, k], bmax, b)
        # the plain definition: the top b bits of the code
        assert np.array_equal(got, idx >> (bmax - b))


def test_plane_bit_positions_brute_force():
    rng = np.random.default_rng(7)
    bmax, K = 5, 200
    idx = rng.integers(0, 1 << bmax, size=(2, K), dtype=np.uint8)
    planes = ap.pack_planes(idx, bmax)
    for p in range(bmax):
        for n in range(2):
            for k in range(ap.kpad(K)):
                word = int(planes[p, n, k // 32])
                bit = (word >> (k % 32)) & 1
                want = ((int(idx[n, k]) >> (bmax - 1 - p)) & 1) if k < K else 0
                assert bit == want


def test_lower_bitwidth_reads_only_top_planes():
    """Dropping to b' reads only planes 0..b'-1: poisoning planes >= b' changes nothing."""
    rng = np.random.default_rng(3)
    bmax, K = 8, 257
    idx = rng.integers(0, 256, size=(4, K), dtype=np.uint8)
    planes = ap.pack_planes(idx, bmax)
    for b in range(1, bmax):
        poisoned = planes.copy()
        poisoned[b:] = 0xFFFFFFFF
        assert np.array_equal(ap.unpack_indices(poisoned, b, K), ap.unpack_indices(planes, b, K))


def test_dequant_lookup():
    lut = np.array([[1.0, -2.0, 0.5, 3.0], [0.25, 0.125, -1.0, 8.0]], dtype=np.float16).view(np.uint16)
    idx = np.array([[3, 0, 2], [1, 1, 3]], dtype=np.uint8)
    W = ap.dequant(idx, lut)
    assert W.tolist() == [[3.0, 1.0, 0.5], [0.125, 0.125, 8.0]]
    assert W.dtype == np.float64
    bits = ap.dequant_fp16_bits(idx, lut)
    assert bits.view(np.float16).astype(np.float64).tolist() == W.tolist()


def test_eq3_hand_example():
    g = load_golden("eq3_bytes.json")
    N, K, bits = g["N"], g["K"], g["bits"]
    assert ap.plane_bytes(N, K) == g["P"]
    for b in bits:
        assert ap.block_bytes(N, K, bits, b) == g["M"][str(b)]
    assert ap.delta_bytes(N, K, bits, 4, 3) == g["delta_4_3"]
    with pytest.raises(ValueError):
        ap.delta_bytes(N, K, bits, 3, 4)


def test_eq3_telescopes():
    """Delta over a chain of single-level steps equals the direct Delta (Eq. 3 is a difference)."""
    bits = (3, 4, 5, 6, 7, 8)
    N, K = 2816, 2048
    direct = ap.delta_bytes(N, K, bits, 8, 3)
    chain = sum(ap.delta_bytes(N, K, bits, b, b - 1) for b in range(4, 9))
    assert direct == chain
    # one level of a block with K=2048: one plane (N*256 B) plus LUT_8 (N*512 B)
    assert ap.delta_bytes(N, K, bits, 8, 7) == N * 256 + N * 256 * 2


def test_read_bytes():
    assert ap.read_bytes(2, 128, 4) == 4 * 32 + 2 * 16 * 2
