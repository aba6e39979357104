"""bench.py's algorithmic bytes, the numerator of its HBM roofline, on a hand-worked layer.

The tiny shape (H = 128, I = 256, E = 8, K = 2, no shared expert): a gate_up block is
N = 512 rows by K = 128 columns, so one bit-plane is 512 * 128 / 8 = 8192 bytes and LUT_b
is 512 * 2^b fp16 entries; a down block is 128 x 256, one plane 4096 bytes.  A forward
reads an active block's top q planes and LUT_q only (PagedWeight Sec. 2.2 and Sec. 3.3);
inactive experts are not read.  With expert 0 active at q = (4, 3) and T = 2 tokens:
  gate_up  4 * 8192 + 512 * 16 * 2 = 49152
  down     3 * 4096 + 128 * 8 * 2  = 14336
  router   E * H * 4 = 4096 (fp32)
  act      2 * T * H * 2 = 1024 (bf16 in and out)
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synthetic as syn  # noqa: E402


def test_layer_bytes_hand_example():
    import bench
    shape = syn.SHAPES["tiny"]
    q = np.full((shape.E, 2), 6, dtype=np.int32)
    q[0] = (4, 3)
    counts = np.zeros(shape.E)
    counts[0] = 3
    b = bench.layer_bytes(shape, q, counts, 2)
    assert (b["gu"], b["dn"], b["sh_gu"], b["sh_dn"], b["router"], b["act"]) == (49152, 14336, 0, 0, 4096, 1024)
    assert b["total"] == 49152 + 14336 + 4096 + 1024 and b["weights"] == 49152 + 14336


def test_layer_bytes_shared_expert_and_ragged_columns():
    """A shared expert is read dense (bf16 -> fp16, 2 bytes a weight) whatever the routing;
    a block whose K is not a multiple of 128 reads its planes padded to 128 columns."""
    import bench
    shape = syn.LayerShape("t2", H=144, E=4, I=200, K=1, Is=64, L=1, bmax=8, bits=(3, 4),
                           sigma_lut=0.02, zipf_a=None, q_rule="uniform")
    q = np.full((shape.E, 2), 3, dtype=np.int32)
    counts = np.array([0, 1, 0, 0])
    b = bench.layer_bytes(shape, q, counts, 1)
    # gate_up: N = 400, K = 144 -> 256 padded columns; down: N = 144, K = 200 -> 256
    assert b["gu"] == 3 * 400 * 256 // 8 + 400 * 8 * 2
    assert b["dn"] == 3 * 144 * 256 // 8 + 144 * 8 * 2
    assert b["sh_gu"] == 2 * 64 * 144 * 2 and b["sh_dn"] == 144 * 64 * 2
