"""The tcgen05 building blocks (tensor memory, shared-memory operand descriptors, MMA with A
from shared memory or from tensor memory, commit, tensor-memory stores and loads) against a
float64 matrix product."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
pw = pytest.importorskip("any_precision_bit_gb300")


@pytest.fixture(scope="module", autouse=True)
def gpu_ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from any_precision_bit_gb300 import _build
    _build.build()


@pytest.mark.parametrize("a_in_tmem", [False, True])
@pytest.mark.parametrize("N,K", [(16, 16), (16, 128), (64, 128), (128, 64), (256, 128)])
def test_tc_gemm_matches_float64(N, K, a_in_tmem):
    rng = np.random.default_rng(N * 1000 + K)
    A = rng.standard_normal((128, K)).astype(np.float16)
    B = rng.standard_normal((N, K)).astype(np.float16)
    ref = A.astype(np.float64) @ B.astype(np.float64).T
    Ad = torch.from_numpy(A.view(np.int16)).cuda()
    Bd = torch.from_numpy(B.view(np.int16)).cuda()
    D = torch.full((128, N), float("nan"), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    pw.pw_tc_selftest(Ad, Bd, N, K, D, err, a_in_tmem=a_in_tmem)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = D.cpu().numpy().astype(np.float64)
    # fp16 products are exact in fp32; K <= 128 fp32 additions
    assert np.allclose(got, ref, rtol=1e-5, atol=1e-4 * np.sqrt(K)), np.abs(got - ref).max()
