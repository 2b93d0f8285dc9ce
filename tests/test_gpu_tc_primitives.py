"""Unit test of the tensor-core building blocks (tcgen05.mma on SW128 K-major
bf16 and fp16 operands, fp32 TMEM accumulators, tcgen05.ld/st) against a host fp64
matmul of the same 16-bit values."""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fp16", [0, 1], ids=["bf16", "fp16"])
@pytest.mark.parametrize("N,K,b_row0", [(64, 64, 0), (64, 128, 0), (128, 128, 0), (128, 64, 0), (64, 128, 64),
                                        (32, 64, 0), (32, 128, 0), (256, 64, 0), (256, 128, 0), (128, 64, 64)])
def test_umma_gemm(N, K, b_row0, fp16):
    import gateddeltanet_layer_gb300 as gdn
    lib = gdn.library()
    fn = lib.gdn_selftest_umma
    fn.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int] * 4 + [ctypes.c_void_p]
    fn.restype = ctypes.c_int
    g = torch.Generator().manual_seed(N * 1000 + K + b_row0)
    dt = torch.float16 if fp16 else torch.bfloat16
    A = torch.randn(128, K, generator=g).to(dt)
    B = torch.randn(b_row0 + N, K, generator=g).to(dt)
    Ad, Bd = A.cuda(), B.cuda()
    D = torch.full((2, 128, N), float("nan"), device="cuda")
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = fn(Ad.data_ptr(), Bd.data_ptr(), D.data_ptr(), flag.data_ptr(), N, K, b_row0, fp16,
            torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
    ref = A.double().numpy() @ B.double().numpy()[b_row0:b_row0 + N].T
    got = D.cpu().double().numpy()
    np.testing.assert_allclose(got[0], ref, rtol=1e-5, atol=1e-4)
    np.testing.assert_allclose(got[1], 2 * ref, rtol=1e-5, atol=2e-4)


@pytest.mark.parametrize("fp16", [0, 1], ids=["bf16", "fp16"])
@pytest.mark.parametrize("N,K", [(128, 128), (128, 64), (64, 64), (256, 128), (128, 32)])
def test_umma_a_from_tensor_memory(N, K, fp16):
    """tcgen05.mma with A in tensor memory (row m in lane m, elements packed two per column)."""
    import gateddeltanet_layer_gb300 as gdn
    lib = gdn.library()
    fn = lib.gdn_selftest_umma_ts
    fn.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int] * 3 + [ctypes.c_void_p]
    fn.restype = ctypes.c_int
    g = torch.Generator().manual_seed(N * 7 + K)
    dt = torch.float16 if fp16 else torch.bfloat16
    A = torch.randn(128, K, generator=g).to(dt)
    B = torch.randn(N, K, generator=g).to(dt)
    Ad, Bd = A.cuda(), B.cuda()
    D = torch.full((128, N), float("nan"), device="cuda")
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert fn(Ad.data_ptr(), Bd.data_ptr(), D.data_ptr(), flag.data_ptr(), N, K, fp16,
              torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
    ref = A.double().numpy() @ B.double().numpy().T
    np.testing.assert_allclose(D.cpu().double().numpy(), ref, rtol=1e-5, atol=1e-4)
