"""The tcgen05 tensor-core GEMM primitive against a float64 reference."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (256, 512, 1024), (512, 768, 4096), (1024, 256, 128)])
def test_tc_gemm_matches_reference(gpu_lib, M, N, K):
    import torch
    import megatron_tensor_block_gb300 as tb
    g = torch.Generator().manual_seed(M + N + K)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    B = (0.05 * torch.randn(N, K, generator=g)).to(torch.bfloat16)
    C = torch.full((M, N), float("nan"), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    tb.tp_gemm_bf16(A.cuda(), B.cuda(), C, M, N, K, device_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = A.double() @ B.double().T
    got = C.double().cpu()
    err = float((got - ref).abs().max() / ref.abs().max())
    assert err < 1e-5, err


def test_tc_gemm_rejects_bad_shapes(gpu_lib):
    import torch
    import megatron_tensor_block_gb300 as tb
    A = torch.zeros(100, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(tb.TpError):
        tb.tp_gemm_bf16(A, A, torch.zeros(100, 100, device="cuda"), 100, 100, 64)


@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (256, 512, 1024), (384, 256, 256)])
def test_tc_gemm_with_n_contiguous_b(gpu_lib, M, N, K):
    # B given as [K, N]: the operand form the prefill attention uses for P @ V
    import torch
    import megatron_tensor_block_gb300 as tb
    g = torch.Generator().manual_seed(7 * M + N + K)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    B = (0.05 * torch.randn(K, N, generator=g)).to(torch.bfloat16)
    C = torch.full((M, N), float("nan"), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    tb.tp_gemm_bf16_kn(A.cuda(), B.cuda(), C, M, N, K, device_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = A.double() @ B.double()
    got = C.double().cpu()
    err = float((got - ref).abs().max() / ref.abs().max())
    assert err < 1e-5, err
