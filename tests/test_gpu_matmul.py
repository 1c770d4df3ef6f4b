"""The general tensor-core product (moe_matmul) in its four operand layouts
against a float64 product of the same bf16 operands."""
import numpy as np
import pytest
import torch

from moe_routing_capacity_gb300 import abi

from helpers import check_close

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("a_mn", [False, True])
@pytest.mark.parametrize("b_mn", [False, True])
@pytest.mark.parametrize("f32", [False, True])
@pytest.mark.parametrize("shape", [(296, 520, 200), (128, 256, 64), (1000, 776, 1064)])
def test_matmul_layouts(a_mn, b_mn, f32, shape):
    M, N, K = shape
    g = torch.Generator().manual_seed(M + N + K)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    B = torch.randn(N, K, generator=g).to(torch.bfloat16)
    ref = A.double() @ B.double().T
    Ad = (A.T.contiguous() if a_mn else A).cuda()
    Bd = (B.T.contiguous() if b_mn else B).cuda()
    out = torch.zeros(M, N, dtype=torch.float32 if f32 else torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    abi.matmul(Ad, Bd, M, N, K, out, status, a_mn=a_mn, b_mn=b_mn)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = out.double().cpu().numpy()
    want = ref.numpy()
    if f32:
        # fp32 accumulation of K products of magnitude ~1
        assert np.abs(got - want).max() <= 1e-3 * np.sqrt(K)
    else:
        check_close("out", got, np.asarray(torch.from_numpy(want).to(torch.bfloat16).double()))
