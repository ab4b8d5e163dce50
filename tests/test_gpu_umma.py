"""tcgen05 building blocks: kind::tf32 MMA with K-major shared-memory operands
(128-byte swizzle) and the TMEM load/store round trip, against torch."""
import pytest
import torch

pytestmark = pytest.mark.gpu


def _tf32(x):
    b = x.contiguous().view(torch.int32)
    return ((b + 0x1000) & ~0x1FFF).view(torch.float32)


@pytest.mark.parametrize("N,Kd", [(64, 128), (128, 64), (256, 128), (32, 32), (128, 128)])
def test_umma_kmajor(N, Kd):
    from kimi_delta_attention_15_gb300 import ops
    torch.manual_seed(N + Kd)
    A = torch.randn(128, Kd, device="cuda")
    B = torch.randn(N, Kd, device="cuda")
    D = ops.umma_selftest(A, B, 0, 0)
    torch.cuda.synchronize()
    ref = _tf32(A).double() @ _tf32(B).double().T
    assert ((D[0].double() - ref).abs().max() / ref.abs().max()).item() < 1e-5
    rows = torch.arange(128, device="cuda").double()[:, None]
    assert (D[1].double() - (2 * D[0].double() + rows)).abs().max().item() < 1e-3
