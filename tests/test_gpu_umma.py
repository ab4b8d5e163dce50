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


def test_tf32_round_matches_hardware_conversion():
    # the kernels round tf32 operands with integer operations; they must equal the
    # hardware conversion (nearest, ties away from zero; NaNs only cleared) bit for bit
    from kimi_delta_attention_15_gb300 import ops
    g = torch.Generator(device="cpu").manual_seed(5)
    bits = torch.randint(-2**31, 2**31 - 1, (1 << 22,), generator=g, dtype=torch.int64)
    special = torch.tensor([
        0x00000000, 0x80000000, 0x00000001, 0x00000fff, 0x00001000, 0x00001001, 0x007ff000, 0x007fffff,
        0x3f800fff, 0x3f801000, 0x3f801001, 0x3f802fff, 0x3f803000, 0x3f7ff000, 0x3f7fefff, 0x3fffffff,
        0x7f7fefff, 0x7f7ff000, 0x7f7fffff, 0x7f800000, 0x7fc00000, 0x80001000, 0xbf801000, 0xbfffffff,
        0xff7fffff, 0xff800000, 0x7f800001, 0x7f801fff, 0x7f802000, 0x7fffffff, 0xffffffff, 0xff801000],
        dtype=torch.int64)
    allbits = torch.cat([bits, special])
    allbits = torch.where(allbits > 0x7FFFFFFF, allbits - (1 << 32), allbits).to(torch.int32)
    x = allbits.view(torch.float32).cuda()
    out, ref = ops.tf32_round_check(x)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int32), ref.view(torch.int32))
