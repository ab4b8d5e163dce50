"""GPU parity of the backward (kda_bwd through the C ABI) against the fp64 oracle,
plus determinism of repeated runs."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import run_fwd_bwd
from parity import check
from kimi_delta_attention_15_gb300 import inputs as I

pytestmark = pytest.mark.gpu

GRADS = ("dq", "dk", "dv", "dg_raw", "dbeta_raw", "dh0", "dA_log", "ddt_bias")


def _compare(inp, out, keys=("o", "hT") + GRADS):
    ref = dict(oracle.forward(inp))
    ref.update(oracle.backward(inp))
    assert out["status"] == 0
    for k in keys:
        check(k, out[k], ref[k])


@pytest.mark.parametrize("idx", [0, 1])
def test_fwd_bwd_small_workloads(idx):
    inp = I.make_inputs(I.WORKLOADS[idx])
    _compare(inp, run_fwd_bwd(inp))


@pytest.mark.parametrize("lengths", [(1,), (2,), (16,), (63,), (64,), (65,), (128,), (129,), (190,)])
def test_fwd_bwd_ragged_single_sequence(lengths):
    inp = I.make_inputs(I.custom(lengths, 3, h0=True, dhT=True), seed=300 + lengths[0])
    out = run_fwd_bwd(inp)
    # dA_log is one scalar per head, a strongly cancelling sum: checked on the
    # workloads with many tokens per head (see test_gpu_large); here per element
    _compare(inp, out, keys=("o", "hT", "dq", "dk", "dv", "dg_raw", "dbeta_raw", "dh0", "ddt_bias"))


def test_fwd_bwd_packed_with_empty_and_tiny_sequences():
    lengths = (70, 0, 1, 64, 0, 130)
    inp = I.make_inputs(I.custom(lengths, 4, h0=True, dhT=True), seed=11)
    out = run_fwd_bwd(inp)
    _compare(inp, out, keys=("o", "hT", "dq", "dk", "dv", "dg_raw", "dbeta_raw", "dh0", "ddt_bias"))
    h0, dhT = inp["h0"].numpy(), inp["dhT"].numpy()
    # empty sequences: hT = h0 and dh0 = dhT exactly
    for n in (1, 4):
        np.testing.assert_array_equal(out["hT"][n].cpu().numpy(), h0[n])
        np.testing.assert_array_equal(out["dh0"][n].cpu().numpy(), dhT[n])


@pytest.mark.parametrize("lengths,G", [((0, 0, 0), 1), ((0,), 1), ((0, 0), 2)])
def test_no_tokens_at_all(lengths, G):
    """Every sequence empty: the token tensors are empty (NULL data pointers), the states pass
    through unchanged (hT = h0, dh0 = dhT) and the parameter gradients are zero."""
    inp = I.make_inputs(I.custom(lengths, 4, h0=True, dhT=True, groups=G), seed=15)
    assert inp["q"].numel() == 0
    out = run_fwd_bwd(inp)
    assert out["status"] == 0
    np.testing.assert_array_equal(out["hT"].cpu().numpy(), inp["h0"].numpy())
    np.testing.assert_array_equal(out["dh0"].cpu().numpy(), inp["dhT"].numpy())
    assert not out["dA_log"].any() and not out["ddt_bias"].any()
    assert out["o"].shape == inp["v"].shape and out["dq"].shape == inp["q"].shape


def test_fwd_bwd_many_short_packed_sequences():
    # 200 sequences of 0..70 tokens: more chunk x head tiles than SMs, so the
    # persistent kernels run several tiles each and reach the empty chunk slots
    # that follow the last real chunk of a packed batch
    rng = np.random.default_rng(14)
    lengths = tuple(int(x) for x in rng.integers(0, 71, size=200))
    inp = I.make_inputs(I.custom(lengths, 2, h0=True, dhT=True), seed=14)
    out = run_fwd_bwd(inp)
    _compare(inp, out, keys=("o", "hT", "dq", "dk", "dv", "dg_raw", "dbeta_raw", "dh0", "ddt_bias"))


def test_thousands_of_packed_sequences():
    # 3,000 sequences of 0..40 tokens: many share a chunk count, so the longest-first scan
    # order (a counting sort with ties in any order) must still be a permutation
    rng = np.random.default_rng(16)
    lengths = tuple(int(x) for x in rng.integers(0, 41, size=3000))
    inp = I.make_inputs(I.custom(lengths, 2, h0=True, dhT=True), seed=16)
    out = run_fwd_bwd(inp)
    _compare(inp, out, keys=("o", "hT", "dq", "dk", "dv", "dg_raw", "dbeta_raw", "dh0", "ddt_bias"))


def test_degenerate_rows():
    """Zero q, k and v rows (padding tokens: q^ = k^ = 0 through the eps of the norm, whose
    gradient is 1/sqrt(eps) times the adjoint), beta ~ 0 (beta_raw = -30) and saturated gates
    (g_raw = +-50), at positions inside, at the start and at the end of chunks."""
    inp = I.make_inputs(I.custom((200,), 3, h0=True, dhT=True), seed=17)
    for r in (0, 5, 64, 130, 199):
        inp["q"][r] = 0
    for r in (7, 63, 65):
        inp["k"][r] = 0
    inp["v"][100:111] = 0
    inp["beta_raw"][10:21] = -30.0
    inp["g_raw"][150:155] = 50.0
    inp["g_raw"][160:165] = -50.0
    out = run_fwd_bwd(inp)
    _compare(inp, out, keys=("o", "hT", "dq", "dk", "dv", "dg_raw", "dbeta_raw", "dh0", "ddt_bias"))


@pytest.mark.parametrize("scale,h0_mult", [(1.0, 1.0), (0.01, 1.0), (0.0883883476, 10.0)])
def test_other_scales_and_a_large_initial_state(scale, h0_mult):
    """Any finite positive output scale is accepted (the pages fix 1/sqrt(128)); an initial
    state ten times the usual size."""
    inp = I.make_inputs(I.custom((150, 40), 2, h0=True, dhT=True), seed=18)
    inp["scale"] = scale
    inp["h0"] = inp["h0"] * h0_mult
    _compare(inp, run_fwd_bwd(inp), keys=("o", "hT", "dq", "dk", "dv", "dg_raw", "dbeta_raw", "dh0", "ddt_bias"))


def test_strong_decay_gate():
    inp = I.make_inputs(I.custom((256,), 2, g_std=4.0, h0=True, dhT=True), seed=12)
    inp["A_log"] = torch.full((2,), float(np.log(16.0)))
    _compare(inp, run_fwd_bwd(inp), keys=("o", "hT", "dq", "dk", "dv", "dg_raw", "dbeta_raw", "dh0", "ddt_bias"))


def test_no_initial_state_no_final_adjoint():
    inp = I.make_inputs(I.custom((100, 50), 2), seed=13)
    assert inp["h0"] is None and inp["dhT"] is None
    _compare(inp, run_fwd_bwd(inp), keys=("o", "hT", "dq", "dk", "dv", "dg_raw", "dbeta_raw", "dh0", "ddt_bias"))


def test_bitwise_deterministic():
    inp = I.make_inputs(I.WORKLOADS[1])
    a = run_fwd_bwd(inp)
    b = run_fwd_bwd(inp)
    for k in ("o", "hT") + GRADS:
        assert torch.equal(a[k], b[k]), k


@pytest.mark.parametrize("lengths", [(17, 33, 65), (300,)])
def test_chunk_size_32_option(lengths):
    """chunk_size = 32 (the other chunk length the Kimi-K3 fused_chunk validator admits) is
    served by the 64-token chunk kernels: the chunk length blocks the computation and does
    not change the function (the oracle's chunk-form pins hold at C = 32 and C = 64), so
    the results equal the oracle within the tolerances and chunk_size = 64 bit for bit."""
    inp = I.make_inputs(I.custom(lengths, 2, h0=True, dhT=True), seed=41)
    inp32 = dict(inp, chunk_size=32)
    out32, out64 = run_fwd_bwd(inp32), run_fwd_bwd(inp)
    _compare(inp, out32, keys=("o", "hT", "dq", "dk", "dv", "dg_raw", "dbeta_raw", "dh0", "ddt_bias"))
    for k in ("o", "hT") + GRADS:
        assert torch.equal(out32[k], out64[k]), k


def test_backward_twice_on_one_forward():
    """kda_bwd may run more than once on the workspace of one kda_fwd (the per-head counters of
    the parameter reduction reset themselves): the second call writes the same gradients."""
    from gpu_helpers import to_dev
    from kimi_delta_attention_15_gb300 import ops
    inp = I.make_inputs(I.custom((300, 70, 129), 3, h0=True, dhT=True), seed=29)
    d = to_dev(inp)
    args = (d["q"], d["k"], d["v"], d["g_raw"], d["beta_raw"], d["A_log"], d["dt_bias"])
    o, hT, ws = ops.fwd(*args, h0=d["h0"], cu_seqlens=d["cu_seqlens"])
    g1 = ops.bwd(*args, d["do"], ws, h0=d["h0"], cu_seqlens=d["cu_seqlens"], dhT=d["dhT"])
    g2 = ops.bwd(*args, d["do"], ws, h0=d["h0"], cu_seqlens=d["cu_seqlens"], dhT=d["dhT"])
    torch.cuda.synchronize()
    assert ops.device_status(ws) == 0
    for k in GRADS:
        assert torch.equal(g1[k], g2[k]), k
