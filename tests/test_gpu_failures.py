"""Failure detection on the GPU without a fault: malformed offsets are caught by
the device-side check (status word, no kernel touches the data), and a wait
that runs out returns KDA_ERR_TIMEOUT through the status word with the CUDA
context still usable."""
import pytest
import torch

from gpu_helpers import run_fwd_bwd
from parity import check
import oracle
from kimi_delta_attention_15_gb300 import inputs as I

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("bad", [[0, 40, 30, 100], [0, 50, 100, 99], [1, 50, 70, 100]])
def test_malformed_offsets_set_device_status(bad):
    from kimi_delta_attention_15_gb300 import ops
    inp = I.make_inputs(I.custom((50, 20, 30), 2), seed=3)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    cu = torch.tensor(bad, dtype=torch.int64, device="cuda")
    o = torch.full_like(d["v"], 7.0)
    _, _, ws = ops.fwd(d["q"], d["k"], d["v"], d["g_raw"], d["beta_raw"], d["A_log"], d["dt_bias"],
                       cu_seqlens=cu, o=o)
    assert ops.device_status(ws) == 6          # KDA_ERR_OFFSETS
    assert torch.all(o == 7.0)                 # no kernel wrote the output
    g = ops.bwd(d["q"], d["k"], d["v"], d["g_raw"], d["beta_raw"], d["A_log"], d["dt_bias"], d["do"], ws,
                cu_seqlens=cu)
    assert ops.device_status(ws) == 6


def test_wait_timeout_reports_status_and_context_survives():
    from kimi_delta_attention_15_gb300 import ops
    ws = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    ops.wait_timeout(ws, 20_000_000)           # 20 ms limit, nothing arrives
    assert ops.device_status(ws) == 7          # KDA_ERR_TIMEOUT
    # the context still works: a normal forward + backward afterwards is correct
    inp = I.make_inputs(I.WORKLOADS[0])
    out = run_fwd_bwd(inp)
    assert out["status"] == 0
    ref = oracle.forward(inp)
    check("o", out["o"], ref["o"])


def _dev(inp):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def _bwd(ops, d, ws, cu=None, grads=None):
    return ops.bwd(d["q"], d["k"], d["v"], d["g_raw"], d["beta_raw"], d["A_log"], d["dt_bias"], d["do"], ws,
                   cu_seqlens=cu, grads=grads)


def test_backward_on_a_zeroed_workspace_reports_stale_and_computes_nothing():
    """A workspace no forward has filled: the backward's first kernel finds no provenance
    stamp, sets KDA_ERR_STALE_WORKSPACE and no later kernel writes a gradient."""
    from kimi_delta_attention_15_gb300 import ops
    inp = I.make_inputs(I.custom((130,), 2), seed=21)
    d = _dev(inp)
    shape = ops._shape_of(d["q"], d["v"], None, 1, ops.SCALE, ops.LOWER_BOUND)
    ws = torch.zeros(ops.workspace_size(shape), dtype=torch.uint8, device="cuda")
    grads = dict(dq=torch.full_like(d["q"], 3.0), dk=torch.full_like(d["k"], 3.0), dv=torch.full_like(d["v"], 3.0),
                 dg_raw=torch.full_like(d["g_raw"], 3.0), dbeta_raw=torch.full_like(d["beta_raw"], 3.0),
                 dA_log=torch.full_like(d["A_log"], 3.0), ddt_bias=torch.full_like(d["dt_bias"], 3.0),
                 dh0=torch.full((1, 2, 128, 128), 3.0, device="cuda"))
    _bwd(ops, d, ws, grads=grads)
    assert ops.device_status(ws) == 9
    for k, t in grads.items():
        assert torch.all(t == 3.0), k


def test_backward_on_a_workspace_of_another_shape_reports_stale():
    """The forward ran on another shape (fewer tokens) in the same, large enough workspace."""
    from kimi_delta_attention_15_gb300 import ops
    big = _dev(I.make_inputs(I.custom((200,), 2), seed=22))
    small = _dev(I.make_inputs(I.custom((130,), 2), seed=23))
    args = lambda d: (d["q"], d["k"], d["v"], d["g_raw"], d["beta_raw"], d["A_log"], d["dt_bias"])
    _, _, ws = ops.fwd(*args(small), workspace=None)
    shape_big = ops._shape_of(big["q"], big["v"], None, 1, ops.SCALE, ops.LOWER_BOUND)
    ws_big = torch.empty(ops.workspace_size(shape_big), dtype=torch.uint8, device="cuda")
    ops.fwd(*args(small), workspace=ws_big)
    assert ops.device_status(ws_big) == 0
    _bwd(ops, big, ws_big)
    assert ops.device_status(ws_big) == 9
    # the same workspace after a forward of the right shape: the backward runs and is correct
    ops.fwd(*args(big), workspace=ws_big)
    g = _bwd(ops, big, ws_big)
    assert ops.device_status(ws_big) == 0
    inp = I.make_inputs(I.custom((200,), 2), seed=22)
    ref = oracle.backward(inp)
    for k in ("dq", "dk", "dv", "dg_raw"):
        check(k, g[k], ref[k])


def test_backward_with_another_lower_bound_reports_stale():
    """Every field of the shape is stamped, also the gate's lower bound."""
    from kimi_delta_attention_15_gb300 import ops
    d = _dev(I.make_inputs(I.custom((100,), 2), seed=24))
    args = (d["q"], d["k"], d["v"], d["g_raw"], d["beta_raw"], d["A_log"], d["dt_bias"])
    _, _, ws = ops.fwd(*args, lower_bound=-5.0)
    ops.bwd(*args, d["do"], ws, lower_bound=-4.0)
    assert ops.device_status(ws) == 9
