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
