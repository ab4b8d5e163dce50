"""kda_fwd + kda_bwd captured in a CUDA graph and replayed.

The launch path neither allocates nor synchronises, so a caller can capture a
training step: after one eager call with the same buffers (which lets the
library set its kernel attributes), the pair is captured on a side stream and
the replay must write exactly what the eager calls wrote (every kernel is
deterministic)."""
import pytest
import torch

from gpu_helpers import to_dev
from kimi_delta_attention_15_gb300 import inputs as I, ops

pytestmark = pytest.mark.gpu


# packed [17, 33, 65] at H=4, T=4096 at H=32, and grouped value heads (a tenth kernel, the
# group reduction of dq, dk, inside the captured step)
WORKLOADS = [I.WORKLOADS[1], I.WORKLOADS[2], I.custom((100, 37, 64), 8, h0=True, dhT=True, groups=4)]


@pytest.mark.parametrize("w", WORKLOADS, ids=[w.name for w in WORKLOADS])
def test_capture_and_replay_matches_eager(w):
    d = to_dev(I.make_inputs(w))
    cu = d["cu_seqlens"] if w.packed else None
    shape = ops.make_shape(w.T, w.H, w.N, groups=w.groups)
    ws = ops.alloc_workspace(shape, d["q"].device)
    o = torch.empty_like(d["v"])
    hT = torch.empty(w.N, w.H, 128, 128, dtype=torch.float32, device=o.device)
    grads = dict(dq=torch.empty_like(d["q"]), dk=torch.empty_like(d["k"]), dv=torch.empty_like(d["v"]),
                 dg_raw=torch.empty_like(d["g_raw"]), dbeta_raw=torch.empty_like(d["beta_raw"]),
                 dA_log=torch.empty_like(d["A_log"]), ddt_bias=torch.empty_like(d["dt_bias"]),
                 dh0=torch.empty_like(hT))
    outs = dict(o=o, hT=hT, **grads)

    def step():
        ops.fwd(d["q"], d["k"], d["v"], d["g_raw"], d["beta_raw"], d["A_log"], d["dt_bias"], h0=d.get("h0"),
                cu_seqlens=cu, workspace=ws, o=o, hT=hT)
        ops.bwd(d["q"], d["k"], d["v"], d["g_raw"], d["beta_raw"], d["A_log"], d["dt_bias"], d["do"], ws,
                h0=d.get("h0"), cu_seqlens=cu, dhT=d.get("dhT"), grads=grads)

    step()
    torch.cuda.synchronize()
    assert ops.device_status(ws) == 0
    eager = {k: v.clone() for k, v in outs.items()}

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()                      # a call on the capture stream before capturing
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for v in outs.values():
        v.zero_()
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    assert ops.device_status(ws) == 0
    for k, v in outs.items():
        assert torch.equal(v, eager[k]), k
