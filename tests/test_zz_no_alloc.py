"""kda_fwd_static_scratch: the forward for callers that cannot allocate device
memory (code inside another runtime's plugin interface, where the host owns
every allocation, or serving loops that must not allocate). It runs the same
kernels on a scratch array compiled into the library. Two calls in a row, on
different workloads, must give what kda_fwd gives with its own workspace,
within the parity tolerances. This file is collected last on purpose."""
import pytest
import torch

from parity import check
from kimi_delta_attention_15_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def _both(inp):
    from kimi_delta_attention_15_gb300 import ops
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    cu = d["cu_seqlens"] if len(inp["lengths"]) > 1 else None
    args = (d["q"], d["k"], d["v"], d["g_raw"], d["beta_raw"], d["A_log"], d["dt_bias"])
    o_s, hT_s = ops.fwd_static_scratch(*args, h0=d["h0"], cu_seqlens=cu)
    torch.cuda.synchronize()
    o_w, hT_w, ws = ops.fwd(*args, h0=d["h0"], cu_seqlens=cu)
    assert ops.device_status(ws) == 0
    torch.cuda.synchronize()
    return (o_s, hT_s), (o_w, hT_w)


def test_static_scratch_forward_matches_workspace_forward_twice():
    for inp in (I.make_inputs(I.WORKLOADS[1]), I.make_inputs(I.custom((200, 3, 90), 2, h0=True), seed=5)):
        (o_s, hT_s), (o_w, hT_w) = _both(inp)
        check("o", o_s, o_w)
        check("hT", hT_s, hT_w)


def test_static_scratch_rejects_too_large_shape():
    from kimi_delta_attention_15_gb300 import ops
    w = I.custom((8192,), 8)
    inp = I.make_inputs(w, seed=1)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    with pytest.raises(ops.KdaError) as e:
        ops.fwd_static_scratch(d["q"], d["k"], d["v"], d["g_raw"], d["beta_raw"], d["A_log"], d["dt_bias"])
    assert e.value.code == 5 and "static scratch holds" in str(e.value)
