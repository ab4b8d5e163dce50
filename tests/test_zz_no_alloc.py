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


def test_static_scratch_single_sequence_and_near_the_limit():
    """A fixed-length input without offsets (its own layout and chunk-table branch), and a
    shape whose forward regions fill most of the array, so that its far end is used."""
    from kimi_delta_attention_15_gb300 import ops
    for w, seed in ((I.custom((130,), 2), 6), (I.custom((2048,), 4), 7)):
        inp = I.make_inputs(w, seed=seed)
        (o_s, hT_s), (o_w, hT_w) = _both(inp)
        assert ops.static_scratch_device_status() == 0
        check("o", o_s, o_w)
        check("hT", hT_s, hT_w)
    sh = ops.make_shape(2048, 5, 1)
    full = ops.workspace_size(sh)
    assert full > ops.STATIC_SCRATCH_BYTES   # the full forward + backward layout would not fit


def test_static_scratch_reports_device_errors():
    """Malformed offsets found on the device land in the scratch array's status word, which
    kda_static_scratch_device_status reads; the next good call clears it."""
    from kimi_delta_attention_15_gb300 import ops
    inp = I.make_inputs(I.custom((50, 20, 30), 2), seed=3)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    args = (d["q"], d["k"], d["v"], d["g_raw"], d["beta_raw"], d["A_log"], d["dt_bias"])
    bad = torch.tensor([0, 40, 30, 100], dtype=torch.int64, device="cuda")
    o = torch.full_like(d["v"], 7.0)
    ops.fwd_static_scratch(*args, cu_seqlens=bad, o=o)
    assert ops.static_scratch_device_status() == 6   # KDA_ERR_OFFSETS
    assert torch.all(o == 7.0)
    ops.fwd_static_scratch(*args, cu_seqlens=d["cu_seqlens"])
    assert ops.static_scratch_device_status() == 0


def test_static_scratch_rejects_too_large_shape():
    from kimi_delta_attention_15_gb300 import ops
    w = I.custom((8192,), 8)
    inp = I.make_inputs(w, seed=1)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    with pytest.raises(ops.KdaError) as e:
        ops.fwd_static_scratch(d["q"], d["k"], d["v"], d["g_raw"], d["beta_raw"], d["A_log"], d["dt_bias"])
    assert e.value.code == 5 and "static scratch holds" in str(e.value)
