"""GPU parity of the forward (kda_fwd through the C ABI) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from parity import check
from kimi_delta_attention_15_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def _dev(inp):
    d = {}
    for k, v in inp.items():
        d[k] = v.cuda() if isinstance(v, torch.Tensor) else v
    return d


def run_fwd(inp):
    from kimi_delta_attention_15_gb300 import ops
    d = _dev(inp)
    packed = len(inp["lengths"]) > 1
    o, hT, ws = ops.fwd(d["q"], d["k"], d["v"], d["g_raw"], d["beta_raw"], d["A_log"], d["dt_bias"],
                        h0=d["h0"], cu_seqlens=d["cu_seqlens"] if packed else None)
    assert ops.device_status(ws) == 0
    torch.cuda.synchronize()
    return o, hT, ws


@pytest.mark.parametrize("idx", [0, 1])
def test_forward_small_workloads(idx):
    w = I.WORKLOADS[idx]
    inp = I.make_inputs(w)
    o, hT, _ = run_fwd(inp)
    ref = oracle.forward(inp)
    check("o", o, ref["o"])
    check("hT", hT, ref["hT"])


@pytest.mark.parametrize("lengths", [(1,), (15,), (16,), (17,), (63,), (64,), (65,), (127,), (128,), (129,),
                                     (200, 0, 1, 64, 70)])
def test_forward_ragged_lengths(lengths):
    w = I.custom(lengths, 2, h0=True)
    inp = I.make_inputs(w, seed=100 + sum(lengths))
    if len(lengths) == 1:
        inp["h0"] = None
    o, hT, _ = run_fwd(inp)
    ref = oracle.forward(inp)
    check("o", o, ref["o"])
    check("hT", hT, ref["hT"])


def test_forward_strong_decay():
    w = I.custom([300], 3, g_std=4.0)
    inp = I.make_inputs(w, seed=7)
    inp["A_log"] = torch.full((3,), float(np.log(16.0)))
    o, hT, _ = run_fwd(inp)
    ref = oracle.forward(inp)
    check("o", o, ref["o"])
    check("hT", hT, ref["hT"])
