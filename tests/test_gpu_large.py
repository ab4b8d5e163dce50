"""Full-size workloads on the GPU (T=4096 H=32; T=8192 H=96; packed
[1300,547,2048,963,271,3063] H=96), run exactly as the benchmark launches
them, checked on sampled heads against the fp64 oracle (the oracle runs only
those heads: every (sequence, head) unit is independent, and the parameter
gradients are per head)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import run_fwd_bwd
from parity import check
from kimi_delta_attention_15_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def _heads(inp, hs):
    sub = {}
    for k, v in inp.items():
        if k in ("q", "k", "v", "g_raw", "do", "beta_raw"):
            sub[k] = v[:, hs]
        elif k in ("A_log", "dt_bias"):
            sub[k] = v[hs]
        elif k in ("h0", "dhT"):
            sub[k] = None if v is None else v[:, hs]
        else:
            sub[k] = v
    return sub


# every head of the three large workloads (the fp64 oracle takes a few seconds per workload on
# the host's cores); the printed line holds each output's normalised max error, relative error
# and cosine
@pytest.mark.parametrize("idx,hs", [(2, list(range(32))), (3, list(range(96))), (4, list(range(96)))])
def test_full_size_all_heads(idx, hs):
    w = I.WORKLOADS[idx]
    inp = I.make_inputs(w)
    out = run_fwd_bwd(inp)
    assert out["status"] == 0
    for k, v in out.items():
        if isinstance(v, torch.Tensor):
            assert torch.isfinite(v.float()).all(), k
    sub = _heads(inp, hs)
    ref = dict(oracle.forward(sub))
    ref.update(oracle.backward(sub))
    rep = {}
    for k in ("o", "dq", "dk", "dv", "dg_raw", "dbeta_raw", "dA_log", "ddt_bias"):
        x = out[k][:, hs] if k not in ("dA_log", "ddt_bias") else out[k][hs]
        check(k, x, ref[k], rep)
    for k in ("hT", "dh0"):
        if ref.get(k) is not None:
            check(k, out[k][:, hs], ref[k], rep)
    print(w.name, {k: tuple(f"{x:.2e}" for x in v) for k, v in rep.items()})


# The other shapes the pages admit: T=17 with 16 heads, T=1024 with 4 heads (every
# head checked), and eight packed sequences of 1024 tokens at 96 heads (sampled heads).
@pytest.mark.parametrize("name,hs", [("fixed_T17_H16", None), ("fixed_T1024_H4", None),
                                     ("varlen_8x1024_H96", [2, 45, 71, 95])])
def test_other_admitted_shapes(name, hs):
    w = next(x for x in I.EXTRA_WORKLOADS if x.name == name)
    inp = I.make_inputs(w, seed=I.BASE_SEED + 100 + I.EXTRA_WORKLOADS.index(w))
    out = run_fwd_bwd(inp)
    assert out["status"] == 0
    sub = inp if hs is None else _heads(inp, hs)
    ref = dict(oracle.forward(sub))
    ref.update(oracle.backward(sub))
    sel = (lambda x: x) if hs is None else (lambda x: x[:, hs])
    for k in ("o", "dq", "dk", "dv", "dg_raw", "dbeta_raw"):
        check(k, sel(out[k]), ref[k])
    for k in ("hT", "dh0"):
        if ref.get(k) is not None and out.get(k) is not None:
            check(k, sel(out[k]), ref[k])
    # a parameter gradient of one head is a sum over all of its tokens: checked where
    # the head has many of them (T=17 leaves too few for the relative criterion)
    if w.T >= 1024:
        for k in ("dA_log", "ddt_bias"):
            x = out[k] if hs is None else out[k][hs]
            check(k, x, ref[k])


# One long chain: 1,024 chunks through each scan at the default lower bound, and a weak
# decay (lb = -0.1, gates in (-0.1, 0): a state with a long memory) over 256 chunks, so that
# a growth of the error along the chain of tf32 state products would show.
@pytest.mark.parametrize("T,lb", [(65536, -5.0), (16384, -0.1)])
def test_long_single_sequence(T, lb):
    w = I.custom((T,), 1, h0=True, dhT=True, name=f"long_T{T}")
    inp = I.make_inputs(w, seed=61)
    inp["lower_bound"] = lb
    out = run_fwd_bwd(inp)
    assert out["status"] == 0
    ref = dict(oracle.forward(inp))
    ref.update(oracle.backward(inp))
    for k in ("o", "hT", "dq", "dk", "dv", "dg_raw", "dbeta_raw", "dh0", "dA_log", "ddt_bias"):
        check(k, out[k], ref[k])


def test_full_size_bitwise_deterministic():
    """T=8192, H=96 twice: every output equal bit for bit (fixed reduction orders, no float
    atomics, every kernel's tile schedule independent of timing)."""
    inp = I.make_inputs(I.WORKLOADS[3])
    a = run_fwd_bwd(inp)
    b = run_fwd_bwd(inp)
    assert a["status"] == 0 and b["status"] == 0
    for k in ("o", "hT", "dq", "dk", "dv", "dg_raw", "dbeta_raw", "dA_log", "ddt_bias", "dh0"):
        assert torch.equal(a[k], b[k]), k
