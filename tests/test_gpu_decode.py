"""Decode step (kda_decode through the C ABI) against the fp64 oracle. One token
per request is a sequence of one token with h0 = the state before and hT = the
state after; T steps of one request are one sequence of T tokens."""
import pytest
import torch

import oracle
from gpu_helpers import to_dev
from parity import check
from kimi_delta_attention_15_gb300 import inputs as I, ops

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n_req,H", [(1, 1), (37, 4), (256, 8)])
def test_decode_batch_one_step(n_req, H):
    inp = I.make_inputs(I.custom((1,) * n_req, H, h0=True), seed=21 + n_req)
    d = to_dev(inp)
    state = d["h0"].clone()
    o = ops.decode(d["q"], d["k"], d["v"], d["g_raw"], d["beta_raw"], d["A_log"], d["dt_bias"], state)
    torch.cuda.synchronize()
    ref = oracle.forward(inp)
    check("o", o, ref["o"])
    check("hT", state, ref["hT"])


@pytest.mark.parametrize("g_std", [1.0, 4.0])
def test_decode_steps_equal_one_sequence(g_std):
    T, H = 70, 4
    inp = I.make_inputs(I.custom((T,), H, g_std=g_std, h0=True), seed=22)
    d = to_dev(inp)
    state = d["h0"].clone()
    outs = []
    for t in range(T):
        tok = {k: d[k][t:t + 1].clone() for k in ("q", "k", "v", "g_raw", "beta_raw")}   # aligned copies
        outs.append(ops.decode(tok["q"], tok["k"], tok["v"], tok["g_raw"], tok["beta_raw"], d["A_log"],
                               d["dt_bias"], state))
    o = torch.cat(outs, 0)
    torch.cuda.synchronize()
    ref = oracle.forward(inp)
    check("o", o, ref["o"])
    check("hT", state, ref["hT"])


def test_decode_matches_forward_of_one_token_sequences():
    n_req, H = 64, 4
    inp = I.make_inputs(I.custom((1,) * n_req, H, h0=True), seed=23)
    d = to_dev(inp)
    o_f, hT_f, _ = ops.fwd(d["q"], d["k"], d["v"], d["g_raw"], d["beta_raw"], d["A_log"], d["dt_bias"],
                           h0=d["h0"], cu_seqlens=d["cu_seqlens"])
    state = d["h0"].clone()
    o_d = ops.decode(d["q"], d["k"], d["v"], d["g_raw"], d["beta_raw"], d["A_log"], d["dt_bias"], state)
    torch.cuda.synchronize()
    check("o", o_d, o_f.float().double().cpu())
    check("hT", state, hT_f.double().cpu())


@pytest.mark.parametrize("n_req,H,G", [(37, 8, 4), (5, 6, 3)])
def test_grouped_decode_matches_the_oracle(n_req, H, G):
    """Grouped value heads: q, k hold H / G heads; value head h reads query/key head h // G."""
    inp = I.make_inputs(I.custom((1,) * n_req, H, h0=True, groups=G), seed=24 + G)
    d = to_dev(inp)
    assert d["q"].shape[1] == H // G
    state = d["h0"].clone()
    o = ops.decode(d["q"], d["k"], d["v"], d["g_raw"], d["beta_raw"], d["A_log"], d["dt_bias"], state)
    torch.cuda.synchronize()
    ref = oracle.forward(inp)
    check("o", o, ref["o"])
    check("hT", state, ref["hT"])
    # the same as the grouped forward over one-token sequences
    o_f, hT_f, _ = ops.fwd(d["q"], d["k"], d["v"], d["g_raw"], d["beta_raw"], d["A_log"], d["dt_bias"],
                           h0=d["h0"], cu_seqlens=d["cu_seqlens"])
    torch.cuda.synchronize()
    check("o", o, o_f.float().double().cpu())
    check("hT", state, hT_f.double().cpu())


def test_decode_other_lower_bound_and_scale():
    """A weak decay (lb = -0.1) and an output scale of 1: the values the oracle reads."""
    inp = I.make_inputs(I.custom((1,) * 40, 4, h0=True), seed=26)
    inp["lower_bound"], inp["scale"] = -0.1, 1.0
    d = to_dev(inp)
    state = d["h0"].clone()
    o = ops.decode(d["q"], d["k"], d["v"], d["g_raw"], d["beta_raw"], d["A_log"], d["dt_bias"], state,
                   scale=1.0, lower_bound=-0.1)
    torch.cuda.synchronize()
    ref = oracle.forward(inp)
    check("o", o, ref["o"])
    check("hT", state, ref["hT"])
