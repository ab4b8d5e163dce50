"""Fixed-length batches without offsets: [B, T, H, 128] token tensors (B sequences of T
tokens, chunks restarting at every sequence) against the oracle, which takes the same
tokens as B packed sequences of length T."""
import pytest
import torch

import oracle
from gpu_helpers import to_dev
from parity import check
from kimi_delta_attention_15_gb300 import inputs as I, ops

pytestmark = pytest.mark.gpu

GRADS = ("dq", "dk", "dv", "dg_raw", "dbeta_raw", "dh0", "dA_log", "ddt_bias")


@pytest.mark.parametrize("B,T,H,G", [(3, 100, 4, 1), (2, 64, 2, 1), (4, 130, 4, 2)])
def test_fixed_length_batch_matches_the_oracle(B, T, H, G):
    inp = I.make_inputs(I.custom((T,) * B, H, h0=True, dhT=True, groups=G), seed=50 + B)
    d = to_dev(inp)
    b4 = {k: d[k].view(B, T, *d[k].shape[1:]) for k in ("q", "k", "v", "g_raw", "beta_raw", "do")}
    o, hT, ws = ops.fwd(b4["q"], b4["k"], b4["v"], b4["g_raw"], b4["beta_raw"], d["A_log"], d["dt_bias"],
                        h0=d["h0"])
    g = ops.bwd(b4["q"], b4["k"], b4["v"], b4["g_raw"], b4["beta_raw"], d["A_log"], d["dt_bias"], b4["do"], ws,
                h0=d["h0"], dhT=d["dhT"])
    assert ops.device_status(ws) == 0
    torch.cuda.synchronize()
    assert o.shape == (B, T, H, 128) and g["dq"].shape == (B, T, H // G, 128)
    ref = dict(oracle.forward(inp))
    ref.update(oracle.backward(inp))
    check("o", o.reshape(B * T, H, 128), ref["o"])
    check("hT", hT, ref["hT"])
    for k in GRADS:
        x = g[k]
        if x.dim() >= 3 and k not in ("dh0",):
            x = x.reshape(B * T, *x.shape[2:])
        check(k, x, ref[k])


def test_fixed_length_batch_equals_packed_offsets():
    """The same tokens through the offset path give the same bits."""
    B, T, H = 3, 90, 4
    inp = I.make_inputs(I.custom((T,) * B, H, h0=True), seed=57)
    d = to_dev(inp)
    b4 = {k: d[k].view(B, T, *d[k].shape[1:]) for k in ("q", "k", "v", "g_raw", "beta_raw", "do")}
    o_b, hT_b, ws_b = ops.fwd(b4["q"], b4["k"], b4["v"], b4["g_raw"], b4["beta_raw"], d["A_log"],
                              d["dt_bias"], h0=d["h0"])
    g_b = ops.bwd(b4["q"], b4["k"], b4["v"], b4["g_raw"], b4["beta_raw"], d["A_log"], d["dt_bias"], b4["do"],
                  ws_b, h0=d["h0"])
    o_p, hT_p, ws_p = ops.fwd(d["q"], d["k"], d["v"], d["g_raw"], d["beta_raw"], d["A_log"], d["dt_bias"],
                              h0=d["h0"], cu_seqlens=d["cu_seqlens"])
    g_p = ops.bwd(d["q"], d["k"], d["v"], d["g_raw"], d["beta_raw"], d["A_log"], d["dt_bias"], d["do"], ws_p,
                  h0=d["h0"], cu_seqlens=d["cu_seqlens"])
    torch.cuda.synchronize()
    assert torch.equal(o_b.reshape(o_p.shape), o_p) and torch.equal(hT_b, hT_p)
    for k in ("dq", "dk", "dv", "dg_raw", "dbeta_raw", "dh0", "dA_log", "ddt_bias"):
        assert torch.equal(g_b[k].reshape(g_p[k].shape), g_p[k]), k
