"""Grouped value heads (G value heads per query/key head): the CUDA path through the C ABI
against the fp64 oracle, and the plain layout as the special case G = 1.

Value head h reads query/key head h // G; dq, dk are the sums over each group."""
import pytest
import torch

import oracle
from gpu_helpers import run_fwd_bwd
from parity import check
from kimi_delta_attention_15_gb300 import inputs as I, ops

pytestmark = pytest.mark.gpu

KEYS = ("o", "hT", "dq", "dk", "dv", "dg_raw", "dbeta_raw", "dh0", "dA_log", "ddt_bias")


def _compare(inp, out):
    ref = dict(oracle.forward(inp))
    ref.update(oracle.backward(inp))
    assert out["status"] == 0
    assert out["dq"].shape == inp["q"].shape and out["dk"].shape == inp["k"].shape
    for k in KEYS:
        if ref.get(k) is None or out.get(k) is None:
            continue
        check(k, out[k], ref[k])


@pytest.mark.parametrize("lengths,H,G", [((200,), 4, 2), ((130,), 4, 4), ((17, 33, 65), 8, 4),
                                         ((64, 1, 127), 6, 3)])
def test_grouped_value_heads_match_the_oracle(lengths, H, G):
    w = I.custom(lengths, H, h0=True, dhT=True, groups=G)
    inp = I.make_inputs(w, seed=31 + G)
    _compare(inp, run_fwd_bwd(inp))


def test_grouped_heads_at_a_multi_chunk_size():
    """Several chunks per sequence and many tiles: T = 1024, 16 value heads in groups of 8."""
    w = I.custom((1024,), 16, groups=8)
    inp = I.make_inputs(w, seed=41)
    _compare(inp, run_fwd_bwd(inp))


def test_grouped_heads_with_repeated_query_key_heads_equal_the_plain_layout():
    """The grouped run equals the plain run with q, k repeated along the head axis: the same
    bits for every output but dq, dk, whose grouped values are the group sums of the plain
    ones (the grouped path sums fp32 partials and rounds once, the plain one rounds each)."""
    G = 2
    w = I.custom((96, 40), 4, h0=True, groups=G)
    inp = I.make_inputs(w, seed=43)
    rep = dict(inp)
    rep["q"] = inp["q"].repeat_interleave(G, dim=1)
    rep["k"] = inp["k"].repeat_interleave(G, dim=1)
    a, b = run_fwd_bwd(inp), run_fwd_bwd(rep)
    for key in ("o", "hT", "dv", "dg_raw", "dbeta_raw", "dh0", "dA_log", "ddt_bias"):
        assert torch.equal(a[key], b[key]), key
    for key in ("dq", "dk"):
        summed = b[key].float().reshape(a[key].shape[0], -1, G, 128).sum(dim=2)
        assert torch.allclose(a[key].float(), summed, rtol=1e-2, atol=1e-2), key


def test_groups_must_divide_the_value_heads():
    w = I.custom((64,), 4, groups=1)
    inp = I.make_inputs(w, seed=1)
    q3 = inp["q"][:, :3].contiguous()
    with pytest.raises(ValueError):
        ops.fwd(q3.cuda(), q3.cuda(), inp["v"].cuda(), inp["g_raw"].cuda(), inp["beta_raw"].cuda(),
                inp["A_log"].cuda(), inp["dt_bias"].cuda())
