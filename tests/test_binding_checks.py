"""The binding's argument checks (CPU): every call pattern the GPU tests use passes the size,
dtype and layout checks and stops only at the device check (the tensors here live on the
CPU), while a wrong head count, size, dtype or layout is refused before any launch."""
import pytest
import torch

from kimi_delta_attention_15_gb300 import inputs as I, ops

DEVICE_MSG = "one CUDA device"


def _fwd(inp, batched=None, **kw):
    t = {k: inp[k] for k in ("q", "k", "v", "g_raw", "beta_raw")}
    cu = inp["cu_seqlens"] if len(inp["lengths"]) > 1 else None
    if batched:
        t = {k: v.view(batched, -1, *v.shape[1:]) for k, v in t.items()}
        cu = None
    t.update(kw)
    return ops.fwd(t["q"], t["k"], t["v"], t["g_raw"], t["beta_raw"], inp["A_log"], inp["dt_bias"],
                   h0=inp.get("h0"), cu_seqlens=cu)


def _bwd(inp, **kw):
    t = {k: inp[k] for k in ("q", "k", "v", "g_raw", "beta_raw", "do")}
    t.update(kw)
    cu = inp["cu_seqlens"] if len(inp["lengths"]) > 1 else None
    ws = torch.empty(1024, dtype=torch.uint8)
    return ops.bwd(t["q"], t["k"], t["v"], t["g_raw"], t["beta_raw"], inp["A_log"], inp["dt_bias"], t["do"],
                   ws, h0=inp.get("h0"), cu_seqlens=cu, dhT=inp.get("dhT"))


CASES = [
    ("fixed_T17_H1", lambda: I.WORKLOADS[0], None),
    ("packed_H4", lambda: I.WORKLOADS[1], None),
    ("grouped_G2", lambda: I.custom((200,), 4, groups=2), None),
    ("grouped_packed_G4", lambda: I.custom((17, 33, 65), 8, h0=True, dhT=True, groups=4), None),
    ("all_empty", lambda: I.custom((0, 0, 0), 4, h0=True, dhT=True), None),
    ("empty_single", lambda: I.custom((0,), 4, h0=True, dhT=True), None),
    ("batched_B3", lambda: I.custom((100,) * 3, 4, h0=True, dhT=True), 3),
    ("batched_grouped", lambda: I.custom((130,) * 4, 4, h0=True, dhT=True, groups=2), 4),
]


@pytest.mark.parametrize("name,make,batched", CASES, ids=[c[0] for c in CASES])
def test_valid_calls_pass_the_size_checks(name, make, batched):
    inp = I.make_inputs(make(), seed=5)
    with pytest.raises(ValueError, match=DEVICE_MSG):
        _fwd(inp, batched)
    if not batched:
        with pytest.raises(ValueError, match=DEVICE_MSG):
            _bwd(inp)


def test_valid_decode_passes_the_size_checks():
    inp = I.make_inputs(I.custom((1,) * 37, 8, h0=True, groups=4), seed=6)
    with pytest.raises(ValueError, match=DEVICE_MSG):
        ops.decode(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta_raw"], inp["A_log"], inp["dt_bias"],
                   inp["h0"].clone())


def test_mistakes_are_refused_before_any_launch():
    inp = I.make_inputs(I.custom((64, 30), 4, h0=True, dhT=True, groups=2), seed=7)
    with pytest.raises(ValueError, match="^k:"):            # k with fewer heads than q
        _fwd(inp, k=inp["k"][:, :1].contiguous())
    with pytest.raises(ValueError, match="^beta_raw:"):
        _fwd(inp, beta_raw=inp["beta_raw"][:50].contiguous())
    with pytest.raises(ValueError, match="must be contiguous"):
        _fwd(inp, q=inp["q"].transpose(0, 1).contiguous().transpose(0, 1))
    with pytest.raises(ValueError, match="^v: dtype"):
        _fwd(inp, v=inp["v"].float())
    bad = dict(inp, A_log=inp["A_log"].double())
    with pytest.raises(ValueError, match="^A_log: dtype"):
        _fwd(bad)
    with pytest.raises(ValueError, match="^do:"):
        _bwd(inp, do=inp["do"][:10].contiguous())
    d = I.make_inputs(I.custom((1,) * 5, 4, h0=True), seed=8)
    with pytest.raises(ValueError, match="^state:"):
        ops.decode(d["q"], d["k"], d["v"], d["g_raw"], d["beta_raw"], d["A_log"], d["dt_bias"], d["h0"][:4].clone())
