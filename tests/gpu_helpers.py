"""Helpers of the GPU parity tests: run the CUDA path through the C ABI binding."""
import torch


def to_dev(inp):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def run_fwd_bwd(inp, want_bwd=True):
    """kda_fwd (+ kda_bwd) on cuda:0 for a dict from kimi_delta_attention_15_gb300.inputs."""
    from kimi_delta_attention_15_gb300 import ops
    d = to_dev(inp)
    packed = len(inp["lengths"]) > 1
    cu = d["cu_seqlens"] if packed else None
    lb = float(inp.get("lower_bound", ops.LOWER_BOUND))   # the oracle reads the same keys
    scale = float(inp.get("scale", ops.SCALE))
    cs = int(inp.get("chunk_size", 64))   # the library's chunk-length option; the oracle has none
    o, hT, ws = ops.fwd(d["q"], d["k"], d["v"], d["g_raw"], d["beta_raw"], d["A_log"], d["dt_bias"],
                        h0=d.get("h0"), cu_seqlens=cu, lower_bound=lb, scale=scale, chunk_size=cs)
    out = dict(o=o, hT=hT)
    if want_bwd:
        g = ops.bwd(d["q"], d["k"], d["v"], d["g_raw"], d["beta_raw"], d["A_log"], d["dt_bias"], d["do"], ws,
                    h0=d.get("h0"), cu_seqlens=cu, dhT=d.get("dhT"), lower_bound=lb, scale=scale,
                    chunk_size=cs)
        out.update(g)
    status = ops.device_status(ws)
    torch.cuda.synchronize()
    out["status"] = status
    return out
