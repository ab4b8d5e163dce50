"""Parity metrics and tolerances shared by the GPU tests.

Tolerances (stated for the KDA path this repository targets):
  bf16 outputs and gradients: normalised max error max|x - x^| / max|x^| <= 1e-2
                              and cosine similarity >= 0.9999;
  fp32 final state, dh0 and parameter gradients: relative error
                              ||x - x^||_2 / ||x^||_2 <= 1e-3;
with x^ the fp64 oracle value. The fp32 tensors are also held to an elementwise
bound, normalised max error <= 1e-2 (the bf16 bar), so that a few wrong elements of a
large tensor, which the normwise criterion would let through, fail too.
"""
import numpy as np

BF16_NMAX = 1e-2
BF16_COS = 0.9999
FP32_REL = 1e-3
FP32_NMAX = 1e-2

BF16_KEYS = ("o", "dq", "dk", "dv", "dg_raw", "dbeta_raw")
FP32_KEYS = ("hT", "dh0", "dA_log", "ddt_bias")


def to_np(x):
    if hasattr(x, "detach"):
        return x.detach().float().cpu().double().numpy()
    return np.asarray(x, dtype=np.float64)


def metrics(x, ref):
    x, ref = to_np(x).ravel(), to_np(ref).ravel()
    den = np.abs(ref).max()
    nmax = np.abs(x - ref).max() / den if den > 0 else np.abs(x).max()
    nr = np.linalg.norm(ref)
    rel = np.linalg.norm(x - ref) / nr if nr > 0 else np.linalg.norm(x)
    nx = np.linalg.norm(x)
    cos = float(x @ ref / (nx * nr)) if nx > 0 and nr > 0 else (1.0 if nx == nr else 0.0)
    return float(nmax), float(rel), cos


def check(name, x, ref, report=None):
    nmax, rel, cos = metrics(x, ref)
    if report is not None:
        report[name] = (nmax, rel, cos)
    if name in FP32_KEYS:
        assert rel <= FP32_REL, f"{name}: rel {rel:.3e} > {FP32_REL}"
        assert nmax <= FP32_NMAX, f"{name}: elementwise nmax {nmax:.3e} > {FP32_NMAX} (rel {rel:.3e})"
    else:
        assert nmax <= BF16_NMAX, f"{name}: nmax {nmax:.3e} > {BF16_NMAX}"
        assert cos >= BF16_COS, f"{name}: cos {cos:.7f} < {BF16_COS}"
    return nmax, rel, cos
