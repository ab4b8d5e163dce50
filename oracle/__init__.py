"""fp64 CPU oracle for the KDA gated delta rule — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The product path (the CUDA library and
its binding) never calls it.

The arithmetic lives in ``kda_oracle.c`` (plain C, fp64, one token at a time).
This module builds it with gcc on first use and exposes:

  forward(inp, ...)   -> dict(o, hT)           fp64 numpy arrays
  backward(inp, ...)  -> dict(dq, dk, dv, dg_raw, dbeta_raw, dA_log, ddt_bias, dh0)

Grouped value heads: q and k may hold fewer heads than v (H_v = G H_qk); value
head h then reads query/key head h // G, and dq, dk are summed over each group.

``inp`` holds fp64 numpy arrays (or anything ``np.asarray`` takes) in the
packed layouts of ``kimi_delta_attention_15_gb300.inputs``. In ``core`` mode
q and k are used as given (no L2 norm), ``g_raw`` is taken as the log-decay g
and ``beta_raw`` as beta itself; A_log and dt_bias are unused.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_LIB = os.path.join(_HERE, "_build", "libkda_oracle.so")
_lock = threading.Lock()
_lib = None

SCALE = 1.0 / np.sqrt(128.0)
LOWER_BOUND = -5.0
EPS = 1e-6

_P = ctypes.POINTER(ctypes.c_double)


class _Args(ctypes.Structure):
    _fields_ = [
        ("N", ctypes.c_int64), ("H", ctypes.c_int64), ("K", ctypes.c_int64), ("V", ctypes.c_int64),
        ("cu", ctypes.POINTER(ctypes.c_int64)),
        ("scale", ctypes.c_double), ("lb", ctypes.c_double), ("eps", ctypes.c_double),
        ("mode", ctypes.c_int), ("nthreads", ctypes.c_int),
        ("q", _P), ("k", _P), ("v", _P), ("gx", _P), ("bx", _P),
        ("A_log", _P), ("dt_bias", _P), ("h0", _P),
        ("o", _P), ("hT", _P),
        ("dO", _P), ("dhT", _P),
        ("dq", _P), ("dk", _P), ("dv", _P), ("dgx", _P), ("dbx", _P),
        ("dA_log_unit", _P), ("ddt_bias_unit", _P), ("dh0", _P),
        ("G", ctypes.c_int64),
    ]


def build(force: bool = False, mutation: int = 0, out: str | None = None) -> str:
    """Compile the oracle with gcc (no fused multiply-add contraction, so the
    result is the same on x86-64 and aarch64). `mutation` > 0 plants one of the
    test mistakes (tests only) into a separate library `out`."""
    lib = out or _LIB
    with _lock:
        if force or mutation or not os.path.exists(lib) or os.path.getmtime(lib) < os.path.getmtime(_SRC):
            os.makedirs(os.path.dirname(lib), exist_ok=True)
            tmp = lib + f".tmp{os.getpid()}"
            subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                                   f"-DKDA_ORACLE_MUTATION={int(mutation)}",
                                   "-shared", "-fPIC", "-pthread", _SRC, "-o", tmp, "-lm"])
            os.replace(tmp, lib)
    return lib


def _bind(path):
    lib = ctypes.CDLL(path)
    lib.kda_oracle_forward.argtypes = [ctypes.POINTER(_Args)]
    lib.kda_oracle_backward.argtypes = [ctypes.POINTER(_Args)]
    lib.kda_oracle_args_size.restype = ctypes.c_size_t
    assert lib.kda_oracle_args_size() == ctypes.sizeof(_Args), "oracle ABI mismatch"
    return lib


_override = None   # a library with a planted mistake, installed by the oracle's own tests


def use_library(path):
    """Tests only: route forward/backward through another build of the oracle
    (None restores the normal one)."""
    global _override
    _override = _bind(path) if path else None


def _load():
    global _lib
    if _override is not None:
        return _override
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        lib.kda_oracle_forward.argtypes = [ctypes.POINTER(_Args)]
        lib.kda_oracle_backward.argtypes = [ctypes.POINTER(_Args)]
        lib.kda_oracle_args_size.restype = ctypes.c_size_t
        assert lib.kda_oracle_args_size() == ctypes.sizeof(_Args), "oracle ABI mismatch"
        _lib = lib
    return _lib


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(x):
    return x.ctypes.data_as(_P) if x is not None else None


def _prepare(inp, mode, nthreads):
    q, k, v = _f64(inp["q"]), _f64(inp["k"]), _f64(inp["v"])
    T, Hk, K = q.shape
    H, V = v.shape[1], v.shape[2]
    assert H % Hk == 0, "value heads must be a multiple of query/key heads"
    cu = np.ascontiguousarray(np.asarray(inp["cu_seqlens"], dtype=np.int64))
    N = cu.shape[0] - 1
    keep = dict(q=q, k=k, v=v, gx=_f64(inp["g_raw"]), bx=_f64(inp["beta_raw"]), cu=cu,
                h0=_f64(inp.get("h0")))
    if mode == "raw":
        keep["A_log"] = _f64(inp["A_log"])
        keep["dt_bias"] = _f64(inp["dt_bias"])
    a = _Args()
    a.N, a.H, a.K, a.V = N, H, K, V
    a.G = H // Hk
    a.cu = cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))
    a.scale = float(inp.get("scale", SCALE))
    a.lb = float(inp.get("lower_bound", LOWER_BOUND))
    a.eps = float(inp.get("eps", EPS))
    a.mode = 1 if mode == "raw" else 0
    a.nthreads = int(nthreads or default_threads())
    for name in ("q", "k", "v", "gx", "bx", "h0"):
        setattr(a, name, _ptr(keep[name]))
    if mode == "raw":
        a.A_log, a.dt_bias = _ptr(keep["A_log"]), _ptr(keep["dt_bias"])
    return a, keep, (T, H, K, V, N)


def forward(inp, mode: str = "raw", nthreads: int | None = None, want_o: bool = True):
    """Token-by-token fp64 forward. Returns dict(o [T,H,V], hT [N,H,V,K])."""
    a, keep, (T, H, K, V, N) = _prepare(inp, mode, nthreads)
    o = np.zeros((T, H, V)) if want_o else None
    hT = np.zeros((N, H, V, K))
    a.o, a.hT = _ptr(o), _ptr(hT)
    _load().kda_oracle_forward(ctypes.byref(a))
    return dict(o=o, hT=hT)


def backward(inp, mode: str = "raw", nthreads: int | None = None):
    """Hand-derived reverse mode of L = sum <o, do> + <hT, dhT> (dhT None = 0).

    Parameter gradients are summed over units (n, h) on the host in a fixed
    order (sequence index ascending), so the result is deterministic."""
    a, keep, (T, H, K, V, N) = _prepare(inp, mode, nthreads)
    dO = _f64(inp["do"])
    dhT = _f64(inp.get("dhT"))
    keep["dO"], keep["dhT"] = dO, dhT
    a.dO, a.dhT = _ptr(dO), _ptr(dhT)
    out = dict(dq=np.zeros((T, H, K)), dk=np.zeros((T, H, K)), dv=np.zeros((T, H, V)),
               dg_raw=np.zeros((T, H, K)), dbeta_raw=np.zeros((T, H)), dh0=np.zeros((N, H, V, K)))
    dA_unit = np.zeros((N, H))
    ddt_unit = np.zeros((N, H, K))
    a.dq, a.dk, a.dv = _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"])
    a.dgx, a.dbx, a.dh0 = _ptr(out["dg_raw"]), _ptr(out["dbeta_raw"]), _ptr(out["dh0"])
    a.dA_log_unit, a.ddt_bias_unit = _ptr(dA_unit), _ptr(ddt_unit)
    _load().kda_oracle_backward(ctypes.byref(a))
    G = a.G
    if G > 1:   # dq, dk per value head -> per query/key head, summed over the group in order
        for name in ("dq", "dk"):
            per = out[name].reshape(T, H // G, G, K)
            acc = per[:, :, 0, :].copy()
            for j in range(1, G):
                acc += per[:, :, j, :]
            out[name] = acc
    dA = np.zeros(H)
    ddt = np.zeros((H, K))
    for n in range(N):          # fixed summation order
        dA += dA_unit[n]
        ddt += ddt_unit[n]
    out["dA_log"], out["ddt_bias"] = dA, ddt
    return out
