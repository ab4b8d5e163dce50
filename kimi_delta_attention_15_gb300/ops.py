"""Thin Python binding of the C ABI in ``include/kda.h``.

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``_build/libkda.so``. PyTorch provides device memory and streams.
Loading fails loudly (RuntimeError) when the library is missing; there is no
fallback path.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

from . import build as _build

KDA_OK = 0
_STATUS = {0: "KDA_OK", 1: "KDA_ERR_NULL", 2: "KDA_ERR_ALIGN", 3: "KDA_ERR_SHAPE",
           4: "KDA_ERR_UNSUPPORTED", 5: "KDA_ERR_WORKSPACE", 6: "KDA_ERR_OFFSETS",
           7: "KDA_ERR_TIMEOUT", 8: "KDA_ERR_CUDA", 9: "KDA_ERR_STALE_WORKSPACE"}

SCALE = 1.0 / math.sqrt(128.0)
LOWER_BOUND = -5.0

_lock = threading.Lock()
_lib = None


class KdaError(RuntimeError):
    def __init__(self, code, where=""):
        self.code = int(code)
        super().__init__(f"{where}: {_STATUS.get(self.code, self.code)}")


class Shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("T", ctypes.c_int64), ("H", ctypes.c_int64),
                ("N", ctypes.c_int64), ("K", ctypes.c_int32), ("V", ctypes.c_int32),
                ("scale", ctypes.c_float), ("lower_bound", ctypes.c_float),
                ("groups", ctypes.c_int32), ("chunk_size", ctypes.c_int32)]


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load ``libkda.so`` (building it first if asked and missing)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if not os.path.exists(path):
            if not build_if_missing:
                raise RuntimeError(f"KDA CUDA library not built: {path}")
            _build.build()
        lib = ctypes.CDLL(path)
        P, S, I64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int64
        lib.kda_workspace_size.argtypes = [ctypes.POINTER(Shape)]
        lib.kda_workspace_size.restype = S
        lib.kda_fwd.argtypes = [ctypes.POINTER(Shape)] + [P] * 11 + [P, S, P]
        lib.kda_fwd.restype = ctypes.c_int
        lib.kda_bwd.argtypes = [ctypes.POINTER(Shape)] + [P] * 19 + [P, S, P]
        lib.kda_bwd.restype = ctypes.c_int
        lib.kda_get_device_status.argtypes = [P, P]
        lib.kda_get_device_status.restype = ctypes.c_int
        lib.kda_status_string.argtypes = [ctypes.c_int]
        lib.kda_status_string.restype = ctypes.c_char_p
        lib.kda_fwd_static_scratch.argtypes = [ctypes.POINTER(Shape)] + [P] * 11 + [P]
        lib.kda_fwd_static_scratch.restype = ctypes.c_int
        lib.kda_static_scratch_device_status.argtypes = [P]
        lib.kda_static_scratch_device_status.restype = ctypes.c_int
        lib.kda_last_error.argtypes = []
        lib.kda_last_error.restype = ctypes.c_char_p
        lib.kda_set_profile_events.argtypes = [P, ctypes.c_int]
        lib.kda_set_profile_events.restype = ctypes.c_int
        lib.kda_diag_wait_timeout.argtypes = [ctypes.c_ulonglong, P, P]
        lib.kda_diag_wait_timeout.restype = ctypes.c_int
        lib.kda_diag_umma_selftest.argtypes = [ctypes.c_int] * 4 + [P, P, P, P]
        lib.kda_diag_umma_selftest.restype = ctypes.c_int
        lib.kda_decode.argtypes = [ctypes.c_longlong] * 3 + [ctypes.c_float, ctypes.c_float] + [P] * 10
        lib.kda_decode.restype = ctypes.c_int
        lib.kda_diag_tf32_round.argtypes = [P, P, P, ctypes.c_longlong, P]
        lib.kda_diag_tf32_round.restype = ctypes.c_int
        _lib = lib
        return lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def make_shape(T: int, H: int, N: int, B: int = 1, scale: float = SCALE,
               lower_bound: float = LOWER_BOUND, groups: int = 1, chunk_size: int = 64) -> Shape:
    """H counts value heads; groups = value heads per query/key head; chunk_size 64 or 32
    (the library computes both with 64-token chunks: the chunk length does not change the
    function)."""
    return Shape(B=B, T=T, H=H, N=N, K=128, V=128, scale=scale, lower_bound=lower_bound, groups=groups,
                 chunk_size=chunk_size)


def workspace_size(shape: Shape) -> int:
    return int(load().kda_workspace_size(ctypes.byref(shape)))


def _check(code, where):
    if code != KDA_OK:
        detail = ""
        if code == 8:
            detail = " (" + load().kda_last_error().decode(errors="replace") + ")"
        raise KdaError(code, where + detail)


def _shape_of(q, v, cu_seqlens, B, scale, lower_bound, chunk_size=64):
    """Shape from the token tensors: H = value heads (v); q, k may hold H / groups heads."""
    H, Hqk = v.shape[-2], q.shape[-2]
    if Hqk <= 0 or H % Hqk != 0:
        raise ValueError(f"value heads ({H}) must be a multiple of query/key heads ({Hqk})")
    G = H // Hqk
    if cu_seqlens is not None:
        return make_shape(q.shape[0], H, cu_seqlens.numel() - 1, 1, scale, lower_bound, G, chunk_size)
    if q.dim() == 4:
        B_, T = q.shape[0], q.shape[1]
        return make_shape(T, H, B_, B_, scale, lower_bound, G, chunk_size)
    return make_shape(q.shape[0] // B, H, B, B, scale, lower_bound, G, chunk_size)


def _validate(specs):
    """Sizes, dtypes and layout of the tensors a call hands to the kernels, which see only
    pointers: (name, tensor or None, element count, dtype or None, optional). Sizes are checked
    as element counts, so [T, H, 128] and [B, T, H, 128] both pass. Every tensor must then be
    contiguous and on one CUDA device. Raises ValueError before anything is launched."""
    present = []
    for name, t, numel, dtype, optional in specs:
        if t is None:
            if not optional:
                raise ValueError(f"{name} is required")
            continue
        if dtype is not None and t.dtype != dtype:
            raise ValueError(f"{name}: dtype {t.dtype}, expected {dtype}")
        if numel is not None and t.numel() != numel:
            raise ValueError(f"{name}: {t.numel()} elements {tuple(t.shape)}, expected {numel}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        present.append((name, t))
    dev = present[0][1].device if present else None
    for name, t in present:
        if t.device.type != "cuda" or t.device != dev:
            raise ValueError(f"{name}: on {t.device}; every tensor must be on one CUDA device ({dev})")


def _token_specs(shape: Shape, q, k, v, g_raw, beta_raw, A_log, dt_bias, h0, cu_seqlens):
    """Specs of the inputs kda_fwd and kda_bwd share."""
    tok, H, N = shape.B * shape.T, shape.H, shape.N
    Hqk = H // max(int(shape.groups), 1)
    bf, f32 = torch.bfloat16, torch.float32
    return [("q", q, tok * Hqk * 128, bf, False), ("k", k, tok * Hqk * 128, bf, False),
            ("v", v, tok * H * 128, bf, False), ("g_raw", g_raw, tok * H * 128, bf, False),
            ("beta_raw", beta_raw, tok * H, bf, False), ("A_log", A_log, H, f32, False),
            ("dt_bias", dt_bias, H * 128, f32, False), ("h0", h0, N * H * 128 * 128, f32, True),
            ("cu_seqlens", cu_seqlens, N + 1, torch.int64, True)]


def alloc_workspace(shape: Shape, device) -> torch.Tensor:
    return torch.empty(workspace_size(shape), dtype=torch.uint8, device=device)


def fwd(q, k, v, g_raw, beta_raw, A_log, dt_bias, h0=None, cu_seqlens=None, *, B: int = 1,
        scale: float = SCALE, lower_bound: float = LOWER_BOUND, workspace=None, o=None,
        hT=None, want_hT: bool = True, stream=None, chunk_size: int = 64):
    """kda_fwd. Token tensors [T, H, 128] bf16 (or [B, T, H, 128]); returns (o, hT, workspace)."""
    lib = load()
    shape = _shape_of(q, v, cu_seqlens, B, scale, lower_bound, chunk_size)
    if workspace is None:
        workspace = alloc_workspace(shape, q.device)
    if o is None:
        o = torch.empty_like(v)
    if hT is None and want_hT:
        hT = torch.empty(shape.N, shape.H, 128, 128, dtype=torch.float32, device=q.device)
    _validate(_token_specs(shape, q, k, v, g_raw, beta_raw, A_log, dt_bias, h0, cu_seqlens)
              + [("o", o, v.numel(), torch.bfloat16, False), ("hT", hT, shape.N * shape.H * 128 * 128,
                                                             torch.float32, True),
                 ("workspace", workspace, None, None, False)])
    code = lib.kda_fwd(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g_raw), _ptr(beta_raw),
                       _ptr(A_log), _ptr(dt_bias), _ptr(h0), _ptr(cu_seqlens), _ptr(o), _ptr(hT),
                       _ptr(workspace), workspace.numel(), _stream_handle(stream))
    _check(code, "kda_fwd")
    return o, hT, workspace


STATIC_SCRATCH_BYTES = 64 * 1024 * 1024


def fwd_static_scratch(q, k, v, g_raw, beta_raw, A_log, dt_bias, h0=None, cu_seqlens=None, *, B: int = 1,
                       scale: float = SCALE, lower_bound: float = LOWER_BOUND, o=None, hT=None,
                       want_hT: bool = True, stream=None):
    """kda_fwd_static_scratch: the forward without a workspace argument, for
    callers that cannot allocate device memory (the scratch is a fixed array
    inside the library). Returns (o, hT)."""
    lib = load()
    shape = _shape_of(q, v, cu_seqlens, B, scale, lower_bound)
    if o is None:
        o = torch.empty_like(v)
    if hT is None and want_hT:
        hT = torch.empty(shape.N, shape.H, 128, 128, dtype=torch.float32, device=q.device)
    _validate(_token_specs(shape, q, k, v, g_raw, beta_raw, A_log, dt_bias, h0, cu_seqlens)
              + [("o", o, v.numel(), torch.bfloat16, False), ("hT", hT, shape.N * shape.H * 128 * 128,
                                                             torch.float32, True)])
    code = lib.kda_fwd_static_scratch(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g_raw),
                                      _ptr(beta_raw), _ptr(A_log), _ptr(dt_bias), _ptr(h0), _ptr(cu_seqlens),
                                      _ptr(o), _ptr(hT), _stream_handle(stream))
    if code == 5:
        raise KdaError(code, "kda_fwd_static_scratch (" + lib.kda_last_error().decode(errors="replace") + ")")
    _check(code, "kda_fwd_static_scratch")
    return o, hT


def bwd(q, k, v, g_raw, beta_raw, A_log, dt_bias, do, workspace, h0=None, cu_seqlens=None,
        dhT=None, *, B: int = 1, scale: float = SCALE, lower_bound: float = LOWER_BOUND,
        grads=None, want_dh0: bool = True, stream=None, chunk_size: int = 64):
    """kda_bwd with the workspace filled by ``fwd``. Returns a dict of gradients."""
    lib = load()
    shape = _shape_of(q, v, cu_seqlens, B, scale, lower_bound, chunk_size)
    if grads is None:
        grads = dict(dq=torch.empty_like(q), dk=torch.empty_like(k), dv=torch.empty_like(v),
                     dg_raw=torch.empty_like(g_raw), dbeta_raw=torch.empty_like(beta_raw),
                     dA_log=torch.empty_like(A_log), ddt_bias=torch.empty_like(dt_bias),
                     dh0=(torch.empty(shape.N, shape.H, 128, 128, dtype=torch.float32,
                                      device=q.device) if want_dh0 else None))
    bf, f32 = torch.bfloat16, torch.float32
    _validate(_token_specs(shape, q, k, v, g_raw, beta_raw, A_log, dt_bias, h0, cu_seqlens)
              + [("do", do, v.numel(), bf, False),
                 ("dhT", dhT, shape.N * shape.H * 128 * 128, f32, True),
                 ("dq", grads.get("dq"), q.numel(), bf, False), ("dk", grads.get("dk"), q.numel(), bf, False),
                 ("dv", grads.get("dv"), v.numel(), bf, False), ("dg_raw", grads.get("dg_raw"), v.numel(), bf, False),
                 ("dbeta_raw", grads.get("dbeta_raw"), beta_raw.numel(), bf, False),
                 ("dA_log", grads.get("dA_log"), shape.H, f32, False),
                 ("ddt_bias", grads.get("ddt_bias"), shape.H * 128, f32, False),
                 ("dh0", grads.get("dh0"), shape.N * shape.H * 128 * 128, f32, True),
                 ("workspace", workspace, None, None, False)])
    code = lib.kda_bwd(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g_raw), _ptr(beta_raw),
                       _ptr(A_log), _ptr(dt_bias), _ptr(h0), _ptr(cu_seqlens), _ptr(do), _ptr(dhT),
                       _ptr(grads["dq"]), _ptr(grads["dk"]), _ptr(grads["dv"]), _ptr(grads["dg_raw"]),
                       _ptr(grads["dbeta_raw"]), _ptr(grads["dA_log"]), _ptr(grads["ddt_bias"]),
                       _ptr(grads.get("dh0")), _ptr(workspace), workspace.numel(),
                       _stream_handle(stream))
    _check(code, "kda_bwd")
    return grads


def decode(q, k, v, g_raw, beta_raw, A_log, dt_bias, state, *, o=None, scale: float = SCALE,
           lower_bound: float = LOWER_BOUND, stream=None):
    """kda_decode: one token per request. v, g_raw [n_req, H, 128] bf16,
    beta_raw [n_req, H] bf16, q, k [n_req, H / groups, 128] bf16 (groups taken
    from the head counts); `state` [n_req, H, 128, 128] fp32 is updated in
    place. Returns o [n_req, H, 128] bf16."""
    n_req, H, Hqk = int(v.shape[0]), int(v.shape[1]), int(q.shape[1])
    if Hqk <= 0 or H % Hqk != 0:
        raise ValueError(f"value heads ({H}) must be a multiple of query/key heads ({Hqk})")
    if o is None:
        o = torch.empty_like(v)
    lib = load()
    bf, f32 = torch.bfloat16, torch.float32
    _validate([("q", q, n_req * Hqk * 128, bf, False), ("k", k, n_req * Hqk * 128, bf, False),
               ("v", v, n_req * H * 128, bf, False), ("g_raw", g_raw, n_req * H * 128, bf, False),
               ("beta_raw", beta_raw, n_req * H, bf, False), ("A_log", A_log, H, f32, False),
               ("dt_bias", dt_bias, H * 128, f32, False), ("state", state, n_req * H * 128 * 128, f32, False),
               ("o", o, n_req * H * 128, bf, False)])
    code = lib.kda_decode(n_req, H, H // Hqk, scale, lower_bound, _ptr(q), _ptr(k), _ptr(v), _ptr(g_raw), _ptr(beta_raw),
                             _ptr(A_log), _ptr(dt_bias), _ptr(state), _ptr(o), _stream_handle(stream))
    _check(code, "kda_decode")
    return o


def device_status(workspace, stream=None) -> int:
    return int(load().kda_get_device_status(_ptr(workspace), _stream_handle(stream)))


def static_scratch_device_status(stream=None) -> int:
    """The device status word of the last fwd_static_scratch call on the current device."""
    return int(load().kda_static_scratch_device_status(_stream_handle(stream)))


def wait_timeout(workspace, limit_ns: int = 20_000_000):
    """Diagnostic: a kernel whose wait runs out sets KDA_ERR_TIMEOUT in `workspace`."""
    _check(load().kda_diag_wait_timeout(limit_ns, _ptr(workspace), _stream_handle()), "kda_diag_wait_timeout")


def tf32_round_check(x):
    """Diagnostics: (library rounding, hardware cvt.rna) of a float32 CUDA tensor."""
    x = x.contiguous()
    out, ref = torch.empty_like(x), torch.empty_like(x)
    _check(load().kda_diag_tf32_round(_ptr(x), _ptr(out), _ptr(ref), x.numel(), _stream_handle()),
           "kda_diag_tf32_round")
    return out, ref


def umma_selftest(A, B, a_mn: int, b_mn: int):
    """Diagnostic: D = A @ B^T through tcgen05 kind::tf32 (see include/kda.h)."""
    lib = load()
    N, Kd = B.shape
    D = torch.empty(2, 128, N, dtype=torch.float32, device=A.device)
    code = lib.kda_diag_umma_selftest(a_mn, b_mn, N, Kd, _ptr(A), _ptr(B), _ptr(D), _stream_handle())
    _check(code, "kda_diag_umma_selftest")
    return D


KERNEL_SLOTS = {
    "fwd_table": (0, 1), "fwd_intra": (1, 2), "fwd_scan": (2, 3),
    "bwd_scan": (4, 5), "bwd_state": (5, 6), "bwd_wy": (6, 7), "bwd_pair": (7, 8), "bwd_reduce": (8, 9),
}


class KernelTimer:
    """Per-kernel CUDA events recorded by the library around its launches
    (kda_set_profile_events). Use as a context manager around one call pair."""

    def __init__(self):
        self.events = [torch.cuda.Event(enable_timing=True) for _ in range(10)]
        for e in self.events:     # torch creates the CUDA event on first record
            e.record()
        torch.cuda.synchronize()
        self._arr = (ctypes.c_void_p * 10)(*[ctypes.c_void_p(e.cuda_event) for e in self.events])

    def __enter__(self):
        load().kda_set_profile_events(self._arr, 10)
        return self

    def __exit__(self, *exc):
        load().kda_set_profile_events(None, 0)

    def times_ms(self):
        return {k: self.events[a].elapsed_time(self.events[b]) for k, (a, b) in KERNEL_SLOTS.items()}
