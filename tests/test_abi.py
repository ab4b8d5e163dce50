"""The C ABI library (no GPU needed): it loads, exports every function that
include/kda.h declares, and rejects bad arguments on the host before any
CUDA call."""
import ctypes
import os
import re

import pytest

from kimi_delta_attention_15_gb300 import build, ops

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "kda.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return ops.load()


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert "kda_fwd" in names and "kda_bwd" in names
    for n in names:
        assert hasattr(lib, n), n


def test_workspace_size(lib):
    s = ops.make_shape(8192, 96, 1)
    n = ops.workspace_size(s)
    assert n > 0 and n % 1024 == 0
    bad = ops.make_shape(8192, 96, 1)
    bad.K = 64
    assert ops.workspace_size(bad) == 0
    bad = ops.make_shape(100, 2, 1, lower_bound=-6.0)
    assert ops.workspace_size(bad) == 0


def _call_fwd(lib, shape, ptr=16, ws_bytes=1 << 40, cu=None, ws=1024):
    p = ctypes.c_void_p(ptr)
    return lib.kda_fwd(ctypes.byref(shape), p, p, p, p, p, p, p, None, cu, p, None, ctypes.c_void_p(ws),
                       ws_bytes, None)


def test_host_validation_codes(lib):
    s = ops.make_shape(64, 2, 1)
    assert _call_fwd(lib, s, ptr=0) == 1                     # NULL
    assert _call_fwd(lib, s, ptr=24) == 2                    # misaligned
    assert _call_fwd(lib, s, ws_bytes=16) == 5               # workspace too small
    assert _call_fwd(lib, s, ws=0) == 5                      # no workspace
    assert _call_fwd(lib, s, ws=1032) == 2                   # misaligned workspace
    u = ops.make_shape(64, 2, 1); u.V = 256
    assert _call_fwd(lib, u) == 4                            # unsupported V
    u = ops.make_shape(64, 2, 1, lower_bound=0.0)
    assert _call_fwd(lib, u) == 4                            # lb must be < 0
    u = ops.make_shape(64, 2, 1, scale=float("nan"))
    assert _call_fwd(lib, u) == 4
    u = ops.make_shape(64, 0, 1)
    assert _call_fwd(lib, u) == 3                            # H = 0
    u = ops.make_shape(64, 2, 3)                             # packed with B = 1, N = 3 needs offsets
    assert _call_fwd(lib, u) == 3
    assert lib.kda_status_string(6) == b"KDA_ERR_OFFSETS"
    u = ops.make_shape(64, 6, 1, groups=4)
    assert _call_fwd(lib, u) == 3                            # groups must divide H
    u = ops.make_shape(64, 6, 1, groups=-1)
    assert _call_fwd(lib, u) == 3
    for cs in (1, 16, 48, 128, -32):
        u = ops.make_shape(64, 2, 1, chunk_size=cs)
        assert _call_fwd(lib, u) == 4                        # chunk length 0, 32 or 64 only
    assert lib.kda_status_string(9) == b"KDA_ERR_STALE_WORKSPACE"


def test_chunk_size_option_accepted_on_the_host(lib):
    """chunk_size 0, 32 and 64 pass the host checks and need the same workspace."""
    sizes = {cs: ops.workspace_size(ops.make_shape(1000, 4, 1, chunk_size=cs)) for cs in (0, 32, 64)}
    assert len(set(sizes.values())) == 1 and sizes[64] > 0
    assert ops.workspace_size(ops.make_shape(1000, 4, 1, chunk_size=16)) == 0


def test_grouped_heads_workspace(lib):
    """groups = 0 reads as 1; grouped heads add the fp32 dq, dk partials of every value head."""
    plain = ops.workspace_size(ops.make_shape(1000, 8, 1))
    assert ops.workspace_size(ops.make_shape(1000, 8, 1, groups=0)) == plain
    assert ops.workspace_size(ops.make_shape(1000, 8, 1, groups=1)) == plain
    grouped = ops.workspace_size(ops.make_shape(1000, 8, 1, groups=4))
    assert grouped >= plain + 2 * 1000 * 8 * 128 * 4
    assert ops.workspace_size(ops.make_shape(1000, 8, 1, groups=3)) == 0


def test_selftest_rejects_bad_shapes(lib):
    p = ctypes.c_void_p(16)
    assert lib.kda_diag_umma_selftest(0, 0, 300, 64, p, p, p, None) == 3
    assert lib.kda_diag_umma_selftest(1, 0, 64, 64, p, p, p, None) == 4


def test_decode_host_validation_codes(lib):
    def call(n=2, H=3, scale=0.088, lb=-5.0, ptr=16, bad=None, groups=1):
        ps = [ctypes.c_void_p(ptr) for _ in range(9)]
        if bad is not None:
            ps[bad] = ctypes.c_void_p(ptr + 8)
        return lib.kda_decode(n, H, groups, scale, lb, *ps, None)
    assert call(groups=2) == 3                # groups must divide H
    assert call(groups=-1) == 3
    assert call(n=-1) == 3                    # negative batch
    assert call(H=0) == 3
    assert call(n=1 << 30, H=8) == 3          # more than 2^31 - 1 units
    assert call(lb=-6.0) == 4                 # lower bound outside [-5, 0)
    assert call(lb=0.0) == 4
    assert call(scale=float("inf")) == 4
    assert call(ptr=0) == 1                   # NULL
    for i in range(9):
        assert call(bad=i) == 2               # each pointer must be 16-byte aligned
    assert call(n=0, ptr=0) == 0              # empty batch: nothing to do


def test_product_path_fails_loudly_without_the_library():
    """No CPU fallback: with the library missing and no way to build it, the binding raises
    instead of computing (run in a fresh interpreter so the loaded library stays untouched)."""
    import subprocess
    import sys
    code = r'''
import sys, torch
sys.path.insert(0, ROOT)
from kimi_delta_attention_15_gb300 import build as B, ops
B.LIB = "/nonexistent/libkda.so"
def no_build(*a, **k):
    raise RuntimeError("nvcc unavailable")
B.build = no_build
x = torch.zeros(64, 2, 128, dtype=torch.bfloat16)
try:
    ops.fwd(x, x, x, x, torch.zeros(64, 2, dtype=torch.bfloat16), torch.zeros(2), torch.zeros(2, 128))
except RuntimeError as e:
    print("raised:", e)
    sys.exit(0)
sys.exit(3)
'''.replace("ROOT", repr(os.path.dirname(os.path.dirname(os.path.abspath(__file__)))))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and "raised" in r.stdout, r.stdout + r.stderr


def test_header_is_plain_c():
    """include/kda.h compiles as C99 (the boundary is a C ABI, not only C++)."""
    import shutil
    import subprocess
    import tempfile
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    src = r'''
#include "kda.h"
int main(void) {
    kda_shape sh = {1, 64, 2, 1, 128, 128, 0.088f, -5.0f, 1, 0};
    size_t (*ws)(const kda_shape*) = kda_workspace_size;
    kda_status (*fwd)(const kda_shape*, const kda_bf16*, const kda_bf16*, const kda_bf16*, const kda_bf16*,
                      const kda_bf16*, const float*, const float*, const float*, const int64_t*, kda_bf16*,
                      float*, void*, size_t, void*) = kda_fwd;
    (void)sh; (void)ws; (void)fwd; (void)kda_bwd; (void)kda_decode; (void)kda_get_device_status;
    return KDA_OK;
}
'''
    with tempfile.TemporaryDirectory() as d:
        p = os.path.join(d, "use_kda.c")
        with open(p, "w") as f:
            f.write(src)
        r = subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", "-pedantic", "-fsyntax-only",
                            "-I", os.path.join(root, "include"), p], capture_output=True, text=True)
        assert r.returncode == 0, r.stderr
