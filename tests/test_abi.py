"""C-ABI checks that need no GPU: the library loads, exports every function include/gla.h declares, and
rejects bad arguments synchronously (before any CUDA work).  Pointers here are fake addresses that the
library only inspects (alignment, overlap) and never dereferences."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def gla():
    from chunkwise_gated_linear_chunked_gb300 import build
    build.build()
    from chunkwise_gated_linear_chunked_gb300 import binding
    return binding


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"^[A-Za-z_][\w\s\*]*?\b(gla_\w+)\s*\(", src, flags=re.M))
    return names


def test_exports_every_declared_symbol(gla):
    names = declared_functions()
    assert {"gla_fwd", "gla_fwd_workspace_size", "gla_get_status", "gla_strerror"} <= names
    lib = gla.lib()
    for n in sorted(names):
        assert hasattr(lib, n), n
    assert set(gla.EXPORTS) == names


def test_strerror_total(gla):
    for code in range(-1, 9):
        assert isinstance(gla.strerror(code), str) and gla.strerror(code)


A = 1 << 20   # fake, 16-byte-aligned device addresses far apart


def call(gla, q=A, k=2 * A, v=3 * A, g=4 * A, o=8 * A, scale=0.125, h0=None, ht=None, cu=None, N=2, B=2,
         T=100, H=2, K=64, V=64, chunk=64, dtype=1, ws=64 * A, wsb=1 << 40):
    p = lambda x: None if x is None else ctypes.c_void_p(x)
    return gla.lib().gla_fwd(p(q), p(k), p(v), p(g), p(o), scale, p(h0), p(ht), p(cu), N, B, T, H, K, V,
                             chunk, dtype, p(ws), wsb, None)


def test_rejects_unsupported_shapes(gla):
    assert call(gla, K=96) == gla.GLA_ERR_UNSUPPORTED
    assert call(gla, V=32) == gla.GLA_ERR_UNSUPPORTED
    assert call(gla, chunk=48) == gla.GLA_ERR_UNSUPPORTED
    assert call(gla, dtype=7) == gla.GLA_ERR_UNSUPPORTED


def test_rejects_invalid_arguments(gla):
    assert call(gla, scale=0.0) == gla.GLA_ERR_INVALID_ARG
    assert call(gla, scale=-1.0) == gla.GLA_ERR_INVALID_ARG
    assert call(gla, scale=float("nan")) == gla.GLA_ERR_INVALID_ARG
    assert call(gla, scale=float("inf")) == gla.GLA_ERR_INVALID_ARG
    assert call(gla, N=3) == gla.GLA_ERR_INVALID_ARG                 # dense: N must equal B
    assert call(gla, cu=40 * A, B=2) == gla.GLA_ERR_INVALID_ARG      # varlen needs B == 1
    assert call(gla, H=0) == gla.GLA_ERR_INVALID_ARG
    assert call(gla, T=-1) == gla.GLA_ERR_INVALID_ARG
    assert call(gla, q=None) == gla.GLA_ERR_INVALID_ARG


def test_rejects_misaligned_pointers(gla):
    assert call(gla, q=A + 8) == gla.GLA_ERR_ALIGNMENT
    assert call(gla, o=8 * A + 4) == gla.GLA_ERR_ALIGNMENT
    assert call(gla, h0=20 * A + 2) == gla.GLA_ERR_ALIGNMENT
    assert call(gla, ws=64 * A + 16) == gla.GLA_ERR_ALIGNMENT        # workspace wants 256 bytes


def test_rejects_missing_or_small_workspace(gla):
    assert call(gla, ws=None) == gla.GLA_ERR_WORKSPACE
    need = gla.workspace_size(2, 100, 2, 64, 64, 2, 64, 1)
    assert need >= 256
    assert call(gla, wsb=need - 1) == gla.GLA_ERR_WORKSPACE


def test_rejects_aliasing(gla):
    assert call(gla, o=A + 256) == gla.GLA_ERR_INVALID_ARG            # o overlaps q
    assert call(gla, h0=20 * A, ht=20 * A + 256) == gla.GLA_ERR_INVALID_ARG   # partial state overlap
    assert call(gla, ht=8 * A + 1024) == gla.GLA_ERR_INVALID_ARG      # ht overlaps o
    assert call(gla, ws=A) == gla.GLA_ERR_INVALID_ARG                 # workspace overlaps inputs


def test_workspace_size_rejects_and_grows(gla):
    assert gla.workspace_size(1, 100, 2, 96, 64, 1, 64, 1) == 0
    small = gla.workspace_size(1, 4096, 1, 128, 128, 1, 64, 1)
    assert small > 256   # one long sequence with one head is split into segments
    assert gla.workspace_size(1, 4096, 1, 128, 128, 8, 64, 1) >= 256


def test_cumsum_rejects(gla):
    f = gla.lib().gla_chunk_local_cumsum
    p = ctypes.c_void_p
    assert f(p(A), p(2 * A), None, 1, 1, 10, 1, 64, 48, 0, None) == gla.GLA_ERR_UNSUPPORTED
    assert f(p(A), p(2 * A), None, 1, 1, 10, 1, 64, 64, 2, None) == gla.GLA_ERR_UNSUPPORTED
    assert f(p(A + 4), p(2 * A), None, 1, 1, 10, 1, 64, 64, 0, None) == gla.GLA_ERR_ALIGNMENT
    assert f(p(A), p(A + 256), None, 1, 1, 10, 1, 64, 64, 0, None) == gla.GLA_ERR_INVALID_ARG


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    """The product path has no fallback: importing the binding with no built library raises."""
    import importlib
    import sys
    from chunkwise_gated_linear_chunked_gb300 import build
    monkeypatch.setattr(build, "LIB", str(tmp_path / "missing.so"))
    sys.modules.pop("chunkwise_gated_linear_chunked_gb300.binding", None)
    try:
        with pytest.raises(ImportError):
            importlib.import_module("chunkwise_gated_linear_chunked_gb300.binding")
    finally:
        sys.modules.pop("chunkwise_gated_linear_chunked_gb300.binding", None)


def bwd(gla, q=A, k=2 * A, v=3 * A, g=4 * A, do=5 * A, scale=0.125, h0=None, dht=None, dq=8 * A, dk=9 * A,
        dv=10 * A, dg=11 * A, dh0=None, cu=None, N=2, B=2, T=100, H=2, K=64, V=64, chunk=64, dtype=1, ws=64 * A,
        wsb=1 << 40):
    p = lambda x: None if x is None else ctypes.c_void_p(x)
    return gla.lib().gla_bwd(p(q), p(k), p(v), p(g), p(do), scale, p(h0), p(dht), p(dq), p(dk), p(dv), p(dg),
                             p(dh0), p(cu), N, B, T, H, K, V, chunk, dtype, p(ws), wsb, None)


def test_bwd_rejects_before_any_cuda_work(gla):
    assert bwd(gla, V=512) == gla.GLA_ERR_UNSUPPORTED                 # value widths 64, 128 and 256 only
    assert bwd(gla, V=192) == gla.GLA_ERR_UNSUPPORTED
    assert bwd(gla, K=96) == gla.GLA_ERR_UNSUPPORTED
    assert bwd(gla, chunk=48) == gla.GLA_ERR_UNSUPPORTED
    assert bwd(gla, dtype=gla.GLA_BF16_OBF16) == gla.GLA_ERR_UNSUPPORTED
    assert bwd(gla, scale=0.0) == gla.GLA_ERR_INVALID_ARG
    assert bwd(gla, N=3) == gla.GLA_ERR_INVALID_ARG
    assert bwd(gla, dq=None) == gla.GLA_ERR_INVALID_ARG
    assert bwd(gla, do=5 * A + 8) == gla.GLA_ERR_ALIGNMENT
    assert bwd(gla, dh0=20 * A + 4) == gla.GLA_ERR_ALIGNMENT
    assert bwd(gla, ws=None) == gla.GLA_ERR_WORKSPACE
    assert gla.bwd_workspace_size(2, 100, 2, 64, 64, 2, 64, 1) > 4096   # chunk states and adjoints
    assert bwd(gla, wsb=4096) == gla.GLA_ERR_WORKSPACE
    assert bwd(gla, dq=A + 256) == gla.GLA_ERR_INVALID_ARG            # dq overlaps q
    assert bwd(gla, dk=8 * A + 256) == gla.GLA_ERR_INVALID_ARG        # dk overlaps dq
    assert bwd(gla, dh0=64 * A) == gla.GLA_ERR_INVALID_ARG            # dh0 overlaps the workspace
    assert bwd(gla, ws=A) == gla.GLA_ERR_INVALID_ARG                  # workspace overlaps inputs
    assert gla.bwd_workspace_size(1, 100, 2, 64, 512, 1, 64, 1) == 0
    # V = 256 runs as two 128-wide value slices that share one slice's workspace
    assert gla.bwd_workspace_size(1, 100, 2, 64, 256, 1, 64, 1) == gla.bwd_workspace_size(1, 100, 2, 64, 128, 1, 64, 1)


def wy(gla, k=A, v=2 * A, beta=3 * A, Am=4 * A, g=5 * A, w=8 * A, u=9 * A, cu=None, N=2, B=2, T=100, H=2, HV=4,
       K=64, V=64, chunk=64, dtype=1, ws=64 * A, wsb=1 << 40):
    p = lambda x: None if x is None else ctypes.c_void_p(x)
    return gla.lib().gla_wy_fwd(p(k), p(v), p(beta), p(Am), p(g), p(w), p(u), p(cu), N, B, T, H, HV, K, V, chunk,
                                dtype, p(ws), wsb, None)


def test_wy_rejects_before_any_cuda_work(gla):
    assert wy(gla, K=96) == gla.GLA_ERR_UNSUPPORTED
    assert wy(gla, V=256) == gla.GLA_ERR_UNSUPPORTED
    assert wy(gla, chunk=128) == gla.GLA_ERR_UNSUPPORTED
    assert wy(gla, dtype=gla.GLA_BF16_GF32) == gla.GLA_ERR_UNSUPPORTED
    assert wy(gla, HV=3) == gla.GLA_ERR_INVALID_ARG                    # value heads not a multiple of key heads
    assert wy(gla, N=3) == gla.GLA_ERR_INVALID_ARG
    assert wy(gla, w=None) == gla.GLA_ERR_INVALID_ARG
    assert wy(gla, beta=3 * A + 2) == gla.GLA_ERR_ALIGNMENT
    assert wy(gla, ws=None) == gla.GLA_ERR_WORKSPACE
    assert wy(gla, w=2 * A + 64) == gla.GLA_ERR_INVALID_ARG            # w overlaps v
    assert wy(gla, u=8 * A + 64) == gla.GLA_ERR_INVALID_ARG            # u overlaps w
    assert wy(gla, ws=A) == gla.GLA_ERR_INVALID_ARG                    # workspace overlaps k
    lib = gla.lib()
    assert lib.gla_wy_workspace_size(100, 2, 48, 0) == 0
    assert lib.gla_wy_workspace_size(1000, 5, 64, 1) > lib.gla_wy_workspace_size(1000, 5, 64, 0)
    assert wy(gla, cu=80 * A, N=3, B=1, wsb=256) == gla.GLA_ERR_WORKSPACE   # varlen needs the chunk table


def ttt(gla, q=A, k=2 * A, v=3 * A, w=4 * A, b=5 * A, eta=6 * A, scale=0.09, eps=1e-6, h0=None, hb0=None, o=8 * A,
        ht=None, hbt=None, cu=None, N=2, B=2, T=100, H=2, D=64, chunk=16, dtype=1, ws=64 * A, wsb=1 << 20):
    p = lambda x: None if x is None else ctypes.c_void_p(x)
    return gla.lib().gla_ttt_linear_fwd(p(q), p(k), p(v), p(w), p(b), p(eta), ctypes.c_float(scale),
                                        ctypes.c_float(eps), p(h0), p(hb0), p(o), p(ht), p(hbt), p(cu), N, B, T, H, D,
                                        chunk, dtype, p(ws), wsb, None)


def test_ttt_rejects_before_any_cuda_work(gla):
    assert ttt(gla, D=96) == gla.GLA_ERR_UNSUPPORTED
    assert ttt(gla, chunk=64) == gla.GLA_ERR_UNSUPPORTED
    assert ttt(gla, dtype=gla.GLA_BF16_GF32) == gla.GLA_ERR_UNSUPPORTED
    assert ttt(gla, scale=0.0) == gla.GLA_ERR_INVALID_ARG
    assert ttt(gla, eps=0.0) == gla.GLA_ERR_INVALID_ARG
    assert ttt(gla, N=3) == gla.GLA_ERR_INVALID_ARG
    assert ttt(gla, o=None) == gla.GLA_ERR_INVALID_ARG
    assert ttt(gla, w=None) == gla.GLA_ERR_INVALID_ARG
    assert ttt(gla, eta=6 * A + 4) == gla.GLA_ERR_ALIGNMENT
    assert ttt(gla, ws=None) == gla.GLA_ERR_WORKSPACE
    assert ttt(gla, wsb=16) == gla.GLA_ERR_WORKSPACE
    assert ttt(gla, o=A + 64) == gla.GLA_ERR_INVALID_ARG                 # o overlaps q
    assert ttt(gla, ht=20 * A, hbt=20 * A + 64) == gla.GLA_ERR_INVALID_ARG   # the two final states overlap
    assert gla.lib().gla_ttt_workspace_size() >= 16


def fwd_host(gla, q=A, k=2 * A, v=3 * A, g=4 * A, o=5 * A, scale=0.09, h0=None, ht=None, cu=None, N=2, B=2, T=100,
             H=4, K=128, V=128, chunk=64, dtype=1, groups=2, ws=64 * A, wsb=1 << 34):
    p = lambda x: None if x is None else ctypes.c_void_p(x)
    return gla.lib().gla_fwd_host(p(q), p(k), p(v), p(g), p(o), ctypes.c_float(scale), p(h0), p(ht), p(cu), N, B, T,
                                  H, K, V, chunk, dtype, groups, p(ws), wsb, None)


def test_host_entry_rejects_before_any_cuda_work(gla):
    assert fwd_host(gla, groups=3) == gla.GLA_ERR_INVALID_ARG            # 4 heads in 3 groups
    assert fwd_host(gla, groups=0) == gla.GLA_ERR_INVALID_ARG
    assert fwd_host(gla, dtype=1 | gla.GLA_HEAD_FIRST) == gla.GLA_ERR_UNSUPPORTED
    assert fwd_host(gla, K=96) == gla.GLA_ERR_UNSUPPORTED
    assert fwd_host(gla, N=3) == gla.GLA_ERR_INVALID_ARG
    assert fwd_host(gla, q=None) == gla.GLA_ERR_INVALID_ARG
    assert fwd_host(gla, scale=0.0) == gla.GLA_ERR_INVALID_ARG
    assert fwd_host(gla, ws=None) == gla.GLA_ERR_WORKSPACE
    assert fwd_host(gla, wsb=1024) == gla.GLA_ERR_WORKSPACE
    assert fwd_host(gla, ws=64 * A + 16) == gla.GLA_ERR_ALIGNMENT
    lib = gla.lib()
    lib.gla_fwd_host_workspace_size.restype = ctypes.c_size_t
    assert lib.gla_fwd_host_workspace_size(2, 100, 4, 128, 128, 2, 64, 1, 3) == 0
    two = lib.gla_fwd_host_workspace_size(2, 100, 4, 128, 128, 2, 64, 1, 2)
    four = lib.gla_fwd_host_workspace_size(2, 100, 4, 128, 128, 2, 64, 1, 4)
    assert 0 < four < two   # device buffers for at most three groups: 3 of 4 heads, against 2 slots of 2
