"""Oracle for the GLA forward and backward passes — TEST INFRASTRUCTURE ONLY.

A plain fp64 CPU implementation (``gla_oracle.c``) of the gated linear attention recurrence, of its
reverse-mode gradients and of the chunk-local gate cumsum, wrapped with ctypes over numpy arrays.  Only ``tests/``, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import this package.  The CUDA library
neither imports nor links it; the two share no code.

Method citations (page "fla/ops/gla/fused_chunk.py"):
  * recurrence / state carry: ``fused_chunk_gla_fwd_kernel`` (state update ``h*exp(G_last) + k_g^T v``,
    output ``q_g h``, initial state load and final state store);
  * intra-chunk term with inclusive diagonal: ``fwd_inner_chunk``;
  * gated operands ``q*exp(G)*scale`` and ``k*exp(G_last-G)``: ``prepare_qg_kg``;
  * chunk-local cumsum in fp32: ``FusedChunkGLAFunction.forward``.
Varlen convention (offsets, per-sequence states): page "fla/ops/ttt/fused_chunk.py",
``fused_chunk_ttt_linear_fwd_kernel`` and ``fused_chunk_ttt_linear``.

TTT-linear forward (``ttt_linear_fwd``): page "fla/ops/ttt/fused_chunk.py", ``fused_chunk_ttt_linear_fwd_kernel``
and the ``norm_residual`` step of ``fused_chunk_ttt_linear`` (pins in ``tests/test_oracle_ttt.py``).

WY representation forward of the gated delta rule (``wy_fwd``): page
"fla/ops/gated_delta_rule/backends/triton_ascend/wy_fast.py", ``recompute_w_u_fwd_kernel_npu`` and
``recompute_w_u_fwd_npu`` (pins in ``tests/test_oracle_wy.py``).

Backward (``gla_bwd``): page "fla/ops/gla/fused_chunk.py", ``fused_chunk_gla_bwd_kernel`` and
``bwd_inner_chunk`` (chunked gradients of the same recurrence) and ``FusedChunkGLAFunction.backward`` (dg from
the reverse cumsum of ``q*dq - k*dk``); the oracle differentiates the plain recurrence step by step instead.

Pins: every function here is checked in ``tests/test_oracle.py`` / ``tests/test_oracle_bwd.py`` against
quantities that do not come from the oracle itself (brute-force quadratic form, the g == 0 closed form,
scalar closed forms, state-split invariance, varlen == separate runs, symmetry invariances, hand-derived
golden fixtures; for the backward: central finite differences of the forward oracle in fp64 and the
gate-gradient identity).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gla_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

F32, BF16, F64, F16 = 0, 1, 2, 3


def build(force: bool = False) -> str:
    """Compile ``gla_oracle.c`` into ``oracle/_build/liboracle.so`` (portable flags, no -march)."""
    os.makedirs(_BUILD, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-fno-fast-math", "-ffp-contract=off", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            p = ctypes.c_void_p
            i = ctypes.c_int
            lib.oracle_gla_fwd.argtypes = [p, p, p, p, i, p, p, p, p, i, i, i, i, i, i,
                                           ctypes.c_double, i]
            lib.oracle_gla_fwd.restype = i
            lib.oracle_chunk_local_cumsum.argtypes = [p, i, p, p, i, i, i, i, i, i]
            lib.oracle_chunk_local_cumsum.restype = i
            _declare_bwd(lib)
            _lib = lib
    return _lib


def _declare_bwd(lib):
    p, i = ctypes.c_void_p, ctypes.c_int
    lib.oracle_gla_bwd.argtypes = [p, p, p, p, p, i, p, p, p, p, p, p, p, p, i, i, i, i, i, i,
                                   ctypes.c_double, i]
    lib.oracle_gla_bwd.restype = i


def _as_stored(x: np.ndarray):
    """Return (contiguous array, dtype code).  bf16 tensors are passed as their raw uint16 words; float64
    inputs (finite-difference checks) are read as they are."""
    x = np.ascontiguousarray(x)
    if x.dtype == np.float32:
        return x, F32
    if x.dtype == np.uint16:
        return x, BF16
    if x.dtype == np.float64:
        return x, F64
    if x.dtype == np.float16:
        return x.view(np.uint16), F16
    raise TypeError(f"oracle inputs must be float32, float16, float64 or bf16 words (uint16), got {x.dtype}")


def _widen(x):
    x = np.ascontiguousarray(x)
    return bf16_words_to_f64(x) if x.dtype == np.uint16 else x.astype(np.float64)


def _common_type(*xs):
    """Inputs of one stored type pass through; mixed types (e.g. 16-bit q, k, v with an fp32 g) are all
    widened exactly to float64."""
    if len({np.asarray(x).dtype for x in xs}) == 1:
        return xs
    return tuple(_widen(x) for x in xs)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def load_variant(path: str):
    """Load a separately compiled copy of ``gla_oracle.c`` (the tests plant mistakes in such copies to
    show that the pins catch them).  Pass the handle as ``lib=`` to :func:`gla_fwd`."""
    lib = ctypes.CDLL(path)
    p, i = ctypes.c_void_p, ctypes.c_int
    lib.oracle_gla_fwd.argtypes = [p, p, p, p, i, p, p, p, p, i, i, i, i, i, i, ctypes.c_double, i]
    lib.oracle_gla_fwd.restype = i
    if hasattr(lib, "oracle_gla_bwd"):
        _declare_bwd(lib)
    return lib


def gla_fwd(q, k, v, g, scale, h0=None, cu_seqlens=None, want_ht=True, nthreads=0, lib=None):
    """fp64 step-by-step GLA forward.

    q, k, g: [B, T, H, K]; v: [B, T, H, V]; all float32 or all bf16 words (uint16).
    h0: optional [N, H, K, V] (float32 or float64; widened to float64).  cu_seqlens: optional int32 [N+1] (host), requires B == 1.
    Returns (o float64 [B, T, H, V], ht float64 [N, H, K, V] or None, threads used).
    """
    q, k, v, g = _common_type(q, k, v, g)
    (q, dt), (k, dk), (v, dv), (g, dg) = map(_as_stored, (q, k, v, g))
    if len({dt, dk, dv, dg}) != 1:
        raise TypeError("q, k, v, g must share one stored type")
    B, T, H, K = q.shape
    V = v.shape[-1]
    if k.shape != q.shape or g.shape != q.shape or v.shape[:3] != q.shape[:3]:
        raise ValueError("shape mismatch between q, k, v, g")
    cu = None
    if cu_seqlens is not None:
        if B != 1:
            raise ValueError("cu_seqlens requires B == 1")
        cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
        N = cu.size - 1
        if cu[0] != 0 or cu[-1] != T or np.any(np.diff(cu) < 0):
            raise ValueError("cu_seqlens must be non-decreasing from 0 to T")
    else:
        N = B
    if h0 is not None:
        h0 = np.ascontiguousarray(h0, dtype=np.float64)  # fp32 widens exactly
        if h0.shape != (N, H, K, V):
            raise ValueError(f"h0 must be [N, H, K, V] = {(N, H, K, V)}, got {h0.shape}")
    o = np.zeros((B, T, H, V), dtype=np.float64)
    ht = np.zeros((N, H, K, V), dtype=np.float64) if want_ht else None
    rc = (lib or _load()).oracle_gla_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), dt, _ptr(h0), _ptr(o), _ptr(ht),
                                _ptr(cu), N, B, T, H, K, V, float(scale), int(nthreads))
    if rc < 0:
        raise RuntimeError(f"oracle_gla_fwd failed ({rc})")
    return o, ht, rc


def gla_bwd(q, k, v, g, do, scale, h0=None, dht=None, cu_seqlens=None, nthreads=0, lib=None):
    """fp64 reverse-mode gradients of the GLA recurrence for L = sum(o * do) + sum(ht * dht).

    q, k, g: [B, T, H, K]; v, do: [B, T, H, V]; all one stored type (float32, bf16 words or float64).
    h0, dht: optional [N, H, K, V] (widened to float64).  Returns float64 (dq, dk, dv, dg, dh0) shaped like
    q, k, v, g and [N, H, K, V].
    """
    q, k, v, g, do = _common_type(q, k, v, g, do)
    arrs = list(map(_as_stored, (q, k, v, g, do)))
    if len({a[1] for a in arrs}) != 1:
        raise TypeError("q, k, v, g, do must share one stored type")
    (q, dt), (k, _), (v, _), (g, _), (do, _) = arrs
    B, T, H, K = q.shape
    V = v.shape[-1]
    if k.shape != q.shape or g.shape != q.shape or v.shape[:3] != q.shape[:3] or do.shape != v.shape:
        raise ValueError("shape mismatch between q, k, v, g, do")
    cu = None
    N = B
    if cu_seqlens is not None:
        if B != 1:
            raise ValueError("cu_seqlens requires B == 1")
        cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
        N = cu.size - 1
        if cu[0] != 0 or cu[-1] != T or np.any(np.diff(cu) < 0):
            raise ValueError("cu_seqlens must be non-decreasing from 0 to T")
    st = []
    for x in (h0, dht):
        if x is not None:
            x = np.ascontiguousarray(x, dtype=np.float64)
            if x.shape != (N, H, K, V):
                raise ValueError(f"states must be [N, H, K, V] = {(N, H, K, V)}, got {x.shape}")
        st.append(x)
    dq = np.zeros(q.shape, np.float64)
    dk = np.zeros(q.shape, np.float64)
    dv = np.zeros(v.shape, np.float64)
    dg = np.zeros(q.shape, np.float64)
    dh0 = np.zeros((N, H, K, V), np.float64)
    rc = (lib or _load()).oracle_gla_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(do), dt, _ptr(st[0]),
                                         _ptr(st[1]), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dg), _ptr(dh0),
                                         _ptr(cu), N, B, T, H, K, V, float(scale), int(nthreads))
    if rc < 0:
        raise RuntimeError(f"oracle_gla_bwd failed ({rc})")
    return dq, dk, dv, dg, dh0


def ttt_linear_fwd(q, k, v, w, b, eta, scale, eps, chunk, h0=None, hb0=None, cu_seqlens=None, nthreads=0,
                   lib=None):
    """fp64 TTT-linear forward (mini-batch gradient descent in chunks of ``chunk`` rows, then the residual
    norm).  q, k, v: [B, T, H, D] (one stored type, or mixed: widened exactly); w, b: [H, D]; eta: [B, T, H]
    (or [..., 1]); h0: [N, H, D, D]; hb0: [N, H, D] (or [N, H, 1, D]).  Returns float64 (o [B, T, H, D],
    ht [N, H, D, D], hbt [N, H, D])."""
    q, k, v = _common_type(q, k, v)
    (q, dt), (k, _), (v, _) = map(_as_stored, (q, k, v))
    B, T, H, D = q.shape
    if k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must share one shape [B, T, H, D] (TTT-linear needs K == V)")
    cu = None
    N = B
    if cu_seqlens is not None:
        cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
        N = cu.size - 1
    f64 = lambda x: None if x is None else np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    w, b = f64(w).reshape(H, D), f64(b).reshape(H, D)
    eta = f64(eta).reshape(B * T, H)
    h0 = None if h0 is None else f64(h0).reshape(N, H, D, D)
    hb0 = None if hb0 is None else f64(hb0).reshape(N, H, D)
    o = np.zeros((B, T, H, D), np.float64)
    ht = np.zeros((N, H, D, D), np.float64)
    hbt = np.zeros((N, H, D), np.float64)
    lib = lib or _load()
    if not getattr(lib, "_ttt_declared", False):
        p_, i_ = ctypes.c_void_p, ctypes.c_int
        lib.oracle_ttt_linear_fwd.argtypes = [p_, p_, p_, i_, p_, p_, p_, ctypes.c_double, ctypes.c_double, p_, p_,
                                              p_, p_, p_, p_, i_, i_, i_, i_, i_, i_, i_]
        lib.oracle_ttt_linear_fwd.restype = i_
        lib._ttt_declared = True
    rc = lib.oracle_ttt_linear_fwd(_ptr(q), _ptr(k), _ptr(v), dt, _ptr(w), _ptr(b), _ptr(eta), float(scale),
                                   float(eps), _ptr(h0), _ptr(hb0), _ptr(o), _ptr(ht), _ptr(hbt), _ptr(cu), N, B, T,
                                   H, D, int(chunk), int(nthreads))
    if rc < 0:
        raise RuntimeError(f"oracle_ttt_linear_fwd failed ({rc})")
    return o, ht, hbt


def wy_fwd(k, v, beta, A, g=None, cu_seqlens=None, nthreads=0, lib=None):
    """fp64 WY representation forward of the gated delta rule: per chunk of BT = A.shape[-1] rows from each
    sequence start, u = A (v * beta) and w = A (k * beta * 2^g).  k: [B, T, H, K]; v: [B, T, HV, V];
    beta: [B, T, HV]; A: [B, T, HV, BT]; g: [B, T, HV] (log2 units) or None.  k, v, beta, A share one stored
    type (mixed types are widened exactly).  Returns float64 (w [B, T, HV, K], u [B, T, HV, V])."""
    k, v, beta, A = _common_type(k, v, beta, A)
    (k, dt), (v, _), (beta, _), (A, _) = map(_as_stored, (k, v, beta, A))
    B, T, H, K = k.shape
    HV, V, BT = v.shape[2], v.shape[3], A.shape[-1]
    if v.shape[:2] != (B, T) or A.shape[:3] != (B, T, HV) or beta.reshape(B, T, -1).shape[2] != HV:
        raise ValueError("wy_fwd: k [B,T,H,K], v [B,T,HV,V], beta [B,T,HV], A [B,T,HV,BT]")
    cu = None
    N = B
    if cu_seqlens is not None:
        cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
        N = cu.size - 1
    g = None if g is None else np.ascontiguousarray(np.asarray(g, dtype=np.float64).reshape(B * T, HV))
    w = np.zeros((B, T, HV, K), np.float64)
    u = np.zeros((B, T, HV, V), np.float64)
    lib = lib or _load()
    if not getattr(lib, "_wy_declared", False):
        p_, i_ = ctypes.c_void_p, ctypes.c_int
        lib.oracle_wy_fwd.argtypes = [p_, p_, p_, p_, i_, p_, p_, p_, p_, i_, i_, i_, i_, i_, i_, i_, i_, i_]
        lib.oracle_wy_fwd.restype = i_
        lib._wy_declared = True
    rc = lib.oracle_wy_fwd(_ptr(k), _ptr(v), _ptr(A), _ptr(beta), dt, _ptr(g), _ptr(w), _ptr(u), _ptr(cu), N, B, T,
                           H, HV, K, V, BT, int(nthreads))
    if rc < 0:
        raise RuntimeError(f"oracle_wy_fwd failed ({rc})")
    return w, u


def chunk_local_cumsum(g, chunk, cu_seqlens=None):
    """fp64 chunk-local inclusive cumsum of g [B, T, H, K], chunks aligned to each sequence start."""
    g, dt = _as_stored(g)
    B, T, H, K = g.shape
    cu = None
    N = B
    if cu_seqlens is not None:
        cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
        N = cu.size - 1
    G = np.zeros(g.shape, dtype=np.float64)
    rc = _load().oracle_chunk_local_cumsum(_ptr(g), dt, _ptr(G), _ptr(cu), N, B, T, H, K, int(chunk))
    if rc != 0:
        raise RuntimeError("oracle_chunk_local_cumsum failed")
    return G


def bf16_words_to_f64(x: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 words (uint16) to float64, independent of torch."""
    return (np.ascontiguousarray(x, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
