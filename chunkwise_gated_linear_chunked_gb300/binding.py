"""Thin ctypes binding of libgla (``include/gla.h``): argument marshalling only.

Every step of the forward runs in libgla's CUDA kernels; torch supplies device memory and streams.  There is
no CPU fallback: if ``_build/libgla.so`` is missing the import fails loudly (run
``chunkwise_gated_linear_chunked_gb300.build.build()`` or ``__graft_entry__.build()`` first).
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from .build import LIB

GLA_OK, GLA_ERR_INVALID_ARG, GLA_ERR_UNSUPPORTED, GLA_ERR_ALIGNMENT, GLA_ERR_WORKSPACE, GLA_ERR_CUDA, \
    GLA_ERR_TIMEOUT, GLA_ERR_RANGE = range(8)
GLA_F32, GLA_BF16, GLA_BF16_OBF16, GLA_F16, GLA_BF16_GF32, GLA_F16_GF32 = 0, 1, 2, 3, 4, 5
GLA_HEAD_FIRST = 0x100   # OR-ed into the dtype code: [B, H, T, *] tensors

EXPORTS = ("gla_fwd", "gla_fwd_workspace_size", "gla_get_status", "gla_strerror", "gla_chunk_local_cumsum",
           "gla_profile_events", "gla_profile_launches", "gla_kernel_name", "gla_fwd_noalloc", "gla_bwd",
           "gla_bwd_workspace_size", "gla_ttt_linear_fwd", "gla_ttt_workspace_size", "gla_wy_fwd",
           "gla_wy_workspace_size", "gla_fwd_host", "gla_fwd_host_workspace_size")

if not os.path.exists(LIB):
    raise ImportError(f"libgla.so not built ({LIB}); call chunkwise_gated_linear_chunked_gb300.build.build()")

_lib = ctypes.CDLL(LIB)
_p, _i, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
_lib.gla_fwd.argtypes = [_p, _p, _p, _p, _p, _f, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _i, _p, _sz, _p]
_lib.gla_fwd.restype = _i
_lib.gla_fwd_workspace_size.argtypes = [_i] * 8
_lib.gla_fwd_workspace_size.restype = _sz
_lib.gla_fwd_host.argtypes = [_p, _p, _p, _p, _p, _f, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _i, _i, _p, _sz, _p]
_lib.gla_fwd_host.restype = _i
_lib.gla_fwd_host_workspace_size.argtypes = [_i] * 9
_lib.gla_fwd_host_workspace_size.restype = _sz
_lib.gla_get_status.argtypes = [_p, _p]
_lib.gla_get_status.restype = _i
_lib.gla_strerror.argtypes = [_i]
_lib.gla_strerror.restype = ctypes.c_char_p
_lib.gla_chunk_local_cumsum.argtypes = [_p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _p]
_lib.gla_chunk_local_cumsum.restype = _i
_lib.gla_profile_events.argtypes = [_p, _i, _p]
_lib.gla_profile_events.restype = _i
_lib.gla_profile_launches.argtypes = []
_lib.gla_profile_launches.restype = _i
_lib.gla_kernel_name.argtypes = [_i]
_lib.gla_kernel_name.restype = ctypes.c_char_p
_lib.gla_bwd.argtypes = [_p, _p, _p, _p, _p, _f, _p, _p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i,
                         _i, _p, _sz, _p]
_lib.gla_bwd.restype = _i
_lib.gla_bwd_workspace_size.argtypes = [_i] * 8
_lib.gla_bwd_workspace_size.restype = _sz
_lib.gla_ttt_linear_fwd.argtypes = [_p, _p, _p, _p, _p, _p, _f, _f, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i,
                                    _i, _p, _sz, _p]
_lib.gla_ttt_linear_fwd.restype = _i
_lib.gla_wy_fwd.argtypes = [_p, _p, _p, _p, _p, _p, _p, _p] + [_i] * 9 + [_p, _sz, _p]
_lib.gla_wy_fwd.restype = _i
_lib.gla_wy_workspace_size.argtypes = [_i, _i, _i, _i]
_lib.gla_wy_workspace_size.restype = _sz
_lib.gla_ttt_workspace_size.argtypes = []
_lib.gla_ttt_workspace_size.restype = _sz


class GlaError(RuntimeError):
    def __init__(self, code: int, what: str = "gla_fwd"):
        self.code = code
        super().__init__(f"{what}: {strerror(code)} (code {code})")


def lib():
    return _lib


def strerror(code: int) -> str:
    return _lib.gla_strerror(int(code)).decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


DTYPE_CODE = {(torch.float32, torch.float32): GLA_F32, (torch.bfloat16, torch.float32): GLA_BF16,
              (torch.bfloat16, torch.bfloat16): GLA_BF16_OBF16, (torch.float16, torch.float32): GLA_F16}

# 16-bit q, k, v with an fp32 g (o fp32)
GF32_CODE = {torch.bfloat16: GLA_BF16_GF32, torch.float16: GLA_F16_GF32}


def _dtype_code(q, g, out_dtype, what):
    """The dtype code of a call: q, k, v share one dtype; g has it too, or is fp32 beside 16-bit q, k, v."""
    if g.dtype == q.dtype:
        code = DTYPE_CODE.get((q.dtype, out_dtype)) if out_dtype is not None else \
            {torch.float32: GLA_F32, torch.bfloat16: GLA_BF16, torch.float16: GLA_F16}.get(q.dtype)
    elif g.dtype == torch.float32 and out_dtype in (None, torch.float32):
        code = GF32_CODE.get(q.dtype)
    else:
        code = None
    if code is None:
        raise GlaError(GLA_ERR_UNSUPPORTED, f"{what} dtypes q {q.dtype}, g {g.dtype} -> {out_dtype}")
    return code


_ws_lock = threading.Lock()
_ws_cache: dict = {}


def workspace_size(B, T, H, K, V, N, chunk=64, dtype=GLA_BF16) -> int:
    return int(_lib.gla_fwd_workspace_size(B, T, H, K, V, N, chunk, dtype))


def get_workspace(nbytes: int, device) -> torch.Tensor:
    """A zero-initialised, cached device workspace of at least ``nbytes`` (one per device and stream use)."""
    device = torch.device(device)
    key = (device.index if device.index is not None else torch.cuda.current_device())
    with _ws_lock:
        ws = _ws_cache.get(key)
        if ws is None or ws.numel() < nbytes:
            ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device)
            _ws_cache[key] = ws
        return ws


def fwd_into(q, k, v, g, o, scale, h0, ht, cu_seqlens, N, B, T, H, K, V, chunk, dtype, workspace,
             stream=None) -> int:
    """Raw call: tensors (or None) are passed as device pointers, sizes as given.  Returns the code."""
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return int(_lib.gla_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(o), float(scale), _ptr(h0), _ptr(ht),
                            _ptr(cu_seqlens), int(N), int(B), int(T), int(H), int(K), int(V), int(chunk),
                            int(dtype), _ptr(workspace), nbytes, _stream_handle(stream)))


def host_workspace_size(B, T, H, K, V, N, chunk, dtype, head_groups) -> int:
    return int(_lib.gla_fwd_host_workspace_size(int(B), int(T), int(H), int(K), int(V), int(N), int(chunk),
                                                int(dtype), int(head_groups)))


def fwd_host_into(q, k, v, g, o, scale, h0, ht, cu_seqlens, N, B, T, H, K, V, chunk, dtype, head_groups, workspace,
                  stream=None) -> int:
    """Raw call of gla_fwd_host: q, k, v, g, o, h0, ht, cu_seqlens are HOST tensors (or None), the workspace a
    device tensor.  Returns the code."""
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("o", o), ("h0", h0), ("ht", ht),
                    ("cu_seqlens", cu_seqlens)):
        if t is not None and (t.is_cuda or not t.is_contiguous()):
            raise GlaError(GLA_ERR_INVALID_ARG, f"gla_fwd_host: {name} must be a contiguous host tensor")
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return int(_lib.gla_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(o), float(scale), _ptr(h0), _ptr(ht),
                                 _ptr(cu_seqlens), int(N), int(B), int(T), int(H), int(K), int(V), int(chunk),
                                 int(dtype), int(head_groups), _ptr(workspace), nbytes, _stream_handle(stream)))


def gla_fwd(q, k, v, g, scale=None, initial_state=None, output_final_state=True, cu_seqlens=None,
            chunk=64, out_dtype=None, stream=None, workspace=None, head_first=False):
    """GLA forward on the GPU.

    q, k, g: [B, T, H, K]; v: [B, T, H, V] (cuda, contiguous, all fp32, all bf16 or all fp16), or
    [B, H, T, *] with head_first=True (with cu_seqlens: [1, H, T, *]).  initial_state: optional fp32 [N, H, K, V].
    cu_seqlens: optional int32 [N+1] cuda offsets (B == 1).  out_dtype: fp32 (default) or, for bf16 inputs,
    bf16.  Returns (o in the layout of the inputs, final_state or None).
    """
    if head_first:
        B, H, T, K = q.shape
    else:
        B, T, H, K = q.shape
    V = v.shape[-1]
    N = B if cu_seqlens is None else cu_seqlens.numel() - 1
    if scale is None:
        scale = K ** -0.5
    out_dtype = out_dtype or torch.float32
    code = _dtype_code(q, g, out_dtype, "gla_fwd")
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g)):
        if (t.dtype != q.dtype and t is not g) or not t.is_cuda or not t.is_contiguous():
            raise GlaError(GLA_ERR_INVALID_ARG, f"gla_fwd: {name} must be a contiguous cuda {q.dtype} tensor")
    o = torch.empty(*((B, H, T, V) if head_first else (B, T, H, V)), dtype=out_dtype, device=q.device)
    ht = torch.empty(N, H, K, V, dtype=torch.float32, device=q.device) if output_final_state else None
    h0 = initial_state
    if h0 is not None and (h0.dtype != torch.float32 or not h0.is_contiguous()):
        raise GlaError(GLA_ERR_INVALID_ARG, "gla_fwd: initial_state must be a contiguous fp32 tensor")
    if cu_seqlens is not None and cu_seqlens.dtype != torch.int32:
        raise GlaError(GLA_ERR_INVALID_ARG, "gla_fwd: cu_seqlens must be int32")
    if workspace is None:
        workspace = get_workspace(workspace_size(B, T, H, K, V, N, chunk, code), q.device)
    if head_first:
        code |= GLA_HEAD_FIRST
    rc = fwd_into(q, k, v, g, o, scale, h0, ht, cu_seqlens, N, B, T, H, K, V, chunk, code, workspace,
                  stream)
    if rc != GLA_OK:
        raise GlaError(rc)
    return o, ht


def bwd_workspace_size(B, T, H, K, V, N, chunk=64, dtype=GLA_BF16) -> int:
    return int(_lib.gla_bwd_workspace_size(B, T, H, K, V, N, chunk, dtype))


def bwd_into(q, k, v, g, do, scale, h0, dht, dq, dk, dv, dg, dh0, cu_seqlens, N, B, T, H, K, V, chunk, dtype,
             workspace, stream=None) -> int:
    """Raw backward call: tensors (or None) are passed as device pointers.  Returns the code."""
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return int(_lib.gla_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(do), float(scale), _ptr(h0), _ptr(dht),
                            _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dg), _ptr(dh0), _ptr(cu_seqlens), int(N), int(B),
                            int(T), int(H), int(K), int(V), int(chunk), int(dtype), _ptr(workspace), nbytes,
                            _stream_handle(stream)))


def gla_bwd(q, k, v, g, do, scale=None, initial_state=None, dht=None, cu_seqlens=None, chunk=64, stream=None,
            workspace=None, want_dh0=True, head_first=False):
    """GLA backward on the GPU for L = sum(o * do) + sum(ht * dht).

    q, k, g: [B, T, H, K]; v, do: [B, T, H, V] (cuda, contiguous, all fp32, bf16 or fp16), or [B, H, T, *]
    with head_first=True.  initial_state and dht: optional fp32 [N, H, K, V].  Returns fp32 (dq, dk, dv, dg,
    dh0 or None), in the layout of the inputs.
    """
    if head_first:
        B, H, T, K = q.shape
    else:
        B, T, H, K = q.shape
    V = v.shape[-1]
    N = B if cu_seqlens is None else cu_seqlens.numel() - 1
    if scale is None:
        scale = K ** -0.5
    code = _dtype_code(q, g, None, "gla_bwd")
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("do", do)):
        if (t.dtype != q.dtype and t is not g) or not t.is_cuda or not t.is_contiguous():
            raise GlaError(GLA_ERR_INVALID_ARG, f"gla_bwd: {name} must be a contiguous cuda {q.dtype} tensor")
    for name, t in (("initial_state", initial_state), ("dht", dht)):
        if t is not None and (t.dtype != torch.float32 or not t.is_contiguous()):
            raise GlaError(GLA_ERR_INVALID_ARG, f"gla_bwd: {name} must be a contiguous fp32 tensor")
    f32 = dict(dtype=torch.float32, device=q.device)
    shk, shv = ((B, H, T, K), (B, H, T, V)) if head_first else ((B, T, H, K), (B, T, H, V))
    dq, dk, dg = (torch.empty(*shk, **f32) for _ in range(3))
    dv = torch.empty(*shv, **f32)
    dh0 = torch.empty(N, H, K, V, **f32) if want_dh0 else None
    if workspace is None:
        workspace = get_workspace(bwd_workspace_size(B, T, H, K, V, N, chunk, code), q.device)
    if head_first:
        code |= GLA_HEAD_FIRST
    rc = bwd_into(q, k, v, g, do, scale, initial_state, dht, dq, dk, dv, dg, dh0, cu_seqlens, N, B, T, H, K, V,
                  chunk, code, workspace, stream)
    if rc != GLA_OK:
        raise GlaError(rc, "gla_bwd")
    return dq, dk, dv, dg, dh0


def ttt_linear_fwd(q, k, v, w, b, eta, scale=None, eps=1e-6, chunk=16, initial_state=None,
                   initial_state_bias=None, output_final_state=True, cu_seqlens=None, stream=None, workspace=None):
    """TTT-linear forward on the GPU.  q, k, v: [B, T, H, D] (cuda, contiguous, fp32 / bf16 / fp16); w, b:
    fp32 [H, D]; eta: fp32 [B, T, H] (or [..., 1]).  Returns fp32 (o [B, T, H, D], ht [N, H, D, D] or None,
    hbt [N, H, D] or None)."""
    B, T, H, D = q.shape
    N = B if cu_seqlens is None else cu_seqlens.numel() - 1
    if scale is None:
        scale = D ** -0.5
    code = {torch.float32: GLA_F32, torch.bfloat16: GLA_BF16, torch.float16: GLA_F16}.get(q.dtype)
    if code is None:
        raise GlaError(GLA_ERR_UNSUPPORTED, f"gla_ttt_linear_fwd dtype {q.dtype}")
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != q.dtype or not t.is_cuda or not t.is_contiguous() or t.shape != q.shape:
            raise GlaError(GLA_ERR_INVALID_ARG, f"gla_ttt_linear_fwd: {name} must be a contiguous cuda tensor like q")
    f32 = lambda x: None if x is None else x.contiguous().float()
    w, b, eta = f32(w), f32(b), f32(eta)
    h0, hb0 = f32(initial_state), f32(initial_state_bias)
    o = torch.empty(B, T, H, D, dtype=torch.float32, device=q.device)
    ht = torch.empty(N, H, D, D, dtype=torch.float32, device=q.device) if output_final_state else None
    hbt = torch.empty(N, H, D, dtype=torch.float32, device=q.device) if output_final_state else None
    if workspace is None:
        workspace = get_workspace(int(_lib.gla_ttt_workspace_size()), q.device)
    nbytes = workspace.numel() * workspace.element_size()
    rc = int(_lib.gla_ttt_linear_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(w), _ptr(b), _ptr(eta), float(scale),
                                     float(eps), _ptr(h0), _ptr(hb0), _ptr(o), _ptr(ht), _ptr(hbt), _ptr(cu_seqlens),
                                     N, B, T, H, D, int(chunk), code, _ptr(workspace), nbytes,
                                     _stream_handle(stream)))
    if rc != GLA_OK:
        raise GlaError(rc, "gla_ttt_linear_fwd")
    return o, ht, hbt


def wy_into(k, v, beta, A, g, w, u, cu_seqlens, N, B, T, H, HV, K, V, chunk, dtype, workspace, stream=None) -> int:
    """Raw call of gla_wy_fwd: tensors (or None) are passed as device pointers, sizes as given.  Returns the
    code."""
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return int(_lib.gla_wy_fwd(_ptr(k), _ptr(v), _ptr(beta), _ptr(A), _ptr(g), _ptr(w), _ptr(u), _ptr(cu_seqlens),
                               int(N), int(B), int(T), int(H), int(HV), int(K), int(V), int(chunk), int(dtype),
                               _ptr(workspace), nbytes, _stream_handle(stream)))


def wy_fwd(k, v, beta, A, g=None, cu_seqlens=None, out_dtype=None, stream=None, workspace=None):
    """WY representation forward of the gated delta rule on the GPU: per chunk of BT = A.shape[-1] rows,
    u = A (v * beta) and w = A (k * beta * 2^g).  k: [B, T, H, K]; v: [B, T, HV, V]; beta: [B, T, HV];
    A: [B, T, HV, BT] (k, v, beta, A: one dtype, fp32 / bf16 / fp16, cuda, contiguous); g: fp32 [B, T, HV]
    (log2 units) or None.  Returns (w [B, T, HV, K], u [B, T, HV, V]) in fp32, or in bf16 when
    ``out_dtype=torch.bfloat16`` with bf16 inputs."""
    B, T, H, K = k.shape
    HV, V, BT = v.shape[2], v.shape[3], A.shape[-1]
    N = B if cu_seqlens is None else cu_seqlens.numel() - 1
    code = {torch.float32: GLA_F32, torch.bfloat16: GLA_BF16, torch.float16: GLA_F16}.get(k.dtype)
    if code is None:
        raise GlaError(GLA_ERR_UNSUPPORTED, f"gla_wy_fwd dtype {k.dtype}")
    odt = torch.float32
    if out_dtype == torch.bfloat16:
        if code != GLA_BF16:
            raise GlaError(GLA_ERR_UNSUPPORTED, "gla_wy_fwd: bf16 outputs need bf16 inputs")
        code, odt = GLA_BF16_OBF16, torch.bfloat16
    for name, t in (("k", k), ("v", v), ("beta", beta), ("A", A)):
        if t.dtype != k.dtype or not t.is_cuda or not t.is_contiguous():
            raise GlaError(GLA_ERR_INVALID_ARG, f"gla_wy_fwd: {name} must be a contiguous cuda tensor of k's dtype")
    if g is not None:
        g = g.contiguous().float()
    w = torch.empty(B, T, HV, K, dtype=odt, device=k.device)
    u = torch.empty(B, T, HV, V, dtype=odt, device=k.device)
    if workspace is None:
        need = int(_lib.gla_wy_workspace_size(T, N, BT, int(cu_seqlens is not None)))
        workspace = get_workspace(max(need, 256), k.device)
    nbytes = workspace.numel() * workspace.element_size()
    rc = int(_lib.gla_wy_fwd(_ptr(k), _ptr(v), _ptr(beta), _ptr(A), _ptr(g), _ptr(w), _ptr(u), _ptr(cu_seqlens), N, B,
                             T, H, HV, K, V, int(BT), code, _ptr(workspace), nbytes, _stream_handle(stream)))
    if rc != GLA_OK:
        raise GlaError(rc, "gla_wy_fwd")
    return w, u


def get_status(workspace, stream=None) -> int:
    return int(_lib.gla_get_status(_ptr(workspace), _stream_handle(stream)))


def chunk_local_cumsum(g, chunk=64, cu_seqlens=None, stream=None):
    B, T, H, K = g.shape
    N = B if cu_seqlens is None else cu_seqlens.numel() - 1
    code = {torch.float32: GLA_F32, torch.bfloat16: GLA_BF16, torch.float16: GLA_F16}.get(g.dtype, GLA_BF16)
    G = torch.empty(B, T, H, K, dtype=torch.float32, device=g.device)
    rc = int(_lib.gla_chunk_local_cumsum(_ptr(g), _ptr(G), _ptr(cu_seqlens), N, B, T, H, K, chunk, code,
                                         _stream_handle(stream)))
    if rc != GLA_OK:
        raise GlaError(rc, "gla_chunk_local_cumsum")
    return G


class KernelTimer:
    """Arms gla_profile_events with CUDA events so each kernel launch of the next gla_fwd calls on this
    thread is bracketed by events on its stream.  ``results()`` (after a synchronize) gives
    [(kernel name, milliseconds)] for the last call."""

    def __init__(self, max_launches=16):
        self.events = [torch.cuda.Event(enable_timing=True) for _ in range(2 * max_launches)]
        for e in self.events:   # torch creates the CUDA event on first record: materialise the handles
            e.record()
        torch.cuda.synchronize()
        handles = [e.cuda_event for e in self.events]
        if not all(handles):
            raise RuntimeError("KernelTimer: could not create CUDA events")
        self._handles = (ctypes.c_void_p * len(self.events))(*handles)
        self._ids = (ctypes.c_int * max_launches)()

    def __enter__(self):
        _lib.gla_profile_events(self._handles, len(self.events), self._ids)
        return self

    def __exit__(self, *exc):
        _lib.gla_profile_events(None, 0, None)

    def results(self):
        n = int(_lib.gla_profile_launches())
        return [(_lib.gla_kernel_name(self._ids[i]).decode(), self.events[2 * i].elapsed_time(self.events[2 * i + 1]))
                for i in range(min(n, len(self.events) // 2))]
