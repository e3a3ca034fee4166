"""gla_fwd_noalloc: the entry point for callers that cannot allocate device memory (their runtime owns all
device memory, or the call path must never hit cudaMalloc).  It must give the same results as gla_fwd with
a caller-provided workspace, also when called twice in a row (the shared scratch keeps the previous call's
contents), and must reject problems whose scratch would not fit its fixed 32 MiB array.

This file is named to be collected last, so a stop-at-first-failure run has already run everything else.
"""
import ctypes

import pytest
import torch

from chunkwise_gated_linear_chunked_gb300.inputs import make_inputs
from parity_util import TOL, as_f64, assert_close, to_device

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 32 << 20


@pytest.fixture(scope="module")
def gla():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from chunkwise_gated_linear_chunked_gb300 import build
    build.build()
    from chunkwise_gated_linear_chunked_gb300 import binding
    f = binding.lib().gla_fwd_noalloc
    p, i = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [p, p, p, p, p, ctypes.c_float, p, p, p, i, i, i, i, i, i, i, i, p]
    f.restype = i
    return binding, f


def _noalloc(gla, inp, o, ht, q, k, v, g, h0, cu):
    binding, f = gla
    ptr = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    B, T = inp.q.shape[0], inp.q.shape[1]
    return f(ptr(q), ptr(k), ptr(v), ptr(g), ptr(o), inp.scale, ptr(h0), ptr(ht), ptr(cu), inp.N, B, T, inp.H,
             inp.K, inp.V, inp.chunk, binding.GLA_BF16,
             ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


CASES = [
    # long single sequences with few heads: split into segments, so the state pass and the scan use the
    # scratch for per-segment states
    dict(B=1, T=3000, H=2, K=128, V=128, h0=True, seed=21),
    # varlen: the slot table lives in the scratch too
    dict(B=1, T=0, H=2, K=128, V=256, h0=True, lengths=[700, 5, 2100, 64], seed=22),
]


def test_noalloc_matches_gla_fwd_on_two_calls_in_a_row(gla):
    binding, _ = gla
    for case in CASES:
        inp = make_inputs("bf16", **case)
        q, k, v, g, h0, cu = to_device(inp)
        o_ref, ht_ref = binding.gla_fwd(q, k, v, g, scale=inp.scale, initial_state=h0, cu_seqlens=cu)
        B, T = inp.q.shape[0], inp.q.shape[1]
        assert 256 < binding.workspace_size(B, T, inp.H, inp.K, inp.V, inp.N) <= SCRATCH_BYTES
        for _ in range(2):
            o = torch.full_like(o_ref, float("nan"))
            ht = torch.full_like(ht_ref, float("nan"))
            assert _noalloc(gla, inp, o, ht, q, k, v, g, h0, cu) == binding.GLA_OK
            torch.cuda.synchronize()
            assert_close(as_f64(o), as_f64(o_ref), TOL["bf16"], "o")
            assert_close(as_f64(ht), as_f64(ht_ref), TOL["bf16"], "ht")


def test_noalloc_rejects_problems_beyond_its_scratch(gla):
    binding, f = gla
    # a varlen pack of many short sequences with one head: every sequence is split into segments, whose
    # states need more than the fixed scratch.  The call must return before enqueuing anything, so the
    # (fake, far apart) pointers are never used.
    shape = None
    for N in (120, 130, 140):
        for T in (N * 256, N * 512):
            if binding.workspace_size(1, T, 1, 128, 256, N) > SCRATCH_BYTES:
                shape = (N, T)
                break
        if shape:
            break
    assert shape is not None
    N, T = shape
    fake = lambda x: ctypes.c_void_p(x << 30)
    rc = f(fake(1), fake(2), fake(3), fake(4), fake(5), 0.1, None, None, fake(6), N, 1, T, 1, 128, 256, 64,
           binding.GLA_BF16, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == binding.GLA_ERR_WORKSPACE
