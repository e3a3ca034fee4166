"""gla_fwd_noalloc: the entry point for callers that cannot allocate device memory (their runtime owns all
device memory, or the call path must never hit cudaMalloc).  It must give the same results as gla_fwd with
a caller-provided workspace and match the oracle, also when called twice in a row and right after other
problems (the shared scratch keeps the previous call's contents), on the tensor-core and the CUDA-core
kernels, and must reject problems whose scratch would not fit its fixed 32 MiB array.

This file is named to be collected last, so a stop-at-first-failure run has already run everything else.
"""
import ctypes

import pytest
import torch

from chunkwise_gated_linear_chunked_gb300.inputs import make_inputs
from parity_util import TOL, as_f64, assert_close, run_oracle, to_device

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
    code = binding.GLA_F32 if inp.dtype == "f32" else binding.GLA_BF16
    return f(ptr(q), ptr(k), ptr(v), ptr(g), ptr(o), inp.scale, ptr(h0), ptr(ht), ptr(cu), inp.N, B, T, inp.H,
             inp.K, inp.V, inp.chunk, code, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


CASES = [
    # long single sequences with few heads: split into segments, so the state pass and the scan use the
    # scratch for per-segment states
    ("bf16", dict(B=1, T=3000, H=2, K=128, V=128, h0=True, seed=21)),
    # varlen: the slot table lives in the scratch too
    ("bf16", dict(B=1, T=0, H=2, K=128, V=256, h0=True, lengths=[700, 5, 2100, 64], seed=22)),
    # fp32 with K = 64: the CUDA-core kernels, whose state pass and segment scan keep per-segment states in
    # the scratch; it runs after the larger calls above, on the scratch they left behind
    ("f32", dict(B=1, T=5000, H=1, K=64, V=128, h0=True, seed=23)),
]


def test_noalloc_matches_gla_fwd_and_the_oracle_on_two_calls_in_a_row(gla):
    binding, _ = gla
    for dtype, case in CASES:
        inp = make_inputs(dtype, **case)
        q, k, v, g, h0, cu = to_device(inp)
        # gla_fwd with a workspace of its own, zeroed for this call
        B, T = inp.q.shape[0], inp.q.shape[1]
        code = binding.GLA_F32 if dtype == "f32" else binding.GLA_BF16
        nbytes = binding.workspace_size(B, T, inp.H, inp.K, inp.V, inp.N, inp.chunk, code)
        assert 256 < nbytes <= SCRATCH_BYTES
        fresh = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
        o_ref, ht_ref = binding.gla_fwd(q, k, v, g, scale=inp.scale, initial_state=h0, cu_seqlens=cu,
                                        workspace=fresh)
        o_or, ht_or = run_oracle(inp)
        for _ in range(2):
            o = torch.full_like(o_ref, float("nan"))
            ht = torch.full_like(ht_ref, float("nan"))
            assert _noalloc(gla, inp, o, ht, q, k, v, g, h0, cu) == binding.GLA_OK
            torch.cuda.synchronize()
            assert_close(as_f64(o), as_f64(o_ref), TOL[dtype], "o vs gla_fwd")
            assert_close(as_f64(ht), as_f64(ht_ref), TOL[dtype], "ht vs gla_fwd")
            assert_close(as_f64(o), o_or, TOL[dtype], "o vs oracle")
            assert_close(as_f64(ht), ht_or, TOL[dtype], "ht vs oracle")


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
