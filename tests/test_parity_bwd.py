"""GPU parity of the backward pass (gla_bwd through the C ABI) against the fp64 backward oracle.

Tolerances (fp32 arithmetic on exactly widened inputs): relative L2 <= 1e-5 for dq, dk, dv and dh0, each a
sum of at most one chunk of intra terms plus a chunk-level scan; dg is a reverse cumulative sum of
(q dq - k dk) over up to T rows, whose rounding grows with T relative to the partial sums: relative L2
<= 1e-4.
"""
import zlib

import numpy as np
import pytest
import torch

import oracle
from chunkwise_gated_linear_chunked_gb300.inputs import make_inputs, stored_numpy
from parity_util import as_f64, errors

pytestmark = pytest.mark.gpu

TOL = {"dq": 1e-5, "dk": 1e-5, "dv": 1e-5, "dh0": 1e-5, "dg": 1e-4}


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _grad_inputs(inp, seed, dht=True):
    g = torch.Generator().manual_seed(seed)
    shape_o = tuple(inp.v.shape)
    do = torch.randn(shape_o, generator=g).to(inp.v.dtype)
    dh = torch.randn(tuple(inp.h0.shape) if inp.h0 is not None else (inp.N, inp.H, inp.K, inp.V),
                     generator=g) * 0.5 if dht else None
    return do, dh


def _run(inp, do, dht):
    from chunkwise_gated_linear_chunked_gb300 import binding
    d = lambda x: None if x is None else x.cuda().contiguous()
    out = binding.gla_bwd(d(inp.q), d(inp.k), d(inp.v), d(inp.g), d(do), scale=inp.scale,
                          initial_state=d(inp.h0), dht=d(dht), cu_seqlens=d(inp.cu_seqlens))
    torch.cuda.synchronize()
    return out


def _oracle(inp, do, dht, heads=None):
    sel = (lambda x: x) if heads is None else (lambda x: x[:, :, heads].contiguous())
    arrs = [stored_numpy(sel(x)) for x in (inp.q, inp.k, inp.v, inp.g, do)]
    st = lambda x: None if x is None else (x.numpy() if heads is None else x[:, heads].contiguous().numpy())
    cu = None if inp.cu_seqlens is None else inp.cu_seqlens.numpy()
    return oracle.gla_bwd(*arrs, inp.scale, h0=st(inp.h0), dht=st(dht), cu_seqlens=cu)


def _check(got, ref):
    for name, x, y in zip(("dq", "dk", "dv", "dg", "dh0"), got, ref):
        rel, mabs = errors(as_f64(x), y)
        assert rel <= TOL[name], f"{name}: rel-L2 {rel:.3e} > {TOL[name]:.0e} (max-abs {mabs:.3e})"


CASES = [
    # dtype, B, T, H, K, V, h0, dht, varlen lengths
    ("f32", 1, 64, 1, 64, 64, False, False, None),
    ("f32", 2, 200, 2, 128, 128, True, True, None),       # ragged last chunk
    ("bf16", 2, 200, 3, 128, 128, True, True, None),
    ("bf16", 1, 1, 2, 64, 128, True, True, None),         # a single row
    ("bf16", 1, 1, 2, 128, 128, True, True, None),        # a single row on the tensor-core path
    ("bf16", 2, 320, 2, 128, 128, False, False, None),    # whole chunks, no initial state or dht
    ("bf16", 1, 33, 1, 128, 128, True, False, None),      # one partial chunk past the anchor row
    ("bf16", 3, 130, 2, 128, 64, False, True, None),
    ("bf16", 1, 700, 2, 64, 64, True, False, None),
    ("bf16", 1, 0, 2, 128, 128, True, True, [1, 63, 64, 65, 0, 130, 300, 2]),   # varlen incl. empty
    ("f32", 1, 0, 1, 64, 64, True, True, [0, 0, 5]),
    ("f16", 2, 200, 2, 128, 128, True, True, None),
    ("f16", 1, 0, 2, 64, 128, True, True, [1, 63, 64, 65, 0, 130]),
]


def _id(c):
    d, B, T, H, K, V, h0, dht, L = c
    return f"{d}-B{B}T{T if L is None else 'var' + str(len(L))}H{H}K{K}V{V}{'-h0' if h0 else ''}{'-dht' if dht else ''}"


@pytest.mark.parametrize("case", CASES, ids=_id)
def test_backward_elementwise(case):
    d, B, T, H, K, V, h0, dht, lengths = case
    seed = zlib.crc32(_id(case).encode()) % 1000
    inp = make_inputs(d, B=B, T=T, H=H, K=K, V=V, h0=h0, lengths=lengths, seed=seed)
    do, dh = _grad_inputs(inp, seed + 1, dht)
    _check(_run(inp, do, dh), _oracle(inp, do, dh))


def test_backward_deterministic_bitwise():
    inp = make_inputs("bf16", B=2, T=300, H=2, K=128, V=128, h0=True, seed=21)
    do, dh = _grad_inputs(inp, 22)
    a, b = _run(inp, do, dh), _run(inp, do, dh)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_backward_large_sampled_heads():
    """B=4 T=2048 H=8 K=V=128 bf16 (the shape of the forward benchmark), heads 0 and 5 against the oracle."""
    inp = make_inputs("bf16", B=4, T=2048, H=8, K=128, V=128, h0=True, seed=23)
    do, dh = _grad_inputs(inp, 24)
    got = _run(inp, do, dh)
    heads = [0, 5]
    ref = _oracle(inp, do, dh, heads=heads)
    sub = [got[0][:, :, heads], got[1][:, :, heads], got[2][:, :, heads], got[3][:, :, heads], got[4][:, heads]]
    _check(sub, ref)
    assert all(torch.isfinite(x).all() for x in got)


V256_CASES = [
    # dtype, B, T, H, K, V, h0, dht, varlen lengths: V = 256 runs as two 128-wide value slices
    ("bf16", 2, 200, 2, 128, 256, True, True, None),                         # tensor-core slices
    ("bf16", 1, 0, 2, 128, 256, True, True, [1, 63, 64, 65, 0, 130, 300, 2]),
    ("f32", 1, 130, 2, 64, 256, False, True, None),                           # CUDA-core slices
]


@pytest.mark.parametrize("case", V256_CASES, ids=_id)
def test_backward_value_width_256(case):
    """dv, dh0 per 128-wide value slice, dq, dk, dg summed over the slices: every element against the oracle."""
    d, B, T, H, K, V, h0, dht, lengths = case
    inp = make_inputs(d, B=B, T=T, H=H, K=K, V=V, h0=h0, lengths=lengths, seed=zlib.crc32(_id(case).encode()) % 1000)
    do, dh = _grad_inputs(inp, zlib.crc32(_id(case).encode()) % 1000 + 1, dht=dht)
    _check(_run(inp, do, dh), _oracle(inp, do, dh))


def test_backward_rejects_unsupported_value_width():
    from chunkwise_gated_linear_chunked_gb300 import binding
    inp = make_inputs("bf16", B=1, T=64, H=1, K=128, V=64, h0=False, seed=25)
    do, _ = _grad_inputs(inp, 26, dht=False)
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    d = lambda x: x.cuda().contiguous()
    f32 = dict(dtype=torch.float32, device="cuda")
    out = [torch.empty(1, 64, 1, 512, **f32) for _ in range(4)]
    rc = binding.bwd_into(d(inp.q), d(inp.k), d(torch.zeros(1, 64, 1, 512, dtype=torch.bfloat16)), d(inp.g),
                          d(torch.zeros(1, 64, 1, 512, dtype=torch.bfloat16)), inp.scale, None, None, out[0], out[1],
                          out[2], out[3], None, None, 1, 1, 64, 1, 128, 512, 64, binding.GLA_BF16, ws)
    assert rc == binding.GLA_ERR_UNSUPPORTED


@pytest.mark.parametrize("d,K,V", [("bf16", 128, 128), ("f32", 64, 128)])
def test_backward_head_first(d, K, V):
    """[B, H, T, *] tensors: gradients are the head-first permutation of the time-major ones."""
    from chunkwise_gated_linear_chunked_gb300 import binding
    inp = make_inputs(d, B=2, T=200, H=2, K=K, V=V, h0=True, seed=27)
    do, dh = _grad_inputs(inp, 28)
    hf = lambda x: x.transpose(1, 2).contiguous().cuda()
    got = binding.gla_bwd(hf(inp.q), hf(inp.k), hf(inp.v), hf(inp.g), hf(do), scale=inp.scale,
                          initial_state=inp.h0.cuda(), dht=dh.cuda(), head_first=True)
    torch.cuda.synchronize()
    got = [x.transpose(1, 2) for x in got[:4]] + [got[4]]
    _check(got, _oracle(inp, do, dh))


@pytest.mark.parametrize("d,K,V", [("bf16", 128, 128), ("f32", 64, 128)])
def test_backward_head_first_varlen(d, K, V):
    """A packed varlen batch in [1, H, T, *]: gradients are the head-first permutation of the time-major ones."""
    from chunkwise_gated_linear_chunked_gb300 import binding
    inp = make_inputs(d, B=1, T=0, H=2, K=K, V=V, h0=True, lengths=[1, 63, 64, 65, 0, 130, 300, 2], seed=33)
    do, dh = _grad_inputs(inp, 34)
    hf = lambda x: x.transpose(1, 2).contiguous().cuda()
    got = binding.gla_bwd(hf(inp.q), hf(inp.k), hf(inp.v), hf(inp.g), hf(do), scale=inp.scale,
                          initial_state=inp.h0.cuda(), dht=dh.cuda(), cu_seqlens=inp.cu_seqlens.cuda(),
                          head_first=True)
    torch.cuda.synchronize()
    got = [x.transpose(1, 2) for x in got[:4]] + [got[4]]
    _check(got, _oracle(inp, do, dh))


@pytest.mark.parametrize("d", ["bf16", "f16"])
def test_backward_fp32_gate(d):
    import dataclasses
    inp = make_inputs(d, B=2, T=200, H=2, K=128, V=128, h0=True, seed=29)
    gen = torch.Generator().manual_seed(30)
    inp = dataclasses.replace(inp, g=torch.nn.functional.logsigmoid(torch.randn(tuple(inp.g.shape), generator=gen)) / 16)
    do, dh = _grad_inputs(inp, 31)
    _check(_run(inp, do, dh), _oracle(inp, do, dh))
