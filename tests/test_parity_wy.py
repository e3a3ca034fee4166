"""GPU parity of the WY-representation forward of the gated delta rule (gla_wy_fwd through the C ABI)
against its fp64 oracle.

Tolerance: fp32 outputs rel-L2 <= 1e-5 (inputs are exact in both; each output is one fp32 sum of at most
64 products; the tensor-core kernel splits each fp32 operand into three bf16 terms, exact to fp32 rounding);
bf16 outputs rel-L2 <= 5e-3 and max-abs <= 2e-2 (one bf16 rounding of values of order 1).
"""
import zlib

import numpy as np
import pytest
import torch

import oracle
from chunkwise_gated_linear_chunked_gb300.inputs import make_wy_inputs, stored_numpy, wy_workload_inputs
from parity_util import as_f64, errors

pytestmark = pytest.mark.gpu
TOL_F32 = 1e-5
TOL_BF16 = (5e-3, 2e-2)


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def run_both(x, out_bf16=False):
    from chunkwise_gated_linear_chunked_gb300 import binding
    dev = lambda t: None if t is None else t.cuda()
    cu = dev(x.cu_seqlens)
    w, u = binding.wy_fwd(dev(x.k), dev(x.v), dev(x.beta), dev(x.A), dev(x.g), cu_seqlens=cu,
                          out_dtype=torch.bfloat16 if out_bf16 else None)
    torch.cuda.synchronize()
    ref = oracle.wy_fwd(*(stored_numpy(t) for t in (x.k, x.v, x.beta, x.A)),
                        None if x.g is None else x.g.double().numpy(),
                        cu_seqlens=None if x.cu_seqlens is None else x.cu_seqlens.numpy())
    return (w, u), ref


def check(got, ref, out_bf16):
    for name, a, b in zip(("w", "u"), got, ref):
        rel, mabs = errors(as_f64(a), b)
        if out_bf16:
            assert rel <= TOL_BF16[0] and mabs <= TOL_BF16[1], f"{name}: rel-L2 {rel:.3e} max-abs {mabs:.3e}"
        else:
            assert rel <= TOL_F32, f"{name}: rel-L2 {rel:.3e} (max-abs {mabs:.3e})"


CASES = [
    # dtype, B, T, H, HV, K, V, BT, gate, lengths, bf16 outputs
    ("f32", 2, 150, 1, 1, 64, 64, 64, True, None, False),                          # ragged last chunk
    ("bf16", 1, 200, 2, 4, 128, 128, 64, True, None, False),                       # shared key heads
    ("f16", 2, 77, 1, 1, 64, 128, 16, False, None, False),                         # no gate, K != V
    ("bf16", 1, 0, 1, 2, 128, 64, 32, True, [1, 31, 32, 33, 0, 130, 7], False),    # varlen incl. empty
    ("bf16", 1, 96, 1, 1, 128, 128, 64, True, None, True),                         # bf16 outputs
    ("f32", 1, 1, 1, 1, 128, 128, 64, True, None, False),                          # a single row
    # bf16 with K == V: the tensor-core kernel (the cases above with bf16 and K == V also take it)
    ("bf16", 2, 77, 1, 1, 64, 64, 16, True, None, False),                          # chunk 16, one block
    ("bf16", 1, 0, 2, 2, 128, 128, 32, True, [5, 32, 0, 70, 1], False),            # chunk 32, varlen
    ("bf16", 3, 100, 1, 3, 128, 128, 64, False, None, True),                       # no gate, bf16 outputs
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}-B{c[1]}T{c[2]}H{c[3]}HV{c[4]}K{c[5]}V{c[6]}-bt{c[7]}")
def test_wy_forward(case):
    d, B, T, H, HV, K, V, BT, gate, lengths, obf = case
    x = make_wy_inputs(d, B=B, T=T, H=H, HV=HV, K=K, V=V, BT=BT, gate=gate, lengths=lengths,
                       seed=zlib.crc32(repr(case).encode()) % 1000)
    got, ref = run_both(x, obf)
    check(got, ref, obf)


def test_wy_full_size_b4_t2k_h8():
    """The benchmark's WY workload (bf16, B=4, T=2048, H=HV=8, K=V=128, chunk 64) in the bench's launch, whole."""
    x = wy_workload_inputs("b4_t2k_h8")
    got, ref = run_both(x)
    check(got, ref, False)


def test_wy_is_deterministic():
    from chunkwise_gated_linear_chunked_gb300 import binding
    x = make_wy_inputs("bf16", B=2, T=300, H=2, HV=2, K=128, V=128, BT=64, seed=3)
    args = [t.cuda() for t in (x.k, x.v, x.beta, x.A, x.g)]
    a = binding.wy_fwd(*args)
    b = binding.wy_fwd(*args)
    assert all(torch.equal(p, q) for p, q in zip(a, b))


def test_wy_bad_offsets_are_reported_and_nothing_is_written():
    from chunkwise_gated_linear_chunked_gb300 import binding
    x = make_wy_inputs("f32", B=1, T=40, H=1, HV=1, K=64, V=64, BT=16, seed=4)
    cu = torch.tensor([0, 30, 20, 40], dtype=torch.int32).cuda()   # decreasing: invalid
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    w, u = binding.wy_fwd(*(t.cuda() for t in (x.k, x.v, x.beta, x.A, x.g)), cu_seqlens=cu, workspace=ws)
    assert binding.get_status(ws) == binding.GLA_ERR_INVALID_ARG
