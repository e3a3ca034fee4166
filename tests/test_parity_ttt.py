"""GPU parity of the TTT-linear forward (gla_ttt_linear_fwd through the C ABI) against its fp64 oracle.

Tolerance: relative L2 <= 1e-4 for o, ht and hbt.  The inner model is updated by a serial fp32 recurrence over
T / chunk mini-batches, each accumulating over D terms and one LayerNorm, so rounding grows with the number of
steps; the shape cases (<= 520 rows, <= 33 steps) and the benchmark's full workload (2048 rows, 128 steps per
head) stay inside that bound.
"""
import zlib

import numpy as np
import pytest
import torch

import oracle
from chunkwise_gated_linear_chunked_gb300.inputs import stored_numpy
from parity_util import as_f64, errors

pytestmark = pytest.mark.gpu
TOL = 1e-4
TORCH = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def make_ttt(dtype, B, T, H, D, h0, lengths, seed):
    g = torch.Generator().manual_seed(seed)
    cu = None
    if lengths is not None:
        B, T = 1, sum(lengths)
        cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32)
    N = B if cu is None else len(lengths)
    q, k, v = (torch.randn(B, T, H, D, generator=g).to(TORCH[dtype]) for _ in range(3))
    w = 1.0 + 0.2 * torch.randn(H, D, generator=g)
    b = 0.1 * torch.randn(H, D, generator=g)
    eta = 0.02 + 0.05 * torch.rand(B, T, H, generator=g)
    s0 = 0.1 * torch.randn(N, H, D, D, generator=g) if h0 else None
    sb0 = 0.1 * torch.randn(N, H, D, generator=g) if h0 else None
    return q, k, v, w, b, eta, s0, sb0, cu


CASES = [
    ("f32", 1, 64, 1, 64, True, None, 16),
    ("f32", 2, 200, 2, 128, True, None, 16),      # ragged last mini-batch
    ("bf16", 2, 130, 2, 128, False, None, 32),
    ("f16", 1, 97, 3, 64, True, None, 16),
    ("bf16", 1, 0, 2, 64, True, [1, 15, 16, 17, 0, 130, 300], 16),   # varlen incl. empty
    # bf16 with D = 128: the tensor-core kernel
    ("bf16", 2, 200, 2, 128, True, None, 16),     # ragged last mini-batch
    ("bf16", 1, 0, 2, 128, True, [1, 15, 16, 17, 0, 130, 300], 16),
    ("bf16", 1, 0, 1, 128, False, [33, 64, 7], 32),
    # the tensor-core kernel's pipeline edges: sequences of one, two and three mini-batches (whole and
    # ragged), at both mini-batch sizes, a dense batch with a ragged tail, and a pack of many short and
    # empty sequences (each CTA then runs at most a few mini-batches)
    ("bf16", 1, 0, 2, 128, True, [16, 32, 48, 1, 2, 3, 31, 33, 47, 49], 16),
    ("bf16", 1, 0, 1, 128, True, [32, 64, 96, 1, 65, 97], 32),
    ("bf16", 3, 50, 4, 128, False, None, 16),
    ("bf16", 1, 0, 2, 128, True, [5] * 40 + [0] * 5 + [16] * 10, 16),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}-B{c[1]}T{c[2]}H{c[3]}D{c[4]}-bt{c[7]}")
def test_ttt_linear_forward(case):
    from chunkwise_gated_linear_chunked_gb300 import binding
    d, B, T, H, D, h0, lengths, chunk = case
    q, k, v, w, b, eta, s0, sb0, cu = make_ttt(d, B, T, H, D, h0, lengths, zlib.crc32(repr(case).encode()) % 1000)
    scale = D ** -0.5
    dev = lambda x: None if x is None else x.cuda()
    o, ht, hbt = binding.ttt_linear_fwd(dev(q), dev(k), dev(v), dev(w), dev(b), dev(eta), scale=scale, eps=1e-6,
                                        chunk=chunk, initial_state=dev(s0), initial_state_bias=dev(sb0),
                                        cu_seqlens=dev(cu))
    torch.cuda.synchronize()
    ref = oracle.ttt_linear_fwd(*(stored_numpy(x) for x in (q, k, v)), w.numpy(), b.numpy(), eta.numpy(), scale,
                                1e-6, chunk, h0=None if s0 is None else s0.numpy(),
                                hb0=None if sb0 is None else sb0.numpy(),
                                cu_seqlens=None if cu is None else cu.numpy())
    for name, x, y in zip(("o", "ht", "hbt"), (o, ht, hbt), ref):
        rel, mabs = errors(as_f64(x), y)
        assert rel <= TOL, f"{name}: rel-L2 {rel:.3e} (max-abs {mabs:.3e})"


def test_ttt_tensor_core_kernel_runs_for_bf16_d128():
    """bf16 q, k, v with D = 128 take the tensor-core kernel (the launch hook names the kernel that ran)."""
    from chunkwise_gated_linear_chunked_gb300 import binding
    q, k, v, w, b, eta, s0, sb0, _ = make_ttt("bf16", 1, 64, 1, 128, True, None, 5)
    timer = binding.KernelTimer()
    with timer:
        binding.ttt_linear_fwd(q.cuda(), k.cuda(), v.cuda(), w.cuda(), b.cuda(), eta.cuda(), chunk=16,
                               initial_state=s0.cuda(), initial_state_bias=sb0.cuda())
    torch.cuda.synchronize()
    assert [n for n, _ in timer.results()] == ["ttt_linear_tc"]


@pytest.mark.parametrize("chunk", [16, 32])
def test_ttt_tensor_core_kernel_is_deterministic(chunk):
    """Repeated calls give bitwise-equal o, ht, hbt: every reduction has a fixed order and the issuing threads'
    products land in their own accumulators, so no result depends on how the roles happen to interleave."""
    from chunkwise_gated_linear_chunked_gb300 import binding
    q, k, v, w, b, eta, s0, sb0, cu = make_ttt("bf16", 1, 0, 4, 128, True, [700, 33, 1, 512, 96], 11 + chunk)
    args = [x.cuda() for x in (q, k, v, w, b, eta)]
    outs = []
    for _ in range(3):
        o, ht, hbt = binding.ttt_linear_fwd(*args, chunk=chunk, initial_state=s0.cuda(),
                                            initial_state_bias=sb0.cuda(), cu_seqlens=cu.cuda())
        torch.cuda.synchronize()
        outs.append([x.cpu() for x in (o, ht, hbt)])
    for other in outs[1:]:
        for x, y in zip(outs[0], other):
            assert torch.equal(x, y)


def test_ttt_bad_offsets_are_reported_not_faulted():
    from chunkwise_gated_linear_chunked_gb300 import binding
    q, k, v, w, b, eta, *_ = make_ttt("f32", 1, 40, 1, 64, False, None, 1)
    cu = torch.tensor([0, 30, 20, 40], dtype=torch.int32).cuda()   # decreasing: invalid
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    binding.ttt_linear_fwd(q.cuda(), k.cuda(), v.cuda(), w.cuda(), b.cuda(), eta.cuda(), cu_seqlens=cu, workspace=ws)
    assert binding.get_status(ws) == binding.GLA_ERR_INVALID_ARG


def test_ttt_full_size_b4_t2k_h8():
    """The benchmark's TTT-linear workload (bf16 q, k, v of B=4, T=2048, H=8, D=128; mini-batch 16: 128 serial
    gradient steps per head) in the bench's launch, whole tensors against the oracle."""
    from chunkwise_gated_linear_chunked_gb300 import binding
    from chunkwise_gated_linear_chunked_gb300.inputs import WORKLOADS, workload_inputs
    inp = workload_inputs("b4_t2k_h8")
    gen = torch.Generator().manual_seed(WORKLOADS["b4_t2k_h8"].seed + 11)   # the bench's draw
    w = 1.0 + 0.2 * torch.randn(inp.H, inp.K, generator=gen)
    b = 0.1 * torch.randn(inp.H, inp.K, generator=gen)
    eta = 0.02 + 0.05 * torch.rand(tuple(inp.q.shape[:3]), generator=gen)
    scale = inp.K ** -0.5
    o, ht, hbt = binding.ttt_linear_fwd(inp.q.cuda(), inp.k.cuda(), inp.v.cuda(), w.cuda(), b.cuda(), eta.cuda(),
                                        scale=scale, eps=1e-6, chunk=16)
    torch.cuda.synchronize()
    ref = oracle.ttt_linear_fwd(*(stored_numpy(x) for x in (inp.q, inp.k, inp.v)), w.numpy(), b.numpy(),
                                eta.numpy(), scale, 1e-6, 16)
    for name, x, y in zip(("o", "ht", "hbt"), (o, ht, hbt), ref):
        rel, mabs = errors(as_f64(x), y)
        assert rel <= TOL, f"{name}: rel-L2 {rel:.3e} (max-abs {mabs:.3e})"
