"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the same seeded inputs.

Small cases compare every element and span several chunks, segments and ragged tails; the full-size
benchmark workloads run in the benchmark's launch configuration and compare every output of every head,
the oracle computing a few heads at a time.
"""
import os
import zlib

import numpy as np
import pytest
import torch

from chunkwise_gated_linear_chunked_gb300.inputs import WORKLOADS, make_inputs, workload_inputs
from parity_util import TOL, TOL_OBF16, as_f64, assert_close, errors, run_gpu, run_oracle, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from chunkwise_gated_linear_chunked_gb300 import build
    build.build()


SMALL = [
    # (dtype, B, T, H, K, V, h0, lengths)
    ("f32", 1, 256, 2, 64, 64, False, None),          # the fp32 workload itself
    ("f32", 2, 200, 3, 128, 128, True, None),         # ragged last chunk (200 = 3*64 + 8)
    ("bf16", 2, 200, 3, 128, 128, True, None),
    ("bf16", 3, 130, 2, 64, 256, True, None),
    ("bf16", 1, 1, 2, 128, 64, True, None),           # a single row
    ("bf16", 1, 64, 1, 128, 128, False, None),        # exactly one chunk
    ("bf16", 1, 3000, 1, 128, 128, True, None),       # one head, long: split into segments + scan
    ("f32", 1, 5000, 1, 64, 128, True, None),
    ("bf16", 1, 0, 2, 64, 64, True, [1, 63, 64, 65, 0, 130, 300, 2]),   # varlen incl. an empty sequence
    ("bf16", 1, 0, 1, 128, 128, True, [3000, 7, 1500]),                  # varlen with segments
    ("f32", 1, 0, 2, 64, 64, False, [0, 0, 5]),
    ("f16", 2, 200, 3, 128, 128, True, None),         # fp16 inputs: tensor-core path
    ("f16", 1, 3000, 1, 128, 256, True, None),        # fp16, segments + scan, V = 256
    ("f16", 2, 130, 2, 64, 64, True, None),           # fp16 on the CUDA-core path
    ("f16", 1, 0, 2, 128, 128, True, [1, 63, 64, 65, 0, 130, 300, 2]),
]


def _case_id(c):
    d, B, T, H, K, V, h0, L = c
    return f"{d}-B{B}T{T if L is None else 'var' + str(len(L))}H{H}K{K}V{V}{'-h0' if h0 else ''}"


@pytest.mark.parametrize("case", SMALL, ids=_case_id)
def test_small_cases_elementwise(case):
    d, B, T, H, K, V, h0, lengths = case
    inp = make_inputs(d, B=B, T=T, H=H, K=K, V=V, h0=h0, lengths=lengths, seed=zlib.crc32(_case_id(case).encode()) % 1000)
    o, ht = run_gpu(inp)
    o_ref, ht_ref = run_oracle(inp)
    assert_close(as_f64(o), o_ref, TOL[d], "o")
    assert_close(as_f64(ht), ht_ref, TOL[d], "ht")


# Start-state scan of the tensor-core path.  On a 152-SM GB300 the planner cuts dense batches whose
# (sequence, head) items leave SMs idle into the fewest segments that fill one wave (16 heads of 4608 rows:
# 9 segments of 512 rows; 40 heads of 4096 rows: 3 segments; one head of 40000 rows: 125 segments), so
# segments are grouped in blocks of 8 and each block starts from the end state published by the block
# before.  Varlen packs are cut into segments of at most 2048 rows; 20 sequences of 4000 rows with 8 heads
# give 320 items, more than one wave, which use blocks of 2.  Every head is compared with the oracle.
# A varlen pack of 40 sequences (lengths 0 .. 2099, including empty and single-row ones).
MANY_LENGTHS = [(i * 677) % 2100 if i % 9 else (i // 9) % 3 for i in range(40)]
SCAN_CASES = [
    ("bf16", 1, 4608, 16, 128, 128, True, None),
    ("bf16", 1, 4096, 40, 128, 128, True, None),
    ("bf16", 2, 2560, 12, 128, 128, False, None),
    ("bf16", 1, 40000, 1, 128, 128, True, None),     # one head: ~125 segments in one wave, 15 block hops
    ("bf16", 1, 0, 2, 128, 128, True, MANY_LENGTHS),
    ("bf16", 1, 0, 1, 128, 256, False, MANY_LENGTHS),
    ("bf16", 1, 0, 8, 128, 128, True, [4000] * 20),   # several waves of items: scan blocks of 2
]


@pytest.mark.parametrize("case", SCAN_CASES, ids=_case_id)
def test_segment_scan_all_heads(case):
    d, B, T, H, K, V, h0, lengths = case
    inp = make_inputs(d, B=B, T=T, H=H, K=K, V=V, h0=h0, lengths=lengths, seed=zlib.crc32(_case_id(case).encode()) % 1000)
    o, ht = run_gpu(inp)
    o_ref, ht_ref = run_oracle(inp)
    assert_close(as_f64(o), o_ref, TOL[d], "o")
    assert_close(as_f64(ht), ht_ref, TOL[d], "ht")


# Balanced pieces of the tensor-core path: on a 152-SM GB300, dense batches whose (sequence, head) units do
# not divide the CTAs evenly, with long enough pieces, are cut into 152 / NV near-equal pieces of the units'
# chunks taken in order; a piece that crosses from one unit into the next runs the next unit's first
# segment, then the previous unit's last.  40 heads of 4096 rows: 5 segments per head at most, 40 pieces
# crossing a head boundary; 33 heads of 5000 rows (ragged last chunk); 3 sequences of 13 heads (pieces
# crossing sequence boundaries); 20 heads with V = 256 (76 pieces per value tile).
PIECE_CASES = [
    ("bf16", 1, 4096, 40, 128, 128, False, None),
    ("bf16", 1, 5000, 33, 128, 128, True, None),
    ("bf16", 3, 4096, 13, 128, 128, True, None),
    ("bf16", 1, 8192, 20, 128, 256, True, None),
    ("f16", 1, 5000, 33, 128, 128, True, None),
]


@pytest.mark.parametrize("case", PIECE_CASES, ids=_case_id)
def test_balanced_pieces_all_heads(case):
    d, B, T, H, K, V, h0, lengths = case
    inp = make_inputs(d, B=B, T=T, H=H, K=K, V=V, h0=h0, lengths=lengths, seed=zlib.crc32(_case_id(case).encode()) % 1000)
    o, ht = run_gpu(inp)
    o_ref, ht_ref = run_oracle(inp)
    assert_close(as_f64(o), o_ref, TOL[d], "o")
    assert_close(as_f64(ht), ht_ref, TOL[d], "ht")
    o2, ht2 = run_gpu(inp)   # the result does not depend on which CTA took which piece
    assert torch.equal(o, o2) and torch.equal(ht, ht2)


@pytest.mark.parametrize("chunk", [16, 32, 128])
def test_chunk_argument_selects_same_tiling(chunk):
    """chunk is accepted as 16, 32, 64 or 128; the kernels tile at 64 rows, so the result is the same."""
    from chunkwise_gated_linear_chunked_gb300 import binding
    inp = make_inputs("bf16", B=1, T=300, H=2, K=128, V=128, h0=True, seed=31)
    q, k, v, g, h0, _ = to_device(inp)
    o64, ht64 = binding.gla_fwd(q, k, v, g, scale=inp.scale, initial_state=h0, chunk=64)
    o, ht = binding.gla_fwd(q, k, v, g, scale=inp.scale, initial_state=h0, chunk=chunk)
    torch.cuda.synchronize()
    assert torch.equal(o, o64) and torch.equal(ht, ht64)


def test_bf16_output_variant():
    inp = make_inputs("bf16", B=2, T=300, H=2, K=128, V=128, h0=True, seed=3)
    o, ht = run_gpu(inp, out_dtype=torch.bfloat16)
    assert o.dtype == torch.bfloat16
    o_ref, ht_ref = run_oracle(inp)
    assert_close(as_f64(o), o_ref, TOL_OBF16, "o(bf16)")
    assert_close(as_f64(ht), ht_ref, TOL["bf16"], "ht")


def test_empty_batch_rows_give_initial_state():
    inp = make_inputs("bf16", B=2, T=0, H=2, K=64, V=128, h0=True, seed=4)
    o, ht = run_gpu(inp)
    assert o.numel() == 0
    assert torch.equal(ht.cpu(), inp.h0)


def test_deterministic_bitwise():
    inp = make_inputs("bf16", B=1, T=2500, H=2, K=128, V=128, h0=True, seed=5)
    o1, h1 = run_gpu(inp)
    o2, h2 = run_gpu(inp)
    assert torch.equal(o1, o2) and torch.equal(h1, h2)


def test_in_place_state_streaming():
    """h0 == ht (same buffer): two halves fed through one state buffer equal the full run."""
    from chunkwise_gated_linear_chunked_gb300 import binding
    inp = make_inputs("bf16", B=2, T=1000, H=2, K=128, V=128, h0=True, seed=6)
    q, k, v, g, h0, _ = to_device(inp)
    state = h0.clone()
    outs = []
    for a, b in ((0, 437), (437, 1000)):
        sl = lambda x: x[:, a:b].contiguous()
        o = torch.empty(2, b - a, 2, 128, device="cuda")
        ws = binding.get_workspace(binding.workspace_size(2, b - a, 2, 128, 128, 2), "cuda")
        rc = binding.fwd_into(sl(q), sl(k), sl(v), sl(g), o, inp.scale, state, state, None, 2, 2, b - a, 2,
                              128, 128, 64, binding.GLA_BF16, ws)
        assert rc == 0
        outs.append(o)
    torch.cuda.synchronize()
    o_ref, ht_ref = run_oracle(inp)
    assert_close(as_f64(torch.cat(outs, 1)), o_ref, TOL["bf16"], "o")
    assert_close(as_f64(state), ht_ref, TOL["bf16"], "ht")


def test_device_side_cu_seqlens_validation():
    """Offsets that do not end at T are caught on the device: status INVALID_ARG, o left untouched."""
    from chunkwise_gated_linear_chunked_gb300 import binding
    inp = make_inputs("bf16", B=1, T=0, H=1, K=64, V=64, lengths=[10, 20], seed=7)
    q, k, v, g, _, _ = to_device(inp)
    bad = torch.tensor([0, 10, 25], dtype=torch.int32, device="cuda")   # T is 30
    o = torch.full((1, 30, 1, 64), 7.0, device="cuda")
    ws = torch.zeros(binding.workspace_size(1, 30, 1, 64, 64, 2), dtype=torch.uint8, device="cuda")
    rc = binding.fwd_into(q, k, v, g, o, inp.scale, None, None, bad, 2, 1, 30, 1, 64, 64, 64,
                          binding.GLA_BF16, ws)
    assert rc == 0
    assert binding.get_status(ws) == binding.GLA_ERR_INVALID_ARG
    assert binding.get_status(ws) == binding.GLA_OK          # the status word is sticky until read
    assert torch.all(o == 7.0)
    good = inp.cu_seqlens.cuda()
    rc = binding.fwd_into(q, k, v, g, o, inp.scale, None, None, good, 2, 1, 30, 1, 64, 64, 64,
                          binding.GLA_BF16, ws)
    assert rc == 0 and binding.get_status(ws) == binding.GLA_OK


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("chunk", [16, 64, 128])
def test_chunk_local_cumsum_kernel(dtype, chunk):
    import oracle
    from chunkwise_gated_linear_chunked_gb300 import binding
    from chunkwise_gated_linear_chunked_gb300.inputs import stored_numpy
    for lengths, B, T in ((None, 2, 333), ([5, 0, 64, 200, 1], 1, 0)):
        inp = make_inputs(dtype, B=B, T=T, H=3, K=64, V=64, lengths=lengths, seed=8)
        cu = None if inp.cu_seqlens is None else inp.cu_seqlens.cuda()
        G = binding.chunk_local_cumsum(inp.g.cuda(), chunk=chunk, cu_seqlens=cu)
        ref = oracle.chunk_local_cumsum(stored_numpy(inp.g), chunk,
                                        None if cu is None else inp.cu_seqlens.numpy())
        # fp32 running sums of at most `chunk` terms of magnitude <= ~0.5
        np.testing.assert_allclose(as_f64(G), ref, rtol=0, atol=2e-6 * chunk)


# --------------------------------------------------------------------------------------------------
# Full-size benchmark workloads (the configuration bench.py times), every head
# --------------------------------------------------------------------------------------------------

@pytest.mark.parametrize("name", list(WORKLOADS))
def test_full_size_workload_all_heads(name):
    """Every output of the benchmark workload against the oracle; the oracle runs a few heads (all sequences
    of them) at a time to bound host memory, and each group must meet the bounds on its own."""
    w = WORKLOADS[name]
    inp = workload_inputs(name)
    o, ht = run_gpu(inp)
    assert torch.isfinite(o).all() and torch.isfinite(ht).all()
    # enough (sequence, head) pairs per group to keep the host cores busy
    group = max(1, min(w.H, (os.cpu_count() or 8) // max(inp.N, 1)))
    for h0 in range(0, w.H, group):
        heads = list(range(h0, min(w.H, h0 + group)))
        o_ref, ht_ref = run_oracle(inp, heads=heads)
        assert_close(as_f64(o[:, :, heads]), o_ref, TOL[w.dtype], f"{name} o heads {heads[0]}..{heads[-1]}")
        assert_close(as_f64(ht[:, heads]), ht_ref, TOL[w.dtype], f"{name} ht heads {heads[0]}..{heads[-1]}")


def test_kernel_timer_brackets_every_launch():
    """The measurement hook records events around each launch of gla_fwd on the call's stream."""
    from chunkwise_gated_linear_chunked_gb300 import binding
    inp = make_inputs("bf16", B=1, T=3000, H=1, K=128, V=128, h0=True, seed=9)   # segments: 3 kernels
    q, k, v, g, h0, _ = to_device(inp)
    timer = binding.KernelTimer()
    with timer:
        o, ht = binding.gla_fwd(q, k, v, g, scale=inp.scale, initial_state=h0)
    torch.cuda.synchronize()
    res = timer.results()
    assert len(res) >= 1 and all(ms > 0 for _, ms in res), res
    assert res[-1][0] in ("fused_tc", "out_ffma"), res
    o2, _ = binding.gla_fwd(q, k, v, g, scale=inp.scale, initial_state=h0)   # disarmed: no events
    torch.cuda.synchronize()
    assert torch.equal(o, o2)


def test_tensor_core_range_check_reports_status():
    """Values outside the fp16 operand range of the tensor-core path are reported, not silently wrong."""
    from chunkwise_gated_linear_chunked_gb300 import binding
    inp = make_inputs("bf16", B=1, T=130, H=1, K=128, V=128, seed=10)
    q, k, v, g, _, _ = to_device(inp)
    v = (v.float() * 1e5).to(torch.bfloat16)
    ws = torch.zeros(binding.workspace_size(1, 130, 1, 128, 128, 1), dtype=torch.uint8, device="cuda")
    o = torch.empty(1, 130, 1, 128, device="cuda")
    rc = binding.fwd_into(q, k, v, g, o, inp.scale, None, None, None, 1, 1, 130, 1, 128, 128, 64,
                          binding.GLA_BF16, ws)
    assert rc == 0
    assert binding.get_status(ws) == binding.GLA_ERR_RANGE
    # in range again: clean status
    q, k, v, g, _, _ = to_device(inp)
    rc = binding.fwd_into(q, k, v, g, o, inp.scale, None, None, None, 1, 1, 130, 1, 128, 128, 64,
                          binding.GLA_BF16, ws)
    assert rc == 0 and binding.get_status(ws) == binding.GLA_OK


HEAD_FIRST_CASES = [
    ("bf16", 2, 200, 3, 128, 128, True, None),    # tensor-core path, ragged chunk
    ("bf16", 3, 4096, 13, 128, 128, True, None),  # balanced pieces crossing heads and sequences
    ("bf16", 1, 3000, 2, 128, 256, True, None),   # segments + scan, V = 256
    ("f16", 2, 130, 2, 128, 128, False, None),
    ("f32", 2, 200, 2, 64, 64, True, None),       # CUDA-core path
]


@pytest.mark.parametrize("case", HEAD_FIRST_CASES, ids=_case_id)
def test_head_first_layout(case):
    """[B, H, T, *] inputs give the head-first permutation of the time-major result (elementwise parity)."""
    from chunkwise_gated_linear_chunked_gb300 import binding
    d, B, T, H, K, V, h0, _ = case
    inp = make_inputs(d, B=B, T=T, H=H, K=K, V=V, h0=h0, seed=zlib.crc32(_case_id(case).encode()) % 1000)
    hf = lambda x: x.transpose(1, 2).contiguous().cuda()
    o, ht = binding.gla_fwd(hf(inp.q), hf(inp.k), hf(inp.v), hf(inp.g), scale=inp.scale,
                            initial_state=None if inp.h0 is None else inp.h0.cuda(), head_first=True)
    torch.cuda.synchronize()
    o_ref, ht_ref = run_oracle(inp)
    assert o.shape == (B, H, T, V)
    assert_close(as_f64(o.transpose(1, 2)), o_ref, TOL[d], "o")
    assert_close(as_f64(ht), ht_ref, TOL[d], "ht")


HEAD_FIRST_VARLEN_CASES = [
    ("bf16", 1, 0, 2, 128, 128, True, [1, 63, 64, 65, 0, 130, 300, 2]),   # tensor-core path
    ("bf16", 1, 0, 1, 128, 256, True, [3000, 7, 1500]),                  # segments + scan, V = 256
    ("f32", 1, 0, 2, 64, 64, True, [5, 0, 200, 64]),                     # CUDA-core path
]


@pytest.mark.parametrize("case", HEAD_FIRST_VARLEN_CASES, ids=_case_id)
def test_head_first_varlen(case):
    """A packed varlen batch in [1, H, T, *] gives the head-first permutation of the time-major result."""
    from chunkwise_gated_linear_chunked_gb300 import binding
    d, B, T, H, K, V, h0, lengths = case
    inp = make_inputs(d, B=B, T=T, H=H, K=K, V=V, h0=h0, lengths=lengths,
                      seed=zlib.crc32(_case_id(case).encode()) % 1000)
    hf = lambda x: x.transpose(1, 2).contiguous().cuda()
    o, ht = binding.gla_fwd(hf(inp.q), hf(inp.k), hf(inp.v), hf(inp.g), scale=inp.scale,
                            initial_state=None if inp.h0 is None else inp.h0.cuda(),
                            cu_seqlens=inp.cu_seqlens.cuda(), head_first=True)
    torch.cuda.synchronize()
    o_ref, ht_ref = run_oracle(inp)
    assert o.shape == (1, H, inp.q.shape[1], V)
    assert_close(as_f64(o.transpose(1, 2)), o_ref, TOL[d], "o")
    assert_close(as_f64(ht), ht_ref, TOL[d], "ht")


GF32_CASES = [
    ("bf16", 2, 200, 2, 128, 128, True, None),      # tensor-core path (two 80 KB stages)
    ("f16", 1, 3000, 1, 128, 256, True, None),      # tensor-core path, segments + scan, V = 256
    ("bf16", 1, 5000, 33, 128, 128, True, None),    # tensor-core path, balanced pieces
    ("bf16", 1, 0, 2, 128, 128, True, [1, 63, 64, 65, 0, 130, 300, 2]),   # tensor-core path, varlen
    ("f16", 1, 3000, 1, 64, 128, True, None),       # K = 64: CUDA-core path
    ("bf16", 1, 0, 2, 64, 64, True, [1, 63, 64, 65, 0, 130, 300, 2]),
]


def _with_fp32_gate(inp, seed):
    """Replace g by an fp32 gate of the same recipe (16-bit q, k, v with fp32 g, as the method allows)."""
    import dataclasses
    gen = torch.Generator().manual_seed(seed)
    g32 = torch.nn.functional.logsigmoid(torch.randn(tuple(inp.g.shape), generator=gen)) / 16
    return dataclasses.replace(inp, g=g32)


@pytest.mark.parametrize("case", GF32_CASES, ids=_case_id)
def test_fp32_gate_with_16bit_inputs(case):
    """16-bit q, k, v with an fp32 g: K == 128 runs the tensor-core kernel (16-bit operands, so the 16-bit
    bound applies, as with a 16-bit g); K == 64 runs the fp32 CUDA-core path (the fp32 bound)."""
    from chunkwise_gated_linear_chunked_gb300 import binding
    d, B, T, H, K, V, h0, lengths = case
    seed = zlib.crc32(_case_id(case).encode()) % 1000
    inp = _with_fp32_gate(make_inputs(d, B=B, T=T, H=H, K=K, V=V, h0=h0, lengths=lengths, seed=seed), seed + 1)
    timer = binding.KernelTimer()
    with timer:
        o, ht = run_gpu(inp)
    names = [n for n, _ in timer.results()]
    o_ref, ht_ref = run_oracle(inp)
    tol = TOL[d] if K == 128 else TOL["f32"]
    assert ("fused_tc" in names) == (K == 128), names
    assert_close(as_f64(o), o_ref, tol, "o")
    assert_close(as_f64(ht), ht_ref, tol, "ht")


def test_fp32_gate_head_first_tensor_cores():
    """fp32 g in the head-first layout on the tensor-core path."""
    from chunkwise_gated_linear_chunked_gb300 import binding
    inp = _with_fp32_gate(make_inputs("bf16", B=2, T=700, H=2, K=128, V=128, h0=True, seed=77), 78)
    hf = lambda x: x.transpose(1, 2).contiguous().cuda()
    o, ht = binding.gla_fwd(hf(inp.q), hf(inp.k), hf(inp.v), hf(inp.g), scale=inp.scale,
                            initial_state=inp.h0.cuda(), head_first=True)
    torch.cuda.synchronize()
    o_ref, ht_ref = run_oracle(inp)
    assert_close(as_f64(o.transpose(1, 2)), o_ref, TOL["bf16"], "o")
    assert_close(as_f64(ht), ht_ref, TOL["bf16"], "ht")
