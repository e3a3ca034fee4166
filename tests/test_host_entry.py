"""gla_fwd_host: the forward on inputs and outputs in host memory, pipelined by head groups, against the oracle
(elementwise) and against gla_fwd on device copies of the same inputs."""
import zlib

import numpy as np
import pytest
import torch

from chunkwise_gated_linear_chunked_gb300.inputs import make_inputs
from parity_util import TOL, as_f64, assert_close, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from chunkwise_gated_linear_chunked_gb300 import build
    build.build()


CASES = [
    # (dtype, B, T, H, K, V, h0, lengths, head_groups)
    ("bf16", 2, 300, 4, 128, 128, True, None, 2),
    ("bf16", 1, 0, 4, 128, 128, True, [1, 63, 200, 0, 130], 4),   # varlen incl. an empty sequence, 1 head a group
    ("bf16", 1, 3000, 10, 128, 128, False, None, 5),               # more groups than slots: slots reused
    ("bf16", 2, 130, 3, 128, 256, True, None, 1),
    ("f32", 2, 200, 4, 64, 64, True, None, 2),                     # CUDA-core path
]


@pytest.mark.parametrize("variant", ["fp32_gate", "bf16_output"])
def test_host_entry_dtype_variants(variant):
    """fp32 g with bf16 q, k, v and bf16 o: the copies size each tensor by its own element type."""
    from chunkwise_gated_linear_chunked_gb300 import binding
    inp = make_inputs("bf16", B=2, T=260, H=4, K=128, V=128, h0=True, seed=91)
    g32 = torch.nn.functional.logsigmoid(torch.randn(inp.g.shape, generator=torch.Generator().manual_seed(5))) / 16
    code = binding.GLA_BF16_GF32 if variant == "fp32_gate" else binding.GLA_BF16_OBF16
    g_host = g32 if variant == "fp32_gate" else inp.g
    B, T, H, K, V, N = 2, 260, 4, 128, 128, 2
    pin = lambda x: x.contiguous().pin_memory()
    out_dtype = torch.bfloat16 if variant == "bf16_output" else torch.float32
    o = torch.empty(B, T, H, V, dtype=out_dtype).pin_memory()
    ht = torch.empty(N, H, K, V).pin_memory()
    ws = torch.zeros(binding.host_workspace_size(B, T, H, K, V, N, 64, code, 2), dtype=torch.uint8, device="cuda")
    rc = binding.fwd_host_into(pin(inp.q), pin(inp.k), pin(inp.v), pin(g_host), o, inp.scale, pin(inp.h0), ht, None,
                               N, B, T, H, K, V, 64, code, 2, ws)
    assert rc == 0
    torch.cuda.synchronize()
    od, htd = binding.gla_fwd(inp.q.cuda(), inp.k.cuda(), inp.v.cuda(), g_host.cuda(), scale=inp.scale,
                              initial_state=inp.h0.cuda(), out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert_close(as_f64(o), as_f64(od), TOL["bf16"], "o vs gla_fwd")
    assert_close(as_f64(ht), as_f64(htd), TOL["bf16"], "ht vs gla_fwd")


def _id(c):
    return f"{c[0]}-B{c[1]}T{c[2]}H{c[3]}K{c[4]}V{c[5]}-G{c[8]}" + ("-var" if c[7] else "")


def _run_host(inp, groups, out_dtype=torch.float32):
    from chunkwise_gated_linear_chunked_gb300 import binding
    pin = lambda x: None if x is None else x.contiguous().pin_memory()
    q, k, v, g, h0, cu = (pin(x) for x in (inp.q, inp.k, inp.v, inp.g, inp.h0, inp.cu_seqlens))
    B, T, H, K, V, N = inp.q.shape[0], inp.q.shape[1], inp.H, inp.K, inp.V, inp.N
    o = torch.empty(B, T, H, V, dtype=out_dtype).pin_memory()
    ht = torch.empty(N, H, K, V, dtype=torch.float32).pin_memory()
    code = binding.GLA_F32 if inp.dtype == "f32" else binding.GLA_BF16
    nb = binding.host_workspace_size(B, T, H, K, V, N, 64, code, groups)
    assert nb > 0
    ws = torch.zeros(nb, dtype=torch.uint8, device="cuda")
    rc = binding.fwd_host_into(q, k, v, g, o, inp.scale, h0, ht, cu, N, B, T, H, K, V, 64, code, groups, ws)
    assert rc == 0, binding.strerror(rc) if hasattr(binding, "strerror") else rc
    torch.cuda.synchronize()
    assert binding.get_status(ws) == binding.GLA_OK
    return o, ht


@pytest.mark.parametrize("case", CASES, ids=_id)
def test_host_entry_matches_oracle_and_device_call(case):
    from chunkwise_gated_linear_chunked_gb300 import binding
    d, B, T, H, K, V, h0, lengths, groups = case
    inp = make_inputs(d, B=B, T=T, H=H, K=K, V=V, h0=h0, lengths=lengths, seed=zlib.crc32(_id(case).encode()) % 1000)
    o, ht = _run_host(inp, groups)
    o_ref, ht_ref = run_oracle(inp)
    assert_close(as_f64(o), o_ref, TOL[d], "o")
    assert_close(as_f64(ht), ht_ref, TOL[d], "ht")
    # the device call on the same inputs: equal within the arithmetic's rounding (the plans may differ)
    dev = lambda x: None if x is None else x.cuda()
    od, htd = binding.gla_fwd(dev(inp.q), dev(inp.k), dev(inp.v), dev(inp.g), scale=inp.scale,
                              initial_state=dev(inp.h0), cu_seqlens=dev(inp.cu_seqlens))
    torch.cuda.synchronize()
    assert_close(as_f64(o), as_f64(od), TOL[d], "o vs gla_fwd")
    assert_close(as_f64(ht), as_f64(htd), TOL[d], "ht vs gla_fwd")


def test_host_entry_one_group_is_the_device_call_bitwise():
    """With one group the host call runs gla_fwd on device copies of the whole tensors: the same bits."""
    from chunkwise_gated_linear_chunked_gb300 import binding
    inp = make_inputs("bf16", B=2, T=700, H=3, K=128, V=128, h0=True, seed=77)
    o, ht = _run_host(inp, 1)
    od, htd = binding.gla_fwd(inp.q.cuda(), inp.k.cuda(), inp.v.cuda(), inp.g.cuda(), scale=inp.scale,
                              initial_state=inp.h0.cuda())
    torch.cuda.synchronize()
    assert torch.equal(o, od.cpu()) and torch.equal(ht, htd.cpu())


def test_host_entry_rejections():
    from chunkwise_gated_linear_chunked_gb300 import binding
    inp = make_inputs("bf16", B=1, T=64, H=4, K=128, V=128, seed=3)
    q, k, v, g = (x.contiguous() for x in (inp.q, inp.k, inp.v, inp.g))
    o = torch.empty(1, 64, 4, 128)
    B, T, H, K, V, N = 1, 64, 4, 128, 128, 1
    code = binding.GLA_BF16
    nb = binding.host_workspace_size(B, T, H, K, V, N, 64, code, 2)
    ws = torch.zeros(nb, dtype=torch.uint8, device="cuda")
    assert binding.host_workspace_size(B, T, H, K, V, N, 64, code, 3) == 0        # 4 heads, 3 groups
    assert binding.fwd_host_into(q, k, v, g, o, inp.scale, None, None, None, N, B, T, H, K, V, 64, code, 3,
                                 ws) == binding.GLA_ERR_INVALID_ARG
    assert binding.fwd_host_into(q, k, v, g, o, inp.scale, None, None, None, N, B, T, H, K, V, 64,
                                 code | binding.GLA_HEAD_FIRST, 2, ws) == binding.GLA_ERR_UNSUPPORTED
    small = ws[: nb // 2]
    assert binding.fwd_host_into(q, k, v, g, o, inp.scale, None, None, None, N, B, T, H, K, V, 64, code, 2,
                                 small) == binding.GLA_ERR_WORKSPACE
