"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI and the fp64 oracle on the
same seeded inputs, and compare with the bounds of the method's contract."""
import numpy as np
import torch

import oracle
from chunkwise_gated_linear_chunked_gb300.inputs import Inputs, stored_numpy

# fp32 inputs: relative L2 <= 1e-5.  bf16 inputs with fp32 state: relative L2 <= 5e-3 and max-abs <= 2e-2.
TOL = {"f32": dict(rel=1e-5, abs=None), "bf16": dict(rel=5e-3, abs=2e-2), "f16": dict(rel=5e-3, abs=2e-2)}
# bf16-stored o is checked on relative L2 only (its own rounding exceeds 2e-2 at |o| >= 8).
TOL_OBF16 = dict(rel=5e-3, abs=None)


def to_device(inp: Inputs, device="cuda"):
    d = lambda x: None if x is None else x.to(device).contiguous()
    return d(inp.q), d(inp.k), d(inp.v), d(inp.g), d(inp.h0), d(inp.cu_seqlens)


def run_gpu(inp: Inputs, out_dtype=torch.float32, want_ht=True):
    from chunkwise_gated_linear_chunked_gb300 import binding
    q, k, v, g, h0, cu = to_device(inp)
    o, ht = binding.gla_fwd(q, k, v, g, scale=inp.scale, initial_state=h0, output_final_state=want_ht,
                            cu_seqlens=cu, chunk=inp.chunk, out_dtype=out_dtype)
    torch.cuda.synchronize()
    return o, ht


def run_oracle(inp: Inputs, heads=None):
    """Oracle outputs for all heads, or for the listed heads only (then shaped [.., len(heads), ..])."""
    sel = (lambda x: x) if heads is None else (lambda x: x[:, :, heads].contiguous())
    args = [stored_numpy(sel(x)) for x in (inp.q, inp.k, inp.v, inp.g)]
    h0 = None
    if inp.h0 is not None:
        h0 = inp.h0.numpy() if heads is None else inp.h0[:, heads].contiguous().numpy()
    cu = None if inp.cu_seqlens is None else inp.cu_seqlens.numpy()
    o, ht, _ = oracle.gla_fwd(*args, inp.scale, h0=h0, cu_seqlens=cu)
    return o, ht


def errors(x, ref):
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    d = x - ref
    n = np.linalg.norm(ref.ravel())
    rel = np.linalg.norm(d.ravel()) / n if n > 0 else np.linalg.norm(d.ravel())
    mx = float(np.max(np.abs(d))) if d.size else 0.0
    return float(rel), mx


def assert_close(x, ref, tol, what=""):
    rel, mx = errors(x, ref)
    assert np.all(np.isfinite(np.asarray(x))), f"{what}: non-finite values"
    assert rel <= tol["rel"], f"{what}: rel-L2 {rel:.3e} > {tol['rel']:.1e} (max-abs {mx:.3e})"
    if tol.get("abs") is not None:
        assert mx <= tol["abs"], f"{what}: max-abs {mx:.3e} > {tol['abs']:.1e} (rel-L2 {rel:.3e})"
    return rel, mx


def as_f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)
