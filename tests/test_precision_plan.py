"""The tensor-core path's precision plan, checked on the CPU against the fp64 oracle.

A numpy model of the chunked algorithm rounds every operand that the tcgen05 kernels form on chip (q~, k~,
k^, S', P) the way the kernels do, accumulates in high precision, and is compared with the oracle on inputs
of the benchmark distribution.  fp16 operands must stay well inside the bf16 parity bounds (rel-L2 5e-3,
max-abs 2e-2); single-rounded bf16 operands must not (which is why the kernels use fp16 operands).
"""
import numpy as np

import oracle
from chunkwise_gated_linear_chunked_gb300.inputs import make_inputs, stored_numpy


def round_fp16(x):
    return np.asarray(x, np.float32).astype(np.float16).astype(np.float64)


def round_bf16(x):
    u = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    u = ((u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000).astype(np.uint32)
    return u.view(np.float32).astype(np.float64)


def chunked_model(q, k, v, g, scale, R, C=64):
    """Chunked GLA for one (sequence, head) with the kernels' rounding points and mid-chunk anchor."""
    T, K = q.shape
    S = np.zeros((K, v.shape[1]))
    o = np.zeros((T, v.shape[1]))
    for c0 in range(0, T, C):
        qc, kc, vc, gc = q[c0:c0 + C], k[c0:c0 + C], v[c0:c0 + C], g[c0:c0 + C]
        n = qc.shape[0]
        G = np.cumsum(gc.astype(np.float32), axis=0, dtype=np.float32).astype(np.float64)
        a = min(C // 2 - 1, n - 1)
        Ga, Gl = G[a], G[n - 1]
        qt = R(qc * np.exp(G - Ga))
        kt = R(kc * np.exp(Ga - G))
        kh = R(kc * np.exp(Gl - G))
        P = R(np.tril(qt @ kt.T))
        o[c0:c0 + n] = scale * (qt @ R(np.exp(Ga)[:, None] * S) + P @ vc)
        S = np.exp(Gl)[:, None] * S + kh.T @ vc
    return o


def _errors(R):
    inp = make_inputs("bf16", B=1, T=2048, H=2, K=128, V=128, seed=1004)
    diffs = []
    for h in range(inp.H):
        f = lambda x: x[0, :, h].float().numpy().astype(np.float64)
        o = chunked_model(f(inp.q), f(inp.k), f(inp.v), f(inp.g), inp.scale, R)
        sel = lambda x: stored_numpy(x[:, :, h:h + 1].contiguous())
        ref, _, _ = oracle.gla_fwd(sel(inp.q), sel(inp.k), sel(inp.v), sel(inp.g), inp.scale)
        diffs.append((o - ref[0, :, 0]).ravel())
        norm = np.linalg.norm(ref)
    d = np.concatenate(diffs)
    return np.linalg.norm(d) / (norm * np.sqrt(inp.H)), np.abs(d).max()


def test_fp16_operands_meet_the_bf16_bounds_with_margin():
    rel, mx = _errors(round_fp16)
    assert rel < 1e-3 and mx < 1e-2, (rel, mx)


def test_single_rounded_bf16_operands_would_not():
    rel, mx = _errors(round_bf16)
    assert mx > 2e-2, (rel, mx)
