"""Pins of the backward oracle (CPU).

The backward oracle differentiates the GLA recurrence step by step (reverse mode).  It is pinned to things
that do not come from that code: central finite differences of the (separately pinned) forward oracle on
fp64 inputs, the closed-form gradients of causal linear attention (all gates zero), and the gate-gradient
identity of the chunked backward of page "fla/ops/gla/fused_chunk.py" (FusedChunkGLAFunction.backward:
dg is the reverse cumsum of q*dq - k*dk, plus the final-state term).  Planted mistakes in copies of the
oracle must each fail at least one pin.
"""
import os
import subprocess

import numpy as np
import pytest

import oracle


def _rand(seed, B, T, H, K, V, h0=True, dht=True, N=None):
    rng = np.random.default_rng(seed)
    q, k = rng.standard_normal((2, B, T, H, K))
    g = -np.abs(rng.standard_normal((B, T, H, K))) * 0.3
    v, do = rng.standard_normal((2, B, T, H, V))
    n = B if N is None else N
    s0 = rng.standard_normal((n, H, K, V)) * 0.5 if h0 else None
    s1 = rng.standard_normal((n, H, K, V)) if dht else None
    return q, k, v, g, do, s0, s1


def _loss(q, k, v, g, h0, do, dht, scale, cu=None, lib=None):
    o, ht, _ = oracle.gla_fwd(q, k, v, g, scale, h0=h0, cu_seqlens=cu)
    L = float((o * do).sum())
    if dht is not None:
        L += float((ht * dht).sum())
    return L


def _fd_check(seed, B, T, H, K, V, h0, dht, cu=None, lib=None):
    N = None if cu is None else len(cu) - 1
    q, k, v, g, do, s0, s1 = _rand(seed, B, T, H, K, V, h0, dht, N)
    scale = 0.7
    grads = oracle.gla_bwd(q, k, v, g, do, scale, h0=s0, dht=s1, cu_seqlens=cu, lib=lib)
    args = [q, k, v, g, s0]
    eps = 1e-6
    for a, name in enumerate(["q", "k", "v", "g", "h0"]):
        x = args[a]
        if x is None:
            continue
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            ap, am = list(args), list(args)
            ap[a], am[a] = xp, xm
            num[idx] = (_loss(*ap, do, s1, scale, cu) - _loss(*am, do, s1, scale, cu)) / (2 * eps)
        ana = grads[a]
        err = np.abs(num - ana).max() / max(1.0, np.abs(num).max())
        assert err < 1e-7, f"{name}: finite-difference mismatch {err:.3e}"


# ----------------------------------------------------------------------------------------------------
# pins, written against a callable so the planted-mistake tests can rerun them on a mutant
# ----------------------------------------------------------------------------------------------------

def pin_finite_differences(lib=None):
    _fd_check(1, 1, 5, 1, 2, 3, True, True, lib=lib)
    _fd_check(2, 2, 3, 2, 3, 2, False, True, lib=lib)
    _fd_check(3, 1, 1, 1, 2, 2, True, False, lib=lib)


def pin_finite_differences_across_checkpoint(lib=None):
    # 70 steps: the backward recomputes states from a checkpoint every 64 steps
    _fd_check(4, 1, 70, 1, 1, 2, True, True, lib=lib)


def pin_finite_differences_varlen(lib=None):
    _fd_check(5, 1, 9, 1, 2, 2, True, True, cu=np.array([0, 4, 4, 9], np.int32), lib=lib)


def pin_linear_attention_closed_form(lib=None):
    """All gates zero: o = scale*(tril(Q K^T) V + Q h0), ht = h0 + K^T V; matrix-form gradients."""
    q, k, v, g, do, s0, s1 = _rand(6, 1, 37, 1, 4, 5)
    g = np.zeros_like(g)
    scale = 0.3
    dq, dk, dv, dg, dh0 = oracle.gla_bwd(q, k, v, g, do, scale, h0=s0, dht=s1, lib=lib)
    Q, Kk, Vv, dO = q[0, :, 0], k[0, :, 0], v[0, :, 0], do[0, :, 0]
    H0, dHT = s0[0, 0], s1[0, 0]
    M = np.tril(np.ones((37, 37)))
    np.testing.assert_allclose(dq[0, :, 0], scale * ((M * (dO @ Vv.T)) @ Kk + dO @ H0.T), rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(dk[0, :, 0], scale * (M * (dO @ Vv.T)).T @ Q + Vv @ dHT.T, rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(dv[0, :, 0], scale * (M * (Q @ Kk.T)).T @ dO + Kk @ dHT, rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(dh0[0, 0], scale * Q.T @ dO + dHT, rtol=1e-11, atol=1e-11)


def pin_gate_gradient_identity(lib=None):
    """dg_t = sum_{s >= t} (q_s*dq_s - k_s*dk_s) + sum_v ht*dht, per sequence (varlen included)."""
    q, k, v, g, do, s0, s1 = _rand(7, 1, 150, 2, 6, 5, N=3)
    cu = np.array([0, 60, 60, 150], np.int32)
    scale = 0.5
    dq, dk, dv, dg, _ = oracle.gla_bwd(q, k, v, g, do, scale, h0=s0, dht=s1, cu_seqlens=cu, lib=lib)
    _, ht, _ = oracle.gla_fwd(q, k, v, g, scale, h0=s0, cu_seqlens=cu)
    term = (q * dq - k * dk)[0]                       # [T, H, K]
    for n in range(3):
        a, b = cu[n], cu[n + 1]
        if a == b:
            continue
        rev = np.cumsum(term[a:b][::-1], axis=0)[::-1]
        ref = rev + (ht[n] * s1[n]).sum(-1)[None]
        np.testing.assert_allclose(dg[0, a:b], ref, rtol=1e-9, atol=1e-9)


PINS = [pin_finite_differences, pin_finite_differences_across_checkpoint, pin_finite_differences_varlen,
        pin_linear_attention_closed_form, pin_gate_gradient_identity]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_backward_pin(pin):
    pin()


def test_backward_reads_stored_types_exactly():
    """bf16 words and fp32 inputs give the gradients of their exactly widened values."""
    from chunkwise_gated_linear_chunked_gb300.inputs import make_inputs, stored_numpy
    inp = make_inputs("bf16", B=1, T=70, H=2, K=8, V=4, h0=True, seed=11)
    q, k, v, g = (stored_numpy(x) for x in (inp.q, inp.k, inp.v, inp.g))
    do = stored_numpy(inp.v.flip(1).contiguous())
    wide = [oracle.bf16_words_to_f64(x) for x in (q, k, v, g, do)]
    a = oracle.gla_bwd(q, k, v, g, do, inp.scale, h0=inp.h0.numpy())
    b = oracle.gla_bwd(*wide, inp.scale, h0=inp.h0.numpy())
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_zero_length_sequence_passes_dht_through():
    q, k, v, g, do, s0, s1 = _rand(8, 1, 4, 1, 2, 2, N=2)
    cu = np.array([0, 0, 4], np.int32)
    *_, dh0 = oracle.gla_bwd(q, k, v, g, do, 0.5, h0=s0, dht=s1, cu_seqlens=cu)
    assert np.array_equal(dh0[0], s1[0])


# ----------------------------------------------------------------------------------------------------
# planted mistakes in the backward: each must fail at least one pin
# ----------------------------------------------------------------------------------------------------

BWD_MUTANTS = {
    "dg_uses_current_state": ("const double *Sp = t > b0 ? blk + (size_t)(t - b0 - 1) * KV : ck + (size_t)m * KV;",
                              "const double *Sp = St;"),
    "adjoint_not_decayed": ("A[(size_t)i * V + j] *= e;", "A[(size_t)i * V + j] *= 1.0;"),
    "dq_without_scale": ("J->dq[kb + i] = J->scale * aq;", "J->dq[kb + i] = aq;"),
    "dht_ignored": ("A[e] = J->dht ? J->dht[st + e] : 0.0;", "A[e] = 0.0;"),
    "dv_from_q": ("av += widen(J->k, kb + i, J->dtype) * A[(size_t)i * V + j];",
                  "av += widen(J->q, kb + i, J->dtype) * A[(size_t)i * V + j];"),
    "output_term_after_grads": (
        "            /* A <- A + scale q_t^T do_t: now dL/dS_t */\n",
        "            if (0) /* A <- A + scale q_t^T do_t: now dL/dS_t */\n"),
}


@pytest.mark.parametrize("name", sorted(BWD_MUTANTS))
def test_backward_pins_catch_planted_mistake(name, tmp_path):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "gla_oracle.c")).read()
    old, new = BWD_MUTANTS[name]
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", str(so),
                           str(path), "-lm"])
    lib = oracle.load_variant(str(so))
    caught = []
    for pin in PINS:
        try:
            pin(lib=lib)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake {name}"


def test_fp16_inputs_widen_exactly():
    """fp16 inputs (including subnormals and large values) give exactly the results of the same values in
    float64: the oracle's half decoder agrees with numpy's conversion, forward and backward."""
    rng = np.random.default_rng(12)
    B, T, H, K, V = 1, 9, 2, 3, 4
    vals = lambda *s: (rng.standard_normal(s) * rng.choice([1e-6, 1e-2, 1.0, 300.0], size=s)).astype(np.float16)
    q, k, v, do = vals(B, T, H, K), vals(B, T, H, K), vals(B, T, H, V), vals(B, T, H, V)
    g = (-np.abs(rng.standard_normal((B, T, H, K))) * 0.2).astype(np.float16)
    q[0, 0, 0, 0] = np.float16(6e-8)       # subnormal
    wide = [x.astype(np.float64) for x in (q, k, v, g, do)]
    o16, ht16, _ = oracle.gla_fwd(q, k, v, g, 0.5)
    o64, ht64, _ = oracle.gla_fwd(*wide[:4], 0.5)
    assert np.array_equal(o16, o64) and np.array_equal(ht16, ht64)
    for x, y in zip(oracle.gla_bwd(q, k, v, g, do, 0.5), oracle.gla_bwd(*wide, 0.5)):
        assert np.array_equal(x, y)
