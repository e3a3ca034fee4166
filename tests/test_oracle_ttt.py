"""Pins of the TTT-linear oracle (CPU).

The oracle runs the kernel's dual form (page "fla/ops/ttt/fused_chunk.py": fused_chunk_ttt_linear_fwd_kernel,
then norm_residual of fused_chunk_ttt_linear).  It is pinned against an independent primal form written here
in numpy: explicit per-row weights W_i = W_c - eta_i * sum_{j<=i} k_j^T grad_j read out as o_i = q_i W_i, with
each gradient obtained by central finite differences of the inner loss (not from the LayerNorm-backward
formula); against the eta == 0 closed form; varlen == separate runs; continuing from (ht, hbt) at a chunk
boundary; and planted mistakes.
"""
import os
import subprocess

import numpy as np
import pytest

import oracle

EPS = 1e-6


def _ln(x, eps=EPS):
    m = x.mean(-1, keepdims=True)
    var = ((x - m) ** 2).mean(-1, keepdims=True)
    return (x - m) / np.sqrt(var + eps)


def _case(seed, B, T, H, D, h0=True):
    rng = np.random.default_rng(seed)
    q, k, v = rng.standard_normal((3, B, T, H, D))
    w = 1.0 + 0.3 * rng.standard_normal((H, D))
    b = 0.2 * rng.standard_normal((H, D))
    eta = 0.05 + 0.1 * rng.random((B, T, H))
    n = B
    s0 = 0.3 * rng.standard_normal((n, H, D, D)) if h0 else None
    sb0 = 0.3 * rng.standard_normal((n, H, D)) if h0 else None
    return q, k, v, w, b, eta, s0, sb0


def primal(q, k, v, w, b, eta, scale, chunk, h0, hb0, cu=None):
    """Mini-batch gradient descent written with explicit weights and finite-difference gradients."""
    B, T, H, D = q.shape
    rows = lambda x: x.reshape(B * T, H, *x.shape[3:]) if x.ndim == 4 else x.reshape(B * T, H)
    Q, Kk, Vv, E = rows(q), rows(k), rows(v), rows(eta)
    bounds = [(n * T, n * T + T) for n in range(B)] if cu is None else list(zip(cu[:-1], cu[1:]))
    o = np.zeros((B * T, H, D))
    ht = np.zeros((len(bounds), H, D, D))
    hbt = np.zeros((len(bounds), H, D))
    for n, (bos, eos) in enumerate(bounds):
        for h in range(H):
            W = np.zeros((D, D)) if h0 is None else h0[n, h].copy()
            bb = np.zeros(D) if hb0 is None else hb0[n, h].copy()
            for r0 in range(bos, eos, chunk):
                r1 = min(r0 + chunk, eos)
                grads = []
                for j in range(r0, r1):
                    kj, vj = Kk[j, h], Vv[j, h]
                    loss = lambda z: 0.5 * np.sum((_ln(z) * w[h] + b[h] + kj - vj) ** 2)
                    z0 = kj @ W + bb
                    gz = np.zeros(D)
                    for c in range(D):
                        dz = np.zeros(D)
                        dz[c] = 1e-5
                        gz[c] = (loss(z0 + dz) - loss(z0 - dz)) / 2e-5
                    grads.append(gz)
                for i in range(r0, r1):
                    Wi = W - E[i, h] * sum(np.outer(Kk[j, h], grads[j - r0]) for j in range(r0, i + 1))
                    bi = bb - E[i, h] * sum(grads[j - r0] for j in range(r0, i + 1))
                    oi = scale * Q[i, h] @ Wi + bi
                    o[i, h] = oi + _ln(oi) * w[h] + b[h]
                el = E[r1 - 1, h]
                W = W - el * sum(np.outer(Kk[j, h], grads[j - r0]) for j in range(r0, r1))
                bb = bb - el * sum(grads)
            ht[n, h], hbt[n, h] = W, bb
    return o.reshape(B, T, H, D), ht, hbt


def pin_primal_form(lib=None):
    for seed, (B, T, H, D, chunk) in enumerate([(1, 7, 1, 3, 3), (2, 10, 2, 4, 4), (1, 9, 1, 2, 16), (1, 5, 1, 3, 1)]):
        q, k, v, w, b, eta, s0, sb0 = _case(seed, B, T, H, D)
        got = oracle.ttt_linear_fwd(q, k, v, w, b, eta, 0.6, EPS, chunk, h0=s0, hb0=sb0, lib=lib)
        ref = primal(q, k, v, w, b, eta, 0.6, chunk, s0, sb0)
        for x, y, name in zip(got, ref, ("o", "ht", "hbt")):
            np.testing.assert_allclose(x, y, rtol=1e-6, atol=1e-6, err_msg=name)


def pin_eta_zero_closed_form(lib=None):
    q, k, v, w, b, eta, s0, sb0 = _case(7, 2, 13, 2, 5)
    eta = np.zeros_like(eta)
    o, ht, hbt = oracle.ttt_linear_fwd(q, k, v, w, b, eta, 0.4, EPS, 4, h0=s0, hb0=sb0, lib=lib)
    pre = np.stack([0.4 * np.einsum("tik,ikv->tiv", q[n], s0[n]) + sb0[n][None] for n in range(2)])
    np.testing.assert_allclose(o, pre + _ln(pre) * w + b, rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(ht, s0)
    np.testing.assert_array_equal(hbt, sb0)


def pin_varlen_is_separate_runs(lib=None):
    q, k, v, w, b, eta, _, _ = _case(8, 1, 23, 2, 4, h0=False)
    cu = np.array([0, 5, 5, 23], np.int32)
    o, ht, hbt = oracle.ttt_linear_fwd(q, k, v, w, b, eta, 0.5, EPS, 4, cu_seqlens=cu, lib=lib)
    for n in range(3):
        a, c = cu[n], cu[n + 1]
        sl = lambda x: x[:, a:c]
        on, htn, hbn = oracle.ttt_linear_fwd(sl(q), sl(k), sl(v), w, b, sl(eta), 0.5, EPS, 4, lib=lib)
        np.testing.assert_array_equal(o[:, a:c], on)
        np.testing.assert_array_equal(ht[n], htn[0])
        np.testing.assert_array_equal(hbt[n], hbn[0])


def pin_state_continuation(lib=None):
    """Running T = 12 equals running 8 rows, then 4 more from (ht, hbt) (8 is a multiple of the chunk)."""
    q, k, v, w, b, eta, s0, sb0 = _case(9, 1, 12, 1, 3)
    full = oracle.ttt_linear_fwd(q, k, v, w, b, eta, 0.5, EPS, 4, h0=s0, hb0=sb0, lib=lib)
    a = oracle.ttt_linear_fwd(q[:, :8], k[:, :8], v[:, :8], w, b, eta[:, :8], 0.5, EPS, 4, h0=s0, hb0=sb0, lib=lib)
    c = oracle.ttt_linear_fwd(q[:, 8:], k[:, 8:], v[:, 8:], w, b, eta[:, 8:], 0.5, EPS, 4, h0=a[1], hb0=a[2], lib=lib)
    np.testing.assert_allclose(full[0], np.concatenate([a[0], c[0]], axis=1), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(full[1], c[1], rtol=1e-12, atol=1e-12)


PINS = [pin_primal_form, pin_eta_zero_closed_form, pin_varlen_is_separate_runs, pin_state_continuation]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_ttt_pin(pin):
    pin()


TTT_MUTANTS = {
    "row_rate_in_update": ("const double el = J->eta[(size_t)(r1 - 1) * H + h];",
                           "const double el = J->eta[(size_t)r0 * H + h];"),
    "no_bias_path": ("kh[c] -= et * (a + 1.0) * V2[(size_t)(s - r0) * D + c];",
                     "kh[c] -= et * a * V2[(size_t)(s - r0) * D + c];"),
    "exclusive_mask": ("for (long s = r0; s <= t; ++s) {", "for (long s = r0; s < t; ++s) {"),
    "no_residual_norm": ("J->o[rb + c] = kh[c] + xh[c] * w[c] + b[c];", "J->o[rb + c] = kh[c];"),
    "no_residual_target": ("(xh[c] * w[c] + b[c] + widen(J->k, rb + c, J->dtype) - widen(J->v, rb + c, J->dtype))",
                           "(xh[c] * w[c] + b[c] - widen(J->v, rb + c, J->dtype))"),
    "ln_grad_sign": ("(D * gv[c] - sg - xh[c] * sgx)", "(D * gv[c] - sg + xh[c] * sgx)"),
}


@pytest.mark.parametrize("name", sorted(TTT_MUTANTS))
def test_ttt_pins_catch_planted_mistake(name, tmp_path):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "gla_oracle.c")).read()
    old, new = TTT_MUTANTS[name]
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", str(so), str(path), "-lm"])
    lib = oracle.load_variant(str(so))
    caught = []
    for pin in PINS:
        try:
            pin(lib=lib)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake {name}"
