"""Pins for the fp64 oracle (CPU only).

Each check compares the oracle with something that does not come from the oracle: a brute-force O(T^2)
quadratic form written from prefix sums of the gates, closed forms (g == 0 is plain causal linear
attention; K = V = 1 with a constant gate; k == 0 leaves only the decayed h0), exact structural
properties of the recurrence (state-split invariance, varlen == separate runs, permutation invariances,
linearity in scale) and hand-derived golden fixtures under tests/golden/.  The last group plants plausible
mistakes in compiled copies of the oracle and checks that the pins catch every one.
"""
import json
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle
from chunkwise_gated_linear_chunked_gb300.inputs import make_inputs, stored_numpy

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def rand_case(rng, B, T, H, K, V, h0=True, gate_scale=1.0 / 16):
    q = rng.standard_normal((B, T, H, K)).astype(np.float32)
    k = rng.standard_normal((B, T, H, K)).astype(np.float32)
    v = rng.standard_normal((B, T, H, V)).astype(np.float32)
    x = rng.standard_normal((B, T, H, K))
    g = (-np.logaddexp(0.0, -x) * gate_scale).astype(np.float32)   # logsigmoid(x) * gate_scale <= 0
    hh = (0.1 * rng.standard_normal((B, H, K, V))).astype(np.float32) if h0 else None
    return q, k, v, g, hh


def rel_err(x, y):
    d = np.linalg.norm((np.asarray(x) - np.asarray(y)).ravel())
    n = np.linalg.norm(np.asarray(y).ravel())
    return d / n if n > 0 else d


# ----------------------------------------------------------------------------------------------------
# Independent reference quantities
# ----------------------------------------------------------------------------------------------------

def brute_force_one(q, k, v, g, scale, h0):
    """O(T^2) quadratic form for one (sequence, head), from prefix sums of g (not from a recurrence):
    o_t = scale * sum_{s<=t} sum_c q_tc k_sc exp(sum_{u=s+1..t} g_uc) v_s
          + scale * sum_c q_tc exp(sum_{u<=t} g_uc) h0[c, :]
    ht  = sum_s diag(exp(sum_{u=s+1..T-1} g_u)) k_s^T v_s + diag(exp(sum_u g_u)) h0."""
    q, k, v, g = (np.asarray(a, dtype=np.float64) for a in (q, k, v, g))
    T, K = q.shape
    V = v.shape[1]
    L = np.concatenate([np.zeros((1, K)), np.cumsum(g, axis=0)])   # L[t+1] = sum_{u<=t} g_u
    o = np.zeros((T, V))
    for t in range(T):
        w = (q[t][None, :] * k[: t + 1] * np.exp(L[t + 1][None, :] - L[1: t + 2])).sum(axis=1)
        o[t] = scale * (w @ v[: t + 1])
        if h0 is not None:
            o[t] += scale * ((q[t] * np.exp(L[t + 1])) @ h0)
    ht = (k * np.exp(L[T][None, :] - L[1: T + 1])).T @ v
    if h0 is not None:
        ht = ht + np.exp(L[T])[:, None] * h0
    return o, ht


def brute_force(q, k, v, g, scale, h0):
    B, T, H, K = q.shape
    V = v.shape[-1]
    o = np.zeros((B, T, H, V))
    ht = np.zeros((B, H, K, V))
    for b in range(B):
        for h in range(H):
            hh = None if h0 is None else np.asarray(h0[b, h], dtype=np.float64)
            o[b, :, h], ht[b, h] = brute_force_one(q[b, :, h], k[b, :, h], v[b, :, h], g[b, :, h],
                                                   scale, hh)
    return o, ht


# ----------------------------------------------------------------------------------------------------
# The pins, written against a callable so the planted-mistake tests can rerun them on a mutant.
# ----------------------------------------------------------------------------------------------------

def pin_quadratic_form(lib=None):
    rng = np.random.default_rng(7)
    for T in (1, 2, 5, 63, 64, 65, 130):
        for K, V in ((1, 1), (2, 8), (8, 2)):
            q, k, v, g, h0 = rand_case(rng, 2, T, 2, K, V, h0=True)
            o, ht, _ = oracle.gla_fwd(q, k, v, g, 0.37, h0=h0, lib=lib)
            ob, hb = brute_force(q, k, v, g, 0.37, h0)
            assert rel_err(o, ob) < 1e-12, (T, K, V, rel_err(o, ob))
            assert rel_err(ht, hb) < 1e-12, (T, K, V, rel_err(ht, hb))


def pin_no_decay_is_causal_linear_attention(lib=None):
    """g == 0: o = scale * (tril(Q K^T) V + Q h0), ht = K^T V + h0 (per sequence and head)."""
    rng = np.random.default_rng(11)
    B, T, H, K, V = 2, 97, 3, 5, 7
    q, k, v, _, h0 = rand_case(rng, B, T, H, K, V)
    g = np.zeros_like(q)
    o, ht, _ = oracle.gla_fwd(q, k, v, g, 0.25, h0=h0, lib=lib)
    for b in range(B):
        for h in range(H):
            Q, Kk, Vv = (x[b, :, h].astype(np.float64) for x in (q, k, v))
            ref = 0.25 * (np.tril(Q @ Kk.T) @ Vv + Q @ h0[b, h])
            assert rel_err(o[b, :, h], ref) < 1e-12
            assert rel_err(ht[b, h], Kk.T @ Vv + h0[b, h]) < 1e-12


def pin_scalar_constant_gate(lib=None):
    """K = V = 1, g_t = gamma: o_t = scale q_t (sum_{s<=t} e^{gamma (t-s)} k_s v_s + e^{gamma (t+1)} h0)."""
    rng = np.random.default_rng(3)
    T = 200
    gamma = np.float32(-0.05)
    q, k, v, _, h0 = rand_case(rng, 1, T, 1, 1, 1)
    g = np.full_like(q, gamma)
    o, ht, _ = oracle.gla_fwd(q, k, v, g, 1.5, h0=h0, lib=lib)
    gm = float(gamma)
    qq, kk, vv = (x.reshape(T).astype(np.float64) for x in (q, k, v))
    h = float(h0.reshape(()))
    t = np.arange(T)
    ref = np.array([1.5 * qq[i] * (np.sum(np.exp(gm * (i - t[: i + 1])) * kk[: i + 1] * vv[: i + 1])
                                   + np.exp(gm * (i + 1)) * h) for i in range(T)])
    assert rel_err(o.reshape(T), ref) < 1e-12
    ht_ref = np.sum(np.exp(gm * (T - 1 - t)) * kk * vv) + np.exp(gm * T) * h
    assert abs(float(ht.reshape(())) - ht_ref) <= 1e-12 * abs(ht_ref)


def pin_initial_state_only(lib=None):
    """k == 0: o_t = scale (q_t * exp(sum_{u<=t} g_u)) h0 and ht = diag(exp(sum g)) h0."""
    rng = np.random.default_rng(5)
    B, T, H, K, V = 1, 150, 2, 6, 4
    q, _, v, g, h0 = rand_case(rng, B, T, H, K, V)
    k = np.zeros_like(q)
    o, ht, _ = oracle.gla_fwd(q, k, v, g, 0.5, h0=h0, lib=lib)
    for h in range(H):
        L = np.cumsum(g[0, :, h].astype(np.float64), axis=0)
        ref = 0.5 * (q[0, :, h] * np.exp(L)) @ h0[0, h]
        assert rel_err(o[0, :, h], ref) < 1e-12
        assert rel_err(ht[0, h], np.exp(L[-1])[:, None] * h0[0, h]) < 1e-12


def pin_state_split(lib=None):
    """Running [0, s) and feeding its ht as h0 to [s, T) reproduces the full run (bit for bit)."""
    rng = np.random.default_rng(13)
    B, T, H, K, V = 2, 130, 2, 4, 3
    q, k, v, g, h0 = rand_case(rng, B, T, H, K, V)
    o, ht, _ = oracle.gla_fwd(q, k, v, g, 0.3, h0=h0, lib=lib)
    for s in (1, 37, 64, 65, 129):
        sl = lambda x, a, b: np.ascontiguousarray(x[:, a:b])
        o1, h1, _ = oracle.gla_fwd(sl(q, 0, s), sl(k, 0, s), sl(v, 0, s), sl(g, 0, s), 0.3, h0=h0, lib=lib)
        o2, h2, _ = oracle.gla_fwd(sl(q, s, T), sl(k, s, T), sl(v, s, T), sl(g, s, T), 0.3, h0=h1, lib=lib)
        assert np.array_equal(np.concatenate([o1, o2], axis=1), o)
        assert np.array_equal(h2, ht)


def pin_varlen_equals_separate(lib=None):
    rng = np.random.default_rng(17)
    lengths = [5, 0, 64, 1, 70]
    T = sum(lengths)
    H, K, V = 2, 3, 4
    q, k, v, g, _ = rand_case(rng, 1, T, H, K, V, h0=False)
    h0 = (0.1 * rng.standard_normal((len(lengths), H, K, V))).astype(np.float32)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    o, ht, _ = oracle.gla_fwd(q, k, v, g, 0.7, h0=h0, cu_seqlens=cu, lib=lib)
    for n, (a, b) in enumerate(zip(cu[:-1], cu[1:])):
        sl = lambda x: np.ascontiguousarray(x[:, a:b])
        on, hn, _ = oracle.gla_fwd(sl(q), sl(k), sl(v), sl(g), 0.7, h0=h0[n: n + 1], lib=lib)
        assert np.array_equal(o[:, a:b], on)
        assert np.array_equal(ht[n: n + 1], hn)
    assert np.array_equal(ht[1], h0[1].astype(np.float64))   # empty sequence: ht = h0


def pin_invariances(lib=None):
    rng = np.random.default_rng(19)
    B, T, H, K, V = 2, 70, 3, 5, 4
    q, k, v, g, h0 = rand_case(rng, B, T, H, K, V)
    o, ht, _ = oracle.gla_fwd(q, k, v, g, 0.5, h0=h0, lib=lib)
    # heads and batch rows are independent problems
    ph, pb = np.array([2, 0, 1]), np.array([1, 0])
    P = lambda x: np.ascontiguousarray(x[pb][:, :, ph])
    o2, ht2, _ = oracle.gla_fwd(P(q), P(k), P(v), P(g), 0.5, h0=np.ascontiguousarray(h0[pb][:, ph]), lib=lib)
    assert np.array_equal(o2, o[pb][:, :, ph]) and np.array_equal(ht2, ht[pb][:, ph])
    # permuting key dims of q, k, g with the rows of h0 leaves o unchanged and permutes ht's rows
    pk = np.array([3, 1, 4, 0, 2])
    Kp = lambda x: np.ascontiguousarray(x[..., pk])
    o3, ht3, _ = oracle.gla_fwd(Kp(q), Kp(k), v, Kp(g), 0.5, h0=np.ascontiguousarray(h0[:, :, pk]), lib=lib)
    assert rel_err(o3, o) < 1e-13 and np.array_equal(ht3, ht[:, :, pk])
    # o is linear in scale, ht does not depend on it (power-of-two factor: exact)
    o4, ht4, _ = oracle.gla_fwd(q, k, v, g, 1.0, h0=h0, lib=lib)
    assert np.array_equal(o4, 2.0 * o) and np.array_equal(ht4, ht)


def load_golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.loads("".join(l for l in f if not l.lstrip().startswith("#")))


def pin_golden(lib=None):
    for name in ("scalar_half_decay.txt", "orientation_h0.txt", "per_key_decay.txt"):
        d = load_golden(name)
        s = d["shape"]
        B, T, H, K, V = s["B"], s["T"], s["H"], s["K"], s["V"]
        arr = lambda key, shp: np.asarray(d[key], dtype=np.float32).reshape(shp)
        h0 = None if d["h0"] is None else arr("h0", (B, H, K, V))
        o, ht, _ = oracle.gla_fwd(arr("q", (B, T, H, K)), arr("k", (B, T, H, K)), arr("v", (B, T, H, V)),
                                  arr("g", (B, T, H, K)), d["scale"], h0=h0, lib=lib)
        np.testing.assert_allclose(o.ravel(), d["o"], rtol=d["rtol"], atol=0, err_msg=name)
        np.testing.assert_allclose(ht.ravel(), d["ht"], rtol=d["rtol"], atol=0, err_msg=name)


PINS = [pin_quadratic_form, pin_no_decay_is_causal_linear_attention, pin_scalar_constant_gate,
        pin_initial_state_only, pin_state_split, pin_varlen_equals_separate, pin_invariances, pin_golden]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()


def test_bf16_inputs_widen_exactly():
    """The oracle reads bf16 words and widens them exactly: same result as the fp32 copy of the values."""
    inp = make_inputs("bf16", B=2, T=77, H=2, K=8, V=4, h0=True, seed=5)
    args16 = [stored_numpy(x) for x in (inp.q, inp.k, inp.v, inp.g)]
    args32 = [x.float().numpy() for x in (inp.q, inp.k, inp.v, inp.g)]
    # independent widening (bit shift) agrees with torch's bf16 -> fp32 conversion
    assert np.array_equal(oracle.bf16_words_to_f64(args16[0]), args32[0].astype(np.float64))
    o16, h16, _ = oracle.gla_fwd(*args16, inp.scale, h0=inp.h0.numpy())
    o32, h32, _ = oracle.gla_fwd(*args32, inp.scale, h0=inp.h0.numpy())
    assert np.array_equal(o16, o32) and np.array_equal(h16, h32)


def test_threads_do_not_change_result():
    rng = np.random.default_rng(23)
    q, k, v, g, h0 = rand_case(rng, 3, 50, 4, 4, 4)
    o1, h1, n1 = oracle.gla_fwd(q, k, v, g, 0.5, h0=h0, nthreads=1)
    o2, h2, n2 = oracle.gla_fwd(q, k, v, g, 0.5, h0=h0, nthreads=5)
    assert n1 == 1 and n2 == 5
    assert np.array_equal(o1, o2) and np.array_equal(h1, h2)


def test_oracle_rejects_bad_arguments():
    rng = np.random.default_rng(1)
    q, k, v, g, _ = rand_case(rng, 2, 8, 1, 2, 2, h0=False)
    with pytest.raises(ValueError):
        oracle.gla_fwd(q, k, v, g, 1.0, cu_seqlens=np.array([0, 8], np.int32))   # B != 1
    with pytest.raises(ValueError):
        oracle.gla_fwd(q[:1], k[:1], v[:1], g[:1], 1.0, cu_seqlens=np.array([0, 9], np.int32))
    with pytest.raises(TypeError):
        oracle.gla_fwd(q.astype(np.int32), k.astype(np.int32), v.astype(np.int32), g.astype(np.int32), 1.0)
    # mixed stored types (the method keeps g's type separate) are widened exactly: same as all-fp64
    mixed = oracle.gla_fwd(q, k, v, g.astype(np.float64), 1.0)[0]
    wide = oracle.gla_fwd(*(x.astype(np.float64) for x in (q, k, v, g)), 1.0)[0]
    assert np.array_equal(mixed, wide)


# ----------------------------------------------------------------------------------------------------
# Chunk-local cumsum
# ----------------------------------------------------------------------------------------------------

def test_chunk_local_cumsum_dense_and_ragged():
    rng = np.random.default_rng(29)
    for T, C in ((1, 64), (63, 64), (64, 64), (130, 64), (50, 16)):
        g = rng.standard_normal((2, T, 3, 5)).astype(np.float32)
        G = oracle.chunk_local_cumsum(g, C)
        ref = np.zeros_like(G)
        for c0 in range(0, T, C):
            ref[:, c0:c0 + C] = np.cumsum(g[:, c0:c0 + C].astype(np.float64), axis=1)
        assert np.allclose(G, ref, rtol=1e-14, atol=1e-14)


def test_chunk_local_cumsum_varlen_restarts_at_sequence_start():
    rng = np.random.default_rng(31)
    lengths = [3, 0, 64, 65, 1]
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    g = rng.standard_normal((1, int(cu[-1]), 2, 3)).astype(np.float32)
    G = oracle.chunk_local_cumsum(g, 64, cu_seqlens=cu)
    for a, b in zip(cu[:-1], cu[1:]):
        Gs = oracle.chunk_local_cumsum(np.ascontiguousarray(g[:, a:b]), 64)
        assert np.array_equal(G[:, a:b], Gs)


def test_chunk_local_cumsum_golden():
    d = load_golden("chunk_cumsum.txt")
    s = d["shape"]
    g = np.asarray(d["g"], dtype=np.float32).reshape(s["B"], s["T"], s["H"], s["K"])
    assert np.array_equal(oracle.chunk_local_cumsum(g, d["chunk"]).ravel(), np.asarray(d["G"], float))


# ----------------------------------------------------------------------------------------------------
# Planted mistakes: each mutant of gla_oracle.c must fail at least one pin.
# ----------------------------------------------------------------------------------------------------

MUTANTS = {
    "decay_after_add": ("row[j] = decay * row[j] + ki * widen(J->v, vb + j, J->dtype);",
                        "row[j] = decay * (row[j] + ki * widen(J->v, vb + j, J->dtype));"),
    "gate_sign": ("const double decay = exp(widen(J->g, kb + i, J->dtype));",
                  "const double decay = exp(-widen(J->g, kb + i, J->dtype));"),
    "dropped_h0": ("S[(size_t)i * V + j] = J->h0 ? J->h0[", "S[(size_t)i * V + j] = 0 ? J->h0["),
    "q_swapped_for_k": ("acc += widen(J->q, kb + i, J->dtype)", "acc += widen(J->k, kb + i, J->dtype)"),
    "previous_token_value": ("ki * widen(J->v, vb + j, J->dtype)",
                             "ki * (t > bos ? widen(J->v, vb - (size_t)H * V + j, J->dtype) : 0.0)"),
    "dropped_scale": ("J->o[vb + j] = J->scale * acc;", "J->o[vb + j] = acc;"),
    "exclusive_diagonal": ("row[j] = decay * row[j] + ki * widen(J->v, vb + j, J->dtype);\n        }\n"
                           "        for (int j = 0; j < V; ++j) {\n            double acc = 0.0;\n"
                           "            for (int i = 0; i < K; ++i)\n"
                           "                acc += widen(J->q, kb + i, J->dtype) * S[(size_t)i * V + j];",
                           "row[j] = decay * row[j] + ki * widen(J->v, vb + j, J->dtype);\n        }\n"
                           "        for (int j = 0; j < V; ++j) {\n            double acc = 0.0;\n"
                           "            for (int i = 0; i < K; ++i)\n"
                           "                acc += widen(J->q, kb + i, J->dtype) * (S[(size_t)i * V + j]"
                           " - widen(J->k, kb + i, J->dtype) * widen(J->v, vb + j, J->dtype));"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "gla_oracle.c")).read()
    old, new = MUTANTS[name]
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
