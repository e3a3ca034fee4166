"""Pins of the WY-representation oracle of the gated delta rule (CPU).

The oracle forms, per chunk of BT rows from each sequence start, u = A (v * beta) and w = A (k * beta * 2^g)
(page "fla/ops/gated_delta_rule/backends/triton_ascend/wy_fast.py": recompute_w_u_fwd_kernel_npu).  It is
pinned by what A means in the gated delta rule and by closed forms, none of which repeats its sum:
  * A = L^-1 for a unit lower-triangular L per chunk (inverted by numpy): then L u = beta v and
    L w = beta 2^g k, checked with numpy products, on dense batches and on varlen packs whose sequences
    start off the chunk grid, with ragged last chunks and shared key heads;
  * A = I: u = beta v and w = beta 2^g k exactly (integer g);
  * A = the all-ones lower triangle: u and w are chunk-local cumulative sums (numpy cumsum);
  * A = the reversal permutation (the upper triangle is used too): u_t = beta_r v_r with r mirrored;
  * key-head sharing: HV value heads over H key heads equals H' = HV with the key heads repeated;
and planted mistakes, each caught by at least one pin.
"""
import os
import subprocess

import numpy as np
import pytest

import oracle


def _bounds(B, T, lengths):
    if lengths is None:
        return [(n * T, n * T + T) for n in range(B)], None
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    return list(zip(cu[:-1].tolist(), cu[1:].tolist())), cu


def _chunks(bounds, BT):
    for bos, eos in bounds:
        for c0 in range(bos, eos, BT):
            yield c0, min(c0 + BT, eos)


def _inputs(seed, B, T, H, HV, K, V, lengths=None, int_gate=False):
    rng = np.random.default_rng(seed)
    if lengths is not None:
        B, T = 1, int(sum(lengths))
    k = rng.standard_normal((B, T, H, K))
    v = rng.standard_normal((B, T, HV, V))
    beta = rng.random((B, T, HV))
    g = np.round(-3 * rng.random((B, T, HV))) if int_gate else -2.0 * rng.random((B, T, HV))
    return k, v, beta, g, B, T


def _fill_A(B, T, HV, BT, bounds, block):
    """A [B, T, HV, BT] whose chunk matrices are block(m=BT, chunk index, head)."""
    A = np.zeros((B * T, HV, BT))
    for ci, (c0, c1) in enumerate(_chunks(bounds, BT)):
        for hv in range(HV):
            M = block(ci, hv)
            A[c0:c1, hv, :] = M[: c1 - c0, :]
    return A.reshape(B, T, HV, BT)


def pin_triangular_solve(lib=None):
    for seed, (B, T, H, HV, K, V, BT, lengths) in enumerate([
            (2, 150, 1, 1, 5, 3, 64, None),
            (1, 0, 2, 4, 4, 6, 16, [1, 15, 16, 17, 0, 40, 7]),
            (1, 0, 1, 2, 3, 3, 64, [63, 65, 130])]):
        k, v, beta, g, B, T = _inputs(seed, B, T, H, HV, K, V, lengths)
        bounds, cu = _bounds(B, T, lengths)
        rng = np.random.default_rng(100 + seed)
        Ls = {}

        def block(ci, hv):
            L = np.eye(BT) + np.tril(0.3 * rng.standard_normal((BT, BT)), -1)
            Ls[ci, hv] = L
            return np.linalg.inv(L)

        A = _fill_A(B, T, HV, BT, bounds, block)
        w, u = oracle.wy_fwd(k, v, beta, A, g, cu_seqlens=cu, lib=lib)
        rows = lambda x: x.reshape(B * T, *x.shape[2:])
        kr, vr, br, gr, wr, ur = map(rows, (k, v, beta, g, w, u))
        for ci, (c0, c1) in enumerate(_chunks(bounds, BT)):
            m = c1 - c0
            for hv in range(HV):
                L = Ls[ci, hv][:m, :m]
                np.testing.assert_allclose(L @ ur[c0:c1, hv], br[c0:c1, hv, None] * vr[c0:c1, hv],
                                           rtol=1e-10, atol=1e-10)
                kk = kr[c0:c1, hv // (HV // H)]
                np.testing.assert_allclose(L @ wr[c0:c1, hv], (br[c0:c1, hv] * 2.0 ** gr[c0:c1, hv])[:, None] * kk,
                                           rtol=1e-10, atol=1e-10)


def pin_identity_closed_form(lib=None):
    B, T, H, HV, K, V, BT = 2, 70, 1, 2, 4, 5, 32
    k, v, beta, g, B, T = _inputs(7, B, T, H, HV, K, V, int_gate=True)
    bounds, _ = _bounds(B, T, None)
    A = _fill_A(B, T, HV, BT, bounds, lambda ci, hv: np.eye(BT))
    w, u = oracle.wy_fwd(k, v, beta, A, g, lib=lib)
    np.testing.assert_array_equal(u, beta[..., None] * v)
    kk = np.repeat(k, HV // H, axis=2)
    np.testing.assert_array_equal(w, (beta * 2.0 ** g)[..., None] * kk)
    w0, _ = oracle.wy_fwd(k, v, beta, A, None, lib=lib)     # no gate: the factor is 1
    np.testing.assert_array_equal(w0, beta[..., None] * kk)


def pin_lower_ones_is_chunk_cumsum(lib=None):
    lengths, H, HV, K, V, BT = [5, 40, 33], 1, 1, 3, 4, 16
    k, v, beta, g, B, T = _inputs(11, 1, 0, H, HV, K, V, lengths)
    bounds, cu = _bounds(B, T, lengths)
    A = _fill_A(B, T, HV, BT, bounds, lambda ci, hv: np.tril(np.ones((BT, BT))))
    w, u = oracle.wy_fwd(k, v, beta, A, g, cu_seqlens=cu, lib=lib)
    for c0, c1 in _chunks(bounds, BT):
        bv = beta[0, c0:c1, 0, None] * v[0, c0:c1, 0]
        bk = (beta[0, c0:c1, 0] * 2.0 ** g[0, c0:c1, 0])[:, None] * k[0, c0:c1, 0]
        np.testing.assert_allclose(u[0, c0:c1, 0], np.cumsum(bv, axis=0), rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(w[0, c0:c1, 0], np.cumsum(bk, axis=0), rtol=1e-12, atol=1e-12)


def pin_full_square_permutation(lib=None):
    B, T, H, HV, K, V, BT = 1, 48, 1, 1, 2, 3, 16
    k, v, beta, g, B, T = _inputs(13, B, T, H, HV, K, V, int_gate=True)
    bounds, _ = _bounds(B, T, None)
    A = _fill_A(B, T, HV, BT, bounds, lambda ci, hv: np.eye(BT)[::-1])
    w, u = oracle.wy_fwd(k, v, beta, A, g, lib=lib)
    for c0, c1 in _chunks(bounds, BT):
        r = np.arange(c1 - 1, c0 - 1, -1)
        np.testing.assert_array_equal(u[0, c0:c1, 0], beta[0, r, 0, None] * v[0, r, 0])
        np.testing.assert_array_equal(w[0, c0:c1, 0], (beta[0, r, 0] * 2.0 ** g[0, r, 0])[:, None] * k[0, r, 0])


def pin_key_head_sharing(lib=None):
    B, T, H, HV, K, V, BT = 2, 50, 2, 4, 3, 2, 16
    k, v, beta, g, B, T = _inputs(17, B, T, H, HV, K, V)
    bounds, _ = _bounds(B, T, None)
    rng = np.random.default_rng(5)
    A = _fill_A(B, T, HV, BT, bounds, lambda ci, hv: rng.standard_normal((BT, BT)))
    w, u = oracle.wy_fwd(k, v, beta, A, g, lib=lib)
    w2, u2 = oracle.wy_fwd(np.repeat(k, HV // H, axis=2), v, beta, A, g, lib=lib)
    np.testing.assert_array_equal(w, w2)
    np.testing.assert_array_equal(u, u2)
    assert not np.allclose(w[:, :, 1], w[:, :, 2])   # heads 1 and 2 read different key heads


def pin_bf16_widens_exactly(lib=None):
    import torch
    B, T, H, HV, K, V, BT = 1, 40, 1, 1, 4, 4, 16
    k, v, beta, g, B, T = _inputs(19, B, T, H, HV, K, V)
    bounds, _ = _bounds(B, T, None)
    rng = np.random.default_rng(9)
    A = _fill_A(B, T, HV, BT, bounds, lambda ci, hv: rng.standard_normal((BT, BT)))
    words = lambda x: torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    exact = lambda x: torch.from_numpy(x).to(torch.bfloat16).double().numpy()
    wa, ua = oracle.wy_fwd(*(words(x) for x in (k, v, beta, A)), g, lib=lib)
    wb, ub = oracle.wy_fwd(*(exact(x) for x in (k, v, beta, A)), g, lib=lib)
    np.testing.assert_array_equal(wa, wb)
    np.testing.assert_array_equal(ua, ub)


PINS = [pin_triangular_solve, pin_identity_closed_form, pin_lower_ones_is_chunk_cumsum, pin_full_square_permutation,
        pin_key_head_sharing, pin_bf16_widens_exactly]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_wy_pin(pin):
    pin()


WY_MUTANTS = {
    "transposed_A": ("widen(J->A, ((size_t)t * HV + hv) * BT + (size_t)(s - c0), J->dtype)",
                     "widen(J->A, ((size_t)s * HV + hv) * BT + (size_t)(t - c0), J->dtype)"),
    "chunks_on_global_grid": ("for (long c0 = first; c0 < end; c0 += BT) {",
                              "for (long c0 = first - first % BT; c0 < end; c0 += BT) {"),
    "natural_exp_gate": ("exp2(J->g[(size_t)s * HV + hv])", "exp(J->g[(size_t)s * HV + hv])"),
    "key_head_modulo": ("hk = hv / (HV / J->H);", "hk = hv % J->H;"),
    "gate_on_u": ("urow[c] += coef * widen(", "urow[c] += coef * decay * widen("),
    "lower_triangle_only": ("for (long s = c0; s < c1; ++s) {", "for (long s = c0; s <= t; ++s) {"),
    "beta_dropped_from_w": ("wrow[c] += coef * decay * widen(J->k",
                            "wrow[c] += coef / widen(J->beta, (size_t)s * HV + hv, J->dtype) * decay * widen(J->k"),
}


@pytest.mark.parametrize("name", sorted(WY_MUTANTS))
def test_wy_pins_catch_planted_mistake(name, tmp_path):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "gla_oracle.c")).read()
    old, new = WY_MUTANTS[name]
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
