"""Pins for the fp64 oracle, checked against what the mathematics fixes.

The pages print no worked numeric example, so every pin here is a closed form,
an invariant, an independent brute-force or library computation, or a finite
difference.  ``test_planted_mistakes_are_caught`` plants plausible mistakes in
a copy of the oracle and checks that at least one pin fails for each.
"""

import math

import numpy as np
import pytest
import torch

from oracle import fa_oracle as orc
from tiled_attention_fa_gb300.inputs import make_qkv

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def rnd(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


# ---------------------------------------------------------------- forward pins

@pytest.mark.parametrize("causal", [False, True])
def test_softmax_rows_sum_to_one(causal):
    # With D = L and V = identity, O is the probability matrix itself.
    L = 24
    q, k = rnd((L, L), 1), rnd((L, L), 2)
    P, _ = orc.unit_forward(q, k, np.eye(L), causal)
    assert np.all(P >= 0)
    np.testing.assert_allclose(P.sum(axis=1), 1.0, atol=1e-12)
    if causal:
        assert np.all(P[np.triu_indices(L, 1)] == 0.0)


@pytest.mark.parametrize("causal", [False, True])
def test_constant_values_give_that_value(causal):
    L, D = 37, 16
    v_row = rnd((D,), 3)
    o, _ = orc.unit_forward(rnd((L, D), 4) * 3, rnd((L, D), 5) * 3,
                            np.tile(v_row, (L, 1)), causal)
    np.testing.assert_allclose(o, np.tile(v_row, (L, 1)), atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_zero_queries_give_mean_of_values(causal):
    L, D = 29, 8
    v = rnd((L, D), 6)
    o, lse = orc.unit_forward(np.zeros((L, D)), rnd((L, D), 7), v, causal)
    if causal:
        want = np.cumsum(v, axis=0) / np.arange(1, L + 1)[:, None]
        want_lse = np.log(np.arange(1, L + 1))
    else:
        want = np.tile(v.mean(axis=0), (L, 1))
        want_lse = np.full(L, math.log(L))
    np.testing.assert_allclose(o, want, atol=1e-12)
    np.testing.assert_allclose(lse, want_lse, atol=1e-12)


def test_causal_first_row_is_first_value():
    L, D = 20, 8
    q, k, v = rnd((L, D), 8), rnd((L, D), 9), rnd((L, D), 10)
    o, lse = orc.unit_forward(q, k, v, True)
    np.testing.assert_allclose(o[0], v[0], atol=1e-14)
    assert lse[0] == pytest.approx(q[0] @ k[0] / math.sqrt(D), abs=1e-13)


def test_two_key_closed_form():
    # Scores [x, 0] give weights [sigmoid(x), 1 - sigmoid(x)] and LSE ln(e^x + 1).
    D = 4
    for x in (-3.0, 0.0, 0.7, 5.0):
        q = np.array([[2.0 * x, 0, 0, 0]])            # q.k0 / sqrt(4) = x
        k = np.array([[1.0, 0, 0, 0], [0, 0, 0, 0]])
        v = np.array([[1.0, 2, 3, 4], [-1.0, 0, 5, 0]])
        o, lse = orc.unit_forward(q, k, v, False)
        p = 1.0 / (1.0 + math.exp(-x))
        np.testing.assert_allclose(o[0], p * v[0] + (1 - p) * v[1], atol=1e-14)
        assert lse[0] == pytest.approx(math.log(math.exp(x) + 1.0), abs=1e-14)


def test_permuting_keys_and_values_together():
    L, D = 33, 16
    q, k, v = rnd((L, D), 11), rnd((L, D), 12), rnd((L, D), 13)
    perm = np.random.default_rng(14).permutation(L)
    o1, l1 = orc.unit_forward(q, k, v, False)
    o2, l2 = orc.unit_forward(q, k[perm], v[perm], False)
    np.testing.assert_allclose(o1, o2, atol=1e-12)
    np.testing.assert_allclose(l1, l2, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_shifting_every_key(causal):
    L, D = 25, 8
    q, k, v = rnd((L, D), 15), rnd((L, D), 16), rnd((L, D), 17)
    c = rnd((D,), 18)
    o1, l1 = orc.unit_forward(q, k, v, causal)
    o2, l2 = orc.unit_forward(q, k + c, v, causal)
    np.testing.assert_allclose(o1, o2, atol=1e-12)
    np.testing.assert_allclose(l2 - l1, q @ c / math.sqrt(D), atol=1e-12)


def brute_force_forward(q, k, v, causal):
    """Straight-line loops over scalars, independent of the oracle's numpy code."""
    B, L, H, D = q.shape
    Hkv = k.shape[2]
    o = np.zeros((B, L, H, D))
    lse = np.zeros((B, H, L))
    for b in range(B):
        for h in range(H):
            hk = h // (H // Hkv)
            for i in range(L):
                s = []
                for j in range(L):
                    if causal and j > i:
                        continue
                    s.append((j, sum(q[b, i, h, d] * k[b, j, hk, d] for d in range(D)) / math.sqrt(D)))
                mx = max(x for _, x in s)
                z = sum(math.exp(x - mx) for _, x in s)
                lse[b, h, i] = mx + math.log(z)
                for d in range(D):
                    o[b, i, h, d] = sum(math.exp(x - mx) / z * v[b, j, hk, d] for j, x in s)
    return o, lse


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("H,Hkv", [(1, 1), (4, 2)])
def test_brute_force_small(causal, H, Hkv):
    B, L, D = 2, 7, 5
    q, k, v = rnd((B, L, H, D), 19), rnd((B, L, Hkv, D), 20), rnd((B, L, Hkv, D), 21)
    o, lse = orc.forward(q, k, v, causal)
    ob, lb = brute_force_forward(q, k, v, causal)
    np.testing.assert_allclose(o, ob, atol=1e-12)
    np.testing.assert_allclose(lse, lb, atol=1e-12)


def torch_reference(q, k, v, do, causal):
    """torch's own float64 attention and autograd, a separately written library path."""
    H, Hkv = q.shape[2], k.shape[2]
    g = H // Hkv
    tq = torch.tensor(q).permute(0, 2, 1, 3).requires_grad_()
    tk = torch.tensor(k).permute(0, 2, 1, 3).requires_grad_()
    tv = torch.tensor(v).permute(0, 2, 1, 3).requires_grad_()
    kk = tk.repeat_interleave(g, dim=1)
    vv = tv.repeat_interleave(g, dim=1)
    out = torch.nn.functional.scaled_dot_product_attention(tq, kk, vv, is_causal=causal)
    out.backward(torch.tensor(do).permute(0, 2, 1, 3))
    f = lambda t: t.detach().permute(0, 2, 1, 3).numpy()
    return f(out), f(tq.grad), f(tk.grad), f(tv.grad)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("H,Hkv", [(2, 2), (4, 1)])
def test_matches_torch_float64_reference(causal, H, Hkv):
    B, L, D = 2, 45, 16
    q, k, v, do = (rnd((B, L, h, D), s) for h, s in ((H, 22), (Hkv, 23), (Hkv, 24), (H, 25)))
    o, _ = orc.forward(q, k, v, causal)
    dq, dk, dv, _ = orc.backward(q, k, v, do, causal)
    to, tdq, tdk, tdv = torch_reference(q, k, v, do, causal)
    for a, b in ((o, to), (dq, tdq), (dk, tdk), (dv, tdv)):
        np.testing.assert_allclose(a, b, atol=1e-11, rtol=1e-9)


def test_gqa_equals_mha_on_repeated_heads():
    B, L, H, Hkv, D = 1, 19, 6, 2, 8
    q, k, v, do = rnd((B, L, H, D), 26), rnd((B, L, Hkv, D), 27), rnd((B, L, Hkv, D), 28), rnd((B, L, H, D), 29)
    kr, vr = np.repeat(k, H // Hkv, axis=2), np.repeat(v, H // Hkv, axis=2)
    for causal in (False, True):
        o1, l1 = orc.forward(q, k, v, causal)
        o2, l2 = orc.forward(q, kr, vr, causal)
        np.testing.assert_allclose(o1, o2, atol=1e-14)
        np.testing.assert_allclose(l1, l2, atol=1e-14)
        dq1, dk1, dv1, _ = orc.backward(q, k, v, do, causal)
        dq2, dk2, dv2, _ = orc.backward(q, kr, vr, do, causal)
        np.testing.assert_allclose(dq1, dq2, atol=1e-13)
        g = H // Hkv
        np.testing.assert_allclose(dk1, dk2.reshape(B, L, Hkv, g, D).sum(axis=3), atol=1e-13)
        np.testing.assert_allclose(dv1, dv2.reshape(B, L, Hkv, g, D).sum(axis=3), atol=1e-13)


# ---------------------------------------------------------------- backward pins

@pytest.mark.parametrize("causal", [False, True])
def test_gradients_match_central_finite_differences(causal):
    B, L, H, Hkv, D = 1, 5, 2, 1, 4
    q, k, v, do = rnd((B, L, H, D), 30), rnd((B, L, Hkv, D), 31), rnd((B, L, Hkv, D), 32), rnd((B, L, H, D), 33)
    dq, dk, dv, _ = orc.backward(q, k, v, do, causal)

    def f(qq, kk, vv):
        return float((orc.forward(qq, kk, vv, causal)[0] * do).sum())

    eps = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = {"q": q, "k": k, "v": v}
            args_m = dict(args_p)
            args_p[name], args_m[name] = xp, xm
            num[idx] = (f(args_p["q"], args_p["k"], args_p["v"]) -
                        f(args_m["q"], args_m["k"], args_m["v"])) / (2 * eps)
        rel = np.abs(num - g).max() / max(1.0, np.abs(g).max())
        assert rel < 1e-6, (name, rel)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_column_sums(causal):
    # sum_j dV_j = sum_i dO_i (rows of P sum to 1); sum_j dK_j = 0 (rows of dS sum to 0).
    B, L, H, Hkv, D = 2, 31, 4, 2, 8
    q, k, v, do = rnd((B, L, H, D), 34), rnd((B, L, Hkv, D), 35), rnd((B, L, Hkv, D), 36), rnd((B, L, H, D), 37)
    _, dk, dv, _ = orc.backward(q, k, v, do, causal)
    g = H // Hkv
    do_sum = do.reshape(B, L, Hkv, g, D).sum(axis=(1, 3))
    np.testing.assert_allclose(dv.sum(axis=1), do_sum, atol=1e-11)
    np.testing.assert_allclose(dk.sum(axis=1), 0.0, atol=1e-11)


def test_delta_is_rowwise_dot_product():
    B, L, H, D = 2, 9, 3, 4
    o, do = rnd((B, L, H, D), 38), rnd((B, L, H, D), 39)
    got = orc.bwd_preprocess(o, do)
    for b in range(B):
        for h in range(H):
            for i in range(L):
                want = sum(o[b, i, h, d] * do[b, i, h, d] for d in range(D))
                assert got[b, h, i] == pytest.approx(want, abs=1e-13)


def test_backward_delta_uses_its_own_output():
    B, L, H, D = 1, 12, 2, 8
    q, k, v, do = rnd((B, L, H, D), 40), rnd((B, L, H, D), 41), rnd((B, L, H, D), 42), rnd((B, L, H, D), 43)
    o, _ = orc.forward(q, k, v, True)
    _, _, _, delta = orc.backward(q, k, v, do, True)
    np.testing.assert_allclose(delta, orc.bwd_preprocess(o, do), atol=1e-13)


def test_row_panels_do_not_change_results():
    L, D = 70, 8
    q, k, v, do = rnd((L, D), 44), rnd((L, D), 45), rnd((L, D), 46), rnd((L, D), 47)
    for causal in (False, True):
        a = orc.unit_backward(q, k, v, do, causal)
        b = orc.unit_backward(q, k, v, do, causal, panel=16)
        for x, y in zip(a, b):
            np.testing.assert_allclose(x, y, atol=1e-13)
        o1, l1 = orc.unit_forward(q, k, v, causal)
        o2, l2 = orc.unit_forward(q, k, v, causal, panel=9)
        np.testing.assert_allclose(o1, o2, atol=1e-14)
        np.testing.assert_allclose(l1, l2, atol=1e-14)


def test_sampled_rows_match_full_rows():
    L, D = 50, 8
    q, k, v = rnd((L, D), 48), rnd((L, D), 49), rnd((L, D), 50)
    rows = np.array([0, 3, 17, 49])
    for causal in (False, True):
        o_full, l_full = orc.unit_forward(q, k, v, causal)
        o_s, l_s = orc.unit_forward(q, k, v, causal, rows=rows)
        np.testing.assert_allclose(o_s, o_full[rows], atol=1e-14)
        np.testing.assert_allclose(l_s, l_full[rows], atol=1e-14)


def test_inputs_are_seeded_and_rounded():
    a = make_qkv(1, 8, 2, 1, 16, "fp16", seed=3)
    b = make_qkv(1, 8, 2, 1, 16, "fp16", seed=3)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    assert a[0].dtype == torch.float16 and a[1].shape == (1, 8, 1, 16)
    c = make_qkv(1, 8, 2, 1, 16, "bf16", seed=3)
    assert c[0].dtype == torch.bfloat16


# ---------------------------------------------------------------- golden fixture

def test_golden_config_small_fixture():
    """Stored oracle values for the B1 H2 L128 D64 fp16 seed-0 case (written by
    tests/golden/make_golden.py, which calls only the oracle)."""
    import json
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "fwd_b1_h2_l128_d64_seed0.json")
    with open(path) as fh:
        gold = json.load(fh)
    q, k, v, _ = make_qkv(1, 128, 2, 2, 64, "fp16", seed=0, with_do=False)
    o, lse = orc.forward(q.double().numpy(), k.double().numpy(), v.double().numpy(), False)
    for rec in gold["rows"]:
        np.testing.assert_allclose(o[0, rec["i"], rec["h"]], rec["o"], atol=1e-12)
        assert lse[0, rec["h"], rec["i"]] == pytest.approx(rec["lse"], abs=1e-12)


# ---------------------------------------------------------------- pins have teeth

def _mutant_forward(kind):
    def fwd(q_bh, k_bh, v_bh, causal, rows=None, panel=4096):
        L, D = q_bh.shape
        scale = {"no_sqrt": 1.0 / D, "no_scale": 1.0}.get(kind, 1.0 / math.sqrt(D))
        kk = k_bh
        S = (q_bh @ kk.T) * scale
        if kind == "transposed":
            S = S.T
        if causal:
            mask = np.arange(L)[None, :] > np.arange(L)[:, None]
            if kind == "mask_below":
                mask = mask.T
            if kind == "mask_inclusive":
                mask = np.arange(L)[None, :] >= np.arange(L)[:, None]
            S = np.where(mask, -np.inf, S)
        m = S.max(axis=1, keepdims=True)
        E = np.exp(S - m)
        if kind == "colsum":
            P = E / E.sum(axis=0, keepdims=True)
        else:
            P = E / E.sum(axis=1, keepdims=True)
        lse = m[:, 0] + np.log(E.sum(axis=1))
        if kind == "lse_no_max":
            lse = np.log(E.sum(axis=1))
        return P @ v_bh, lse
    return fwd


def _forward_pins(fwd):
    """Run the forward pins against ``fwd``; return True when they all pass."""
    try:
        L, D = 12, 12
        for causal in (False, True):
            P, _ = fwd(rnd((L, D), 1), rnd((L, D), 2), np.eye(L), causal)
            np.testing.assert_allclose(P.sum(axis=1), 1.0, atol=1e-12)
            v = rnd((L, D), 6)
            o, lse = fwd(np.zeros((L, D)), rnd((L, D), 7), v, causal)
            want = (np.cumsum(v, axis=0) / np.arange(1, L + 1)[:, None]) if causal else np.tile(v.mean(0), (L, 1))
            np.testing.assert_allclose(o, want, atol=1e-12)
            want_lse = np.log(np.arange(1, L + 1)) if causal else np.full(L, math.log(L))
            np.testing.assert_allclose(lse, want_lse, atol=1e-12)
        B, L2, D2 = 1, 6, 3
        q, k, v = rnd((B, L2, 1, D2), 19), rnd((B, L2, 1, D2), 20), rnd((B, L2, 1, D2), 21)
        for causal in (False, True):
            ob, lb = brute_force_forward(q, k, v, causal)
            o, lse = fwd(q[0, :, 0], k[0, :, 0], v[0, :, 0], causal)
            np.testing.assert_allclose(o, ob[0, :, 0], atol=1e-12)
            np.testing.assert_allclose(lse, lb[0, 0], atol=1e-12)
        return True
    except AssertionError:
        return False


def test_planted_mistakes_are_caught():
    assert _forward_pins(orc.unit_forward), "pins must pass on the oracle itself"
    for kind in ("no_sqrt", "no_scale", "transposed", "mask_below", "mask_inclusive",
                 "colsum", "lse_no_max"):
        assert not _forward_pins(_mutant_forward(kind)), f"planted mistake {kind!r} not caught"


def _mutant_backward(kind):
    def bwd(q_bh, k_bh, v_bh, do_bh, causal, panel=4096):
        L, D = q_bh.shape
        inv = 1.0 / math.sqrt(D)
        S = (q_bh @ k_bh.T) * inv
        if causal:
            S = np.where(np.arange(L)[None, :] > np.arange(L)[:, None], -np.inf, S)
        m = S.max(axis=1, keepdims=True)
        E = np.exp(S - m)
        P = E / E.sum(axis=1, keepdims=True)
        O = P @ v_bh
        dl = (O * do_bh).sum(axis=1)
        dv = (P @ do_bh) if kind == "dv_untransposed" else (P.T @ do_bh)
        dP = do_bh @ v_bh.T
        dS = P * dP if kind == "no_delta" else P * (dP - dl[:, None])
        dq = dS @ k_bh * (1.0 if kind == "dq_unscaled" else inv)
        dk = (dS @ q_bh if kind == "dk_untransposed" else dS.T @ q_bh) * inv
        return dq, dk, dv
    return bwd


def _backward_pins(bwd):
    try:
        L, D = 5, 4
        q, k, v, do = rnd((L, D), 60), rnd((L, D), 61), rnd((L, D), 62), rnd((L, D), 63)
        for causal in (False, True):
            dq, dk, dv = bwd(q, k, v, do, causal)[:3]
            np.testing.assert_allclose(dv.sum(axis=0), do.sum(axis=0), atol=1e-11)
            np.testing.assert_allclose(dk.sum(axis=0), 0.0, atol=1e-11)

            def f(qq, kk, vv):
                return float((orc.unit_forward(qq, kk, vv, causal)[0] * do).sum())
            eps = 1e-6
            for i, (x, g) in enumerate(((q, dq), (k, dk), (v, dv))):
                num = np.zeros_like(x)
                for idx in np.ndindex(x.shape):
                    args_p, args_m = [q, k, v], [q, k, v]
                    xp, xm = x.copy(), x.copy()
                    xp[idx] += eps
                    xm[idx] -= eps
                    args_p[i], args_m[i] = xp, xm
                    num[idx] = (f(*args_p) - f(*args_m)) / (2 * eps)
                assert np.abs(num - g).max() / max(1.0, np.abs(g).max()) < 1e-6
        return True
    except AssertionError:
        return False


def test_planted_backward_mistakes_are_caught():
    assert _backward_pins(orc.unit_backward), "pins must pass on the oracle itself"
    for kind in ("dv_untransposed", "no_delta", "dq_unscaled", "dk_untransposed"):
        assert not _backward_pins(_mutant_backward(kind)), f"planted mistake {kind!r} not caught"


# ---------------------------------------------------------------- storage rounding

@pytest.mark.parametrize("fmt,tdt", [("fp16", torch.float16), ("bf16", torch.bfloat16)])
def test_storage_round_matches_torch_casts(fmt, tdt):
    rng = np.random.default_rng(70)
    x = rng.standard_normal(20000) * np.exp(rng.uniform(-8, 8, 20000))
    want = torch.tensor(x, dtype=torch.float32).to(tdt).double().numpy()
    np.testing.assert_array_equal(orc.storage_round(x, fmt), want)


def test_storage_round_ties_and_identity():
    # bf16 keeps 8 significant bits: 1 + 2^-8 is a tie between 1 and 1 + 2^-7 -> even (1.0);
    # 1 + 3 * 2^-8 is a tie between 1 + 2^-7 and 1 + 2^-6 -> even (1 + 2^-6).
    assert orc.storage_round(np.array([1 + 2.0 ** -8]), "bf16")[0] == 1.0
    assert orc.storage_round(np.array([1 + 3 * 2.0 ** -8]), "bf16")[0] == 1 + 2.0 ** -6
    assert orc.storage_round(np.array([1 + 2.0 ** -11]), "fp16")[0] == 1.0
    vals = np.array([0.0, -2.5, 0.09375, 1024.0])
    for fmt in ("fp16", "bf16", None):
        np.testing.assert_array_equal(orc.storage_round(vals, fmt), vals)


def test_rounded_delta_only_moves_delta():
    # Rounding O before Delta leaves dV unchanged and moves Delta by at most the rounding.
    B, L, H, D = 1, 40, 2, 16
    q, k, v, do = (rnd((B, L, H, D), s) for s in (80, 81, 82, 83))
    dq0, dk0, dv0, d0 = orc.backward(q, k, v, do, True)
    dq1, dk1, dv1, d1 = orc.backward(q, k, v, do, True, o_round="bf16")
    np.testing.assert_array_equal(dv0, dv1)
    o, _ = orc.forward(q, k, v, True)
    bound = 2.0 ** -9 * np.einsum("blhd->bhl", np.abs(o * do))
    assert np.all(np.abs(d1 - d0) <= bound + 1e-15)
    assert np.abs(d1 - d0).max() > 0


@pytest.mark.parametrize("fmt,tdt", [("bf16", torch.bfloat16), ("fp16", torch.float16)])
def test_cast_p_only_moves_dv(fmt, tdt):
    # P cast for the dV product: dV equals P (torch's softmax, cast by torch) times dO;
    # dQ, dK and Delta are those of the exact P.
    B, L, H, Hkv, D = 1, 33, 4, 2, 16
    q, k, v, do = (rnd((B, L, h, D), s) for h, s in ((H, 90), (Hkv, 91), (Hkv, 92), (H, 93)))
    dq0, dk0, dv0, d0 = orc.backward(q, k, v, do, True)
    dq1, dk1, dv1, d1 = orc.backward(q, k, v, do, True, p_round=fmt)
    np.testing.assert_array_equal(dq0, dq1)
    np.testing.assert_array_equal(dk0, dk1)
    np.testing.assert_array_equal(d0, d1)
    qt, kt, dot = (torch.from_numpy(x) for x in (q, k, do))
    mask = torch.ones(L, L, dtype=torch.bool).tril()
    ref = torch.zeros(B, L, Hkv, D, dtype=torch.float64)
    for h in range(H):
        hk = h // (H // Hkv)
        s = qt[0, :, h] @ kt[0, :, hk].T / math.sqrt(D)
        p = torch.softmax(s.masked_fill(~mask, float("-inf")), dim=1)
        ref[0, :, hk] += p.to(torch.float32).to(tdt).double().T @ dot[0, :, h]
    np.testing.assert_allclose(dv1, ref.numpy(), rtol=1e-12, atol=1e-12)
    assert np.abs(dv1 - dv0).max() > 0


def test_cast_p_exact_when_p_is_representable():
    # Zero queries: row i of P is 1/L (non-causal, L a power of two) -- exact in 16 bits.
    B, L, H, D = 1, 32, 2, 8
    q = np.zeros((B, L, H, D))
    k, v, do = (rnd((B, L, H, D), s) for s in (94, 95, 96))
    for fmt in ("bf16", "fp16"):
        _, _, dv0, _ = orc.backward(q, k, v, do, False)
        _, _, dv1, _ = orc.backward(q, k, v, do, False, p_round=fmt)
        np.testing.assert_allclose(dv1, dv0, rtol=0, atol=1e-14)


def _torch_unit(qt, kt, vt, dot, h, hk, causal):
    """Independent float64 torch computation of one (b=0, h) unit: S, E = exp(S - m),
    row sum l, P, dP, exact O."""
    L, D = qt.shape[1], qt.shape[3]
    s = qt[0, :, h] @ kt[0, :, hk].T / math.sqrt(D)
    if causal:
        s = s.masked_fill(~torch.ones(L, L, dtype=torch.bool).tril(), float("-inf"))
    m = s.max(dim=1, keepdim=True).values
    e = torch.exp(s - m)
    l = e.sum(dim=1, keepdim=True)
    p = e / l
    return e, l, p, dot[0, :, h] @ vt[0, :, hk].T, p @ vt[0, :, hk]


@pytest.mark.parametrize("fmt,tdt", [("bf16", torch.bfloat16), ("fp16", torch.float16)])
@pytest.mark.parametrize("causal", [False, True])
def test_forward_cast_matches_torch(fmt, tdt, causal):
    # O = cast(exp(S - m)) V / l with l the unrounded row sum; LSE is unchanged.
    B, L, H, Hkv, D = 1, 37, 4, 2, 16
    q, k, v = (rnd((B, L, h, D), s) for h, s in ((H, 100), (Hkv, 101), (Hkv, 102)))
    o0, lse0 = orc.forward(q, k, v, causal)
    o1, lse1 = orc.forward(q, k, v, causal, p_round=fmt)
    np.testing.assert_array_equal(lse0, lse1)
    qt, kt, vt = (torch.from_numpy(x) for x in (q, k, v))
    for h in range(H):
        hk = h // (H // Hkv)
        e, l, _, _, _ = _torch_unit(qt, kt, vt, qt, h, hk, causal)
        want = (e.to(torch.float32).to(tdt).double() @ vt[0, :, hk]) / l
        np.testing.assert_allclose(o1[0, :, h], want.numpy(), rtol=1e-12, atol=1e-12)
    # the cast moves O by at most half an ulp of each weight: |dO| <= u sum_j P_j |V_j|
    u = {"bf16": 2.0 ** -8, "fp16": 2.0 ** -11}[fmt]
    p = np.stack([_torch_unit(qt, kt, vt, qt, h, h // (H // Hkv), causal)[2].numpy()
                  for h in range(H)], axis=1)                     # [L, H, L]
    bound = u * np.einsum("ihj,jhd->ihd", p, np.abs(np.repeat(v[0], H // Hkv, axis=1)))
    assert np.all(np.abs(o1[0] - o0[0]) <= bound + 1e-15)
    assert np.abs(o1 - o0).max() > 0


def test_forward_cast_exact_when_weights_are_representable():
    # Zero queries: exp(S - m) = 1 on every visible key, exact in 16 bits.
    B, L, H, D = 1, 32, 2, 8
    q = np.zeros((B, L, H, D))
    k, v = (rnd((B, L, H, D), s) for s in (103, 104))
    for causal in (False, True):
        o0, _ = orc.forward(q, k, v, causal)
        for fmt in ("bf16", "fp16"):
            o1, _ = orc.forward(q, k, v, causal, p_round=fmt)
            np.testing.assert_allclose(o1, o0, rtol=0, atol=1e-14)


@pytest.mark.parametrize("fmt,tdt", [("bf16", torch.bfloat16), ("fp16", torch.float16)])
def test_forward_cast_in_backward_moves_delta(fmt, tdt):
    # fwd_p_round forms the O behind Delta with the forward's cast: Delta is the row dot
    # product of (cast(exp(S - m)) V / l, stored) with dO; dV does not depend on Delta.
    B, L, H, D = 1, 30, 2, 16
    q, k, v, do = (rnd((B, L, H, D), s) for s in (110, 111, 112, 113))
    _, _, dv0, d0 = orc.backward(q, k, v, do, True)
    _, _, dv1, d1 = orc.backward(q, k, v, do, True, o_round=fmt, fwd_p_round=fmt)
    np.testing.assert_array_equal(dv0, dv1)
    qt, kt, vt, dot = (torch.from_numpy(x) for x in (q, k, v, do))
    for h in range(H):
        e, l, _, _, _ = _torch_unit(qt, kt, vt, dot, h, h, True)
        o = ((e.to(torch.float32).to(tdt).double() @ vt[0, :, h]) / l).to(torch.float32).to(tdt)
        want = (o.double() * dot[0, :, h]).sum(dim=1)
        np.testing.assert_allclose(d1[0, h], want.numpy(), rtol=1e-12, atol=1e-12)
    assert np.abs(d1 - d0).max() > 0


# ---------------------------------------------------------------- fewer queries than keys

def _suffix_case(seed, B=1, L=23, Lq=7, H=2, Hkv=1, D=8):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, L, H, D))
    k = rng.standard_normal((B, L, Hkv, D))
    v = rng.standard_normal((B, L, Hkv, D))
    do = rng.standard_normal((B, L, H, D))
    do[:, : L - Lq] = 0.0       # only the last Lq query rows carry a gradient
    return q, k, v, do, Lq


def test_suffix_queries_match_the_full_causal_problem():
    # The last Lq rows of a causal L x L problem are the (Lq, Lk=L) problem with
    # past_len = L - Lq: same O, LSE; with dO zero on the other rows, same dQ
    # rows and the same dK, dV.
    q, k, v, do, Lq = _suffix_case(90)
    L = q.shape[1]
    o_full, l_full = orc.forward(q, k, v, True)
    o_suf, l_suf = orc.forward(q[:, L - Lq:], k, v, True)
    np.testing.assert_allclose(o_suf, o_full[:, L - Lq:], atol=1e-13)
    np.testing.assert_allclose(l_suf, l_full[:, :, L - Lq:], atol=1e-13)
    dq_f, dk_f, dv_f, _ = orc.backward(q, k, v, do, True)
    dq_s, dk_s, dv_s, _ = orc.backward(q[:, L - Lq:], k, v, do[:, L - Lq:], True)
    np.testing.assert_allclose(dq_s, dq_f[:, L - Lq:], atol=1e-13)
    np.testing.assert_allclose(dk_s, dk_f, atol=1e-13)
    np.testing.assert_allclose(dv_s, dv_f, atol=1e-13)


def test_single_query_causal_sees_every_key():
    rng = np.random.default_rng(91)
    q, k, v = rng.standard_normal((1, 8)), rng.standard_normal((30, 8)), rng.standard_normal((30, 8))
    oc, lc = orc.unit_forward(q, k, v, True)
    on, ln_ = orc.unit_forward(q, k, v, False)
    np.testing.assert_allclose(oc, on, atol=1e-14)
    np.testing.assert_allclose(lc, ln_, atol=1e-14)


def test_fewer_queries_non_causal_matches_torch():
    rng = np.random.default_rng(92)
    B, Lq, Lk, H, Hkv, D = 2, 9, 21, 4, 2, 16
    q, k, v, do = (rng.standard_normal(s) for s in ((B, Lq, H, D), (B, Lk, Hkv, D), (B, Lk, Hkv, D), (B, Lq, H, D)))
    o, _ = orc.forward(q, k, v, False)
    dq, dk, dv, _ = orc.backward(q, k, v, do, False)
    to, tdq, tdk, tdv = torch_reference(q, k, v, do, False)
    for a, b in ((o, to), (dq, tdq), (dk, tdk), (dv, tdv)):
        np.testing.assert_allclose(a, b, atol=1e-11, rtol=1e-9)


def test_fewer_queries_gradients_match_finite_differences():
    rng = np.random.default_rng(93)
    B, Lq, Lk, H, Hkv, D = 1, 3, 6, 2, 1, 4
    q, k, v, do = (rng.standard_normal(s) for s in ((B, Lq, H, D), (B, Lk, Hkv, D), (B, Lk, Hkv, D), (B, Lq, H, D)))
    dq, dk, dv, _ = orc.backward(q, k, v, do, True)

    def f(qq, kk, vv):
        return float((orc.forward(qq, kk, vv, True)[0] * do).sum())
    eps = 1e-6
    for i, (x, g) in enumerate(((q, dq), (k, dk), (v, dv))):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            args_p, args_m = [q, k, v], [q, k, v]
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p[i], args_m[i] = xp, xm
            num[idx] = (f(*args_p) - f(*args_m)) / (2 * eps)
        assert np.abs(num - g).max() / max(1.0, np.abs(g).max()) < 1e-6


def test_top_left_alignment_is_caught():
    # A planted mistake: aligning the causal mask top-left for Lq < Lk.
    q, k, v, _, Lq = _suffix_case(94)
    L = q.shape[1]

    def top_left(q_bh, k_bh, v_bh):
        S = unit_scores_top_left(q_bh, k_bh)
        P = np.exp(S - S.max(axis=1, keepdims=True))
        return (P / P.sum(axis=1, keepdims=True)) @ v_bh

    def unit_scores_top_left(q_bh, k_bh):
        return orc.unit_scores(q_bh, k_bh, True, past=0)

    o_full, _ = orc.forward(q, k, v, True)
    wrong = top_left(q[0, L - Lq:, 0], k[0, :, 0], v[0, :, 0])
    assert not np.allclose(wrong, o_full[0, L - Lq:, 0], atol=1e-6)


def test_key_slices_merged_by_lse_equal_the_whole():
    # Split-KV decoding rests on this identity: attention over disjoint key
    # slices, merged with weights exp(LSE_s - LSE) where LSE = ln sum_s exp(LSE_s),
    # is attention over all keys (checked on the oracle's own forward).
    rng = np.random.default_rng(95)
    Lq, Lk, D = 3, 50, 8
    q, k, v = rng.standard_normal((Lq, D)), rng.standard_normal((Lk, D)), rng.standard_normal((Lk, D))
    o_all, l_all = orc.unit_forward(q, k, v, False)
    cuts = [0, 7, 8, 31, 50]
    parts = [orc.unit_forward(q, k[a:b], v[a:b], False) for a, b in zip(cuts[:-1], cuts[1:])]
    lses = np.stack([p[1] for p in parts])            # [slices, Lq]
    lse = np.log(np.exp(lses).sum(axis=0))
    w = np.exp(lses - lse)                            # [slices, Lq]
    o = sum(w[s][:, None] * parts[s][0] for s in range(len(parts)))
    np.testing.assert_allclose(lse, l_all, atol=1e-13)
    np.testing.assert_allclose(o, o_all, atol=1e-13)


# ---------------------------------------------------------------- FP8 (E4M3) inputs

E4M3_HAND = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x0F: 1.875 * 2.0 ** -6,
             0x38: 1.0, 0x3C: 1.5, 0x40: 2.0, 0x7E: 448.0, 0x80: -0.0, 0xB8: -1.0, 0xFE: -448.0}


def test_e4m3_decode_matches_torch_on_every_code():
    codes = np.arange(256, dtype=np.uint8)
    mine = orc.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    assert np.isnan(mine).sum() == 2                       # 0x7F and 0xFF only
    ok = ~np.isnan(ref)
    assert np.array_equal(mine[ok], ref[ok])


def test_e4m3_decode_hand_values():
    for code, val in E4M3_HAND.items():
        got = orc.e4m3_decode(np.array([code], dtype=np.uint8))[0]
        assert got == val and math.copysign(1.0, got) == math.copysign(1.0, val), hex(code)


def _fp8_case(seed, B=1, Lq=9, Lk=23, H=4, Hkv=2, D=16):
    """Random E4M3 codes with exponent field <= 8 (|x| < 4, no NaN)."""
    rng = np.random.default_rng(seed)

    def codes(shape):
        sign = rng.integers(0, 2, shape) << 7
        exp = rng.integers(0, 9, shape) << 3
        man = rng.integers(0, 8, shape)
        return (sign | exp | man).astype(np.uint8)
    return codes((B, Lq, H, D)), codes((B, Lk, Hkv, D)), codes((B, Lk, Hkv, D))


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_forward_is_forward_of_dequantised_inputs(causal):
    q8, k8, v8 = _fp8_case(101)
    o, lse = orc.forward_fp8(q8, k8, v8, 0.5, 0.25, 3.0, causal)
    assert not np.isnan(o).any()
    v_scaled_o, _ = orc.forward_fp8(q8, k8, v8, 0.5, 0.25, 6.0, causal)
    np.testing.assert_allclose(v_scaled_o, 2.0 * o, rtol=1e-14, atol=0)          # V scale is linear
    o2, lse2 = orc.forward_fp8(q8, k8, v8, 0.25, 0.5, 3.0, causal)
    np.testing.assert_allclose(o2, o, atol=1e-13)                                # only qs*ks matters
    np.testing.assert_allclose(lse2, lse, atol=1e-13)
    o3, lse3 = orc.forward_fp8(q8, k8, v8, 1.0, 0.25, 3.0, causal)               # doubles every score
    qd = orc.e4m3_decode(q8)
    ref3, ref_l3 = orc.forward(qd, orc.e4m3_decode(k8) * 0.25, orc.e4m3_decode(v8) * 3.0, causal)
    np.testing.assert_allclose(o3, ref3, atol=1e-13)
    np.testing.assert_allclose(lse3, ref_l3, atol=1e-13)


def test_planted_e4m3_mistakes_are_caught():
    codes = np.arange(256, dtype=np.uint8)
    torch_ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()

    def bias8(c):          # exponent bias 8 instead of 7
        return orc.e4m3_decode(c) / 2.0

    def implicit_one(c):   # subnormals decoded with the implicit leading 1
        c = np.asarray(c)
        e = (c >> 3) & 0xF
        v = orc.e4m3_decode(c)
        return np.where(e == 0, np.sign(v + 0.0) * np.ldexp(1.0 + (c & 7) / 8.0, -6), v)

    def no_sign(c):
        return np.abs(orc.e4m3_decode(c))

    def mant16(c):         # mantissa read as sixteenths
        c = np.asarray(c)
        e = ((c >> 3) & 0xF).astype(np.int64)
        return np.where(e == 0, orc.e4m3_decode(c), np.ldexp(1.0 + (c & 7) / 16.0, e - 7))

    for bad in (bias8, implicit_one, no_sign, mant16):
        vals = bad(codes)
        ok = ~np.isnan(torch_ref)
        hand_fail = any(bad(np.array([k], dtype=np.uint8))[0] != v for k, v in E4M3_HAND.items())
        torch_fail = not np.array_equal(vals[ok], torch_ref[ok])
        assert hand_fail and torch_fail, bad.__name__


def test_fp8_inputs_are_seeded_codes_with_amax_scales():
    from tiled_attention_fa_gb300.inputs import make_qkv_fp8
    a = make_qkv_fp8(1, 3, 40, 4, 2, 16, seed=5)
    b = make_qkv_fp8(1, 3, 40, 4, 2, 16, seed=5)
    for x, y in zip(a, b):
        assert (x == y).all() if isinstance(x, torch.Tensor) else x == y
    for codes, s in zip(a[:3], a[3:]):
        vals = orc.e4m3_decode(codes.numpy())
        assert not np.isnan(vals).any() and np.abs(vals).max() == 448.0 and s > 0


# ---------------------------------------------------------------- intermediates for error bounds

def _torch_scores_grad(q, k, v, do, causal):
    """Independent torch float64 autograd of f = sum(O o dO) through the score matrix:
    returns (P, dS = df/dS) for one unit, with S = Q K^T / sqrt(D), bottom-right causal."""
    qt, kt, vt, dot = (torch.from_numpy(x) for x in (q, k, v, do))
    Lq, Lk, D = q.shape[0], k.shape[0], q.shape[1]
    s = (qt @ kt.T / math.sqrt(D)).detach().requires_grad_(True)
    if causal:
        mask = torch.arange(Lk)[None, :] > torch.arange(Lq)[:, None] + (Lk - Lq)
        sm = s.masked_fill(mask, float("-inf"))
    else:
        sm = s
    p = torch.softmax(sm, dim=1)
    (p @ vt * dot).sum().backward()
    return p.detach().numpy(), s.grad.numpy()


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Lq,Lk", [(9, 9), (5, 13), (1, 4)])
def test_unit_probs_match_torch_softmax(causal, Lq, Lk):
    rng = np.random.default_rng(120 + Lq + Lk)
    q, k = rng.standard_normal((Lq, 8)), rng.standard_normal((Lk, 8))
    P, E, l = orc.unit_probs(q, k, causal)
    want, _ = _torch_scores_grad(q, k, rng.standard_normal((Lk, 8)), rng.standard_normal((Lq, 8)),
                                 causal)
    np.testing.assert_allclose(P, want, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(E.max(axis=1), 1.0, rtol=0, atol=0)  # largest entry is exp(0)
    np.testing.assert_allclose(E / l[:, None], P, rtol=1e-15, atol=0)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Lq,Lk", [(11, 11), (6, 14)])
def test_backward_parts_match_autograd(causal, Lq, Lk):
    # dS is the gradient of sum(O o dO) with respect to the scores (torch autograd,
    # independent of the oracle); its rows sum to zero; dQ, dK from the parts equal the
    # finite-difference-pinned unit_backward.
    rng = np.random.default_rng(130 + Lq + Lk + int(causal))
    D = 8
    q, k, v = rng.standard_normal((Lq, D)), rng.standard_normal((Lk, D)), rng.standard_normal((Lk, D))
    do = rng.standard_normal((Lq, D))
    parts = orc.unit_backward_parts(q, k, v, do, causal)
    P, dS_ref = _torch_scores_grad(q, k, v, do, causal)
    np.testing.assert_allclose(parts["P"], P, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(parts["dS"], dS_ref, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(parts["dS"].sum(axis=1), 0.0, atol=1e-13)
    np.testing.assert_allclose(parts["dP"], do @ v.T, rtol=1e-14, atol=1e-14)
    dq, dk, dv, delta, o, _ = orc.unit_backward(q, k, v, do, causal)
    np.testing.assert_allclose(parts["O"], o, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(parts["Delta"], delta, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(parts["dS"] @ k / math.sqrt(D), dq, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(parts["dS"].T @ q / math.sqrt(D), dk, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(parts["P"].T @ do, dv, rtol=1e-12, atol=1e-13)


def test_backward_parts_teeth():
    # A dS without Delta, or with the probabilities transposed, breaks the zero row sums
    # or the autograd comparison.
    rng = np.random.default_rng(140)
    q, k, v, do = (rng.standard_normal((10, 8)) for _ in range(4))
    parts = orc.unit_backward_parts(q, k, v, do, True)
    _, dS_ref = _torch_scores_grad(q, k, v, do, True)
    no_delta = parts["P"] * parts["dP"]
    assert np.abs(no_delta.sum(axis=1)).max() > 1e-3
    transposed = parts["P"].T * (parts["dP"] - parts["Delta"][:, None])
    assert np.abs(transposed - dS_ref).max() > 1e-3
