"""Shared helpers for the GPU parity tests: seeded inputs, oracle calls and
the element-wise tolerance check (|gpu - ref| <= atol + rtol * |ref|)."""

import numpy as np
import torch

from oracle import fa_oracle as orc
from tiled_attention_fa_gb300.inputs import make_qkv

# Tolerances: O, dQ, dK, dV rtol = atol = 1e-2; LSE 1e-3 absolute.
RTOL = 1e-2
ATOL = 1e-2
LSE_ATOL = 1e-3


# Unit roundoff of the 16-bit storage formats (round to nearest): half an ulp of 1.
UNIT_ROUNDOFF = {"fp16": 2.0 ** -11, "bf16": 2.0 ** -8}


def cited_casts(dtype):
    """Oracle backward options for the 16-bit casts the pages print before their GEMMs:
    the forward's exp(S - m) tile before PV and the stored O behind Delta
    (forward page, K/V tile loop; backward page, preprocess), P^T before dV
    (backward page, main kernel).  The pages print no cast of dS."""
    return dict(o_round=dtype, fwd_p_round=dtype, p_round=dtype)


def excess_over(got, ref, rtol=RTOL, atol=ATOL, extra=0.0):
    """Element-wise |got - ref| - (atol + rtol |ref| + extra)  (<= 0 where within tolerance)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return np.abs(got - ref) - (atol + rtol * np.abs(ref) + extra)


def assert_close(got, ref, rtol=RTOL, atol=ATOL, name="x", extra=0.0):
    """|got - ref| <= atol + rtol |ref| + extra element-wise (extra: an array of derived
    rounding bounds, or 0)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    excess = excess_over(got, ref, rtol, atol, extra)
    if excess.max() > 0:
        idx = np.unravel_index(int(np.argmax(excess)), excess.shape)
        bad = int((excess > 0).sum())
        raise AssertionError(
            f"{name}: {bad}/{excess.size} elements out of tolerance; worst at {idx}: "
            f"got {got[idx]:.6g} ref {ref[idx]:.6g} (max abs err {np.abs(got - ref).max():.3g})")


def to64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def inputs(B, L, H, Hkv, D, dtype, seed, device="cuda"):
    q, k, v, do = make_qkv(B, L, H, Hkv, D, dtype, seed)
    host = tuple(to64(x) for x in (q, k, v, do))
    dev = tuple(x.to(device) for x in (q, k, v, do))
    return host, dev


def bwd_rounding_bound(q, k, v, do, causal, fmt, modelled=(), with_var=False):
    """Element-wise first-order bound on how far a kernel that rounds to ``fmt`` at
    the method's points can move dQ, dK, dV from the exact oracle (BSHD float64 inputs;
    returns arrays shaped like dQ, dK, dV).  With u the unit roundoff of ``fmt``:

      forward O:  e_O = u |O| + u P|V|          (stored O; exp tile cast before PV)
      Delta:      e_D_i  = sum_d |dO_id| e_O_id
      dS:         e_S_ij = P_ij e_D_i + u |dS_ij| (Delta's error; dS cast before dK, dQ)
      dQ = e_S |K| / sqrt(D),  dK = e_S^T |Q| / sqrt(D),  dV = u P^T |dO|  (P cast before dV)

    summed over the query heads of a K/V group for dK and dV.  ``modelled`` names the
    roundings the reference already applies ("o" for the forward's cast and stored O,
    "p" for P before dV), which are then left out.  With ``with_var`` it also returns
    the variances of the same errors when every rounding error is independent and
    uniform on [-u|x|, u|x|] (variance u^2 x^2 / 3), propagated through the same sums.
    P, dS, O come from the oracle (exact); this function only does the bound's
    arithmetic."""
    u = UNIT_ROUNDOFF[fmt]
    B, Lq, H, D = q.shape
    Lk, Hkv = k.shape[1], k.shape[2]
    eq = np.zeros((B, Lq, H, D))
    ek = np.zeros((B, Lk, Hkv, D))
    ev = np.zeros((B, Lk, Hkv, D))
    vq, vk, vv = np.zeros_like(eq), np.zeros_like(ek), np.zeros_like(ev)
    for b in range(B):
        for h in range(H):
            hk = orc.kv_head(h, H, Hkv)
            pt = orc.unit_backward_parts(q[b, :, h], k[b, :, hk], v[b, :, hk], do[b, :, h], causal)
            P, dS = pt["P"], pt["dS"]
            Kb, Qb, Vb, dOb = k[b, :, hk], q[b, :, h], v[b, :, hk], do[b, :, h]
            if "o" in modelled:
                e_s = u * np.abs(dS)
                s2_s = (u * dS) ** 2 / 3
            else:
                e_o = u * (np.abs(pt["O"]) + P @ np.abs(Vb))
                e_d = (np.abs(dOb) * e_o).sum(axis=1)
                e_s = P * e_d[:, None] + u * np.abs(dS)
                if with_var:
                    s2_o = u * u * (pt["O"] ** 2 + (P ** 2) @ (Vb ** 2)) / 3
                    s2_d = (dOb ** 2 * s2_o).sum(axis=1)
                    s2_s = P ** 2 * s2_d[:, None] + (u * dS) ** 2 / 3
            eq[b, :, h] = e_s @ np.abs(Kb) / np.sqrt(D)
            ek[b, :, hk] += e_s.T @ np.abs(Qb) / np.sqrt(D)
            if "p" not in modelled:
                ev[b, :, hk] += u * (P.T @ np.abs(dOb))
            if with_var:
                vq[b, :, h] = s2_s @ Kb ** 2 / D
                vk[b, :, hk] += s2_s.T @ Qb ** 2 / D
                if "p" not in modelled:
                    vv[b, :, hk] += u * u * ((P ** 2).T @ dOb ** 2) / 3
    if with_var:
        return (eq, ek, ev), (vq, vk, vv)
    return eq, ek, ev


def check_backward(got, q, k, v, do, causal, dtype, name=""):
    """dQ, dK, dV (float64 arrays, BSHD) against the exact fp64 oracle: within
    1e-2 + 1e-2 |ref| element-wise for fp16 (the stated tolerance).  For bf16, whose
    8-bit significand alone moves early-causal-key gradients by about that much, the
    same plus the first-order bound of the kernel's bf16 roundings (bwd_rounding_bound),
    and the RMS error over each output at most twice the RMS of those roundings'
    propagated standard deviation.  Returns the largest excess over the plain 1e-2 bound."""
    ref = orc.backward(q, k, v, do, causal)[:3]
    if dtype == "bf16":
        extra, var = bwd_rounding_bound(q, k, v, do, causal, dtype, with_var=True)
    else:
        extra, var = (0, 0, 0), None
    worst = -np.inf
    for i, (nm, g, r, e) in enumerate(zip(("dQ", "dK", "dV"), got, ref, extra)):
        worst = max(worst, float(excess_over(g, r).max()))
        assert_close(g, r, name=f"{nm}{name} (exact oracle)", extra=e)
        if var is not None:
            rms = float(np.sqrt(np.mean((np.asarray(g, dtype=np.float64) - r) ** 2)))
            sig = float(np.sqrt(np.mean(var[i])))
            assert rms <= 2.0 * sig + 1e-6, (
                f"{nm}{name}: RMS error {rms:.3g} above twice the RMS rounding deviation {sig:.3g}")
    return worst


def check_backward_cited(got, q, k, v, do, causal, dtype, name=""):
    """Second check: the oracle with the casts the pages print (cited_casts), within
    1e-2 + 1e-2 |ref| plus the bound of the one rounding it does not model (dS cast
    to the input type before dK and dQ)."""
    ref = orc.backward(q, k, v, do, causal, **cited_casts(dtype))[:3]
    extra = bwd_rounding_bound(q, k, v, do, causal, dtype, modelled=("o", "p"))
    for nm, g, r, e in zip(("dQ", "dK", "dV"), got, ref, extra):
        assert_close(g, r, name=f"{nm}{name} (oracle with the printed casts)", extra=e)


def oracle_units_fwd(q, k, v, causal, units):
    """Oracle O [L, D] and LSE [L] for each (b, h) in ``units``."""
    H, Hkv = q.shape[2], k.shape[2]
    out = {}
    for b, h in units:
        hk = orc.kv_head(h, H, Hkv)
        out[(b, h)] = orc.unit_forward(q[b, :, h], k[b, :, hk], v[b, :, hk], causal)
    return out



# ---------------------------------------------------------------- E4M3 inputs
#
# The FP8 forward rounds each probability p (scaled so that the row max is at
# most 1, or up to 2^8 under a stale running max) to E4M3 before the PV
# product, while l sums the unrounded p.  Per key the rounding error, in
# units where the row's true max gives p = 1, is at most
#     e(p) = 2^-4 p            for p >= 2^-6   (3-bit mantissa, half an ulp)
#     e(p) = min(p, 2^-10)     below            (subnormal spacing 2^-9)
# and a stale max only scales p up, which cannot raise that bound.  So
#     |O_gpu - O| <= sum_j e(p_j)/l |V_j| + (Lk 2^-24 + 2^-16) sum_j P_j |V_j|
#                    + u_out |O| + 1e-5
# element-wise (fp32 accumulation, exp2 and S rounding in the second term,
# the output cast in the third).  That bound is worst-case (every error the
# same sign), so the tests also compare the root-mean-square error over the
# whole output with the RMS of the rounding's standard deviation, taking each
# key's error as uniform on [-e, e]: sigma^2 = sum_j (e_j/l)^2 V_j^2 / 3.

E4M3_REL = 2.0 ** -4
E4M3_SUB = 2.0 ** -10
E4M3_NORMAL_MIN = 2.0 ** -6
OUT_ULP = {"bf16": 2.0 ** -8, "fp16": 2.0 ** -10}


def fp8_unit_reference(q, k, v, causal):
    """Exact O [Lq, D] and LSE [Lq] of one (b, h) unit (dequantised float64 inputs)
    from the oracle, with the element-wise bound and error variance above computed
    from the oracle's probabilities (E = exp(S - m), l, P = E / l)."""
    Lk = k.shape[0]
    O, lse = orc.unit_forward(q, k, v, causal)
    P, p, l = orc.unit_probs(q, k, causal)
    e = np.where(p >= E4M3_NORMAL_MIN, E4M3_REL * p, np.minimum(p, E4M3_SUB)) / l[:, None]
    bound = e @ np.abs(v) + (Lk * 2.0 ** -24 + 2.0 ** -16) * (P @ np.abs(v))
    var = (e ** 2 @ v ** 2) / 3.0
    return O, lse, bound, var


class Fp8Check:
    """Accumulates element-wise and RMS checks of FP8-forward outputs."""

    def __init__(self, out: str):
        self.u = OUT_ULP[out]
        self.sq_err = 0.0
        self.sq_sigma = 0.0
        self.n = 0

    def unit(self, o_gpu, lse_gpu, q, k, v, causal, name="O"):
        O, lse, bound, var = fp8_unit_reference(q, k, v, causal)
        tol = bound + self.u * np.abs(O) + 1e-5
        err = np.abs(np.asarray(o_gpu, dtype=np.float64) - O)
        assert np.all(np.isfinite(o_gpu)), f"{name}: non-finite values"
        if np.any(err > tol):
            idx = np.unravel_index(int(np.argmax(err - tol)), err.shape)
            raise AssertionError(f"{name}: {int((err > tol).sum())} elements above the E4M3 bound; "
                                 f"worst at {idx}: got {o_gpu[idx]:.6g} ref {O[idx]:.6g} "
                                 f"bound {tol[idx]:.3g}")
        assert_close(lse_gpu, lse, rtol=0, atol=LSE_ATOL, name=f"LSE of {name}")
        self.sq_err += float((err ** 2).sum())
        self.sq_sigma += float((var + (self.u * O) ** 2 / 12.0).sum())
        self.n += err.size

    def finish(self):
        rms_err = (self.sq_err / self.n) ** 0.5
        rms_sigma = (self.sq_sigma / self.n) ** 0.5
        assert rms_err <= 2.0 * rms_sigma + 1e-6, (
            f"RMS error {rms_err:.3g} above twice the RMS rounding deviation {rms_sigma:.3g}")
        return rms_err, rms_sigma
