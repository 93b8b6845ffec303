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


def kernel_casts(dtype):
    """Oracle backward options for the 16-bit casts the method puts before its GEMMs:
    the forward's exp(S - m) tile and the stored O behind Delta, P^T before dV, dS
    before dK and dQ."""
    return dict(o_round=dtype, fwd_p_round=dtype, p_round=dtype, ds_round=dtype)


def assert_close(got, ref, rtol=RTOL, atol=ATOL, name="x"):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    excess = np.abs(got - ref) - (atol + rtol * np.abs(ref))
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
    """Exact O [Lq, D] and LSE [Lq] of one (b, h) unit (dequantised float64
    inputs), with the element-wise bound and error variance above."""
    Lq, Lk = q.shape[0], k.shape[0]
    S = orc.unit_scores(q, k, causal, 0, Lk - Lq)
    m = S.max(axis=1, keepdims=True)
    p = np.exp(S - m)
    l = p.sum(axis=1, keepdims=True)
    P = p / l
    O = P @ v
    lse = (m + np.log(l))[:, 0]
    e = np.where(p >= E4M3_NORMAL_MIN, E4M3_REL * p, np.minimum(p, E4M3_SUB)) / l
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
