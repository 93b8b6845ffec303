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

