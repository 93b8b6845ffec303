"""CPU checks of the backward comparison used by the GPU tests: a simulated
kernel (torch float64 arithmetic with the 16-bit casts a tensor-core backward
makes -- the forward's exp tile before PV, the stored O, P before dV, dS
before dK and dQ) passes the exact-oracle check (1e-2 for fp16; 1e-2 plus the
derived rounding bound for bf16) and the check against the oracle with the
printed casts, and plausible mistakes fail."""

import math

import numpy as np
import pytest
import torch

from tests.helpers import check_backward, check_backward_cited

CAST = {"fp16": torch.float16, "bf16": torch.bfloat16}


def simulated_backward(q, k, v, do, causal, fmt, mistake=None):
    """dQ, dK, dV [BSHD float64] the way a 16-bit tensor-core kernel forms them."""
    dt = CAST[fmt]
    c = lambda x: x.to(torch.float32).to(dt).double()  # noqa: E731
    qt, kt, vt, dot = (torch.from_numpy(x) for x in (q, k, v, do))
    B, L, H, D = q.shape
    Hkv = k.shape[2]
    dq, dk, dv = torch.zeros_like(qt), torch.zeros_like(kt), torch.zeros_like(vt)
    for b in range(B):
        for h in range(H):
            hk = h // (H // Hkv)
            s = qt[b, :, h] @ kt[b, :, hk].T / math.sqrt(D)
            if causal:
                s = s.masked_fill(~torch.ones(L, L, dtype=torch.bool).tril(), float("-inf"))
            m = s.max(dim=1, keepdim=True).values
            e = torch.exp(s - m)
            l = e.sum(dim=1, keepdim=True)
            p = e / l
            o = c((c(e) @ vt[b, :, hk]) / l)                 # forward: cast tile, stored O
            delta = (o * dot[b, :, h]).sum(dim=1, keepdim=True)
            if mistake == "no_delta":
                delta = delta * 0
            dp = dot[b, :, h] @ vt[b, :, hk].T
            ds = c(p * (dp - delta))
            if mistake == "ds_gain":
                ds = ds * 1.25
            if mistake == "ds_small_gain":
                ds = ds * 1.02
            dq[b, :, h] = ds @ kt[b, :, hk] / math.sqrt(D)
            dk[b, :, hk] += ds.T @ qt[b, :, h] / math.sqrt(D)
            pv = c(p) if mistake != "p_untransposed" else c(p).T
            dv[b, :, hk] += pv.T @ dot[b, :, h]
    return dq.numpy(), dk.numpy(), dv.numpy()


def case(seed, B=1, L=160, H=4, Hkv=2, D=64):
    rng = np.random.default_rng(seed)
    q, do = rng.standard_normal((B, L, H, D)), rng.standard_normal((B, L, H, D))
    k, v = rng.standard_normal((B, L, Hkv, D)), rng.standard_normal((B, L, Hkv, D))
    q, k, v, do = (torch.from_numpy(x).to(torch.float16).double().numpy() for x in (q, k, v, do))
    return q, k, v, do


@pytest.mark.parametrize("fmt", ["fp16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
def test_simulated_kernel_passes(fmt, causal):
    q, k, v, do = case(1 + int(causal))
    got = simulated_backward(q, k, v, do, causal, fmt)
    check_backward(got, q, k, v, do, causal, fmt)
    check_backward_cited(got, q, k, v, do, causal, fmt)


@pytest.mark.parametrize("mistake", ["no_delta", "ds_gain", "p_untransposed"])
@pytest.mark.parametrize("fmt", ["fp16", "bf16"])
def test_planted_mistakes_fail(mistake, fmt):
    q, k, v, do = case(3)
    got = simulated_backward(q, k, v, do, True, fmt, mistake=mistake)
    with pytest.raises(AssertionError):
        check_backward(got, q, k, v, do, True, fmt)
    with pytest.raises(AssertionError):
        check_backward_cited(got, q, k, v, do, True, fmt)


def test_small_bf16_mistake_fails_the_rms_check():
    # A 2% gain on dS stays inside bf16's element-wise allowance but not the RMS model.
    q, k, v, do = case(4)
    got = simulated_backward(q, k, v, do, True, "bf16", mistake="ds_small_gain")
    with pytest.raises(AssertionError, match="RMS"):
        check_backward(got, q, k, v, do, True, "bf16")
