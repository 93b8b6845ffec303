"""CPU checks of the FP8-forward error model used by the GPU tests: a
simulated kernel (the oracle's exact P rounded to E4M3 by torch's cast, l
from the unrounded P) passes both checks, and plausible mistakes fail one."""

import numpy as np
import pytest
import torch

from oracle import fa_oracle as orc
from tests.helpers import Fp8Check
from tiled_attention_fa_gb300.inputs import make_qkv_fp8


def simulated(q, k, v, causal, stale=0.0, unmask_next=False, v_gain=1.0):
    """O, LSE the way the kernel forms them: p = exp(S - m + stale) rounded to
    E4M3, l = sum of the unrounded p.  Options plant mistakes."""
    Lq, Lk = q.shape[0], k.shape[0]
    S = orc.unit_scores(q, k, causal, 0, Lk - Lq + (1 if unmask_next else 0))
    m = S.max(axis=1, keepdims=True)
    p = np.exp(S - m + stale)
    l = p.sum(axis=1, keepdims=True)
    pr = torch.from_numpy(p).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    o = (pr @ v) / l * v_gain
    o = torch.from_numpy(o).to(torch.bfloat16).to(torch.float64).numpy()
    return o, (m + np.log(l))[:, 0] - stale


def units(seed, Lq, Lk, causal):
    q8, k8, v8, qs, ks, vs = make_qkv_fp8(1, Lq, Lk, 2, 1, 128, seed=seed)
    q = orc.e4m3_decode(q8.numpy()) * qs
    k = orc.e4m3_decode(k8.numpy()) * ks
    v = orc.e4m3_decode(v8.numpy()) * vs
    return [(q[0, :, h], k[0, :, 0], v[0, :, 0]) for h in range(2)]


@pytest.mark.parametrize("stale", [0.0, 3.0])
@pytest.mark.parametrize("causal", [False, True])
def test_simulated_rounding_passes(causal, stale):
    chk = Fp8Check("bf16")
    for q, k, v in units(1, 200, 300, causal):
        o, lse = simulated(q, k, v, causal, stale=stale)
        chk.unit(o, lse, q, k, v, causal)
    chk.finish()


@pytest.mark.parametrize("mistake", ["unmask_next", "v_gain", "p_not_rounded_as_bf16_swap"])
def test_planted_mistakes_fail(mistake):
    chk = Fp8Check("bf16")
    causal = True
    with pytest.raises(AssertionError):
        for q, k, v in units(2, 200, 300, causal):
            if mistake == "unmask_next":
                o, lse = simulated(q, k, v, causal, unmask_next=True)
            elif mistake == "v_gain":
                o, lse = simulated(q, k, v, causal, v_gain=1.25)
            else:  # neighbouring keys' probabilities swapped (a packing-order slip)
                perm = np.arange(k.shape[0]).reshape(-1, 2)[:, ::-1].reshape(-1)
                o, lse = simulated(q, k, v[perm], causal)
            chk.unit(o, lse, q, k, v, causal)
        chk.finish()
