"""Backward parity: preprocess (Delta) and dQ/dK/dV against the fp64 oracle.

The GPU backward consumes the GPU forward's O and LSE; the oracle recomputes
its own from the same inputs."""

import numpy as np
import pytest
import torch

import tiled_attention_fa_gb300 as fa
from tests.helpers import assert_close, check_backward, check_backward_cited, inputs, to64
from oracle import fa_oracle as orc

pytestmark = pytest.mark.gpu


def gpu_fwd_bwd(qd, kd, vd, dod, causal):
    o, lse = fa.fwd(qd, kd, vd, causal)
    dq, dk, dv, delta = fa.attention_backward(qd, kd, vd, o, lse, dod, causal)
    torch.cuda.synchronize()
    fa.check_device_error()
    return o, lse, dq, dk, dv, delta


def run_and_compare(B, L, H, Hkv, D, dtype, causal, seed):
    (q, k, v, do), (qd, kd, vd, dod) = inputs(B, L, H, Hkv, D, dtype, seed)
    o, lse, dq, dk, dv, delta = gpu_fwd_bwd(qd, kd, vd, dod, causal)
    got = (to64(dq), to64(dk), to64(dv))
    # The exact oracle (fp16 at 1e-2; bf16 with its derived rounding allowance), then
    # the oracle with the casts the pages print (forward exp tile and stored O behind
    # Delta, P before dV) with only the dS cast's allowance.
    check_backward(got, q, k, v, do, causal, dtype)
    check_backward_cited(got, q, k, v, do, causal, dtype)
    # Delta of the GPU's own O against the oracle's: O is within the forward
    # tolerance (atol + rtol |O|) per element, so Delta is within
    # sum_d |dO_d| (atol + rtol |O_d|) of the exact value.
    ro, _ = orc.forward(q, k, v, causal)
    rdelta = orc.bwd_preprocess(ro, do)
    bound = np.einsum("blhd->bhl", np.abs(do) * (1e-2 + 1e-2 * np.abs(ro)))
    assert np.all(np.abs(to64(delta) - rdelta) <= bound), "Delta"


def test_preprocess_matches_definition(cuda_lib):
    for (B, L, H, D, dt) in [(2, 77, 3, 64, "fp16"), (1, 300, 4, 128, "bf16"), (3, 1, 2, 128, "fp16")]:
        g = torch.Generator().manual_seed(L)
        dtt = torch.float16 if dt == "fp16" else torch.bfloat16
        o = torch.randn(B, L, H, D, generator=g).to(dtt)
        do = torch.randn(B, L, H, D, generator=g).to(dtt)
        acc = torch.full((fa.workspace_size(B, L, H, D) // 4,), 7.0, device="cuda")
        delta = fa.bwd_preprocess(o.cuda(), do.cuda(), dq_accum=acc)
        torch.cuda.synchronize()
        ref = orc.bwd_preprocess(to64(o), to64(do))
        assert_close(to64(delta), ref, rtol=1e-5, atol=1e-4, name="Delta")
        assert torch.count_nonzero(acc).item() == 0, "accumulator not zeroed"


@pytest.mark.parametrize("B,L,H,D,dt", [(8, 1024, 5, 64, "fp16"), (1, 1000, 7, 128, "bf16"),
                                         (2, 77, 3, 64, "fp16"), (1, 4096, 32, 128, "fp16")])
def test_preprocess_head_groups(cuda_lib, B, L, H, D, dt):
    """Shapes whose (batch, chunk) pairs alone would not fill the GPU, so the
    preprocess splits the heads into groups, some of them partial (H = 5, 7)."""
    g = torch.Generator().manual_seed(B * L + H)
    dtt = torch.float16 if dt == "fp16" else torch.bfloat16
    o = torch.randn(B, L, H, D, generator=g).to(dtt)
    do = torch.randn(B, L, H, D, generator=g).to(dtt)
    acc = torch.full((fa.workspace_size(B, L, H, D) // 4,), 7.0, device="cuda")
    delta = fa.bwd_preprocess(o.cuda(), do.cuda(), dq_accum=acc)
    torch.cuda.synchronize()
    ref = orc.bwd_preprocess(to64(o), to64(do))
    assert_close(to64(delta), ref, rtol=1e-5, atol=1e-4, name="Delta")
    assert torch.count_nonzero(acc).item() == 0, "accumulator not zeroed"


def test_smallest_case(cuda_lib):
    run_and_compare(1, 128, 2, 2, 64, "fp16", False, 0)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("L", [1, 17, 127, 128, 129, 255, 256, 300, 513])
def test_ragged_lengths(cuda_lib, L, causal, D):
    run_and_compare(1, L, 2, 2, D, "fp16", causal, seed=100 + L)


@pytest.mark.parametrize("H,Hkv", [(1, 1), (4, 1), (8, 2)])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
def test_heads_and_dtypes(cuda_lib, H, Hkv, dtype, causal):
    run_and_compare(2, 384, H, Hkv, 128, dtype, causal, seed=H * 10 + Hkv)
    run_and_compare(2, 320, H, Hkv, 64, dtype, causal, seed=H * 10 + Hkv + 1)


def test_unzeroed_accumulator_path(cuda_lib):
    """fa_bwd zeroes a dirty workspace itself when told it is not zeroed."""
    (q, k, v, do), (qd, kd, vd, dod) = inputs(1, 256, 2, 1, 64, "fp16", 3)
    o, lse = fa.fwd(qd, kd, vd, True)
    delta = fa.bwd_preprocess(o, dod)
    acc = torch.full((fa.workspace_size(1, 256, 2, 64) // 4,), 3.0, device="cuda")
    dq, dk, dv = fa.bwd(qd, kd, vd, o, dod, lse, delta, True, dq_accum=acc, accum_zeroed=False)
    check_backward((to64(dq), to64(dk), to64(dv)), q, k, v, do, True, "fp16")
