"""Forward parity: the CUDA path against the fp64 oracle, element by element."""

import numpy as np
import pytest
import torch

import tiled_attention_fa_gb300 as fa
from tests.helpers import LSE_ATOL, assert_close, inputs, oracle_units_fwd, to64
from oracle import fa_oracle as orc

pytestmark = pytest.mark.gpu


def run_and_compare(B, L, H, Hkv, D, dtype, causal, seed, units=None):
    (q, k, v, _), (qd, kd, vd, _) = inputs(B, L, H, Hkv, D, dtype, seed)
    o, lse = fa.fwd(qd, kd, vd, causal)
    torch.cuda.synchronize()
    fa.check_device_error()
    o, lse = to64(o), to64(lse)
    if units is None:
        ro, rl = orc.forward(q, k, v, causal)
        assert_close(o, ro, name="O")
        assert_close(lse, rl, rtol=0, atol=LSE_ATOL, name="LSE")
    else:
        ref = oracle_units_fwd(q, k, v, causal, units)
        for (b, h), (ro, rl) in ref.items():
            assert_close(o[b, :, h], ro, name=f"O[{b},:,{h}]")
            assert_close(lse[b, h], rl, rtol=0, atol=LSE_ATOL, name=f"LSE[{b},{h}]")
    return o, lse


def test_smallest_case_b1_h2_l128_d64(cuda_lib):
    """Forward only, non-causal MHA: B=1, H=2, L=128, D=64, fp16, seed 0."""
    run_and_compare(1, 128, 2, 2, 64, "fp16", False, 0)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("L", [1, 17, 127, 128, 129, 200, 255, 256, 257, 300, 513])
def test_ragged_lengths(cuda_lib, L, causal, D):
    run_and_compare(1, L, 2, 1, D, "fp16", causal, seed=L)


@pytest.mark.parametrize("H,Hkv", [(1, 1), (4, 1), (8, 2)])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
def test_heads_and_dtypes(cuda_lib, H, Hkv, dtype, causal):
    run_and_compare(2, 384, H, Hkv, 128, dtype, causal, seed=H * 10 + Hkv)
    run_and_compare(2, 320, H, Hkv, 64, dtype, causal, seed=H * 10 + Hkv + 1)


def test_many_items_per_cta(cuda_lib):
    """More work items than SMs, so each persistent CTA runs several items."""
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    H = max(2, (3 * n_sm) // 2)  # B*H*pairs > 2 * SMs with L=512 (two pairs)
    for causal in (False, True):
        run_and_compare(1, 512, H, 2 if H % 2 == 0 else 1, 64, "fp16", causal, seed=5,
                        units=[(0, 0), (0, H // 2), (0, H - 1)])


def test_special_values(cuda_lib):
    """Constant V gives that value; Q = 0 gives the (causal) running mean of V."""
    B, L, H, D = 1, 300, 2, 128
    v_row = torch.randn(D, generator=torch.Generator().manual_seed(1)).half()
    q = torch.randn(B, L, H, D, generator=torch.Generator().manual_seed(2)).half().cuda()
    k = torch.randn(B, L, H, D, generator=torch.Generator().manual_seed(3)).half().cuda()
    v = v_row.expand(B, L, H, D).contiguous().cuda()
    for causal in (False, True):
        o, _ = fa.fwd(q, k, v, causal)
        assert_close(to64(o), np.broadcast_to(v_row.double().numpy(), (B, L, H, D)), name="O")
    vr = torch.randn(B, L, H, D, generator=torch.Generator().manual_seed(4)).half()
    o, lse = fa.fwd(torch.zeros_like(q), k, vr.cuda(), True)
    want = np.cumsum(vr.double().numpy(), axis=1) / np.arange(1, L + 1)[None, :, None, None]
    assert_close(to64(o), want, name="O")
    assert_close(to64(lse), np.broadcast_to(np.log(np.arange(1, L + 1)), (B, H, L)),
                 rtol=0, atol=LSE_ATOL, name="LSE")


def test_large_scores_stay_finite(cuda_lib):
    """Scores of magnitude ~1e3 exercise the rescale path without overflow."""
    B, L, H, D = 1, 640, 2, 64
    g = torch.Generator().manual_seed(7)
    q = (torch.randn(B, L, H, D, generator=g) * 8).half()
    k = (torch.randn(B, L, H, D, generator=g) * 8).half()
    v = torch.randn(B, L, H, D, generator=g).half()
    for causal in (False, True):
        o, lse = fa.fwd(q.cuda(), k.cuda(), v.cuda(), causal)
        ro, rl = orc.forward(to64(q), to64(k), to64(v), causal)
        assert_close(to64(o), ro, name="O")
        assert_close(to64(lse), rl, rtol=1e-5, atol=LSE_ATOL, name="LSE")


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("causal", [False, True])
def test_row_max_rising_every_tile(cuda_lib, D, dtype, causal):
    """Scores that rise by ~20 (natural log) across every 128-key tile: every
    row's running max grows past the 2^8 rescale threshold at each K/V tile,
    always at the tile's last keys, so O is rescaled at every step (after
    the first half of P is stored and before the tensor core adds PV)."""
    B, L, H = 1, 640, 2
    g = torch.Generator().manual_seed(21)
    alpha = 20.0 / (128 * D ** 0.5)  # score rise per key: q . k_j / sqrt(D) ~ sqrt(D) * alpha * j
    ramp = alpha * torch.arange(L, dtype=torch.float32).view(1, L, 1, 1)
    q = (1 + 0.1 * torch.randn(B, L, H, D, generator=g)).to(dtype)
    k = (ramp * (1 + 0.1 * torch.randn(B, L, H, D, generator=g))).to(dtype)
    v = torch.randn(B, L, H, D, generator=g).to(dtype)
    o, lse = fa.fwd(q.cuda(), k.cuda(), v.cuda(), causal)
    ro, rl = orc.forward(to64(q), to64(k), to64(v), causal)
    assert np.isfinite(to64(o)).all()
    assert_close(to64(o), ro, name="O")
    assert_close(to64(lse), rl, rtol=1e-5, atol=LSE_ATOL, name="LSE")


def test_repeated_calls_are_deterministic(cuda_lib):
    (_, _, _, _), (qd, kd, vd, _) = inputs(2, 700, 4, 2, 128, "bf16", 11)
    o1, l1 = fa.fwd(qd, kd, vd, True)
    o2, l2 = fa.fwd(qd, kd, vd, True)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
