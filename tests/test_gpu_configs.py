"""Parity at the benchmark configurations' full sizes.

The GPU runs each whole configuration through the same entry points the
benchmark times; the oracle recomputes sampled (batch, head) units exactly and
the kernels' outputs for those units are compared element by element.  On all
heads, the backward outputs are also checked against invariants that hold at
any size: sum_j dV_j = sum_i dO_i and sum_j dK_j = 0 per (batch, kv-head)."""

import pytest
import torch

import tiled_attention_fa_gb300 as fa
from oracle import fa_oracle as orc
from tests.helpers import LSE_ATOL, assert_close, kernel_casts
from tiled_attention_fa_gb300.inputs import make_qkv

pytestmark = pytest.mark.gpu


def unit64(t, b, h):
    return t[b, :, h].to(torch.float64).numpy()


def check_fwd_units(q, k, v, o, lse, causal, units):
    H, Hkv = q.shape[2], k.shape[2]
    o, lse = o.cpu(), lse.cpu()
    for b, h in units:
        hk = orc.kv_head(h, H, Hkv)
        ro, rl = orc.unit_forward(unit64(q, b, h), unit64(k, b, hk), unit64(v, b, hk), causal,
                                  panel=2048)
        assert_close(unit64(o, b, h), ro, name=f"O[{b},:,{h}]")
        assert_close(lse[b, h].double().numpy(), rl, rtol=0, atol=LSE_ATOL, name=f"LSE[{b},{h}]")


def check_bwd_units(q, k, v, do, dq, dk, dv, causal, units, dtype):
    """MHA units: the K/V head of (b, h) receives gradient only from query head h."""
    dq, dk, dv = dq.cpu(), dk.cpu(), dv.cpu()
    for b, h in units:
        rq, rk, rv, _, _, _ = orc.unit_backward(unit64(q, b, h), unit64(k, b, h), unit64(v, b, h),
                                                unit64(do, b, h), causal, panel=2048,
                                                **kernel_casts(dtype))
        assert_close(unit64(dv, b, h), rv, name=f"dV[{b},:,{h}]")
        assert_close(unit64(dk, b, h), rk, name=f"dK[{b},:,{h}]")
        assert_close(unit64(dq, b, h), rq, name=f"dQ[{b},:,{h}]")


def check_bwd_invariants(do, dk, dv, H, Hkv):
    """sum over keys of dV equals sum over queries (of the group) of dO; sum of dK is 0."""
    B, L = do.shape[0], do.shape[1]
    g = H // Hkv
    do_sum = do.double().reshape(B, L, Hkv, g, -1).sum(dim=(1, 3))
    dv_sum = dv.double().sum(dim=1)
    dv_abs = dv.double().abs().sum(dim=1) + do.double().abs().reshape(B, L, Hkv, g, -1).sum(dim=(1, 3))
    assert torch.all((dv_sum - do_sum).abs() <= 1e-3 * dv_abs + 1e-2), "sum dV != sum dO"
    dk_sum = dk.double().sum(dim=1)
    dk_abs = dk.double().abs().sum(dim=1)
    assert torch.all(dk_sum.abs() <= 1e-3 * dk_abs + 1e-2), "sum dK != 0"
    for t in (dk, dv):
        assert torch.isfinite(t).all()


def run_fwd_bwd(q, k, v, do, causal, with_bwd=True):
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o, lse = fa.fwd(qd, kd, vd, causal)
    out = {"o": o, "lse": lse}
    if with_bwd:
        dod = do.cuda()
        dq, dk, dv, _ = fa.attention_backward(qd, kd, vd, o, lse, dod, causal)
        out.update(dq=dq, dk=dk, dv=dv, do=dod)
    torch.cuda.synchronize()
    fa.check_device_error()
    return out


@pytest.fixture(scope="module")
def mha_b8_l4096():
    """Forward MHA B=8, H=32, L=4096, D=128, fp16 (the benchmark's workload)."""
    return make_qkv(8, 4096, 32, 32, 128, "fp16", seed=0)


@pytest.mark.parametrize("causal", [False, True])
def test_mha_b8_h32_l4096_d128_fp16(cuda_lib, mha_b8_l4096, causal):
    q, k, v, do = mha_b8_l4096
    out = run_fwd_bwd(q, k, v, do, causal)
    check_fwd_units(q, k, v, out["o"], out["lse"], causal, [(0, 0), (3, 17), (7, 31)])
    check_bwd_units(q, k, v, do, out["dq"], out["dk"], out["dv"], causal, [(0, 5), (6, 30)], "fp16")
    check_bwd_invariants(out["do"], out["dk"], out["dv"], 32, 32)


def test_gqa_b4_h32_hkv8_l4096_d128_bf16_causal(cuda_lib):
    """Forward GQA causal, groups of 4 query heads per K/V head, bf16."""
    q, k, v, _ = make_qkv(4, 4096, 32, 8, 128, "bf16", seed=1, with_do=False)
    out = run_fwd_bwd(q, k, v, None, True, with_bwd=False)
    check_fwd_units(q, k, v, out["o"], out["lse"], True, [(0, 0), (1, 3), (2, 4), (3, 31)])


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_b8_h32_l1024_d64_fp16(cuda_lib, causal):
    """Backward MHA B=8, H=32, L=1024, D=64 fp16, O and LSE from the forward."""
    q, k, v, do = make_qkv(8, 1024, 32, 32, 64, "fp16", seed=2 + int(causal))
    out = run_fwd_bwd(q, k, v, do, causal)
    check_fwd_units(q, k, v, out["o"], out["lse"], causal, [(0, 0), (7, 31)])
    check_bwd_units(q, k, v, do, out["dq"], out["dk"], out["dv"], causal,
                    [(0, 0), (2, 9), (5, 20), (7, 31)], "fp16")
    check_bwd_invariants(out["do"], out["dk"], out["dv"], 32, 32)


@pytest.mark.parametrize("L", [1024, 4096, 8192, 16384])
def test_long_sequence_b1_h32_d128_causal(cuda_lib, L):
    """Long-sequence forward + backward, causal, B=1, H=32, D=128 (hidden 4096)."""
    q, k, v, do = make_qkv(1, L, 32, 32, 128, "fp16", seed=10 + L)
    out = run_fwd_bwd(q, k, v, do, True)
    units = [(0, 0), (0, 31)] if L > 4096 else [(0, 0), (0, 13), (0, 31)]
    check_fwd_units(q, k, v, out["o"], out["lse"], True, units)
    check_bwd_units(q, k, v, do, out["dq"], out["dk"], out["dv"], True, units[:2], "fp16")
    check_bwd_invariants(out["do"], out["dk"], out["dv"], 32, 32)
