"""Parity at the benchmark configurations' full sizes.

The GPU runs each whole configuration through the same entry points the
benchmark times; the exact fp64 oracle recomputes (batch, head) units -- all
of them where the host finishes them in well under a minute, otherwise a
deterministic spread of at least eight -- on a pool of host processes, and
the kernels' outputs for those units are compared element by element
(O, dQ, dK, dV within 1e-2 + 1e-2 |ref|, LSE within 1e-3).  On all heads, the
backward outputs are also checked against invariants that hold at any size:
sum_j dV_j = sum_i dO_i and sum_j dK_j = 0 per (batch, kv-head)."""

import pytest
import torch

import tiled_attention_fa_gb300 as fa
from tests.oracle_pool import check_backward_units, check_forward_units
from tiled_attention_fa_gb300.inputs import make_qkv

pytestmark = pytest.mark.gpu


def all_units(B, H):
    return [(b, h) for b in range(B) for h in range(H)]


def spread(B, H, n):
    """n deterministic (b, h) units spread over the batch and the heads."""
    total = B * H
    idx = sorted({(i * total) // n + (i * 7) % max(1, total // n) for i in range(n)})
    return [(i // H, i % H) for i in idx]


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
    """The whole configuration on the GPU; outputs back on the host."""
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o, lse = fa.fwd(qd, kd, vd, causal)
    out = {"o": o, "lse": lse}
    if with_bwd:
        dod = do.cuda()
        dq, dk, dv, _ = fa.attention_backward(qd, kd, vd, o, lse, dod, causal)
        out.update(dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    fa.check_device_error()
    return {name: t.cpu() for name, t in out.items()}


@pytest.fixture(scope="module")
def mha_b8_l4096():
    """Forward MHA B=8, H=32, L=4096, D=128, fp16 (the benchmark's workload)."""
    return make_qkv(8, 4096, 32, 32, 128, "fp16", seed=0)


@pytest.mark.parametrize("causal", [False, True])
def test_mha_b8_h32_l4096_d128_fp16(cuda_lib, mha_b8_l4096, causal):
    q, k, v, do = mha_b8_l4096
    out = run_fwd_bwd(q, k, v, do, causal)
    check_forward_units(q, k, v, out["o"], out["lse"], causal, all_units(8, 32))
    check_backward_units(q, k, v, do, out["dq"], out["dk"], out["dv"], causal, spread(8, 32, 16))
    check_bwd_invariants(do, out["dk"], out["dv"], 32, 32)


def test_gqa_b4_h32_hkv8_l4096_d128_bf16_causal(cuda_lib):
    """Forward GQA causal, groups of 4 query heads per K/V head, bf16."""
    q, k, v, _ = make_qkv(4, 4096, 32, 8, 128, "bf16", seed=1, with_do=False)
    out = run_fwd_bwd(q, k, v, None, True, with_bwd=False)
    check_forward_units(q, k, v, out["o"], out["lse"], True, spread(4, 32, 16))


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_b8_h32_l1024_d64_fp16(cuda_lib, causal):
    """Backward MHA B=8, H=32, L=1024, D=64 fp16, O and LSE from the forward: every unit."""
    q, k, v, do = make_qkv(8, 1024, 32, 32, 64, "fp16", seed=2 + int(causal))
    out = run_fwd_bwd(q, k, v, do, causal)
    check_forward_units(q, k, v, out["o"], out["lse"], causal, all_units(8, 32))
    check_backward_units(q, k, v, do, out["dq"], out["dk"], out["dv"], causal, all_units(8, 32))
    check_bwd_invariants(do, out["dk"], out["dv"], 32, 32)


@pytest.mark.parametrize("L", [1024, 4096, 8192, 16384])
def test_long_sequence_b1_h32_d128_causal(cuda_lib, L):
    """Long-sequence forward + backward, causal, B=1, H=32, D=128 (hidden 4096):
    every head up to L = 4096, sixteen forward and eight backward heads beyond."""
    q, k, v, do = make_qkv(1, L, 32, 32, 128, "fp16", seed=10 + L)
    out = run_fwd_bwd(q, k, v, do, True)
    fwd_units = all_units(1, 32) if L <= 4096 else spread(1, 32, 16)
    bwd_units = all_units(1, 32) if L <= 4096 else spread(1, 32, 8)
    panel = 1024 if L > 8192 else 2048
    check_forward_units(q, k, v, out["o"], out["lse"], True, fwd_units, panel=panel)
    check_backward_units(q, k, v, do, out["dq"], out["dk"], out["dv"], True, bwd_units,
                         panel=panel)
    check_bwd_invariants(do, out["dk"], out["dv"], 32, 32)
