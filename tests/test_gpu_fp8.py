"""FP8 (E4M3) forward against the oracle's exact attention of the dequantised
inputs.  The kernel rounds P to E4M3 before the PV product, so O is checked
against the element-wise error bound and the RMS error model of
``tests.helpers.Fp8Check`` (derived from that rounding); LSE, formed from the
unrounded probabilities, keeps the 1e-3 absolute tolerance."""

import pytest
import torch

import tiled_attention_fa_gb300 as fa
from oracle import fa_oracle as orc
from tests.helpers import Fp8Check, to64
from tiled_attention_fa_gb300 import _lib
from tiled_attention_fa_gb300.inputs import make_qkv_fp8

pytestmark = pytest.mark.gpu

OUT = {"bf16": torch.bfloat16, "fp16": torch.float16}


def run(B, Lq, Lk, H, Hkv, causal, out, seed, units=None):
    q8, k8, v8, qs, ks, vs = make_qkv_fp8(B, Lq, Lk, H, Hkv, 128, seed=seed)
    o, lse = fa.fwd_fp8(q8.cuda(), k8.cuda(), v8.cuda(), qs, ks, vs, causal, out_dtype=OUT[out])
    torch.cuda.synchronize()
    fa.check_device_error()
    o, lse = o.cpu(), lse.cpu()
    q8, k8, v8 = q8.numpy(), k8.numpy(), v8.numpy()
    chk = Fp8Check(out)
    if units is None:
        units = [(b, h) for b in range(B) for h in range(H)]
    for b, h in units:
        hk = orc.kv_head(h, H, Hkv)
        chk.unit(to64(o[b, :, h]), to64(lse[b, h]), orc.e4m3_decode(q8[b, :, h]) * qs,
                 orc.e4m3_decode(k8[b, :, hk]) * ks, orc.e4m3_decode(v8[b, :, hk]) * vs, causal,
                 name=f"O[{b},:,{h}]")
    return chk.finish()


CASES = [
    # B, Lq, Lk, H, Hkv
    (1, 128, 128, 2, 2),
    (1, 300, 300, 4, 2),      # ragged, two Q tiles + tail
    (1, 1, 1, 1, 1),          # one query, one key
    (2, 17, 700, 4, 1),       # fewer queries than keys (bottom-right causal)
    (1, 513, 513, 2, 1),
    (2, 1000, 1000, 8, 2),
]


@pytest.mark.parametrize("out", ["bf16", "fp16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,Lq,Lk,H,Hkv", CASES)
def test_fp8_forward_matches_oracle(cuda_lib, B, Lq, Lk, H, Hkv, causal, out):
    run(B, Lq, Lk, H, Hkv, causal, out, seed=B * 7919 + Lq * 31 + Lk + int(causal))


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_b8_h32_l4096_d128_full(cuda_lib, causal):
    """The FP8 benchmark's workload at full size, sampled (batch, head) units."""
    run(8, 4096, 4096, 32, 32, causal, "bf16", seed=77 + int(causal),
        units=[(0, 0), (3, 17), (7, 31)])


def test_fp8_gqa_b4_h32_hkv8_l4096(cuda_lib):
    run(4, 4096, 4096, 32, 8, True, "bf16", seed=78, units=[(0, 0), (1, 3), (2, 4), (3, 31)])


def test_fp8_scales_act_on_the_right_operands(cuda_lib):
    """Doubling q_scale while halving k_scale leaves O unchanged; doubling
    v_scale doubles O and leaves LSE unchanged (up to output rounding)."""
    q8, k8, v8, qs, ks, vs = make_qkv_fp8(1, 256, 256, 2, 2, 128, seed=3)
    q8, k8, v8 = q8.cuda(), k8.cuda(), v8.cuda()
    o1, l1 = fa.fwd_fp8(q8, k8, v8, qs, ks, vs, True)
    o2, l2 = fa.fwd_fp8(q8, k8, v8, qs * 2, ks / 2, vs, True)
    o3, l3 = fa.fwd_fp8(q8, k8, v8, qs, ks, vs * 2, True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.allclose(l1, l2, atol=1e-5, rtol=0)
    assert torch.equal(o3.float(), 2 * o1.float()) and torch.equal(l1, l3)


def test_fp8_argument_errors(cuda_lib):
    q8, k8, v8, qs, ks, vs = make_qkv_fp8(1, 64, 64, 2, 2, 128, seed=4)
    q8, k8, v8 = q8.cuda(), k8.cuda(), v8.cuda()
    for bad in (0.0, -1.0, float("inf"), float("nan")):
        with pytest.raises(_lib.FAError) as e:
            fa.fwd_fp8(q8, k8, v8, bad, ks, vs)
        assert e.value.status == _lib.FA_ERR_INVALID_ARG
    q64 = torch.zeros(1, 64, 2, 64, dtype=torch.uint8, device="cuda")
    k64 = torch.zeros(1, 64, 2, 64, dtype=torch.uint8, device="cuda")
    with pytest.raises(_lib.FAError) as e:
        fa.fwd_fp8(q64, k64, k64, 1.0, 1.0, 1.0)
    assert e.value.status == _lib.FA_ERR_UNSUPPORTED
