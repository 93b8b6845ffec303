"""Forward and backward with several work items per persistent CTA, compared
whole against the fp64 oracle.

The backward's CTAs are persistent: each takes work units (one K/V tile, or
under causal masking the pair of K/V tiles j and n_kv-1-j of one head) in
turn, reloading K/V, writing the finished unit's dK/dV and draining its last
dQ tile while the next unit starts.  These shapes have more units than the
GPU has SMs, so every hand-off between units runs, and the whole outputs are
compared (the full-size configuration tests sample (batch, head) units)."""

import pytest
import torch

import tiled_attention_fa_gb300 as fa
from tests.helpers import LSE_ATOL, assert_close, check_backward, inputs, to64
from tests.test_gpu_bwd import gpu_fwd_bwd
from oracle import fa_oracle as orc

pytestmark = pytest.mark.gpu


def units(B, L, Hkv, causal):
    n_kv = (L + 127) // 128
    return B * Hkv * ((n_kv + 1) // 2 if causal else n_kv)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,L,H,Hkv,D,dtype", [
    (4, 1024, 16, 16, 64, "fp16"),    # 512 (256 causal) units: several per CTA
    (8, 640, 8, 8, 64, "bf16"),       # n_kv = 5: the middle tile is a unit of its own
    (32, 768, 8, 2, 128, "bf16"),     # grouped heads: 4 query heads per K/V tile
])
def test_backward_many_units_per_cta(cuda_lib, B, L, H, Hkv, D, dtype, causal):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert units(B, L, Hkv, causal) > sms, "shape must give some CTA more than one unit"
    (q, k, v, do), (qd, kd, vd, dod) = inputs(B, L, H, Hkv, D, dtype, seed=B * L + H + int(causal))
    _, _, dq, dk, dv, _ = gpu_fwd_bwd(qd, kd, vd, dod, causal)
    check_backward((to64(dq), to64(dk), to64(dv)), q, k, v, do, causal, dtype)


def fwd_items(B, L, H):
    return B * H * ((L + 255) // 256)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,L,H,Hkv,D,dtype", [
    (4, 1024, 32, 8, 64, "bf16"),     # 512 items; at D = 64 Q lives in TMEM and the next
                                      # item's Q loads while the current one runs
    (3, 900, 40, 8, 64, "fp16"),      # ragged length, group of 5
    (2, 768, 64, 64, 128, "fp16"),    # 384 items at D = 128
])
def test_forward_many_items_per_cta(cuda_lib, B, L, H, Hkv, D, dtype, causal):
    """The forward's persistent CTAs take items (batch, head, pair of Q tiles)
    in turn; these shapes give every CTA several, so each hand-off between
    items (Q buffers reloaded, at D = 64 while the previous item still runs)
    is compared element by element."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert fwd_items(B, L, H) > 2 * sms, "shape must give CTAs several items"
    (q, k, v, _), (qd, kd, vd, _) = inputs(B, L, H, Hkv, D, dtype, seed=7 * B + L + H + int(causal))
    o, lse = fa.fwd(qd, kd, vd, causal)
    torch.cuda.synchronize()
    fa.check_device_error()
    ro, rl = orc.forward(q, k, v, causal)
    assert_close(to64(o), ro, name="O")
    assert_close(to64(lse), rl, rtol=0, atol=LSE_ATOL, name="LSE")
