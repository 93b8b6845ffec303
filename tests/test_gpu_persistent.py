"""Backward with several work units per persistent CTA, compared whole
against the fp64 oracle.

The backward's CTAs are persistent: each takes work units (one K/V tile, or
under causal masking the pair of K/V tiles j and n_kv-1-j of one head) in
turn, reloading K/V, writing the finished unit's dK/dV and draining its last
dQ tile while the next unit starts.  These shapes have more units than the
GPU has SMs, so every hand-off between units runs, and the whole outputs are
compared (the full-size configuration tests sample (batch, head) units)."""

import pytest
import torch

from tests.helpers import assert_close, inputs, kernel_casts, to64
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
    rq, rk, rv, _ = orc.backward(q, k, v, do, causal, **kernel_casts(dtype))
    assert_close(to64(dv), rv, name="dV")
    assert_close(to64(dk), rk, name="dK")
    assert_close(to64(dq), rq, name="dQ")
