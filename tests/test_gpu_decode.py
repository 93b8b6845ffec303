"""Split-KV decoding (few queries, long key/value sequence) against the
oracle's forward: the sliced computation and its log-sum-exp merge must give
the forward's O and LSE (causal offset past_len = Lk - Lq)."""

import numpy as np
import pytest
import torch

import tiled_attention_fa_gb300 as fa
from oracle import fa_oracle as orc
from tests.helpers import LSE_ATOL, assert_close, to64
from tiled_attention_fa_gb300 import _lib
from tiled_attention_fa_gb300.inputs import make_qkv_kv

pytestmark = pytest.mark.gpu


def slices(B, Lq, Lk, H, Hkv, D):
    """Key slices per (batch, K/V head) the library plans on this GPU, recovered
    from the workspace size (fp32 partial O and LSE per slice, 256-byte padded)."""
    rows = B * H * Lq
    ws = fa.decode_workspace_size(B, Lq, Lk, H, Hkv, D)
    for ns in range(1, (Lk + 127) // 128 + 1):
        pad = lambda x: (x + 255) // 256 * 256  # noqa: E731
        if pad(ns * rows * D * 4) + pad(ns * rows * 4) == ws:
            return ns
    raise AssertionError(f"workspace size {ws} matches no slice count")


def check(B, Lq, Lk, H, Hkv, D, dtype, causal, seed, workspace=None):
    q, k, v, _ = make_qkv_kv(B, Lq, Lk, H, Hkv, D, dtype, seed)
    qd, kd, vd = (x.cuda() for x in (q, k, v))
    o, lse = fa.decode(qd, kd, vd, causal, workspace=workspace)
    torch.cuda.synchronize()
    fa.check_device_error()
    ro, rl = orc.forward(to64(q), to64(k), to64(v), causal)
    assert_close(to64(o), ro, name="O")
    assert_close(to64(lse), rl, rtol=0, atol=LSE_ATOL, name="LSE")


CASES = [
    # B, Lq, Lk, H, Hkv, D, dtype
    (2, 1, 4096, 32, 8, 128, "bf16"),    # GQA decode, 4 query heads per K/V head
    (1, 1, 1, 8, 8, 128, "fp16"),        # one key, one packed row
    (1, 1, 100, 4, 1, 64, "fp16"),       # fewer keys than one tile
    (3, 4, 1000, 16, 4, 64, "bf16"),     # 16 packed rows, ragged last tile
    (1, 16, 8197, 8, 1, 128, "fp16"),    # 128 packed rows, one-tile slices, 5-key tail slice
    (2, 2, 3000, 64, 1, 128, "fp16"),    # multi-query: 64 heads share one K/V head
    (4, 1, 16384, 32, 32, 128, "fp16"),  # MHA decode, one row per CTA
    (1, 8, 65536, 8, 1, 128, "bf16"),    # long context
    (2, 3, 777, 6, 2, 64, "fp16"),       # 9 packed rows, odd sizes
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,Lq,Lk,H,Hkv,D,dtype", CASES)
def test_decode_matches_oracle(cuda_lib, B, Lq, Lk, H, Hkv, D, dtype, causal):
    check(B, Lq, Lk, H, Hkv, D, dtype, causal, seed=B * 1000 + Lq * 10 + Lk + int(causal))


def test_slices_cover_masked_tail(cuda_lib):
    """With one (batch, K/V head) and 65 tiles the plan cuts the keys into many
    slices; under causal masking the 5-key tail slice holds no visible key for
    the first queries, whose partial LSE is -inf and must drop out of the merge."""
    assert slices(1, 16, 8197, 8, 1, 128) > 8
    check(1, 16, 8197, 8, 1, 128, "fp16", True, seed=5)


def test_workspace_reused_across_calls(cuda_lib):
    """One caller workspace serves consecutive calls with different inputs."""
    ws = torch.empty(fa.decode_workspace_size(2, 4, 5000, 32, 8, 128), device="cuda",
                     dtype=torch.uint8)
    check(2, 4, 5000, 32, 8, 128, "bf16", True, seed=1, workspace=ws)
    check(2, 4, 5000, 32, 8, 128, "bf16", False, seed=2, workspace=ws)
    check(2, 1, 300, 32, 8, 128, "bf16", True, seed=3, workspace=ws)   # smaller problem, same buffer


def test_decode_rejects_short_workspace(cuda_lib):
    q, k, v, _ = make_qkv_kv(1, 1, 2048, 8, 2, 128, "fp16", 0)
    qd, kd, vd = (x.cuda() for x in (q, k, v))
    small = torch.empty(256, device="cuda", dtype=torch.uint8)
    with pytest.raises(_lib.FAError) as e:
        fa.decode(qd, kd, vd, False, workspace=small)
    assert e.value.status == _lib.FA_ERR_SCRATCH_TOO_SMALL


@pytest.mark.parametrize("causal", [False, True])
def test_decode_b16_h32_hkv8_lk16384_d128_bf16_full(cuda_lib, causal):
    """The decoding benchmark's workload at full size, every (batch, head) row
    against the oracle."""
    B, Lq, Lk, H, Hkv, D = 16, 1, 16384, 32, 8, 128
    check(B, Lq, Lk, H, Hkv, D, "bf16", causal, seed=42 + int(causal))


def test_decode_long_b1_lk131072(cuda_lib):
    """Long context: B=1, 8 K/V heads, 131072 keys, GQA 4 queries per K/V head."""
    q, k, v, _ = make_qkv_kv(1, 1, 131072, 32, 8, 128, "bf16", 7)
    qd, kd, vd = (x.cuda() for x in (q, k, v))
    o, lse = fa.decode(qd, kd, vd, True)
    torch.cuda.synchronize()
    fa.check_device_error()
    q64, k64, v64 = to64(q), to64(k), to64(v)
    for h in (0, 5, 31):
        hk = orc.kv_head(h, 32, 8)
        ro, rl = orc.unit_forward(q64[0, :, h], k64[0, :, hk], v64[0, :, hk], True)
        assert_close(to64(o)[0, :, h], ro, name=f"O[h={h}]")
        assert_close(to64(lse)[0, h], rl, rtol=0, atol=LSE_ATOL, name=f"LSE[h={h}]")
    assert np.isfinite(to64(o)).all()


def test_two_stage_calls_match_decode(cuda_lib):
    """fa_decode_slices then fa_decode_merge give fa_decode's result bit for bit."""
    q, k, v, _ = make_qkv_kv(2, 2, 5000, 16, 4, 64, "fp16", 11)
    qd, kd, vd = (x.cuda() for x in (q, k, v))
    o1, l1 = fa.decode(qd, kd, vd, True)
    ws = fa.alloc_decode_workspace(2, 2, 5000, 16, 4, 64, qd.device)
    o2, l2 = torch.empty_like(o1), torch.empty_like(l1)
    fa.decode_slices(qd, kd, vd, ws, True)
    fa.decode_merge(ws, o2, l2, 5000, 4)
    torch.cuda.synchronize()
    fa.check_device_error()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
