"""Fewer queries than keys (prefill against a key/value cache): the queries
are the last Lq positions, causal offset past_len = Lk - Lq.  Forward and
backward against the oracle; non-causal also with Lq > Lk."""

import ctypes

import pytest
import torch

import tiled_attention_fa_gb300 as fa
from oracle import fa_oracle as orc
from tests.helpers import LSE_ATOL, assert_close, check_backward, to64
from tiled_attention_fa_gb300 import _lib
from tiled_attention_fa_gb300.inputs import storage_dtype

pytestmark = pytest.mark.gpu


def make(B, Lq, Lk, H, Hkv, D, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    dt = storage_dtype(dtype)
    q = torch.randn(B, Lq, H, D, generator=g).to(dt)
    k = torch.randn(B, Lk, Hkv, D, generator=g).to(dt)
    v = torch.randn(B, Lk, Hkv, D, generator=g).to(dt)
    do = torch.randn(B, Lq, H, D, generator=g).to(dt)
    return q, k, v, do


CASES = [(1, 300), (17, 129), (128, 640), (200, 513), (129, 1000), (256, 4096)]


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Lq,Lk", CASES)
def test_forward_backward(cuda_lib, Lq, Lk, causal, D):
    q, k, v, do = make(1, Lq, Lk, 4, 2, D, "fp16", seed=Lq * 7 + Lk)
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    o, lse = fa.fwd(qd, kd, vd, causal)
    dq, dk, dv, _ = fa.attention_backward(qd, kd, vd, o, lse, dod, causal)
    torch.cuda.synchronize()
    fa.check_device_error()
    q64, k64, v64, do64 = (to64(x) for x in (q, k, v, do))
    ro, rl = orc.forward(q64, k64, v64, causal)
    assert_close(to64(o), ro, name="O")
    assert_close(to64(lse), rl, rtol=0, atol=LSE_ATOL, name="LSE")
    check_backward((to64(dq), to64(dk), to64(dv)), q64, k64, v64, do64, causal, "fp16")


@pytest.mark.parametrize("Lq,Lk", [(300, 100), (513, 129)])
def test_more_queries_than_keys_non_causal(cuda_lib, Lq, Lk):
    q, k, v, do = make(2, Lq, Lk, 2, 2, 128, "bf16", seed=Lq + Lk)
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    o, lse = fa.fwd(qd, kd, vd, False)
    dq, dk, dv, _ = fa.attention_backward(qd, kd, vd, o, lse, dod, False)
    q64, k64, v64, do64 = (to64(x) for x in (q, k, v, do))
    ro, rl = orc.forward(q64, k64, v64, False)
    assert_close(to64(o), ro, name="O")
    check_backward((to64(dq), to64(dk), to64(dv)), q64, k64, v64, do64, False, "bf16")


def test_causal_needs_at_least_as_many_keys(cuda_lib):
    t = torch.empty(64, device="cuda", dtype=torch.float16)
    p = ctypes.c_void_p(t.data_ptr())
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert cuda_lib.fa_fwd_kv(p, p, p, p, p, 1, 200, 100, 2, 2, 64, 1, 0, s) == _lib.FA_ERR_INVALID_ARG
