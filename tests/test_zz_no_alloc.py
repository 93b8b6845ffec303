"""fa_bwd_noalloc: the backward for callers that cannot allocate device memory
at call time (a plugin inside a host application that owns all GPU memory,
or a serving path that must not allocate after start-up).  It keeps the dQ
accumulator in a fixed array inside the library instead of a caller
workspace.  Checked through the C ABI against fa_bwd with a workspace, on two
calls in a row (the second call must not see the first call's sums).

This file sorts last so that a run stopping at its first failure has already
run every other test."""

import ctypes

import pytest
import torch

from tests.helpers import assert_close, inputs, to64
from tiled_attention_fa_gb300 import _lib

pytestmark = pytest.mark.gpu


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("B,L,H,Hkv,D,causal", [(1, 300, 4, 2, 128, True), (2, 513, 2, 1, 64, False)])
def test_noalloc_matches_workspace_backward(cuda_lib, B, L, H, Hkv, D, causal):
    lib = cuda_lib
    _, (q, k, v, do) = inputs(B, L, H, Hkv, D, "fp16", seed=L + D)
    dev = q.device
    o = torch.empty_like(q)
    lse = torch.empty(B, H, L, device=dev, dtype=torch.float32)
    delta = torch.empty_like(lse)
    acc = torch.empty(lib.fa_bwd_workspace_size(B, L, H, D) // 4, device=dev, dtype=torch.float32)
    dims = (B, L, H, Hkv, D, int(causal), _lib.FA_F16)
    assert lib.fa_fwd(_p(q), _p(k), _p(v), _p(o), _p(lse), *dims, _stream()) == _lib.FA_OK
    assert lib.fa_bwd_preprocess(_p(o), _p(do), _p(delta), _p(acc), B, L, H, D, _lib.FA_F16,
                                 _stream()) == _lib.FA_OK
    ref = [torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)]
    assert lib.fa_bwd(_p(q), _p(k), _p(v), _p(o), _p(do), _p(lse), _p(delta),
                      *(_p(t) for t in ref), _p(acc), 0, *dims, _stream()) == _lib.FA_OK
    # The flow of a caller that allocates nothing: Delta from the preprocess
    # with no accumulator, then the no-allocation backward.
    delta2 = torch.full_like(lse, float("nan"))
    assert lib.fa_bwd_preprocess(_p(o), _p(do), _p(delta2), None, B, L, H, D, _lib.FA_F16,
                                 _stream()) == _lib.FA_OK
    for call in range(2):
        got = [torch.full_like(q, float("nan")), torch.full_like(k, float("nan")),
               torch.full_like(v, float("nan"))]
        st = lib.fa_bwd_noalloc(_p(q), _p(k), _p(v), _p(o), _p(do), _p(lse), _p(delta2),
                                *(_p(t) for t in got), *dims, _stream())
        assert st == _lib.FA_OK, lib.fa_status_string(st)
        torch.cuda.synchronize()
        assert lib.fa_check_device_error(_stream()) == _lib.FA_OK
        for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
            assert_close(to64(g), to64(r), name=f"{name} (call {call + 1})")


def test_noalloc_rejects_problems_beyond_its_scratch(cuda_lib):
    lib = cuda_lib
    # B=1, H=32, L=4096, D=128 needs exactly the 64 MiB; one more 128-row tile does not fit.
    assert lib.fa_bwd_workspace_size(1, 4096, 32, 128) == _lib.FA_NOALLOC_SCRATCH_BYTES
    t = torch.empty(16, device="cuda", dtype=torch.float16)
    st = lib.fa_bwd_noalloc(*([_p(t)] * 10), 1, 4097, 32, 32, 128, 0, _lib.FA_F16, _stream())
    assert st == _lib.FA_ERR_SCRATCH_TOO_SMALL
