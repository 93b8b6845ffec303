"""Failure detection without a GPU fault: a bounded wait that nothing
completes gives up, the host reads FA_ERR_DEVICE_TIMEOUT with the site id,
and the context keeps working (a normal call afterwards still matches)."""

import ctypes

import pytest
import torch

import tiled_attention_fa_gb300 as fa
from tests.helpers import assert_close, inputs, to64
from oracle import fa_oracle as orc
from tiled_attention_fa_gb300 import _lib

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_and_reports(cuda_lib):
    lib = cuda_lib
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.fa_check_device_error(s) == _lib.FA_OK           # clean state
    assert lib.fa_selftest_bounded_wait(20_000_000, s) == _lib.FA_OK
    assert lib.fa_check_device_error(s) == _lib.FA_ERR_DEVICE_TIMEOUT
    assert lib.fa_last_error_site() == 900
    assert lib.fa_check_device_error(s) == _lib.FA_OK           # the word was cleared
    # The context is still usable: a forward afterwards matches the oracle.
    (q, k, v, _), (qd, kd, vd, _) = inputs(1, 200, 2, 1, 64, "fp16", 4)
    o, lse = fa.fwd(qd, kd, vd, True)
    ro, rl = orc.forward(q, k, v, True)
    assert_close(to64(o), ro, name="O")


def test_python_binding_raises_on_device_timeout(cuda_lib):
    lib = cuda_lib
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.fa_selftest_bounded_wait(1_000_000, s) == _lib.FA_OK
    with pytest.raises(_lib.FAError, match="site 900"):
        fa.check_device_error()
    fa.check_device_error()  # cleared
