"""Host-side checks of the C ABI (no GPU): the library builds and loads, it
exports every function include/fa.h declares, and argument validation rejects
bad calls before anything reaches the device."""

import os

import pytest

from tiled_attention_fa_gb300 import _lib


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(_lib.LIB_PATH):
        from tiled_attention_fa_gb300 import build
        build.build(quiet=True)
    return _lib.load()


def test_exports_every_declared_function(lib):
    names = _lib.header_functions()
    assert {"fa_fwd", "fa_bwd_preprocess", "fa_bwd", "fa_bwd_workspace_size"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/fa.h but not exported"


def test_status_strings(lib):
    for code in range(5):
        assert lib.fa_status_string(code)
    assert b"sm_103a" in lib.fa_version()


def test_workspace_size(lib):
    assert lib.fa_bwd_workspace_size(8, 4096, 32, 128) == 8 * 32 * 4096 * 128 * 4
    assert lib.fa_bwd_workspace_size(1, 1, 1, 64) == 128 * 64 * 4   # padded to one 128-row tile
    assert lib.fa_bwd_workspace_size(2, 129, 3, 64) == 2 * 3 * 256 * 64 * 4
    assert lib.fa_bwd_workspace_size(0, 128, 1, 64) == 0


FAKE = 0x10000  # never dereferenced: every call below fails validation first


@pytest.mark.parametrize("args,want", [
    # (Q, K, V, O, LSE, B, L, H, Hkv, D, causal, dtype)
    ((None, FAKE, FAKE, FAKE, FAKE, 1, 128, 2, 2, 64, 0, 0), _lib.FA_ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, None, 1, 128, 2, 2, 64, 0, 0), _lib.FA_ERR_INVALID_ARG),
    ((FAKE + 8, FAKE, FAKE, FAKE, FAKE, 1, 128, 2, 2, 64, 0, 0), _lib.FA_ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 0, 128, 2, 2, 64, 0, 0), _lib.FA_ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 1, 0, 2, 2, 64, 0, 0), _lib.FA_ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 1, 128, 3, 2, 64, 0, 0), _lib.FA_ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 1, 128, 2, 2, 96, 0, 0), _lib.FA_ERR_UNSUPPORTED),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 1, 128, 2, 2, 64, 0, 7), _lib.FA_ERR_UNSUPPORTED),
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 20, 1 << 20, 1 << 12, 1, 128, 0, 0), _lib.FA_ERR_INVALID_ARG),
])
def test_fwd_argument_errors(lib, args, want):
    assert lib.fa_fwd(*args, None) == want


def test_bwd_argument_errors(lib):
    ok = [FAKE] * 11
    base = ok + [1, 1, 128, 4, 2, 64, 0, 0]
    assert lib.fa_bwd(*(ok[:10] + [None] + base[11:]), None) == _lib.FA_ERR_INVALID_ARG  # no workspace
    bad_d = list(base)
    bad_d[16] = 80
    assert lib.fa_bwd(*bad_d, None) == _lib.FA_ERR_UNSUPPORTED
    bad_h = list(base)
    bad_h[14] = 3
    assert lib.fa_bwd(*bad_h, None) == _lib.FA_ERR_INVALID_ARG
    assert lib.fa_bwd_preprocess(None, FAKE, FAKE, None, 1, 128, 2, 64, 0, None) == _lib.FA_ERR_INVALID_ARG
    assert lib.fa_bwd_preprocess(FAKE, FAKE, FAKE, FAKE + 4, 1, 128, 2, 64, 0, None) == _lib.FA_ERR_INVALID_ARG
    assert lib.fa_bwd_preprocess(FAKE, FAKE, FAKE, None, 1, 128, 2, 64, 3, None) == _lib.FA_ERR_UNSUPPORTED


def test_product_path_has_no_oracle_or_cpu_fallback():
    """The package never imports the oracle and every compute call goes through the library."""
    import tiled_attention_fa_gb300 as pkg
    root = os.path.dirname(pkg.__file__)
    for dirpath, _, files in os.walk(root):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f), encoding="utf-8").read()
                assert "import oracle" not in src and "from oracle" not in src, f


def test_decode_argument_errors(lib):
    """fa_decode rejects bad calls (and a short workspace) before any launch."""
    big = 1 << 30
    # (Q, K, V, O, LSE, ws, ws_bytes, B, Lq, Lk, H, Hkv, D, causal, dtype)
    base = [FAKE] * 6 + [big, 2, 1, 4096, 32, 8, 128, 0, 1]

    def call(**kw):
        a = list(base)
        names = ["Q", "K", "V", "O", "LSE", "ws", "ws_bytes", "B", "Lq", "Lk", "H", "Hkv", "D",
                 "causal", "dtype"]
        for key, val in kw.items():
            a[names.index(key)] = val
        return lib.fa_decode(*a, None)

    assert call(ws=None) == _lib.FA_ERR_INVALID_ARG
    assert call(ws=FAKE + 4) == _lib.FA_ERR_INVALID_ARG
    assert call(Q=None) == _lib.FA_ERR_INVALID_ARG
    assert call(H=30) == _lib.FA_ERR_INVALID_ARG             # H % Hkv != 0
    assert call(D=96) == _lib.FA_ERR_UNSUPPORTED
    assert call(Lq=33) == _lib.FA_ERR_UNSUPPORTED           # g * Lq = 132 > 128 packed rows
    assert call(Lq=8, Lk=4, causal=1) == _lib.FA_ERR_INVALID_ARG  # causal needs Lk >= Lq
    assert call(ws_bytes=0) == _lib.FA_ERR_SCRATCH_TOO_SMALL
    need = lib.fa_decode_workspace_size(2, 1, 4096, 32, 8, 128)
    assert need >= 2 * 32 * 1 * 129 * 4                      # one slice at least
    assert call(ws_bytes=need - 1) == _lib.FA_ERR_SCRATCH_TOO_SMALL
    assert lib.fa_decode_workspace_size(0, 1, 4096, 32, 8, 128) == 0
    assert lib.fa_decode_workspace_size(2, 1, 4096, 32, 8, 80) == 0
