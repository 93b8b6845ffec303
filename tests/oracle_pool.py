"""A pool of host processes that run the fp64 oracle on many (batch, head) units
at once and compare each with the GPU's output for that unit.

The processes are started with ``spawn`` (a process forked after CUDA has been
initialised in the parent can hang) and each keeps its BLAS to one thread, so
the pool spreads whole units over the host cores.  Workers import only numpy
and the oracle; the GPU outputs travel to them as float32 arrays (exact for
16-bit values) and only the verdicts come back."""

import multiprocessing as mp
import os
from concurrent.futures import ProcessPoolExecutor

import numpy as np

from oracle import fa_oracle as orc

_POOL = None
_BLAS_ENV = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")


def _cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def pool() -> ProcessPoolExecutor:
    global _POOL
    if _POOL is None:
        saved = {k: os.environ.get(k) for k in _BLAS_ENV}
        for k in _BLAS_ENV:
            os.environ[k] = "1"
        try:
            n = max(1, min(16, _cores()))
            _POOL = ProcessPoolExecutor(max_workers=n, mp_context=mp.get_context("spawn"))
            # start every worker now, while the single-thread BLAS setting is in the environment
            list(_POOL.map(_ping, range(n)))
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v
    return _POOL


def _ping(_):
    return os.getpid()


def _worst(got, ref, rtol, atol):
    got = np.asarray(got, dtype=np.float64)
    if not np.all(np.isfinite(got)):
        return float("inf"), "non-finite values"
    ex = np.abs(got - ref) - (atol + rtol * np.abs(ref))
    i = np.unravel_index(int(np.argmax(ex)), ex.shape)
    return float(ex[i]), f"worst at {i}: got {got[i]:.6g} ref {ref[i]:.6g}"


def _fwd_task(args):
    tag, q, k, v, o, lse, causal, panel = args
    ro, rl = orc.unit_forward(q, k, v, causal, panel=panel)
    return [(f"O{tag}",) + _worst(o, ro, 1e-2, 1e-2),
            (f"LSE{tag}",) + _worst(lse, rl, 0.0, 1e-3)]


def _bwd_task(args):
    tag, q, k, v, do, dq, dk, dv, causal, panel = args
    rq, rk, rv, _, _, _ = orc.unit_backward(q, k, v, do, causal, panel=panel)
    return [(f"dQ{tag}",) + _worst(dq, rq, 1e-2, 1e-2),
            (f"dK{tag}",) + _worst(dk, rk, 1e-2, 1e-2),
            (f"dV{tag}",) + _worst(dv, rv, 1e-2, 1e-2)]


def _f32(t):
    return t.float().numpy() if hasattr(t, "float") else np.asarray(t, dtype=np.float32)


def check_forward_units(q, k, v, o, lse, causal, units, panel=2048):
    """O and LSE of each (b, h) in ``units`` against the exact oracle (1e-2 / 1e-3).
    Tensors are CPU torch tensors, BSHD (LSE [B, H, L])."""
    H, Hkv = q.shape[2], k.shape[2]
    tasks = []
    for b, h in units:
        hk = orc.kv_head(h, H, Hkv)
        tasks.append((f"[{b},:,{h}]", _f32(q[b, :, h]), _f32(k[b, :, hk]), _f32(v[b, :, hk]),
                      _f32(o[b, :, h]), _f32(lse[b, h]), causal, panel))
    _raise_on(pool().map(_fwd_task, tasks))


def check_backward_units(q, k, v, do, dq, dk, dv, causal, units, panel=2048):
    """dQ, dK, dV of MHA units (the K/V head of (b, h) receives gradient from query
    head h alone) against the exact oracle, 1e-2 + 1e-2 |ref| element-wise."""
    assert q.shape[2] == k.shape[2], "unit-wise dK / dV comparison needs one query head per K/V head"
    tasks = [(f"[{b},:,{h}]", _f32(q[b, :, h]), _f32(k[b, :, h]), _f32(v[b, :, h]),
              _f32(do[b, :, h]), _f32(dq[b, :, h]), _f32(dk[b, :, h]), _f32(dv[b, :, h]),
              causal, panel) for b, h in units]
    _raise_on(pool().map(_bwd_task, tasks))


def _raise_on(results):
    bad = [r for res in results for r in res if r[1] > 0]
    if bad:
        bad.sort(key=lambda r: -r[1])
        lines = "; ".join(f"{n}: excess {e:.3g}, {msg}" for n, e, msg in bad[:5])
        raise AssertionError(f"{len(bad)} output(s) out of tolerance: {lines}")
