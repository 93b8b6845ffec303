"""Python binding of the C ABI: argument marshalling only.

Every function takes torch CUDA tensors (PyTorch supplies device memory and
the current stream), checks layout and dtype, and calls the matching C entry
point.  All arithmetic runs in the library's CUDA kernels; there is no CPU or
framework fallback.  ``HostRunner`` serves callers whose data lives on the
host: it copies through pinned host memory around the same calls;
``HostPipeline`` does the same for a sequence of batches with the copies of
one batch overlapping the kernels of its neighbours.
"""

from __future__ import annotations

import torch

from . import _lib

_DT = {torch.float16: _lib.FA_F16, torch.bfloat16: _lib.FA_BF16}


def _dtype_code(t: torch.Tensor) -> int:
    try:
        return _DT[t.dtype]
    except KeyError as e:
        raise TypeError(f"dtype {t.dtype} unsupported: use float16 or bfloat16") from e


def _need(t: torch.Tensor, name: str, shape=None, dtype=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def fwd(q, k, v, causal: bool = False, out=None, lse=None, stream=None):
    """O, LSE = attention(Q, K, V).  q [B, Lq, H, D]; k, v [B, Lk, Hkv, D].

    Lq < Lk means the queries are the last Lq positions (causal offset
    Lk - Lq); Lq == Lk is the square case."""
    B, L, H, D = q.shape
    Lk, Hkv = k.shape[1], k.shape[2]
    _need(q, "q")
    _need(k, "k", (B, Lk, Hkv, D), q.dtype)
    _need(v, "v", (B, Lk, Hkv, D), q.dtype)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(B, H, L, device=q.device, dtype=torch.float32)
    _need(out, "out", q.shape, q.dtype)
    _need(lse, "lse", (B, H, L), torch.float32)
    lib = _lib.load()
    if Lk == L:
        st = lib.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                        B, L, H, Hkv, D, int(bool(causal)), _dtype_code(q), _stream(stream))
        _lib.check("fa_fwd", st)
    else:
        st = lib.fa_fwd_kv(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                           lse.data_ptr(), B, L, Lk, H, Hkv, D, int(bool(causal)),
                           _dtype_code(q), _stream(stream))
        _lib.check("fa_fwd_kv", st)
    return out, lse


def decode_workspace_size(B: int, Lq: int, Lk: int, H: int, Hkv: int, D: int) -> int:
    """Bytes of the partial-result workspace ``decode`` needs on the current device."""
    return int(_lib.load().fa_decode_workspace_size(B, Lq, Lk, H, Hkv, D))


_OUT = {torch.float16: _lib.FA_F16, torch.bfloat16: _lib.FA_BF16}


def _codes(t: torch.Tensor, name: str, shape=None):
    """E4M3 codes: a uint8 or float8_e4m3fn CUDA tensor."""
    if t.dtype not in (torch.uint8, torch.float8_e4m3fn):
        raise TypeError(f"{name} must hold E4M3 codes (uint8 or float8_e4m3fn), got {t.dtype}")
    _need(t, name, shape)


def fwd_fp8(q8, k8, v8, q_scale: float, k_scale: float, v_scale: float, causal: bool = False,
            out_dtype=torch.bfloat16, out=None, lse=None, stream=None):
    """O, LSE = attention of E4M3 inputs with per-tensor scales: the forward of
    decode(q8) * q_scale, decode(k8) * k_scale, decode(v8) * v_scale.
    q8 [B, Lq, H, 128]; k8, v8 [B, Lk, Hkv, 128]; O in ``out_dtype``."""
    B, L, H, D = q8.shape
    Lk, Hkv = k8.shape[1], k8.shape[2]
    _codes(q8, "q8")
    _codes(k8, "k8", (B, Lk, Hkv, D))
    _codes(v8, "v8", (B, Lk, Hkv, D))
    if out_dtype not in _OUT:
        raise TypeError("out_dtype must be torch.float16 or torch.bfloat16")
    if out is None:
        out = torch.empty(B, L, H, D, device=q8.device, dtype=out_dtype)
    if lse is None:
        lse = torch.empty(B, H, L, device=q8.device, dtype=torch.float32)
    _need(out, "out", (B, L, H, D), out_dtype)
    _need(lse, "lse", (B, H, L), torch.float32)
    st = _lib.load().fa_fwd_fp8(q8.data_ptr(), k8.data_ptr(), v8.data_ptr(), float(q_scale),
                                float(k_scale), float(v_scale), out.data_ptr(), lse.data_ptr(), B, L,
                                Lk, H, Hkv, D, int(bool(causal)), _OUT[out_dtype], _stream(stream))
    _lib.check("fa_fwd_fp8", st)
    return out, lse


def _decode_shapes(q, k, v):
    B, Lq, H, D = q.shape
    Lk, Hkv = k.shape[1], k.shape[2]
    _need(q, "q")
    _need(k, "k", (B, Lk, Hkv, D), q.dtype)
    _need(v, "v", (B, Lk, Hkv, D), q.dtype)
    return B, Lq, Lk, H, Hkv, D


def _decode_outputs(q, B, Lq, H, out, lse):
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(B, H, Lq, device=q.device, dtype=torch.float32)
    _need(out, "out", q.shape, q.dtype)
    _need(lse, "lse", (B, H, Lq), torch.float32)
    return out, lse


def _nbytes(t) -> int:
    _need(t, "workspace")
    return t.numel() * t.element_size()


def alloc_decode_workspace(B, Lq, Lk, H, Hkv, D, device) -> torch.Tensor:
    """A byte tensor large enough for ``decode`` on ``device``."""
    with torch.cuda.device(device):
        n = decode_workspace_size(B, Lq, Lk, H, Hkv, D)
    return torch.empty(max(n, 16), device=device, dtype=torch.uint8)


def decode(q, k, v, causal: bool = False, out=None, lse=None, workspace=None, stream=None):
    """Split-KV decoding: O, LSE = attention(Q, K, V) for few queries against
    many keys.  q [B, Lq, H, D]; k, v [B, Lk, Hkv, D] with (H / Hkv) * Lq <= 128.
    Same result and masking rule as ``fwd``.  ``workspace`` (a CUDA byte
    tensor of at least ``decode_workspace_size`` bytes) is allocated when not
    given."""
    B, Lq, Lk, H, Hkv, D = _decode_shapes(q, k, v)
    out, lse = _decode_outputs(q, B, Lq, H, out, lse)
    if workspace is None:
        workspace = alloc_decode_workspace(B, Lq, Lk, H, Hkv, D, q.device)
    st = _lib.load().fa_decode(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                               lse.data_ptr(), workspace.data_ptr(), _nbytes(workspace), B, Lq, Lk,
                               H, Hkv, D, int(bool(causal)), _dtype_code(q), _stream(stream))
    _lib.check("fa_decode", st)
    return out, lse


def decode_slices(q, k, v, workspace, causal: bool = False, stream=None):
    """First stage of ``decode``: per-slice partial O and LSE into ``workspace``."""
    B, Lq, Lk, H, Hkv, D = _decode_shapes(q, k, v)
    st = _lib.load().fa_decode_slices(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                      workspace.data_ptr(), _nbytes(workspace), B, Lq, Lk, H, Hkv,
                                      D, int(bool(causal)), _dtype_code(q), _stream(stream))
    _lib.check("fa_decode_slices", st)


def decode_merge(workspace, out, lse, Lk: int, Hkv: int, stream=None):
    """Second stage of ``decode``: merge the slices into ``out`` [B, Lq, H, D]
    and ``lse`` [B, H, Lq] for a key length Lk and Hkv K/V heads."""
    B, Lq, H, D = out.shape
    _need(out, "out")
    _need(lse, "lse", (B, H, Lq), torch.float32)
    st = _lib.load().fa_decode_merge(workspace.data_ptr(), _nbytes(workspace), out.data_ptr(),
                                     lse.data_ptr(), B, Lq, Lk, H, Hkv, D, _dtype_code(out),
                                     _stream(stream))
    _lib.check("fa_decode_merge", st)


def workspace_size(B: int, L: int, H: int, D: int) -> int:
    """Bytes of the fp32 dQ accumulator the backward needs."""
    return int(_lib.load().fa_bwd_workspace_size(B, L, H, D))


def alloc_workspace(B: int, L: int, H: int, D: int, device) -> torch.Tensor:
    n = workspace_size(B, L, H, D) // 4
    return torch.empty(n, device=device, dtype=torch.float32)


def bwd_preprocess(o, do, delta=None, dq_accum=None, stream=None):
    """Delta[b, h, i] = sum_d O[b, i, h, d] dO[b, i, h, d]; optionally zero dq_accum."""
    B, L, H, D = o.shape
    _need(o, "o")
    _need(do, "do", o.shape, o.dtype)
    if delta is None:
        delta = torch.empty(B, H, L, device=o.device, dtype=torch.float32)
    _need(delta, "delta", (B, H, L), torch.float32)
    acc_ptr = 0
    if dq_accum is not None:
        _need(dq_accum, "dq_accum", dtype=torch.float32)
        if dq_accum.numel() * 4 < workspace_size(B, L, H, D):
            raise ValueError("dq_accum is smaller than workspace_size()")
        acc_ptr = dq_accum.data_ptr()
    st = _lib.load().fa_bwd_preprocess(o.data_ptr(), do.data_ptr(), delta.data_ptr(), acc_ptr or None,
                                       B, L, H, D, _dtype_code(o), _stream(stream))
    _lib.check("fa_bwd_preprocess", st)
    return delta


def bwd(q, k, v, o, do, lse, delta, causal: bool = False, dq=None, dk=None, dv=None,
        dq_accum=None, accum_zeroed: bool = False, stream=None):
    """dQ, dK, dV of the forward.  ``dq_accum`` is the fp32 workspace; unless
    ``accum_zeroed`` (fa_bwd_preprocess zeroed it) the call zeroes it first."""
    B, L, H, D = q.shape
    Lk, Hkv = k.shape[1], k.shape[2]
    _need(q, "q")
    for name, t, shp in (("k", k, (B, Lk, Hkv, D)), ("v", v, (B, Lk, Hkv, D)), ("do", do, q.shape)):
        _need(t, name, shp, q.dtype)
    _need(lse, "lse", (B, H, L), torch.float32)
    _need(delta, "delta", (B, H, L), torch.float32)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _need(dq, "dq", q.shape, q.dtype)
    _need(dk, "dk", k.shape, q.dtype)
    _need(dv, "dv", v.shape, q.dtype)
    if dq_accum is None:
        dq_accum = alloc_workspace(B, L, H, D, q.device)
        accum_zeroed = False
    _need(dq_accum, "dq_accum", dtype=torch.float32)
    if dq_accum.numel() * 4 < workspace_size(B, L, H, D):
        raise ValueError("dq_accum is smaller than workspace_size()")
    lib = _lib.load()
    ptrs = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr() if o is not None else None,
            do.data_ptr(), lse.data_ptr(), delta.data_ptr(), dq.data_ptr(), dk.data_ptr(),
            dv.data_ptr(), dq_accum.data_ptr(), 0 if accum_zeroed else 1)
    if Lk == L:
        st = lib.fa_bwd(*ptrs, B, L, H, Hkv, D, int(bool(causal)), _dtype_code(q), _stream(stream))
        _lib.check("fa_bwd", st)
    else:
        st = lib.fa_bwd_kv(*ptrs, B, L, Lk, H, Hkv, D, int(bool(causal)), _dtype_code(q),
                           _stream(stream))
        _lib.check("fa_bwd_kv", st)
    return dq, dk, dv


def bwd_main(q, k, v, do, lse, delta, dq_accum, causal: bool = False, dk=None, dv=None,
             accum_zeroed: bool = True, stream=None):
    """Stage 2 alone: dK, dV and the fp32 dQ accumulator (added into)."""
    B, L, H, D = q.shape
    Hkv = k.shape[2]
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for name, t in (("q", q), ("k", k), ("v", v), ("do", do), ("lse", lse), ("delta", delta),
                    ("dk", dk), ("dv", dv), ("dq_accum", dq_accum)):
        _need(t, name)
    if dq_accum.numel() * 4 < workspace_size(B, L, H, D):
        raise ValueError("dq_accum is smaller than workspace_size()")
    st = _lib.load().fa_bwd_main(q.data_ptr(), k.data_ptr(), v.data_ptr(), do.data_ptr(),
                                 lse.data_ptr(), delta.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                                 dq_accum.data_ptr(), 0 if accum_zeroed else 1, B, L, H, Hkv, D,
                                 int(bool(causal)), _dtype_code(q), _stream(stream))
    _lib.check("fa_bwd_main", st)
    return dk, dv


def bwd_postprocess(dq_accum, dq, stream=None):
    """Stage 3 alone: dQ (BSHD, input dtype) from the fp32 accumulator."""
    B, L, H, D = dq.shape
    _need(dq, "dq")
    _need(dq_accum, "dq_accum", dtype=torch.float32)
    st = _lib.load().fa_bwd_postprocess(dq_accum.data_ptr(), dq.data_ptr(), B, L, H, D,
                                        _dtype_code(dq), _stream(stream))
    _lib.check("fa_bwd_postprocess", st)
    return dq


def attention_backward(q, k, v, o, lse, do, causal: bool = False, dq_accum=None, stream=None):
    """Preprocess + backward in one call (Delta computed here, accumulator zeroed in the same pass)."""
    B, L, H, D = q.shape
    if dq_accum is None:
        dq_accum = alloc_workspace(B, L, H, D, q.device)
    delta = bwd_preprocess(o, do, dq_accum=dq_accum, stream=stream)
    dq, dk, dv = bwd(q, k, v, o, do, lse, delta, causal, dq_accum=dq_accum, accum_zeroed=True,
                     stream=stream)
    return dq, dk, dv, delta


def check_device_error(stream=None) -> None:
    """Synchronise and raise if a kernel gave up a bounded wait since the last check."""
    lib = _lib.load()
    st = lib.fa_check_device_error(_stream(stream))
    if st != _lib.FA_OK:
        raise _lib.FAError(f"device (site {lib.fa_last_error_site()})", st)


class HostRunner:
    """Forward + backward for host-resident tensors through pinned buffers.

    ``run(q, k, v, do)`` copies the CPU inputs to the device, runs the
    forward, the preprocess and the backward, and copies O, LSE, dQ, dK, dV
    back into pinned host tensors (returned).  Device buffers are allocated
    once per shape and reused.
    """

    def __init__(self, B, L, H, Hkv, D, dtype=torch.float16, causal=False, device="cuda",
                 Lk=None):
        self.causal = causal
        dev = torch.device(device)
        Lk = L if Lk is None else Lk
        self.q = torch.empty(B, L, H, D, dtype=dtype, device=dev)
        self.k = torch.empty(B, Lk, Hkv, D, dtype=dtype, device=dev)
        self.v = torch.empty_like(self.k)
        self.do = torch.empty_like(self.q)
        self.o = torch.empty_like(self.q)
        self.lse = torch.empty(B, H, L, dtype=torch.float32, device=dev)
        self.delta = torch.empty_like(self.lse)
        self.dq = torch.empty_like(self.q)
        self.dk = torch.empty_like(self.k)
        self.dv = torch.empty_like(self.k)
        self.acc = alloc_workspace(B, L, H, D, dev)
        pin = dict(pin_memory=True)
        self.h_out = {
            "o": torch.empty(self.o.shape, dtype=dtype, **pin),
            "lse": torch.empty(self.lse.shape, dtype=torch.float32, **pin),
            "dq": torch.empty(self.dq.shape, dtype=dtype, **pin),
            "dk": torch.empty(self.dk.shape, dtype=dtype, **pin),
            "dv": torch.empty(self.dv.shape, dtype=dtype, **pin),
        }

    def h2d_bytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in (self.q, self.k, self.v, self.do))

    def d2h_bytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in self.h_out.values())

    def run(self, q, k, v, do, stream=None):
        for dst, src in ((self.q, q), (self.k, k), (self.v, v), (self.do, do)):
            dst.copy_(src, non_blocking=True)
        fwd(self.q, self.k, self.v, self.causal, out=self.o, lse=self.lse, stream=stream)
        bwd_preprocess(self.o, self.do, delta=self.delta, dq_accum=self.acc, stream=stream)
        bwd(self.q, self.k, self.v, self.o, self.do, self.lse, self.delta, self.causal,
            dq=self.dq, dk=self.dk, dv=self.dv, dq_accum=self.acc, accum_zeroed=True,
            stream=stream)
        for name, src in (("o", self.o), ("lse", self.lse), ("dq", self.dq), ("dk", self.dk),
                          ("dv", self.dv)):
            self.h_out[name].copy_(src, non_blocking=True)
        return self.h_out


class HostPipeline:
    """Forward + backward over a stream of host-resident batches, with each
    batch's copies overlapping its neighbours' kernels.

    ``submit(q, k, v, do)`` enqueues one step (pinned host inputs) and returns
    the pinned host tensors its O, LSE, dQ, dK, dV will land in; ``wait()``
    blocks until every submitted step is done.  ``depth`` sets of device
    buffers rotate: step s uploads into set s % depth on an upload stream, runs
    the forward, preprocess and backward on the compute stream once its inputs
    are in and the set's previous outputs have been read back, and reads its
    results back on a download stream.  A step's host outputs are valid after
    ``wait()`` (or once the step ``depth`` later has been submitted and has
    started its download) and are reused by step s + depth.
    """

    def __init__(self, B, L, H, Hkv, D, dtype=torch.float16, causal=False, device="cuda",
                 Lk=None, depth=2):
        self.causal = causal
        self.depth = depth
        dev = torch.device(device)
        Lk = L if Lk is None else Lk
        self.sets = []
        pin = dict(pin_memory=True)
        for _ in range(depth):
            d = {"q": torch.empty(B, L, H, D, dtype=dtype, device=dev),
                 "k": torch.empty(B, Lk, Hkv, D, dtype=dtype, device=dev)}
            d["v"] = torch.empty_like(d["k"])
            d["do"] = torch.empty_like(d["q"])
            d["o"] = torch.empty_like(d["q"])
            d["lse"] = torch.empty(B, H, L, dtype=torch.float32, device=dev)
            d["delta"] = torch.empty_like(d["lse"])
            d["dq"] = torch.empty_like(d["q"])
            d["dk"] = torch.empty_like(d["k"])
            d["dv"] = torch.empty_like(d["k"])
            d["acc"] = alloc_workspace(B, L, H, D, dev)
            d["h_out"] = {n: torch.empty(d[n].shape, dtype=d[n].dtype, **pin)
                          for n in ("o", "lse", "dq", "dk", "dv")}
            d["in_ready"] = torch.cuda.Event()
            d["computed"] = torch.cuda.Event()
            d["read_back"] = torch.cuda.Event()
            d["used"] = False
            self.sets.append(d)
        self.up = torch.cuda.Stream(device=dev)
        self.compute = torch.cuda.Stream(device=dev)
        self.down = torch.cuda.Stream(device=dev)
        self.n = 0

    def h2d_bytes(self) -> int:
        d = self.sets[0]
        return sum(d[n].numel() * d[n].element_size() for n in ("q", "k", "v", "do"))

    def d2h_bytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in self.sets[0]["h_out"].values())

    def submit(self, q, k, v, do):
        d = self.sets[self.n % self.depth]
        self.n += 1
        if d["used"]:
            self.up.wait_event(d["computed"])  # the set's previous step has read its inputs
        with torch.cuda.stream(self.up):
            for name, src in (("q", q), ("k", k), ("v", v), ("do", do)):
                d[name].copy_(src, non_blocking=True)
            d["in_ready"].record(self.up)
        self.compute.wait_event(d["in_ready"])
        if d["used"]:
            self.compute.wait_event(d["read_back"])  # its previous outputs are on the host
        fwd(d["q"], d["k"], d["v"], self.causal, out=d["o"], lse=d["lse"], stream=self.compute)
        bwd_preprocess(d["o"], d["do"], delta=d["delta"], dq_accum=d["acc"], stream=self.compute)
        bwd(d["q"], d["k"], d["v"], d["o"], d["do"], d["lse"], d["delta"], self.causal,
            dq=d["dq"], dk=d["dk"], dv=d["dv"], dq_accum=d["acc"], accum_zeroed=True,
            stream=self.compute)
        d["computed"].record(self.compute)
        self.down.wait_event(d["computed"])
        with torch.cuda.stream(self.down):
            for name, dst in d["h_out"].items():
                dst.copy_(d[name], non_blocking=True)
            d["read_back"].record(self.down)
        d["used"] = True
        return d["h_out"]

    def wait(self):
        for st in (self.up, self.compute, self.down):
            st.synchronize()


class DecodeHostRunner:
    """Split-KV decoding for host-resident tensors through pinned buffers.

    ``run(q, k, v)`` copies the CPU inputs to the device, runs ``decode`` and
    copies O and LSE back into pinned host tensors (returned).  Device buffers
    and the workspace are allocated once and reused.
    """

    def __init__(self, B, Lq, Lk, H, Hkv, D, dtype=torch.bfloat16, causal=False, device="cuda"):
        self.causal = causal
        dev = torch.device(device)
        self.q = torch.empty(B, Lq, H, D, dtype=dtype, device=dev)
        self.k = torch.empty(B, Lk, Hkv, D, dtype=dtype, device=dev)
        self.v = torch.empty_like(self.k)
        self.o = torch.empty_like(self.q)
        self.lse = torch.empty(B, H, Lq, dtype=torch.float32, device=dev)
        self.ws = alloc_decode_workspace(B, Lq, Lk, H, Hkv, D, dev)
        pin = dict(pin_memory=True)
        self.h_out = {"o": torch.empty(self.o.shape, dtype=dtype, **pin),
                      "lse": torch.empty(self.lse.shape, dtype=torch.float32, **pin)}

    def h2d_bytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in (self.q, self.k, self.v))

    def d2h_bytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in self.h_out.values())

    def run(self, q, k, v, stream=None):
        for dst, src in ((self.q, q), (self.k, k), (self.v, v)):
            dst.copy_(src, non_blocking=True)
        decode(self.q, self.k, self.v, self.causal, out=self.o, lse=self.lse, workspace=self.ws,
               stream=stream)
        self.h_out["o"].copy_(self.o, non_blocking=True)
        self.h_out["lse"].copy_(self.lse, non_blocking=True)
        return self.h_out


class Fp8HostRunner:
    """FP8 forward for host-resident E4M3 codes through pinned buffers:
    ``run(q8, k8, v8, q_scale, k_scale, v_scale)`` copies the codes in, runs
    ``fwd_fp8`` and copies O and LSE back into pinned host tensors."""

    def __init__(self, B, Lq, Lk, H, Hkv, D=128, out_dtype=torch.bfloat16, causal=False,
                 device="cuda"):
        self.causal = causal
        dev = torch.device(device)
        self.q8 = torch.empty(B, Lq, H, D, dtype=torch.uint8, device=dev)
        self.k8 = torch.empty(B, Lk, Hkv, D, dtype=torch.uint8, device=dev)
        self.v8 = torch.empty_like(self.k8)
        self.o = torch.empty(B, Lq, H, D, dtype=out_dtype, device=dev)
        self.lse = torch.empty(B, H, Lq, dtype=torch.float32, device=dev)
        pin = dict(pin_memory=True)
        self.h_out = {"o": torch.empty(self.o.shape, dtype=out_dtype, **pin),
                      "lse": torch.empty(self.lse.shape, dtype=torch.float32, **pin)}

    def h2d_bytes(self) -> int:
        return sum(t.numel() for t in (self.q8, self.k8, self.v8))

    def d2h_bytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in self.h_out.values())

    def run(self, q8, k8, v8, q_scale, k_scale, v_scale, stream=None):
        for dst, src in ((self.q8, q8), (self.k8, k8), (self.v8, v8)):
            dst.copy_(src, non_blocking=True)
        fwd_fp8(self.q8, self.k8, self.v8, q_scale, k_scale, v_scale, self.causal,
                out_dtype=self.o.dtype, out=self.o, lse=self.lse, stream=stream)
        self.h_out["o"].copy_(self.o, non_blocking=True)
        self.h_out["lse"].copy_(self.lse, non_blocking=True)
        return self.h_out
