"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle runs.

This module holds no attention arithmetic: it only draws iid N(0, 1) values
with a seeded CPU ``torch.Generator`` and rounds them to the storage dtype, so
the CUDA path and the CPU oracle see the same bytes.

Recipe (the pages benchmark on random tensors of the attention shapes, with no
dataset): Q [B, L, H, D], then K and V [B, L, Hkv, D], then dO [B, L, H, D],
drawn in that order from one generator seeded with ``seed``, in float32, then
cast with round-to-nearest-even to fp16 or bf16.
"""

from __future__ import annotations

import torch

_DTYPES = {"fp16": torch.float16, "bf16": torch.bfloat16,
           "f16": torch.float16, torch.float16: torch.float16,
           torch.bfloat16: torch.bfloat16}


def storage_dtype(dt) -> torch.dtype:
    """Map 'fp16' / 'bf16' (or a torch dtype) to the torch storage dtype."""
    try:
        return _DTYPES[dt]
    except KeyError as e:
        raise ValueError(f"unsupported dtype {dt!r}: use fp16 or bf16") from e


def make_qkv(B: int, L: int, H: int, Hkv: int, D: int, dtype="fp16",
             seed: int = 0, with_do: bool = True):
    """Return (q, k, v, do) CPU tensors; do is None when ``with_do`` is False."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    dt = storage_dtype(dtype)
    q = torch.randn(B, L, H, D, generator=g, dtype=torch.float32).to(dt)
    k = torch.randn(B, L, Hkv, D, generator=g, dtype=torch.float32).to(dt)
    v = torch.randn(B, L, Hkv, D, generator=g, dtype=torch.float32).to(dt)
    do = None
    if with_do:
        do = torch.randn(B, L, H, D, generator=g, dtype=torch.float32).to(dt)
    return q, k, v, do


def make_qkv_kv(B: int, Lq: int, Lk: int, H: int, Hkv: int, D: int, dtype="fp16",
                seed: int = 0, with_do: bool = False):
    """Like ``make_qkv`` with Lq query positions and Lk key positions (same
    draw order: Q, K, V, then dO)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    dt = storage_dtype(dtype)
    q = torch.randn(B, Lq, H, D, generator=g, dtype=torch.float32).to(dt)
    k = torch.randn(B, Lk, Hkv, D, generator=g, dtype=torch.float32).to(dt)
    v = torch.randn(B, Lk, Hkv, D, generator=g, dtype=torch.float32).to(dt)
    do = None
    if with_do:
        do = torch.randn(B, Lq, H, D, generator=g, dtype=torch.float32).to(dt)
    return q, k, v, do


def make_qkv_fp8(B: int, Lq: int, Lk: int, H: int, Hkv: int, D: int, seed: int = 0):
    """E4M3 inputs with one fp32 scale per tensor: (q8, k8, v8, q_scale, k_scale,
    v_scale), the codes as uint8 CPU tensors.  Q, K, V are drawn as in
    ``make_qkv_kv``; each tensor's scale is its largest magnitude over 448 (the
    largest E4M3 value) and its codes are torch's round-to-nearest cast of
    x / scale to float8_e4m3fn."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    q = torch.randn(B, Lq, H, D, generator=g, dtype=torch.float32)
    k = torch.randn(B, Lk, Hkv, D, generator=g, dtype=torch.float32)
    v = torch.randn(B, Lk, Hkv, D, generator=g, dtype=torch.float32)
    out = []
    scales = []
    for x in (q, k, v):
        s = float(x.abs().max()) / 448.0 if x.numel() else 1.0
        s = s if s > 0 else 1.0
        out.append((x / s).to(torch.float8_e4m3fn).view(torch.uint8))
        scales.append(s)
    return out[0], out[1], out[2], scales[0], scales[1], scales[2]


def make_unit(L: int, D: int, dtype="fp16", seed: int = 0, group: int = 1):
    """One (batch, kv-head) unit with ``group`` query heads: shapes [1, L, group, D]
    for Q/dO and [1, L, 1, D] for K/V.  Used for small, fast cases."""
    return make_qkv(1, L, group, 1, D, dtype, seed)
