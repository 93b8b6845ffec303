"""fp64 CPU oracle for scaled-dot-product attention, forward and backward.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this module: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code with the CUDA path and imports nothing from the package.

What it computes, written out from its plain definition (no tiling, no online
softmax, no fusion):

* Forward, per (batch b, query head h), following the core-formula section of
  "使用 TileLang 在 AMD GPU 上快速开发高性能 Flash Attention" (score
  computation, optional causal mask, softmax, output) and the PyTorch
  reference function described on the same page:

      S = Q_bh K_{b,hk}^T / sqrt(D)              (full L x L matrix)
      S[i, j] = -inf  for j > i + past_len        (causal; past_len = Lk - Lq)
      m_i = max_j S_ij
      P_ij = exp(S_ij - m_i) / sum_j exp(S_ij - m_i)   (two-pass softmax)
      O = P V_{b,hk}                              (explicit matmul)

  Queries may be fewer than keys (Lq <= Lk): following the causal-mask
  section of "TileLang性能分析报告：H100上FlashAttention吞吐量达1.2PFlops"
  (query index = row + past_len, key visible iff query index >= key index)
  with past_len = Lk - Lq, i.e. the queries are the last Lq positions of the
  Lk-long sequence (bottom-right aligned; top-left when Lq = Lk).

  with the grouped-query head map hk = h // (H // Hkv): the page's kernel
  reads the K/V head whose index is the query head divided by the group
  size, and its PyTorch reference repeats each K/V head group-size times
  along the head axis, which is the same map.

* LSE (the pages only name the tensor ``lse`` as an input of the backward
  kernel in "TileLang与机器学习训练：反向传播算子优化案例", section
  算子拆分与流水线设计): reading taken here is the natural-log log-sum-exp of
  the scaled, masked scores, LSE_i = m_i + ln sum_j exp(S_ij - m_i).

* Backward preprocess, same page and section: Delta_i = sum_d O_id dO_id.
  The printed snippet multiplies an O block by a transposed dO block and
  row-sums the product, which taken literally mixes different rows; the
  reading used here is the per-row dot product that the softmax gradient
  needs.

* Delta is formed from the stored forward output.  The pages' pipeline keeps
  the forward Output tensor in the input dtype (fp16 in the printed kernel)
  and the preprocess reads that tensor; ``o_round`` lets the backward round
  its own O to that storage format before forming Delta (None = exact O).

* The dV product: the main backward kernel of the same page (section
  算子拆分与流水线设计) casts the transposed probabilities to the input type
  before the dV GEMM (its qkT_cast operand), as the forward page casts P
  before the PV GEMM; ``p_round`` lets the backward round P to that storage
  format for the dV product only (None = exact P).

* The forward's cast: the forward kernel of "使用 TileLang 在 AMD GPU 上快速
  开发高性能 Flash Attention" (section K/V Tile 遍历与核心计算; the buffer is
  allocated in the input type in section Q Tile 处理与缓存初始化) copies the
  exponentiated score tile into that buffer before multiplying it with V,
  and divides by the row sum only when it writes the output.  ``unit_forward``'s ``p_round``
  rounds the unnormalised exp(S - m) (m the row max; the row sum stays
  unrounded) to that format before the PV product; the backward's
  ``fwd_p_round`` forms the O behind Delta the same way.  Reading taken
  here: the tile is cast relative to the final row max; an online kernel
  casts it relative to its running max, which is the same value for rows
  whose maximum lies in the first key tile they visit and otherwise only
  moves which way each value rounds.

* The dK and dQ products: the pages print no cast of dS, so the oracle
  has none; its dS is exact.  (A kernel that multiplies a 16-bit dS on the
  tensor cores differs from it by that rounding, which the tests bound.)

* Intermediates for error bounds: ``unit_probs`` returns the probability
  matrix of one unit together with exp(S - m) and its row sum, and
  ``unit_backward_parts`` the matrices of the backward definition (P, dP,
  Delta, dS, exact O).  They are the same arithmetic as ``unit_forward`` and
  ``unit_backward``, exposed so that tests can bound a kernel's roundings
  with exact values; nothing in them is specific to a kernel.

* Backward (the page elides every step after the dV product): the analytic
  gradient of O = softmax(S) V,

      dV = P^T dO,  dP = dO V^T,  dS = P o (dP - Delta 1^T),
      dQ = dS K / sqrt(D),  dK = dS^T Q / sqrt(D),

  with dK and dV of a KV head summed over the query heads of its group (what
  differentiating through the head repeat gives).

* FP8 forward (page "TileLang性能分析报告：H100上FlashAttention吞吐量达1.2PFlops",
  section 生产环境部署建议, item 1, which names FP8 mixed precision and an FP8
  example and gives nothing more): reading taken here is attention over
  inputs given as 8-bit E4M3 codes with one fp32 scale per tensor, i.e. the
  forward above applied to decode(Q8) * q_scale, decode(K8) * k_scale,
  decode(V8) * v_scale.  decode follows the E4M3 format of the OCP 8-bit
  floating point specification (the variant without infinities): sign in
  bit 7, a 4-bit exponent with bias 7 in bits 6-3, a 3-bit mantissa in bits
  2-0; exponent 0 holds the subnormals m/8 * 2^-6; exponent 15 with mantissa
  7 is NaN.  The result is the exact attention of the dequantised inputs;
  a kernel that rounds P to E4M3 before the PV product differs from it by
  that rounding, for which the tests carry an error bound.

All arithmetic is numpy float64; matmul and exp are library primitives.  For
very long sequences the per-unit functions may process query rows in panels:
each row's softmax still sees all of its keys, so the result is the same
computation, only with the row loop split.
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "kv_head",
    "unit_scores",
    "unit_forward",
    "unit_backward",
    "forward",
    "backward",
    "bwd_preprocess",
    "storage_round",
    "unit_probs",
    "unit_backward_parts",
    "e4m3_decode",
    "forward_fp8",
]


def kv_head(h: int, H: int, Hkv: int) -> int:
    """K/V head that query head ``h`` reads (grouped-query map h -> h // groups)."""
    if H % Hkv != 0:
        raise ValueError(f"H={H} is not a multiple of Hkv={Hkv}")
    return h // (H // Hkv)


def storage_round(x: np.ndarray, fmt) -> np.ndarray:
    """Round float64 values to a 16-bit storage format and back.

    fmt None: unchanged.  Otherwise the value is rounded to binary32 first and
    then to the 16-bit format with round-to-nearest-even -- the two steps a
    kernel takes when it stores an fp32 result: "fp16" is IEEE binary16
    (numpy's cast), "bf16" is bfloat16, the upper 16 bits of a binary32.
    """
    x = np.asarray(x, dtype=np.float64)
    if fmt is None:
        return x
    if fmt == "fp16":
        return x.astype(np.float32).astype(np.float16).astype(np.float64)
    if fmt == "bf16":
        b = x.astype(np.float32).view(np.uint32).astype(np.uint64)
        b = (b + 0x7FFF + ((b >> 16) & 1)) & 0xFFFF0000
        return b.astype(np.uint32).view(np.float32).astype(np.float64)
    raise ValueError(f"unknown storage format {fmt!r}")


def _as64(x) -> np.ndarray:
    a = np.asarray(x, dtype=np.float64)
    return a


def unit_scores(q_bh: np.ndarray, k_bh: np.ndarray, causal: bool,
                row0: int = 0, past: int = 0) -> np.ndarray:
    """Scaled, masked score rows S[row0:row0+n, :] for one (b, h).

    q_bh: [n, D] query rows row0..row0+n-1; k_bh: [Lk, D] all keys.
    Causal: key j is visible to query i iff j <= i + past.
    """
    n, D = q_bh.shape
    Lk = k_bh.shape[0]
    S = (q_bh @ k_bh.T) / np.sqrt(D)
    if causal:
        i = np.arange(row0, row0 + n)[:, None]
        j = np.arange(Lk)[None, :]
        S = np.where(j > i + past, -np.inf, S)
    return S


def _softmax_rows(S: np.ndarray):
    """Two-pass row softmax: returns P, row max m, row sum of exp(S - m)."""
    m = S.max(axis=1, keepdims=True)
    E = np.exp(S - m)
    s = E.sum(axis=1, keepdims=True)
    return E / s, m[:, 0], s[:, 0]


def _output(S, P, m, s, v_bh, p_round):
    """O = P V, or with the unnormalised tile cast first: cast(exp(S - m)) V / s."""
    if p_round is None:
        return P @ v_bh
    return (storage_round(np.exp(S - m[:, None]), p_round) @ v_bh) / s[:, None]


def unit_forward(q_bh, k_bh, v_bh, causal: bool, rows=None, panel: int = 4096, p_round=None):
    """O and LSE rows of one (b, h).

    q_bh [Lq, D], k_bh / v_bh [Lk, D] (already the K/V head this query head
    reads), Lq <= Lk under causal masking.  ``rows`` (optional int array)
    restricts the output to those query rows; the keys are always all Lk.
    ``p_round`` (None, "fp16", "bf16"): the format exp(S - m) is cast to
    before the PV product, O = cast(exp(S - m)) V / sum_j exp(S_ij - m_i).
    Returns (O [n, D], LSE [n]).
    """
    q_bh, k_bh, v_bh = _as64(q_bh), _as64(k_bh), _as64(v_bh)
    Lq, Lk = q_bh.shape[0], k_bh.shape[0]
    past = Lk - Lq
    rows = np.arange(Lq) if rows is None else np.asarray(rows)
    outs_o, outs_l = [], []
    for p0 in range(0, len(rows), panel):
        r = rows[p0:p0 + panel]
        S = (q_bh[r] @ k_bh.T) / np.sqrt(q_bh.shape[1])
        if causal:
            S = np.where(np.arange(Lk)[None, :] > r[:, None] + past, -np.inf, S)
        P, m, s = _softmax_rows(S)
        outs_o.append(_output(S, P, m, s, v_bh, p_round))
        outs_l.append(m + np.log(s))
    if not outs_o:
        return np.zeros((0, q_bh.shape[1])), np.zeros((0,))
    return np.concatenate(outs_o), np.concatenate(outs_l)


def unit_backward(q_bh, k_bh, v_bh, do_bh, causal: bool, panel: int = 4096, o_round=None,
                  p_round=None, fwd_p_round=None):
    """Gradients of one (b, h) pair against its K/V head.

    q_bh, do_bh [Lq, D]; k_bh, v_bh [Lk, D] (Lq <= Lk under causal masking).
    Returns (dQ [Lq, D], dK [Lk, D], dV [Lk, D], Delta [Lq], O [Lq, D], LSE [Lq]).
    The oracle recomputes its own O and Delta; nothing comes from a kernel.
    Formats (None, "fp16", "bf16"): ``o_round`` is the storage format of the
    O that Delta is formed from and ``fwd_p_round`` the forward's cast of
    exp(S - m) that made that O; ``p_round`` the format P is cast to for the
    dV product.  The returned O is the exact one.
    """
    q_bh, k_bh, v_bh, do_bh = (_as64(x) for x in (q_bh, k_bh, v_bh, do_bh))
    Lq, D = q_bh.shape
    Lk = k_bh.shape[0]
    past = Lk - Lq
    inv = 1.0 / np.sqrt(D)
    dq = np.zeros((Lq, D))
    dk = np.zeros((Lk, D))
    dv = np.zeros((Lk, D))
    o = np.zeros((Lq, D))
    lse = np.zeros((Lq,))
    delta = np.zeros((Lq,))
    for r0 in range(0, Lq, panel):
        r = np.arange(r0, min(Lq, r0 + panel))
        S = (q_bh[r] @ k_bh.T) * inv
        if causal:
            S = np.where(np.arange(Lk)[None, :] > r[:, None] + past, -np.inf, S)
        P, m, s = _softmax_rows(S)
        O = P @ v_bh
        o[r] = O
        lse[r] = m + np.log(s)
        dO = do_bh[r]
        Os = storage_round(_output(S, P, m, s, v_bh, fwd_p_round), o_round)  # stored O
        dl = (Os * dO).sum(axis=1)              # Delta_i = sum_d O_id dO_id
        delta[r] = dl
        dv += storage_round(P, p_round).T @ dO  # dV = P^T dO (P cast for the product)
        dP = dO @ v_bh.T                        # dP = dO V^T
        dS = P * (dP - dl[:, None])             # dS = P o (dP - Delta)
        dq[r] = (dS @ k_bh) * inv               # dQ = dS K / sqrt(D)
        dk += (dS.T @ q_bh[r]) * inv            # dK = dS^T Q / sqrt(D)
    return dq, dk, dv, delta, o, lse


def unit_probs(q_bh, k_bh, causal: bool):
    """Softmax parts of one (b, h): P [Lq, Lk] (rows sum to 1), E = exp(S - m)
    with m the row max (so every row's largest entry is 1), and l [Lq], the
    row sum of E (P = E / l).  Lq <= Lk under causal masking, bottom-right
    aligned as in ``unit_forward``."""
    q_bh, k_bh = _as64(q_bh), _as64(k_bh)
    S = unit_scores(q_bh, k_bh, causal, 0, k_bh.shape[0] - q_bh.shape[0])
    m = S.max(axis=1, keepdims=True)
    E = np.exp(S - m)
    l = E.sum(axis=1)
    return E / l[:, None], E, l


def unit_backward_parts(q_bh, k_bh, v_bh, do_bh, causal: bool):
    """The matrices of the backward definition for one (b, h), all exact:
    returns a dict with P [Lq, Lk], dP = dO V^T, Delta [Lq] (from the exact
    O), dS = P o (dP - Delta 1^T) and O = P V.  dQ = dS K / sqrt(D) and
    dK = dS^T Q / sqrt(D) follow from them as in ``unit_backward``."""
    q_bh, k_bh, v_bh, do_bh = (_as64(x) for x in (q_bh, k_bh, v_bh, do_bh))
    P, _, _ = unit_probs(q_bh, k_bh, causal)
    O = P @ v_bh
    dP = do_bh @ v_bh.T
    delta = (O * do_bh).sum(axis=1)
    dS = P * (dP - delta[:, None])
    return {"P": P, "dP": dP, "Delta": delta, "dS": dS, "O": O}


def forward(q, k, v, causal: bool, p_round=None):
    """Full forward over BSHD tensors.

    q [B, Lq, H, D]; k, v [B, Lk, Hkv, D].  Returns O [B, Lq, H, D] and
    LSE [B, H, Lq] (float64); ``p_round`` as in ``unit_forward``.
    """
    q, k, v = _as64(q), _as64(k), _as64(v)
    B, L, H, D = q.shape
    Hkv = k.shape[2]
    o = np.zeros((B, L, H, D))
    lse = np.zeros((B, H, L))
    for b in range(B):
        for h in range(H):
            hk = kv_head(h, H, Hkv)
            o[b, :, h, :], lse[b, h, :] = unit_forward(
                q[b, :, h, :], k[b, :, hk, :], v[b, :, hk, :], causal, p_round=p_round)
    return o, lse


def bwd_preprocess(o, do):
    """Delta[b, h, i] = sum_d O[b, i, h, d] * dO[b, i, h, d], as [B, H, L]."""
    o, do = _as64(o), _as64(do)
    return np.einsum("blhd,blhd->bhl", o, do)


def backward(q, k, v, do, causal: bool, o_round=None, p_round=None, fwd_p_round=None):
    """Full backward over BSHD tensors.

    q, do [B, Lq, H, D]; k, v [B, Lk, Hkv, D].  Returns dQ [B, Lq, H, D],
    dK [B, Lk, Hkv, D], dV [B, Lk, Hkv, D], Delta [B, H, Lq] (from the
    oracle's own O).  The format options are those of ``unit_backward``.
    """
    q, k, v, do = _as64(q), _as64(k), _as64(v), _as64(do)
    B, L, H, D = q.shape
    Lk, Hkv = k.shape[1], k.shape[2]
    dq = np.zeros((B, L, H, D))
    dk = np.zeros((B, Lk, Hkv, D))
    dv = np.zeros((B, Lk, Hkv, D))
    delta = np.zeros((B, H, L))
    for b in range(B):
        for h in range(H):
            hk = kv_head(h, H, Hkv)
            gq, gk, gv, dl, _, _ = unit_backward(
                q[b, :, h, :], k[b, :, hk, :], v[b, :, hk, :], do[b, :, h, :], causal,
                o_round=o_round, p_round=p_round, fwd_p_round=fwd_p_round)
            dq[b, :, h, :] = gq
            dk[b, :, hk, :] += gk                 # group heads sum into their KV head
            dv[b, :, hk, :] += gv
            delta[b, h, :] = dl
    return dq, dk, dv, delta


def e4m3_decode(codes) -> np.ndarray:
    """float64 value of each E4M3 code (uint8 array): (-1)^s * 2^(e-7) * (1 + m/8)
    for exponent field e in 1..15, (-1)^s * 2^-6 * m/8 for e = 0, NaN for the
    all-ones exponent and mantissa."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    normal = sign * np.ldexp(1.0 + m / 8.0, (e - 7).astype(np.int64))
    subnormal = sign * np.ldexp(m / 8.0, -6)
    val = np.where(e == 0, subnormal, normal)
    return np.where((e == 15) & ((c & 0x7) == 7), np.nan, val)


def forward_fp8(q8, k8, v8, q_scale: float, k_scale: float, v_scale: float, causal: bool):
    """Forward on per-tensor-scaled E4M3 inputs: ``forward`` of the decoded
    values times their scales.  q8 [B, Lq, H, D], k8, v8 [B, Lk, Hkv, D] as
    uint8 codes.  Returns O [B, Lq, H, D], LSE [B, H, Lq] (float64)."""
    return forward(e4m3_decode(q8) * float(q_scale), e4m3_decode(k8) * float(k_scale),
                   e4m3_decode(v8) * float(v_scale), causal)
