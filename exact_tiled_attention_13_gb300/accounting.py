"""Work and traffic accounting for the attention forward pass.

FLOPs: each head does two contractions, S = Q K^T (2 N^2 d) and O = P V (2 N^2 d_v),
so 2 N^2 (d + d_v) per head; a causal mask keeps half of the score matrix, so the
count is halved. The method stays quadratic in work; only the N x N intermediates
leave HBM ("Compilers and kernels", section "FlashAttention rewrites the algorithm
around IO": exactness and the remark that the arithmetic is still quadratic).

Algorithmic bytes (the traffic a kernel that reads every input once and writes every
output once must move): Q, K, V in bf16, O in its output dtype, LSE in fp32, and the
dense fp32 bias C when there is one. S and P count zero bytes: keeping them on chip
is the method. The materialised alternative writes S and reads it, writes P and reads
it ("AI Infra ch. 5", section 5.3 "FlashAttention", the L = 8192, d = 128 example).
"""
from __future__ import annotations

BF16 = 2
F32 = 4
MiB = 1 << 20
GiB = 1 << 30


def allowed_pairs(N: int, causal: bool, Nk: int | None = None) -> float:
    """(query, key) pairs that take part, per head. Without a mask Nq * Nk. With the causal
    mask (query i sees keys j <= i + Nk - Nq) the continuous count Nq Nk - Nq^2 / 2 when
    Nq <= Nk and Nk^2 / 2 otherwise; for Nq = Nk both give the usual N^2 / 2."""
    Nq, Nk = N, (N if Nk is None else Nk)
    if not causal:
        return float(Nq) * Nk
    if Nq <= Nk:
        return float(Nq) * Nk - 0.5 * float(Nq) * Nq
    return 0.5 * float(Nk) * Nk


def flops(BH: int, N: int, d: int, dv: int, causal: bool, Nk: int | None = None) -> float:
    """Algorithmic FLOPs of one forward pass: 2 (d + dv) per allowed (query, key) pair,
    i.e. 2 BH N^2 (d + dv), halved when causal, for N queries and N keys."""
    return 2.0 * BH * allowed_pairs(N, causal, Nk) * (d + dv)


def required_bytes(BH: int, N: int, d: int, dv: int, out_bytes: int, lse: bool = True,
                   dense_bias: bool = False, key_bias: bool = False, Nk: int | None = None) -> int:
    """Bytes of reading Q (N rows), K and V (Nk rows, default N) in bf16 and the bias (fp32
    C [N, Nk] or vector [Nk]) once and writing O and LSE once."""
    Nk = N if Nk is None else Nk
    b = BH * N * d * BF16 + BH * Nk * (d + dv) * BF16 + BH * N * dv * out_bytes
    if lse:
        b += BH * N * F32
    if dense_bias:
        b += BH * N * Nk * F32
    if key_bias:
        b += BH * Nk * F32
    return b


def bwd_flops(BH: int, N: int, d: int, dv: int, causal: bool, Nk: int | None = None) -> float:
    """Algorithmic FLOPs of one backward pass: the five products S = Q K^T (d), dP = dO V^T
    (dv), dV = P^T dO (dv), dK = dS^T Q (d) and dQ = dS K (d), 2 (3 d + 2 dv) per allowed
    pair. Recomputing S and dP a second time (the dQ kernel) is not counted."""
    return 2.0 * BH * allowed_pairs(N, causal, Nk) * (3 * d + 2 * dv)


def bwd_required_bytes(BH: int, N: int, d: int, dv: int, o_bytes: int, dense_bias: bool = False,
                       key_bias: bool = False, Nk: int | None = None) -> int:
    """Bytes of reading Q, K, V, dO (bf16), O (its dtype), LSE and the bias once and writing
    dQ, dK, dV (fp32) once."""
    Nk = N if Nk is None else Nk
    b = BH * N * d * BF16 + BH * Nk * (d + dv) * BF16 + BH * N * dv * (BF16 + o_bytes) + BH * N * F32
    b += BH * N * d * F32 + BH * Nk * (d + dv) * F32
    if dense_bias:
        b += BH * N * Nk * F32
    if key_bias:
        b += BH * Nk * F32
    return b


def materialized_intermediate_bytes(N: int, elem_bytes: int = F32) -> dict:
    """Sizes of S and P for one head and the traffic of writing and re-reading both."""
    s = N * N * elem_bytes
    return {"S": s, "P": s, "roundtrip": 4 * s}


def roofline_time_s(F: float, Q_bytes: float, peak_flops: float, peak_bytes_per_s: float) -> float:
    """Lower bound T >= max(F / P_max, Q / B_max) ("Compilers and kernels", roofline section)."""
    return max(F / peak_flops, Q_bytes / peak_bytes_per_s)
