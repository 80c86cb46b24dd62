"""Seeded synthetic inputs for the attention forward path.

This module only makes input bytes. It holds none of the attention arithmetic, so
both the CPU oracle and the CUDA path can be fed from it without sharing any of
the computation they are compared on.

Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014) used as a counter-based stream, u = (x >> 11 + 1) * 2^-53
in (0, 1], and the Box-Muller transform (Box and Muller 1958) for normal deviates.
Every tensor gets its own stream: seed = base + 100 * workload_id + tensor_id
(Q=0, K=1, V=2, C=3, key-padding mask=4).

Values follow the synthetic workloads of the attention pages: Q, K, V i.i.d. N(0,1)
rounded to bf16 (round to nearest, ties to even), optionally multiplied by a power
of two before rounding (exact in bf16), and for the dense-bias workload an fp32
N(0,1) bias with a random key-padding mask (-inf with probability p per key).
"""
from __future__ import annotations

import concurrent.futures
import dataclasses
import math
import os

import numpy as np

BASE_SEED = 20261202
TENSOR_ID = {"Q": 0, "K": 1, "V": 2, "C": 3, "mask": 4, "ckey": 5, "dO": 6}

MODE_NONE, MODE_CAUSAL, MODE_DENSE, MODE_KEY = 0, 1, 2, 4
MODE_SHARED = 8  # with MODE_DENSE: one [Nq, Nk] bias for every head (the inputs are the same)
MODE_NAMES = {MODE_NONE: "none", MODE_CAUSAL: "causal", MODE_DENSE: "dense_bias",
              MODE_KEY: "key_bias", MODE_CAUSAL | MODE_DENSE: "causal_dense_bias",
              MODE_CAUSAL | MODE_KEY: "causal_key_bias"}

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 21


def splitmix64(seed: int, start: int, count: int) -> np.ndarray:
    """Outputs start..start+count-1 of the SplitMix64 stream for `seed` (uint64)."""
    with np.errstate(over="ignore"):
        idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + idx * _GAMMA
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def uniform01(seed: int, start: int, count: int) -> np.ndarray:
    """Uniform doubles in (0, 1] from the top 53 bits of each SplitMix64 output."""
    x = splitmix64(seed, start, count) >> np.uint64(11)
    return (x.astype(np.float64) + 1.0) * (2.0 ** -53)


def _normal_chunk(seed: int, out: np.ndarray, count: int, p0: int, pn: int) -> None:
    u = uniform01(seed, 2 * p0, 2 * pn)
    r = np.sqrt(-2.0 * np.log(u[0::2]))
    th = (2.0 * math.pi) * u[1::2]
    z = np.empty(2 * pn, dtype=np.float64)
    z[0::2] = r * np.cos(th)
    z[1::2] = r * np.sin(th)
    lo = 2 * p0
    hi = min(count, lo + 2 * pn)
    out[lo:hi] = z[: hi - lo].astype(np.float32)


def normal_f32(seed: int, count: int) -> np.ndarray:
    """`count` standard normal deviates (Box-Muller on consecutive uniform pairs), as fp32.

    Element k depends only on (seed, k): chunks are generated independently (in
    parallel threads for large counts) and the result does not depend on chunking.
    """
    out = np.empty(count, dtype=np.float32)
    pairs = (count + 1) // 2
    starts = list(range(0, pairs, _CHUNK))
    jobs = [(p0, min(_CHUNK, pairs - p0)) for p0 in starts]
    if len(jobs) <= 1:
        for p0, pn in jobs:
            _normal_chunk(seed, out, count, p0, pn)
        return out
    with concurrent.futures.ThreadPoolExecutor(max_workers=min(len(jobs), _threads())) as ex:
        list(ex.map(lambda j: _normal_chunk(seed, out, count, j[0], j[1]), jobs))
    return out


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest, ties to even. Inputs are finite."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> the fp32 values they encode (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic attention workload: shapes, mask mode, output dtype and value recipe."""

    name: str
    B: int
    H: int
    N: int
    d: int
    dv: int
    mode: int
    out_dtype: str  # "bf16" or "f32"
    qk_mult: float = 1.0
    p_mask: float = 0.0
    Nk: int = 0             # keys per head; 0: as many as queries (N)
    split_kv: bool = False  # launched as a split forward pass (key ranges + merge)
    backward: bool = False  # the step is the backward pass (dQ, dK, dV for a seeded dO)

    @property
    def BH(self) -> int:
        return self.B * self.H

    @property
    def Nkv(self) -> int:
        return self.Nk or self.N

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


# The five synthetic workloads of the attention forward benchmark.
WORKLOADS = {
    1: Workload("single_head_n256_d64_nomask", 1, 1, 256, 64, 64, MODE_NONE, "f32"),
    2: Workload("b4h16_n2048_d128_causal", 4, 16, 2048, 128, 128, MODE_CAUSAL, "bf16"),
    3: Workload("b2h32_n8192_d128_causal", 2, 32, 8192, 128, 128, MODE_CAUSAL, "bf16"),
    4: Workload("b1h8_n4096_d64_dv128_dense_bias_keypad", 1, 8, 4096, 64, 128, MODE_DENSE, "f32",
                p_mask=0.3),
    5: Workload("b1h16_n16384_d128_nomask_qk_x4", 1, 16, 16384, 128, 128, MODE_NONE, "f32",
                qk_mult=4.0),
    # Workload 4's key padding as a per-key vector (bias c_j ~ N(0,1), -inf with p = 0.3)
    # instead of a dense N x N array.
    6: Workload("b1h8_n4096_d64_dv128_key_bias_keypad", 1, 8, 4096, 64, 128, MODE_KEY, "f32",
                p_mask=0.3),
    # A 128-query block at the end of a 65536-key sequence (causal mask aligned at the
    # last key), 8 heads: one query tile per head, so the keys are split into ranges.
    7: Workload("b1h8_nq128_nk65536_d128_causal_splitkv", 1, 8, 128, 128, 128, MODE_CAUSAL,
                "bf16", Nk=65536, split_kv=True),
    # The backward pass of workload 2 (O bf16 from the forward pass, dO ~ N(0,1) in bf16).
    8: Workload("b4h16_n2048_d128_causal_bwd", 4, 16, 2048, 128, 128, MODE_CAUSAL, "bf16",
                backward=True),
}


def seed_for(workload_id: int, tensor: str, base: int = BASE_SEED) -> int:
    return base + 100 * workload_id + TENSOR_ID[tensor]


def bf16_tensor(seed: int, shape, mult: float = 1.0) -> np.ndarray:
    """bf16 bit patterns of shape `shape`: N(0,1) in fp32, times `mult`, rounded to bf16."""
    n = int(np.prod(shape))
    x = normal_f32(seed, n)
    if mult != 1.0:
        x = (x.astype(np.float64) * mult).astype(np.float32)
    return bf16_bits(x).reshape(shape)


def dense_bias(seed_c: int, seed_mask: int, BH: int, N: int, p_mask: float) -> np.ndarray:
    """fp32 additive bias C[BH, N, N] ~ N(0,1) with a key-padding mask folded in.

    Each key j of head bh is forbidden (C[bh, :, j] = -inf) with probability p_mask,
    one Bernoulli draw per (bh, j). If a head ends up with every key forbidden, key 0
    is allowed again (its bias value restored) so that every row keeps an allowed key.
    """
    C = normal_f32(seed_c, BH * N * N).reshape(BH, N, N)
    if p_mask > 0.0:
        u = uniform01(seed_mask, 0, BH * N).reshape(BH, N)
        masked = u <= p_mask
        for bh in range(BH):
            if masked[bh].all():
                masked[bh, 0] = False
        C[np.broadcast_to(masked[:, None, :], C.shape)] = -np.inf
    return C


def key_bias(seed_c: int, seed_mask: int, BH: int, Nk: int, p_mask: float, std: float = 1.0) -> np.ndarray:
    """fp32 per-key bias c[BH, Nk] ~ N(0, std^2) with key padding: each key is forbidden
    (-inf) with probability p_mask; a head that lost every key gets key 0 back."""
    c = normal_f32(seed_c, BH * Nk).reshape(BH, Nk)
    if std != 1.0:
        c = (c.astype(np.float64) * std).astype(np.float32)
    if p_mask > 0.0:
        masked = uniform01(seed_mask, 0, BH * Nk).reshape(BH, Nk) <= p_mask
        for bh in range(BH):
            if masked[bh].all():
                masked[bh, 0] = False
        c[masked] = -np.inf
    return c


def make_inputs(w: Workload, workload_id: int, base: int = BASE_SEED) -> dict:
    """Seeded inputs of workload `w`: Q, K, V as bf16 bit arrays, C fp32 or None."""
    BH, N, Nk = w.BH, w.N, w.Nkv
    Q = bf16_tensor(seed_for(workload_id, "Q", base), (BH, N, w.d), w.qk_mult)
    K = bf16_tensor(seed_for(workload_id, "K", base), (BH, Nk, w.d), w.qk_mult)
    V = bf16_tensor(seed_for(workload_id, "V", base), (BH, Nk, w.dv))
    C = ckey = None
    if w.mode & MODE_DENSE:
        if Nk != N:
            raise ValueError("the dense-bias recipe is square (Nq = Nk)")
        C = dense_bias(seed_for(workload_id, "C", base), seed_for(workload_id, "mask", base),
                       BH, N, w.p_mask)
    if w.mode & MODE_KEY:
        ckey = key_bias(seed_for(workload_id, "ckey", base), seed_for(workload_id, "mask", base),
                        BH, Nk, w.p_mask)
    out = {"Q": Q, "K": K, "V": V, "C": C, "ckey": ckey, "scale": w.scale, "mode": w.mode}
    if w.backward:
        out["dO"] = bf16_tensor(seed_for(workload_id, "dO", base), (BH, N, w.dv))
    return out


def random_case(seed: int, BH: int, N: int, d: int, dv: int, mode: int, qk_mult: float = 1.0,
                p_mask: float = 0.0) -> dict:
    """A seeded case of arbitrary shape (for parity tests at small and ragged sizes)."""
    w = Workload("case", 1, BH, N, d, dv, mode, "f32", qk_mult, p_mask)
    return make_inputs(w, 0, base=seed)


def random_case_ex(seed: int, BH: int, Nq: int, Nk: int, d: int, dv: int, mode: int,
                   qk_mult: float = 1.0, p_mask: float = 0.0) -> dict:
    """A seeded case with Nq queries and Nk keys; C is [BH, Nq, Nk], ckey [BH, Nk]."""
    Q = bf16_tensor(seed + TENSOR_ID["Q"], (BH, Nq, d), qk_mult)
    K = bf16_tensor(seed + TENSOR_ID["K"], (BH, Nk, d), qk_mult)
    V = bf16_tensor(seed + TENSOR_ID["V"], (BH, Nk, dv))
    C = ckey = None
    if mode & MODE_DENSE:
        C = normal_f32(seed + TENSOR_ID["C"], BH * Nq * Nk).reshape(BH, Nq, Nk)
        if p_mask > 0.0:
            masked = uniform01(seed + TENSOR_ID["mask"], 0, BH * Nk).reshape(BH, Nk) <= p_mask
            masked[:, 0] = False
            C[np.broadcast_to(masked[:, None, :], C.shape)] = -np.inf
    if mode & MODE_KEY:
        ckey = key_bias(seed + TENSOR_ID["ckey"], seed + TENSOR_ID["mask"], BH, Nk, p_mask)
    return {"Q": Q, "K": K, "V": V, "C": C, "ckey": ckey, "scale": 1.0 / math.sqrt(d),
            "mode": mode}
