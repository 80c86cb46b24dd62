"""CPU fp64 oracle for exact attention (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may
import this package. The CUDA product path never does. The arithmetic lives in
``attn_oracle.c`` (plain C, fp64, one query row at a time with the whole row of S
and P materialised), compiled here with gcc on first use; this module only
marshals numpy arrays.

Definition followed: "Compilers and kernels", section "FlashAttention rewrites the
algorithm around IO":
S = Q K^T * scale + C, m_i = max_j S_ij, l_i = sum_j exp(S_ij - m_i),
P = exp(S - m) / l, O = P V; LSE_i = m_i + ln l_i is reported beside O.
Second, test-only path: the blockwise online recurrence of the same section and
the (m, l, u) form of "AI Infra ch. 5", section 5.3, Example 5-6. Backward pass: the
gradients dQ, dK, dV of that definition by the chain rule, recomputing S and P from
the kept row statistics (the same section's remark on the backward pass).

Every function is pinned by the ``-m "not gpu"`` tests in tests/test_oracle_pins.py
(invariants, closed forms, special cases, the pages' worked numbers and brute force).
"""
from __future__ import annotations

import ctypes
import hashlib
import os
import subprocess
import threading

import numpy as np

MODE_NONE, MODE_CAUSAL, MODE_DENSE, MODE_KEY = 0, 1, 2, 4

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_lock = threading.Lock()
_default = None


def source_text() -> str:
    with open(_SRC, "r") as f:
        return f.read()


def build(src_text: str | None = None) -> str:
    """Compile the oracle C source (the committed file unless `src_text` is given) into a
    shared library cached by source hash; return its path."""
    text = source_text() if src_text is None else src_text
    digest = hashlib.sha256(text.encode()).hexdigest()[:16]
    os.makedirs(_BUILD_DIR, exist_ok=True)
    so = os.path.join(_BUILD_DIR, f"liboracle_{digest}.so")
    if not os.path.exists(so):
        tmp_c = os.path.join(_BUILD_DIR, f"src_{digest}_{os.getpid()}.c")
        with open(tmp_c, "w") as f:
            f.write(text)
        tmp = so + f".tmp{os.getpid()}"
        # -ffp-contract=off keeps every multiply and add a separately rounded fp64 op.
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
               tmp_c, "-o", tmp, "-lm"]
        try:
            subprocess.run(cmd, check=True)
            os.replace(tmp, so)
        finally:
            if os.path.exists(tmp_c):
                os.remove(tmp_c)
    return so


def _bind(path: str):
    lib = ctypes.CDLL(path)
    p = ctypes.c_void_p
    i64 = ctypes.c_int64
    dbl = ctypes.c_double
    lib.oracle_attention.argtypes = [p, p, p, ctypes.c_int, p, i64, i64, i64, i64, dbl, p, i64,
                                     p, p, ctypes.c_int]
    lib.oracle_attention.restype = ctypes.c_int
    lib.oracle_attention_ex.argtypes = [p, p, p, ctypes.c_int, p, p, i64, i64, i64, i64, i64, dbl,
                                        p, i64, p, p, ctypes.c_int]
    lib.oracle_attention_ex.restype = ctypes.c_int
    lib.oracle_attention_head.argtypes = [p, p, p, ctypes.c_int, p, i64, i64, i64, dbl, p, p,
                                          p, p]
    lib.oracle_attention_head.restype = ctypes.c_int
    lib.oracle_online_blocks.argtypes = [p, p, i64, i64, p, ctypes.c_int, p, p, p, p]
    lib.oracle_online_blocks.restype = ctypes.c_int
    lib.oracle_online_step.argtypes = [p, p, p, i64, dbl, p]
    lib.oracle_online_step.restype = None
    lib.oracle_online_merge.argtypes = [dbl, dbl, p, dbl, dbl, p, i64, p, p, p]
    lib.oracle_online_merge.restype = None
    lib.oracle_attention_bwd.argtypes = [p, p, p, p, ctypes.c_int, p, p, i64, i64, i64, i64, i64,
                                         dbl, p, i64, p, i64, p, i64, p, p, p, ctypes.c_int]
    lib.oracle_attention_bwd.restype = ctypes.c_int
    return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _bits(a, shape_len):
    a = np.ascontiguousarray(a, dtype=np.uint16)
    if a.ndim != shape_len:
        raise ValueError(f"expected a {shape_len}-d bf16 bit array, got shape {a.shape}")
    return a


class Oracle:
    """numpy front end of one compiled copy of the oracle C source."""

    def __init__(self, src_text: str | None = None):
        self.lib = _bind(build(src_text))

    def attention(self, Q, K, V, mode, C, scale, rows=None, nthreads=0):
        """O (fp64 [nrows, dv]) and LSE (fp64 [nrows]) by the definition.

        Q, K: bf16 bit arrays [BH, N, d]; V: [BH, N, dv]; C: fp32 [BH, N, N] for DENSE.
        rows: optional flat row ids bh * N + i (int64); None evaluates every row, and the
        outputs are then shaped [BH, N, dv] and [BH, N].
        Returns (O, LSE, threads_used).
        """
        Q, K, V = _bits(Q, 3), _bits(K, 3), _bits(V, 3)
        BH, N, d = Q.shape
        dv = V.shape[2]
        if K.shape != (BH, N, d) or V.shape[:2] != (BH, N):
            raise ValueError("inconsistent Q/K/V shapes")
        Cc = None
        if mode == MODE_DENSE:
            Cc = np.ascontiguousarray(C, dtype=np.float32)
            if Cc.shape != (BH, N, N):
                raise ValueError("C must be [BH, N, N]")
        rows_arr = None
        nrows = BH * N
        if rows is not None:
            rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
            nrows = rows_arr.size
        O = np.empty((nrows, dv), dtype=np.float64)
        LSE = np.empty(nrows, dtype=np.float64)
        used = self.lib.oracle_attention(_ptr(Q), _ptr(K), _ptr(V), int(mode), _ptr(Cc), BH, N, d,
                                         dv, float(scale), _ptr(rows_arr), nrows, _ptr(O),
                                         _ptr(LSE), int(nthreads))
        if used < 0:
            raise ValueError("oracle_attention rejected its arguments")
        if rows is None:
            O = O.reshape(BH, N, dv)
            LSE = LSE.reshape(BH, N)
        return O, LSE, used

    def attention_ex(self, Q, K, V, mode, C, ckey, scale, rows=None, nthreads=0):
        """Queries and keys of their own lengths; mode is a bit set of CAUSAL (key j >
        i + Nk - Nq forbidden), DENSE (C fp32 [BH, Nq, Nk]) and KEY (ckey fp32 [BH, Nk]).
        Q: bf16 bits [BH, Nq, d]; K: [BH, Nk, d]; V: [BH, Nk, dv]. Returns (O, LSE, threads)
        shaped [BH, Nq, dv] / [BH, Nq], or [nrows, dv] / [nrows] for a row subset."""
        Q, K, V = _bits(Q, 3), _bits(K, 3), _bits(V, 3)
        BH, Nq, d = Q.shape
        Nk, dv = K.shape[1], V.shape[2]
        if K.shape != (BH, Nk, d) or V.shape[:2] != (BH, Nk):
            raise ValueError("inconsistent Q/K/V shapes")
        Cc = kk = None
        if mode & MODE_DENSE:
            Cc = np.ascontiguousarray(C, dtype=np.float32)
            if Cc.shape != (BH, Nq, Nk):
                raise ValueError("C must be [BH, Nq, Nk]")
        if mode & MODE_KEY:
            kk = np.ascontiguousarray(ckey, dtype=np.float32)
            if kk.shape != (BH, Nk):
                raise ValueError("ckey must be [BH, Nk]")
        rows_arr = None
        nrows = BH * Nq
        if rows is not None:
            rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
            nrows = rows_arr.size
        O = np.empty((nrows, dv), dtype=np.float64)
        LSE = np.empty(nrows, dtype=np.float64)
        used = self.lib.oracle_attention_ex(_ptr(Q), _ptr(K), _ptr(V), int(mode), _ptr(Cc), _ptr(kk),
                                            BH, Nq, Nk, d, dv, float(scale), _ptr(rows_arr), nrows,
                                            _ptr(O), _ptr(LSE), int(nthreads))
        if used < 0:
            raise ValueError("oracle_attention_ex rejected its arguments")
        if rows is None:
            O = O.reshape(BH, Nq, dv)
            LSE = LSE.reshape(BH, Nq)
        return O, LSE, used

    def attention_bwd(self, Q, K, V, dO, mode, C, ckey, scale, heads=None, qrows=None,
                      krows=None, nthreads=0):
        """Gradients of O = softmax(scale Q K^T + C) V for the loss gradient dO (bf16 bits
        [BH, Nq, dv]): returns (dQ, dK, dV, threads), fp64, shaped [nheads, nq_sel, d],
        [nheads, nk_sel, d], [nheads, nk_sel, dv] for the selected heads, query rows (dQ)
        and keys (dK, dV); None selects all of them."""
        Q, K, V, dO = _bits(Q, 3), _bits(K, 3), _bits(V, 3), _bits(dO, 3)
        BH, Nq, d = Q.shape
        Nk, dv = K.shape[1], V.shape[2]
        if K.shape != (BH, Nk, d) or V.shape[:2] != (BH, Nk) or dO.shape != (BH, Nq, dv):
            raise ValueError("inconsistent Q/K/V/dO shapes")
        Cc = kk = None
        if mode & MODE_DENSE:
            Cc = np.ascontiguousarray(C, dtype=np.float32)
            if Cc.shape != (BH, Nq, Nk):
                raise ValueError("C must be [BH, Nq, Nk]")
        if mode & MODE_KEY:
            kk = np.ascontiguousarray(ckey, dtype=np.float32)
            if kk.shape != (BH, Nk):
                raise ValueError("ckey must be [BH, Nk]")

        def sel(a, n):
            return (None, n) if a is None else (np.ascontiguousarray(a, dtype=np.int64), len(a))

        h_arr, nh = sel(heads, BH)
        q_arr, nq = sel(qrows, Nq)
        k_arr, nk = sel(krows, Nk)
        dQ = np.empty((nh, nq, d))
        dK = np.empty((nh, nk, d))
        dV = np.empty((nh, nk, dv))
        used = self.lib.oracle_attention_bwd(_ptr(Q), _ptr(K), _ptr(V), _ptr(dO), int(mode),
                                             _ptr(Cc), _ptr(kk), BH, Nq, Nk, d, dv, float(scale),
                                             _ptr(h_arr), nh, _ptr(q_arr), nq, _ptr(k_arr), nk,
                                             _ptr(dQ), _ptr(dK), _ptr(dV), int(nthreads))
        if used < 0:
            raise ValueError("oracle_attention_bwd rejected its arguments")
        return dQ, dK, dV, used

    def attention_head(self, Q, K, V, mode, C, scale):
        """S, P (fp64 [N, N]), O ([N, dv]) and LSE ([N]) of one head, all materialised."""
        Q, K, V = _bits(Q, 2), _bits(K, 2), _bits(V, 2)
        N, d = Q.shape
        dv = V.shape[1]
        Cc = None
        if mode == MODE_DENSE:
            Cc = np.ascontiguousarray(C, dtype=np.float32).reshape(N, N)
        S = np.empty((N, N))
        P = np.empty((N, N))
        O = np.empty((N, dv))
        LSE = np.empty(N)
        rc = self.lib.oracle_attention_head(_ptr(Q), _ptr(K), _ptr(V), int(mode), _ptr(Cc), N, d,
                                            dv, float(scale), _ptr(S), _ptr(P), _ptr(O), _ptr(LSE))
        if rc != 0:
            raise ValueError("oracle_attention_head rejected its arguments")
        return S, P, O, LSE

    def online_blocks(self, s, v, blk, T, order=None):
        """Blockwise recurrence over one row: returns (O_i, m_T, l_T)."""
        s = np.ascontiguousarray(s, dtype=np.float64)
        v = np.ascontiguousarray(v, dtype=np.float64)
        if v.ndim == 1:
            v = np.ascontiguousarray(v[:, None])
        blk = np.ascontiguousarray(blk, dtype=np.int32)
        order_arr = None if order is None else np.ascontiguousarray(order, dtype=np.int32)
        n, dv = v.shape
        O = np.empty(dv)
        m = ctypes.c_double()
        l = ctypes.c_double()
        rc = self.lib.oracle_online_blocks(_ptr(s), _ptr(v), n, dv, _ptr(blk), int(T),
                                           _ptr(order_arr), _ptr(O), ctypes.byref(m),
                                           ctypes.byref(l))
        if rc != 0:
            raise ValueError("oracle_online_blocks: a block with no allowed key came first")
        return O, m.value, l.value

    def online_step(self, m, l, u, s, v):
        """One (m, l, u) update with a new element (score s, value vector v)."""
        u = np.array(u, dtype=np.float64, ndmin=1)
        v = np.ascontiguousarray(np.array(v, dtype=np.float64, ndmin=1))
        mm = ctypes.c_double(m)
        ll = ctypes.c_double(l)
        self.lib.oracle_online_step(ctypes.byref(mm), ctypes.byref(ll), _ptr(u), u.size, float(s),
                                    _ptr(v))
        return mm.value, ll.value, u

    def online_merge(self, state1, state2):
        """Merge two (m, l, u) partial states of disjoint key sets."""
        m1, l1, u1 = state1
        m2, l2, u2 = state2
        u1 = np.ascontiguousarray(np.array(u1, dtype=np.float64, ndmin=1))
        u2 = np.ascontiguousarray(np.array(u2, dtype=np.float64, ndmin=1))
        u = np.empty_like(u1)
        m = ctypes.c_double()
        l = ctypes.c_double()
        self.lib.oracle_online_merge(float(m1), float(l1), _ptr(u1), float(m2), float(l2),
                                     _ptr(u2), u1.size, ctypes.byref(m), ctypes.byref(l), _ptr(u))
        return m.value, l.value, u


def default() -> Oracle:
    """The oracle built from the committed source."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle()
        return _default


def attention(*args, **kwargs):
    return default().attention(*args, **kwargs)


def attention_ex(*args, **kwargs):
    return default().attention_ex(*args, **kwargs)


def attention_bwd(*args, **kwargs):
    return default().attention_bwd(*args, **kwargs)


def attention_head(*args, **kwargs):
    return default().attention_head(*args, **kwargs)


def online_blocks(*args, **kwargs):
    return default().online_blocks(*args, **kwargs)


def online_step(*args, **kwargs):
    return default().online_step(*args, **kwargs)


def online_merge(*args, **kwargs):
    return default().online_merge(*args, **kwargs)
