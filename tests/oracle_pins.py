"""Pins for the CPU oracle: facts fixed by the attention pages and by mathematics.

Each pin takes an ``oracle.Oracle`` and raises AssertionError when the oracle
breaks the fact it checks. tests/test_oracle_pins.py runs them on the committed
oracle; tests/test_oracle_mutants.py runs them on copies of the oracle source with
a planted mistake and requires that some pin fails for every mistake.

Sources of the facts:
  * "Compilers and kernels", section "FlashAttention rewrites the algorithm around
    IO": the definition of
    S, P, O, m, l; the assumption of at least one allowed key per row; the blockwise
    recurrence over blocks that partition the allowed keys and its exactness.
  * "AI Infra ch. 5 Operators and runtime", section 5.3, Example 5-6
    and Exercise 5-3 (the (m, l, u) update), and section 5.4 (two blocks holding 1
    and 3 cannot be merged without their statistics).
  * Closed forms and invariants of softmax attention (rows of P sum to 1, constant V,
    uniform weights, shift invariance, key permutation), and brute force in 50-digit
    arithmetic on tiny inputs.
"""
from __future__ import annotations

import itertools
import json
import math
import os

import numpy as np

import synth

NONE, CAUSAL, DENSE = synth.MODE_NONE, synth.MODE_CAUSAL, synth.MODE_DENSE
EPS = np.finfo(np.float64).eps
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _vals(bits):
    return synth.bf16_to_f32(bits).astype(np.float64)


def _case(seed, N, d, dv, mode, p_mask=0.0, qk_mult=1.0, BH=1):
    return synth.random_case(seed, BH, N, d, dv, mode, qk_mult, p_mask)


def _head(c, h=0):
    C = None if c["C"] is None else c["C"][h]
    return c["Q"][h], c["K"][h], c["V"][h], C


def _scores_numpy(Q, K, C, mode, scale):
    """S recomputed with a numpy matmul (used only where a pin needs a single score)."""
    S = scale * (_vals(Q) @ _vals(K).T)
    N = S.shape[0]
    if mode == CAUSAL:
        S = S + np.where(np.arange(N)[None, :] > np.arange(N)[:, None], -np.inf, 0.0)
    elif mode == DENSE:
        S = S + C.astype(np.float64)
    return S


def _set_partitions(items):
    """Every partition of the list `items` into non-empty blocks."""
    if not items:
        yield []
        return
    first, rest = items[0], items[1:]
    for part in _set_partitions(rest):
        for k in range(len(part)):
            yield part[:k] + [[first] + part[k]] + part[k + 1:]
        yield [[first]] + part


def pin_p_rows_sum_to_one(orc):
    """Rows of P are probability vectors: P >= 0 and sum_j P_ij = 1 within 4 N eps."""
    for seed, N, mode in [(11, 1, NONE), (12, 7, CAUSAL), (13, 33, DENSE), (14, 50, NONE),
                          (15, 40, CAUSAL)]:
        c = _case(seed, N, 16, 8, mode, p_mask=0.3)
        Q, K, V, C = _head(c)
        S, P, O, L = orc.attention_head(Q, K, V, mode, C, c["scale"])
        assert np.all(P >= 0.0)
        assert np.all(np.abs(P.sum(axis=1) - 1.0) <= 4 * N * EPS), (seed, P.sum(axis=1))
        # O is the P-weighted combination of the rows of V.
        assert np.allclose(O, P @ _vals(V), rtol=0, atol=64 * N * EPS)


def pin_constant_v(orc):
    """If every v_j equals the same vector c, then O_i = c for any Q, K and C."""
    for seed, N, mode, cval in [(21, 13, NONE, 1.5), (22, 29, CAUSAL, -0.375), (23, 17, DENSE, 3.0)]:
        c = _case(seed, N, 32, 5, mode, p_mask=0.4)
        Q, K, _, C = _head(c)
        row = synth.bf16_bits(np.array([cval, -2.0 * cval, 0.5, 7.0, -1.25], dtype=np.float32))
        V = np.tile(row, (N, 1))
        _, _, O, _ = orc.attention_head(Q, K, V, mode, C, c["scale"])
        expect = _vals(row)
        assert np.allclose(O, expect[None, :], rtol=8 * N * EPS, atol=0), (seed, O[:2])


def pin_single_allowed_key(orc):
    """A row with exactly one allowed key j returns O_i = v_j exactly and LSE_i = S_ij."""
    N, d, dv = 9, 16, 6
    c = _case(31, N, d, dv, DENSE)
    Q, K, V, C = _head(c)
    C = C.copy()
    rng = np.random.default_rng(31)
    keep = rng.integers(0, N, size=N)
    mask = np.full((N, N), -np.inf, dtype=np.float32)
    mask[np.arange(N), keep] = C[np.arange(N), keep]
    _, _, O, L = orc.attention_head(Q, K, V, DENSE, mask, c["scale"])
    Vv = _vals(V)
    assert np.array_equal(O, Vv[keep]), "O_i must equal v_j of the only allowed key"
    S = _scores_numpy(Q, K, mask, DENSE, c["scale"])
    assert np.allclose(L, S[np.arange(N), keep], rtol=0, atol=1e-12)
    # Causal row 0 may only see key 0.
    c2 = _case(32, 5, d, dv, CAUSAL)
    Q2, K2, V2, _ = _head(c2)
    _, _, O2, L2 = orc.attention_head(Q2, K2, V2, CAUSAL, None, c2["scale"])
    assert np.array_equal(O2[0], _vals(V2)[0])
    assert math.isclose(L2[0], c2["scale"] * float(_vals(Q2)[0] @ _vals(K2)[0]), rel_tol=0,
                        abs_tol=1e-12)


def pin_uniform_weights(orc):
    """Q = 0 and C = 0 give uniform weights: O_i = mean_j v_j, LSE_i = ln N (causal: ln(i+1))."""
    N, d, dv = 23, 8, 7
    c = _case(41, N, d, dv, NONE)
    _, K, V, _ = _head(c)
    Q0 = np.zeros((N, d), dtype=np.uint16)
    Vv = _vals(V)
    _, _, O, L = orc.attention_head(Q0, K, V, NONE, None, c["scale"])
    assert np.allclose(O, Vv.mean(axis=0)[None, :], rtol=0, atol=16 * N * EPS)
    assert np.allclose(L, math.log(N), rtol=0, atol=4 * EPS)
    _, _, Oc, Lc = orc.attention_head(Q0, K, V, CAUSAL, None, c["scale"])
    for i in range(N):
        assert np.allclose(Oc[i], Vv[: i + 1].mean(axis=0), rtol=0, atol=16 * N * EPS), i
        assert math.isclose(Lc[i], math.log(i + 1), rel_tol=0, abs_tol=4 * EPS), i


def pin_shift_invariance(orc):
    """Adding kappa_i to row i of C leaves O_i unchanged and adds kappa_i to LSE_i."""
    N, d, dv = 19, 16, 4
    c = _case(51, N, d, dv, DENSE)
    Q, K, V, _ = _head(c)
    rng = np.random.default_rng(51)
    # Multiples of 1/64 below 8 in magnitude and shifts in quarters stay exact in fp32.
    C = (np.round(rng.standard_normal((N, N)) * 64.0) / 64.0).astype(np.float32)
    C[rng.random((N, N)) < 0.25] = -np.inf
    C[:, 0] = 0.5
    kappa = (rng.integers(-12, 13, size=N) / 4.0).astype(np.float32)
    C2 = (C + kappa[:, None]).astype(np.float32)
    _, _, O1, L1 = orc.attention_head(Q, K, V, DENSE, C, c["scale"])
    _, _, O2, L2 = orc.attention_head(Q, K, V, DENSE, C2, c["scale"])
    assert np.allclose(O1, O2, rtol=0, atol=64 * EPS * np.abs(O1).max())
    assert np.allclose(L2 - L1, kappa.astype(np.float64), rtol=0, atol=1e-13)


def pin_blockwise_equals_full(orc):
    """The recurrence over any partition of the allowed keys into blocks, in any block
    order, gives the full-softmax O_i and m_T + ln l_T = LSE_i."""
    rng = np.random.default_rng(61)
    for N in range(1, 7):
        for rep in range(2):
            c = _case(600 + 10 * N + rep, N, 8, 3, DENSE, p_mask=0.0)
            Q, K, V, C = _head(c)
            C = C.copy()
            forbidden = rng.random(N) < 0.3
            forbidden[rng.integers(0, N)] = False
            C[:, forbidden] = -np.inf
            S, _, O, L = orc.attention_head(Q, K, V, DENSE, C, c["scale"])
            Vv = _vals(V)
            i = int(rng.integers(0, N))
            allowed = [j for j in range(N) if not forbidden[j]]
            for part in _set_partitions(allowed):
                T = len(part)
                blk = np.full(N, -1, dtype=np.int32)
                for t, block in enumerate(part):
                    blk[block] = t
                orders = [list(range(T)), list(reversed(range(T)))]
                orders.append(list(rng.permutation(T)))
                for order in orders:
                    Ob, m, l = orc.online_blocks(S[i], Vv, blk, T, order)
                    assert np.allclose(Ob, O[i], rtol=0, atol=32 * N * EPS), (N, part, order)
                    assert math.isclose(m + math.log(l), L[i], rel_tol=0, abs_tol=1e-14)
                    # m_T is the running maximum, so it ends at the row maximum m_i.
                    assert m == S[i].max(), (m, S[i].max())
    # Random contiguous partitions (tiles) of longer rows, scores of large magnitude.
    for N in (8, 17, 64):
        c = _case(700 + N, N, 32, 4, NONE, qk_mult=4.0)
        Q, K, V, C = _head(c)
        S, _, O, L = orc.attention_head(Q, K, V, NONE, None, c["scale"])
        Vv = _vals(V)
        for rep in range(8):
            cuts = sorted(set(rng.integers(1, N, size=int(rng.integers(0, min(N - 1, 8) + 1)))))
            bounds = [0] + list(cuts) + [N]
            blk = np.empty(N, dtype=np.int32)
            for t in range(len(bounds) - 1):
                blk[bounds[t]:bounds[t + 1]] = t
            i = int(rng.integers(0, N))
            Ob, m, l = orc.online_blocks(S[i], Vv, blk, len(bounds) - 1)
            assert np.allclose(Ob, O[i], rtol=0, atol=64 * N * EPS * max(1.0, np.abs(O[i]).max()))
            assert math.isclose(m + math.log(l), L[i], rel_tol=0, abs_tol=1e-12)
            assert m == S[i].max()
    # Tiles whose maxima differ by thousands (scores ~1e4): alpha must stay <= 1, so the
    # recurrence cannot overflow whatever the order of the tiles.
    c = _case(777, 48, 64, 4, NONE, qk_mult=32.0)
    Q, K, V, _ = _head(c)
    S, _, O, L = orc.attention_head(Q, K, V, NONE, None, c["scale"])
    Vv = _vals(V)
    blk = np.repeat(np.arange(6, dtype=np.int32), 8)
    for i in range(48):
        for order in (list(range(6)), list(reversed(range(6)))):
            Ob, m, l = orc.online_blocks(S[i], Vv, blk, 6, order)
            assert np.isfinite(Ob).all() and np.isfinite(l), (i, order)
            assert np.allclose(Ob, O[i], rtol=0, atol=1e-12 * max(1.0, np.abs(O[i]).max()))


def pin_exercise_5_3(orc):
    """The page's single-step update with the element of Exercise 5-3 (score ln 4, value 5)."""
    with open(os.path.join(GOLDEN, "exercise_5_3.json")) as f:
        g = json.load(f)
    prior, el, exp_ = g["prior"], g["element"], g["expected"]
    m, l, u = orc.online_step(prior["m"], prior["l"], prior["u"], math.log(4.0), el["value"])
    assert math.isclose(m, math.log(4.0), rel_tol=0, abs_tol=1e-15)
    assert math.isclose(l, exp_["l_new"], rel_tol=1e-15)
    assert np.allclose(u, exp_["u_new"], rtol=1e-15, atol=0)
    assert np.allclose(u / l, exp_["output"], rtol=1e-15, atol=0)
    # The same value from the blockwise recurrence with one element per block.
    O, m2, l2 = orc.online_blocks(np.array([0.0, math.log(4.0)]), np.array([[1.0], [5.0]]),
                                  np.array([0, 1]), 2)
    assert np.allclose(O, exp_["output"], rtol=1e-15, atol=0)
    assert math.isclose(l2, exp_["l_new"], rel_tol=1e-15)


def pin_one_and_three(orc):
    """Blocks holding 1 and 3: block-local outputs are 1 and 3 either way, and only the
    kept (m, l, u) statistics recover 7/3 (weights 1:2) or 5/3 (weights 2:1)."""
    with open(os.path.join(GOLDEN, "one_and_three.json")) as f:
        g = json.load(f)
    ln2 = math.log(2.0)
    expected = {"7/3": 7.0 / 3.0, "5/3": 5.0 / 3.0}
    for case in g["cases"]:
        s = [ln2 if x == "ln 2" else float(x) for x in case["scores"]]
        v = case["values"]
        st1 = (s[0], 1.0, [v[0]])  # a block of one element: m = s, l = e^0 = 1, u = v
        st2 = (s[1], 1.0, [v[1]])
        assert [st1[2][0] / st1[1], st2[2][0] / st2[1]] == g["block_local_outputs"]
        m, l, u = orc.online_merge(st1, st2)
        assert math.isclose(u[0] / l, expected[case["expected"]], rel_tol=4 * EPS)
        O, _, _ = orc.online_blocks(np.array(s), np.array([[v[0]], [v[1]]]), np.array([0, 1]), 2)
        assert math.isclose(O[0], expected[case["expected"]], rel_tol=4 * EPS)


def pin_merge_of_partial_states(orc):
    """Partial states of two disjoint key sets of a row, merged with their (m, l, u)
    statistics, give the full-row O_i, m_i and l_i (any split, unequal l's)."""
    rng = np.random.default_rng(161)
    c = _case(161, 30, 16, 5, NONE, qk_mult=2.0)
    Q, K, V, _ = _head(c)
    S, _, O, L = orc.attention_head(Q, K, V, NONE, None, c["scale"])
    Vv = _vals(V)
    for i in range(0, 30, 3):
        side = rng.random(30) < rng.uniform(0.1, 0.9)
        side[0], side[1] = True, False
        states = []
        for sel in (side, ~side):
            blk = np.where(sel, 0, -1).astype(np.int32)
            Ob, m, l = orc.online_blocks(S[i], Vv, blk, 1)
            states.append((m, l, Ob * l))
        m, l, u = orc.online_merge(states[0], states[1])
        assert m == S[i].max()
        assert math.isclose(m + math.log(l), L[i], rel_tol=0, abs_tol=1e-13)
        assert np.allclose(u / l, O[i], rtol=0, atol=1e-13)


def pin_bruteforce_tiny(orc):
    """Tiny problems against 50-digit arithmetic (mpmath), relative error <= 1e-13."""
    import mpmath

    mpmath.mp.dps = 50
    for seed, N, d, dv, mode in [(81, 1, 4, 3, NONE), (82, 3, 5, 2, CAUSAL), (83, 5, 3, 4, DENSE),
                                 (84, 8, 6, 5, NONE), (85, 8, 4, 7, DENSE), (86, 6, 7, 3, CAUSAL)]:
        c = _case(seed, N, d, dv, mode, p_mask=0.3, qk_mult=2.0)
        Q, K, V, C = _head(c)
        _, _, O, L = orc.attention_head(Q, K, V, mode, C, c["scale"])
        Qv, Kv, Vv = _vals(Q), _vals(K), _vals(V)
        sc = mpmath.mpf(c["scale"])
        for i in range(N):
            srow = []
            for j in range(N):
                if mode == CAUSAL and j > i:
                    srow.append(None)
                    continue
                if mode == DENSE and np.isneginf(C[i, j]):
                    srow.append(None)
                    continue
                acc = mpmath.mpf(0)
                for k in range(d):
                    acc += mpmath.mpf(float(Qv[i, k])) * mpmath.mpf(float(Kv[j, k]))
                sij = sc * acc
                if mode == DENSE:
                    sij += mpmath.mpf(float(C[i, j]))
                srow.append(sij)
            if all(x is None for x in srow):
                assert np.all(O[i] == 0.0) and np.isneginf(L[i])
                continue
            w = [mpmath.exp(x) if x is not None else mpmath.mpf(0) for x in srow]
            tot = mpmath.fsum(w)
            for col in range(dv):
                ref = mpmath.fsum(w[j] * mpmath.mpf(float(Vv[j, col])) for j in range(N)) / tot
                assert abs(O[i, col] - float(ref)) <= 1e-13 * max(1.0, abs(float(ref))), \
                    (seed, i, col, O[i, col], float(ref))
            assert abs(L[i] - float(mpmath.log(tot))) <= 1e-13 * max(1.0, abs(float(mpmath.log(tot))))


def pin_two_keys_logistic(orc):
    """N = 2 without a mask: P_i0 = 1 / (1 + e^{S_i1 - S_i0}) (the logistic function)."""
    c = _case(91, 2, 16, 3, NONE, qk_mult=2.0)
    Q, K, V, _ = _head(c)
    S, P, O, _ = orc.attention_head(Q, K, V, NONE, None, c["scale"])
    Vv = _vals(V)
    for i in range(2):
        p0 = 1.0 / (1.0 + math.exp(S[i, 1] - S[i, 0]))
        assert math.isclose(P[i, 0], p0, rel_tol=4 * EPS)
        assert np.allclose(O[i], p0 * Vv[0] + (1.0 - p0) * Vv[1], rtol=0, atol=8 * EPS * 4)


def pin_large_scores(orc):
    """Scores of magnitude ~1e4: no overflow; a row whose top score leads by more than 60
    returns the top key's v exactly (every other weight is below e^-60)."""
    c = _case(101, 24, 64, 8, NONE, qk_mult=32.0)
    Q, K, V, _ = _head(c)
    S, P, O, L = orc.attention_head(Q, K, V, NONE, None, c["scale"])
    assert np.isfinite(O).all() and np.isfinite(L).all()
    assert np.abs(S).max() > 1e3
    Vv = _vals(V)
    checked = 0
    for i in range(24):
        order = np.argsort(S[i])
        if S[i, order[-1]] - S[i, order[-2]] > 60.0:
            assert np.array_equal(O[i], Vv[order[-1]]), i
            assert math.isclose(L[i], S[i, order[-1]], rel_tol=4 * EPS)
            checked += 1
    assert checked >= 3


def pin_causal_is_triangular_bias(orc):
    """The causal mode equals a dense C with -inf above the diagonal and 0 elsewhere."""
    c = _case(111, 37, 16, 9, CAUSAL, BH=2)
    N = 37
    tri = np.where(np.arange(N)[None, :] > np.arange(N)[:, None], -np.inf, 0.0).astype(np.float32)
    C = np.broadcast_to(tri, (2, N, N)).copy()
    O1, L1, _ = orc.attention(c["Q"], c["K"], c["V"], CAUSAL, None, c["scale"])
    O2, L2, _ = orc.attention(c["Q"], c["K"], c["V"], DENSE, C, c["scale"])
    assert np.array_equal(O1, O2) and np.array_equal(L1, L2)


def pin_scale_wiring(orc):
    """S = scale * Q K^T: doubling Q (exact in bf16) and halving the scale changes nothing;
    and with K = Q = e_1 rows the score is exactly `scale`."""
    c = _case(121, 11, 16, 4, NONE, BH=2)
    Q2 = synth.bf16_bits(2.0 * synth.bf16_to_f32(c["Q"]))
    O1, L1, _ = orc.attention(c["Q"], c["K"], c["V"], NONE, None, c["scale"])
    O2, L2, _ = orc.attention(Q2, c["K"], c["V"], NONE, None, c["scale"] / 2.0)
    assert np.array_equal(O1, O2) and np.array_equal(L1, L2)
    # Two keys, one of them equal to the query direction: S_i0 = scale, S_i1 = 0.
    e1 = np.zeros((2, 4), dtype=np.float32)
    e1[:, 0] = 1.0
    Qb = synth.bf16_bits(e1)
    Kb = synth.bf16_bits(np.array([[1, 0, 0, 0], [0, 1, 0, 0]], dtype=np.float32))
    Vb = synth.bf16_bits(np.array([[1.0], [0.0]], dtype=np.float32))
    S, _, O, L = orc.attention_head(Qb, Kb, Vb, NONE, None, 0.75)
    assert S[0, 0] == 0.75 and S[0, 1] == 0.0
    assert math.isclose(O[0, 0], 1.0 / (1.0 + math.exp(-0.75)), rel_tol=4 * EPS)
    assert math.isclose(L[0], math.log(math.exp(0.75) + 1.0), rel_tol=4 * EPS)


def pin_key_permutation(orc):
    """Permuting the keys (rows of K and V with the columns of C) leaves O and LSE unchanged."""
    rng = np.random.default_rng(131)
    for mode in (NONE, DENSE):
        c = _case(131 + mode, 21, 16, 6, mode, p_mask=0.3)
        Q, K, V, C = _head(c)
        perm = rng.permutation(21)
        C2 = None if C is None else C[:, perm]
        _, _, O1, L1 = orc.attention_head(Q, K, V, mode, C, c["scale"])
        _, _, O2, L2 = orc.attention_head(Q, K[perm], V[perm], mode, C2, c["scale"])
        assert np.allclose(O1, O2, rtol=0, atol=1e-13)
        assert np.allclose(L1, L2, rtol=0, atol=1e-13)


def pin_row_subset_and_threads(orc):
    """Evaluating a subset of rows, or with another thread count, gives identical bits."""
    c = _case(141, 45, 32, 16, CAUSAL, BH=3)
    O, L, _ = orc.attention(c["Q"], c["K"], c["V"], CAUSAL, None, c["scale"], nthreads=4)
    O1, L1, used = orc.attention(c["Q"], c["K"], c["V"], CAUSAL, None, c["scale"], nthreads=1)
    assert used == 1
    assert np.array_equal(O, O1) and np.array_equal(L, L1)
    rows = np.array([0, 44, 45, 89, 134, 70], dtype=np.int64)
    Os, Ls, _ = orc.attention(c["Q"], c["K"], c["V"], CAUSAL, None, c["scale"], rows=rows)
    assert np.array_equal(Os, O.reshape(-1, 16)[rows])
    assert np.array_equal(Ls, L.reshape(-1)[rows])


def pin_no_allowed_key(orc):
    """Outside the pages' assumption (a row with no allowed key) the defined result is
    O_i = 0 and LSE_i = -inf; the other rows are unaffected."""
    c = _case(151, 6, 8, 3, DENSE)
    Q, K, V, C = _head(c)
    C = C.copy()
    C[2, :] = -np.inf
    _, _, O, L = orc.attention_head(Q, K, V, DENSE, C, c["scale"])
    assert np.array_equal(O[2], np.zeros(3)) and np.isneginf(L[2])
    assert np.isfinite(O).all() and np.isfinite(np.delete(L, 2)).all()


# ------------------------------------------------------------------ rectangular and key bias
def _case_ex(seed, BH, Nq, Nk, d, dv, mode, p_mask=0.0, qk_mult=1.0):
    return synth.random_case_ex(seed, BH, Nq, Nk, d, dv, mode, qk_mult, p_mask)


def pin_key_bias_is_a_broadcast_dense_bias(orc):
    """A per-key bias c_j is the dense bias C_ij = c_j for every row: identical bits."""
    for mode_extra in (0, CAUSAL):
        c = _case_ex(171 + mode_extra, 2, 37, 37, 16, 8, synth.MODE_KEY | mode_extra, p_mask=0.3)
        C = np.broadcast_to(c["ckey"][:, None, :], (2, 37, 37)).copy()
        O1, L1, _ = orc.attention_ex(c["Q"], c["K"], c["V"], synth.MODE_KEY | mode_extra, None,
                                     c["ckey"], c["scale"])
        O2, L2, _ = orc.attention_ex(c["Q"], c["K"], c["V"], DENSE | mode_extra, C, None, c["scale"])
        assert np.array_equal(O1, O2) and np.array_equal(L1, L2)


def pin_rows_depend_only_on_their_query(orc):
    """Without a causal mask, a problem holding any subset of a square problem's queries
    (same keys, values and bias columns) returns exactly those rows."""
    N = 29
    c = _case_ex(181, 2, N, N, 16, 6, synth.MODE_KEY, p_mask=0.2)
    O, L, _ = orc.attention_ex(c["Q"], c["K"], c["V"], synth.MODE_KEY, None, c["ckey"], c["scale"])
    rows = np.array([3, 0, 17, 28, 9])
    Os, Ls, _ = orc.attention_ex(np.ascontiguousarray(c["Q"][:, rows]), c["K"], c["V"],
                                 synth.MODE_KEY, None, c["ckey"], c["scale"])
    assert np.array_equal(Os, O[:, rows]) and np.array_equal(Ls, L[:, rows])


def pin_causal_offset(orc):
    """Causal with Nq != Nk aligns the last query with the last key: query i may see keys
    j <= i + Nk - Nq. It equals a dense bias with that -inf pattern, and it reproduces the
    square causal problem on the rows the two share."""
    for Nq, Nk in ((13, 40), (40, 13), (1, 17), (25, 25)):
        c = _case_ex(191 + Nq, 2, Nq, Nk, 16, 5, CAUSAL)
        off = Nk - Nq
        tri = np.where(np.arange(Nk)[None, :] > np.arange(Nq)[:, None] + off, -np.inf, 0.0)
        C = np.broadcast_to(tri.astype(np.float32), (2, Nq, Nk)).copy()
        O1, L1, _ = orc.attention_ex(c["Q"], c["K"], c["V"], CAUSAL, None, None, c["scale"])
        O2, L2, _ = orc.attention_ex(c["Q"], c["K"], c["V"], DENSE, C, None, c["scale"])
        assert np.array_equal(O1, O2) and np.array_equal(L1, L2), (Nq, Nk)
        # Shared rows with the square causal problem over the same keys.
        Qsq = synth.bf16_tensor(777 + Nq, (2, Nk, 16))
        if Nq <= Nk:
            Qsq[:, Nk - Nq:] = c["Q"]
            Osq, Lsq, _ = orc.attention_ex(Qsq, c["K"], c["V"], CAUSAL, None, None, c["scale"])
            assert np.array_equal(O1, Osq[:, Nk - Nq:]) and np.array_equal(L1, Lsq[:, Nk - Nq:])
            # The last query sees every key: the unmasked result.
            On, Ln, _ = orc.attention_ex(c["Q"], c["K"], c["V"], NONE, None, None, c["scale"])
            assert np.array_equal(O1[:, -1], On[:, -1]) and np.array_equal(L1[:, -1], Ln[:, -1])
        else:
            # The first Nq - Nk queries have no allowed key: O = 0, LSE = -inf.
            assert np.all(O1[:, :Nq - Nk] == 0.0) and np.all(np.isneginf(L1[:, :Nq - Nk]))
            Osq, Lsq, _ = orc.attention_ex(np.ascontiguousarray(c["Q"][:, Nq - Nk:]), c["K"],
                                           c["V"], CAUSAL, None, None, c["scale"])
            assert np.array_equal(O1[:, Nq - Nk:], Osq) and np.array_equal(L1[:, Nq - Nk:], Lsq)


def pin_bias_terms_add(orc):
    """Causal with a dense bias is the dense bias plus the causal -inf pattern; a key bias
    plus a dense bias is their sum (exact in fp64 for these fp32 values)."""
    Nq, Nk = 21, 30
    c = _case_ex(201, 2, Nq, Nk, 16, 4, CAUSAL | DENSE, p_mask=0.2)
    off = Nk - Nq
    tri = np.where(np.arange(Nk)[None, :] > np.arange(Nq)[:, None] + off, -np.inf, 0.0)
    C2 = (c["C"] + tri[None].astype(np.float32)).astype(np.float32)
    O1, L1, _ = orc.attention_ex(c["Q"], c["K"], c["V"], CAUSAL | DENSE, c["C"], None, c["scale"])
    O2, L2, _ = orc.attention_ex(c["Q"], c["K"], c["V"], DENSE, C2, None, c["scale"])
    assert np.array_equal(O1, O2) and np.array_equal(L1, L2)
    rng = np.random.default_rng(201)
    ck = (np.round(rng.standard_normal((2, Nk)) * 8) / 8).astype(np.float32)
    Cq = (np.round(rng.standard_normal((2, Nq, Nk)) * 8) / 8).astype(np.float32)
    O3, L3, _ = orc.attention_ex(c["Q"], c["K"], c["V"], DENSE | synth.MODE_KEY, Cq, ck, c["scale"])
    O4, L4, _ = orc.attention_ex(c["Q"], c["K"], c["V"], DENSE, (Cq + ck[:, None, :]).astype(np.float32),
                                 None, c["scale"])
    assert np.allclose(O3, O4, rtol=0, atol=1e-15) and np.allclose(L3, L4, rtol=0, atol=1e-14)


def pin_bruteforce_rectangular(orc):
    """Nq != Nk with causal, key and dense terms against 50-digit arithmetic."""
    import mpmath

    mpmath.mp.dps = 50
    for seed, Nq, Nk, mode in [(211, 3, 7, CAUSAL | synth.MODE_KEY), (212, 6, 4, CAUSAL | DENSE),
                               (213, 5, 8, synth.MODE_KEY), (214, 2, 9, CAUSAL)]:
        c = _case_ex(seed, 1, Nq, Nk, 5, 3, mode, p_mask=0.3, qk_mult=2.0)
        O, L, _ = orc.attention_ex(c["Q"], c["K"], c["V"], mode, c["C"], c["ckey"], c["scale"])
        Qv, Kv, Vv = _vals(c["Q"][0]), _vals(c["K"][0]), _vals(c["V"][0])
        for i in range(Nq):
            w = []
            for j in range(Nk):
                if (mode & CAUSAL) and j > i + (Nk - Nq):
                    w.append(mpmath.mpf(0))
                    continue
                sij = mpmath.mpf(c["scale"]) * mpmath.fsum(
                    mpmath.mpf(float(Qv[i, k])) * mpmath.mpf(float(Kv[j, k])) for k in range(5))
                if mode & DENSE:
                    if np.isneginf(c["C"][0, i, j]):
                        w.append(mpmath.mpf(0))
                        continue
                    sij += mpmath.mpf(float(c["C"][0, i, j]))
                if mode & synth.MODE_KEY:
                    if np.isneginf(c["ckey"][0, j]):
                        w.append(mpmath.mpf(0))
                        continue
                    sij += mpmath.mpf(float(c["ckey"][0, j]))
                w.append(mpmath.exp(sij))
            tot = mpmath.fsum(w)
            if tot == 0:
                assert np.all(O[0, i] == 0.0) and np.isneginf(L[0, i])
                continue
            for col in range(3):
                ref = mpmath.fsum(w[j] * mpmath.mpf(float(Vv[j, col])) for j in range(Nk)) / tot
                assert abs(O[0, i, col] - float(ref)) <= 1e-13 * max(1.0, abs(float(ref))), (seed, i)
            assert abs(L[0, i] - float(mpmath.log(tot))) <= 1e-13 * max(1.0, abs(float(mpmath.log(tot))))


# ---------------------------------------------------------------- backward pass
KEY = synth.MODE_KEY


def _bwd_case(seed, BH, Nq, Nk, d, dv, mode, p_mask=0.0):
    c = _case_ex(seed, BH, Nq, Nk, d, dv, mode, p_mask)
    c["dO"] = synth.bf16_tensor(seed + 17, (BH, Nq, dv))
    return c


def _bwd(orc, c, **kw):
    return orc.attention_bwd(c["Q"], c["K"], c["V"], c["dO"], c["mode"], c["C"], c["ckey"],
                             c["scale"], **kw)


def pin_bwd_finite_differences(orc):
    """Every gradient entry equals the central difference of the loss sum(dO * O) in
    60-digit arithmetic (step 1e-20), on tiny problems of every mask kind, queries
    and keys of their own lengths: <= 1e-11 relative."""
    import mpmath

    mpmath.mp.dps = 60
    h = mpmath.mpf("1e-20")
    for seed, Nq, Nk, mode, p_mask in ((11, 3, 4, NONE, 0.0), (12, 3, 4, CAUSAL, 0.0),
                                       (13, 4, 3, CAUSAL, 0.0), (14, 3, 4, DENSE, 0.3),
                                       (15, 3, 5, KEY | CAUSAL, 0.3)):
        d, dv = 3, 2
        c = _bwd_case(seed, 1, Nq, Nk, d, dv, mode, p_mask)
        dQ, dK, dV, _ = _bwd(orc, c)
        Qv, Kv, Vv, G = (_vals(c[k])[0] for k in ("Q", "K", "V", "dO"))
        sc = mpmath.mpf(c["scale"])

        def loss(Qm, Km, Vm):
            tot = mpmath.mpf(0)
            for i in range(Nq):
                w = []
                for j in range(Nk):
                    if (mode & CAUSAL) and j > i + (Nk - Nq):
                        w.append(None)
                        continue
                    sij = sc * mpmath.fsum(Qm[i][k] * Km[j][k] for k in range(d))
                    if mode & DENSE:
                        cij = float(c["C"][0, i, j])
                        if cij == -math.inf:
                            w.append(None)
                            continue
                        sij += mpmath.mpf(cij)
                    if mode & KEY:
                        cj = float(c["ckey"][0, j])
                        if cj == -math.inf:
                            w.append(None)
                            continue
                        sij += mpmath.mpf(cj)
                    w.append(sij)
                live = [x for x in w if x is not None]
                if not live:
                    continue
                e = [mpmath.exp(x) if x is not None else mpmath.mpf(0) for x in w]
                z = mpmath.fsum(e)
                for col in range(dv):
                    o = mpmath.fsum(e[j] * Vm[j][col] for j in range(Nk)) / z
                    tot += mpmath.mpf(float(G[i, col])) * o
            return tot

        base = {"Q": [[mpmath.mpf(float(x)) for x in r] for r in Qv],
                "K": [[mpmath.mpf(float(x)) for x in r] for r in Kv],
                "V": [[mpmath.mpf(float(x)) for x in r] for r in Vv]}
        for name, grad in (("Q", dQ[0]), ("K", dK[0]), ("V", dV[0])):
            for r in range(grad.shape[0]):
                for col in range(grad.shape[1]):
                    plus = {k: [list(row) for row in v] for k, v in base.items()}
                    minus = {k: [list(row) for row in v] for k, v in base.items()}
                    plus[name][r][col] += h
                    minus[name][r][col] -= h
                    fd = float((loss(plus["Q"], plus["K"], plus["V"]) -
                                loss(minus["Q"], minus["K"], minus["V"])) / (2 * h))
                    assert abs(grad[r, col] - fd) <= 1e-11 * max(1.0, abs(fd)), (
                        name, seed, r, col, grad[r, col], fd)


def pin_bwd_key_gradients_sum_to_zero(orc):
    """Adding one vector to every key adds a constant to each row of S (softmax does not
    change), so the key gradients of a head sum to zero, for every mask kind."""
    for seed, Nq, Nk, mode, pm in ((21, 40, 40, NONE, 0.0), (22, 33, 70, CAUSAL, 0.0),
                                   (23, 50, 30, CAUSAL, 0.0), (24, 20, 45, DENSE, 0.3),
                                   (25, 31, 64, KEY | CAUSAL, 0.3)):
        c = _bwd_case(seed, 2, Nq, Nk, 16, 8, mode, pm)
        dQ, dK, dV, _ = _bwd(orc, c)
        scale = np.abs(dK).max()
        assert np.abs(dK.sum(axis=1)).max() <= 1e-12 * max(1.0, scale) * Nk, (seed, dK.sum(axis=1))


def pin_bwd_value_gradients_sum_to_dO(orc):
    """Rows of P sum to 1, so sum_j dV_j = sum over rows with an allowed key of dO_i."""
    for seed, Nq, Nk, mode in ((31, 40, 40, NONE), (32, 50, 30, CAUSAL), (33, 17, 64, KEY)):
        c = _bwd_case(seed, 2, Nq, Nk, 16, 8, mode, 0.3 if mode & KEY else 0.0)
        dQ, dK, dV, _ = _bwd(orc, c)
        G = _vals(c["dO"])
        live = np.ones((2, Nq), dtype=bool)
        if mode & CAUSAL and Nq > Nk:
            live[:, :Nq - Nk] = False  # rows that see no key
        want = (G * live[:, :, None]).sum(axis=1)
        assert np.abs(dV.sum(axis=1) - want).max() <= 1e-12 * Nq, seed


def pin_bwd_uniform_weights(orc):
    """Q = 0 and no mask: P_ij = 1/Nk, so dV_j = mean_i-free sum_i dO_i / Nk, dK = 0, and
    dQ_i = scale / Nk * sum_j (dO_i . (v_j - vbar)) k_j (closed form)."""
    c = _bwd_case(41, 1, 12, 20, 8, 6, NONE)
    c["Q"] = np.zeros_like(c["Q"])
    dQ, dK, dV, _ = _bwd(orc, c)
    K, V, G = _vals(c["K"])[0], _vals(c["V"])[0], _vals(c["dO"])[0]
    Nk = K.shape[0]
    assert np.abs(dV[0] - G.sum(axis=0)[None, :] / Nk).max() <= 1e-14
    assert np.abs(dK).max() == 0.0
    vbar = V.mean(axis=0)
    want = c["scale"] / Nk * ((G @ (V - vbar).T) @ K)
    assert np.abs(dQ[0] - want).max() <= 1e-13


def pin_bwd_single_and_no_key_rows(orc):
    """A row with one allowed key has a one-hot P, so dS_i = 0 and dQ_i = 0; a row with no
    allowed key (Nq > Nk, causal) has the constant output 0 and gradient 0 everywhere."""
    c = _bwd_case(51, 1, 20, 20, 8, 8, CAUSAL)
    dQ, dK, dV, _ = _bwd(orc, c)
    assert np.all(dQ[0, 0] == 0.0)  # query 0 sees key 0 only
    c = _bwd_case(52, 1, 30, 10, 8, 8, CAUSAL)
    dQ, dK, dV, _ = _bwd(orc, c)
    assert np.all(dQ[0, :20] == 0.0) and np.all(dQ[0, 20] == 0.0)  # none, then one key
    # The keyless rows' dO does not reach dV or dK.
    c2 = dict(c)
    c2["dO"] = c["dO"].copy()
    c2["dO"][0, :20] = synth.bf16_tensor(999, (20, 8))
    _, dK2, dV2, _ = _bwd(orc, c2)
    assert np.array_equal(dK, dK2) and np.array_equal(dV, dV2)


def pin_bwd_selection_and_threads(orc):
    """Selected heads, query rows and keys, and any thread count, give the same bits."""
    c = _bwd_case(61, 3, 37, 45, 8, 16, CAUSAL | KEY, 0.2)
    dQ, dK, dV, _ = _bwd(orc, c, nthreads=1)
    heads, qr, kr = [2, 0], [36, 0, 17], [44, 3, 3, 10]
    sQ, sK, sV, _ = _bwd(orc, c, heads=heads, qrows=qr, krows=kr, nthreads=3)
    assert np.array_equal(sQ, dQ[heads][:, qr]) and np.array_equal(sK, dK[heads][:, kr])
    assert np.array_equal(sV, dV[heads][:, kr])
    tQ, tK, tV, _ = _bwd(orc, c, nthreads=7)
    assert np.array_equal(tQ, dQ) and np.array_equal(tK, dK) and np.array_equal(tV, dV)


ALL_PINS = [
    pin_p_rows_sum_to_one,
    pin_constant_v,
    pin_single_allowed_key,
    pin_uniform_weights,
    pin_shift_invariance,
    pin_blockwise_equals_full,
    pin_exercise_5_3,
    pin_one_and_three,
    pin_merge_of_partial_states,
    pin_bruteforce_tiny,
    pin_two_keys_logistic,
    pin_large_scores,
    pin_causal_is_triangular_bias,
    pin_scale_wiring,
    pin_key_permutation,
    pin_row_subset_and_threads,
    pin_no_allowed_key,
    pin_key_bias_is_a_broadcast_dense_bias,
    pin_rows_depend_only_on_their_query,
    pin_causal_offset,
    pin_bias_terms_add,
    pin_bruteforce_rectangular,
    pin_bwd_finite_differences,
    pin_bwd_key_gradients_sum_to_zero,
    pin_bwd_value_gradients_sum_to_dO,
    pin_bwd_uniform_weights,
    pin_bwd_single_and_no_key_rows,
    pin_bwd_selection_and_threads,
]
