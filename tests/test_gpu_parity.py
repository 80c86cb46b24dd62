"""CUDA path vs the fp64 oracle, element by element, on seeded inputs (needs a GB300).

Sizes span several 128-row tiles and ragged tails; modes cover no mask, causal, and
a dense bias with key-padding -inf (through TMA when N % 4 == 0, read directly
otherwise). Edge cases: N = 1, whole masked tiles, single allowed keys, rows with no
allowed key, large-magnitude scores, determinism, concurrent streams, and
perturbations that must (or must not) change given outputs.
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_helpers import compare, device_inputs, run_gpu

pytestmark = pytest.mark.gpu

NONE, CAUSAL, DENSE = synth.MODE_NONE, synth.MODE_CAUSAL, synth.MODE_DENSE

# (BH, N, d, dv, mode, out_f32, qk_mult, p_mask)
CASES = [
    (1, 1, 64, 64, NONE, True, 1.0, 0.0),
    (2, 17, 64, 64, NONE, True, 1.0, 0.0),
    (1, 128, 128, 128, NONE, True, 1.0, 0.0),
    (2, 129, 128, 128, CAUSAL, False, 1.0, 0.0),
    (1, 255, 64, 128, DENSE, True, 1.0, 0.3),
    (2, 256, 64, 128, DENSE, True, 1.0, 0.3),
    (1, 300, 128, 64, CAUSAL, True, 1.0, 0.0),
    (2, 1000, 128, 128, CAUSAL, False, 1.0, 0.0),
    (3, 384, 64, 64, CAUSAL, True, 1.0, 0.0),
    (1, 512, 128, 128, NONE, True, 4.0, 0.0),
    (1, 640, 64, 128, DENSE, True, 1.0, 0.3),
    (1, 127, 128, 128, DENSE, False, 1.0, 0.5),
    (2, 200, 128, 64, NONE, False, 1.0, 0.0),
    (1, 513, 64, 64, CAUSAL, False, 2.0, 0.0),
    (1, 1024, 128, 128, NONE, True, 4.0, 0.0),
    (1, 768, 128, 64, DENSE, True, 1.0, 0.3),
    (1, 96, 64, 128, CAUSAL, True, 1.0, 0.0),
    (5, 130, 64, 128, NONE, False, 1.0, 0.0),
]


def _id(c):
    BH, N, d, dv, mode, f32, mult, pm = c
    return f"bh{BH}-n{N}-d{d}-dv{dv}-{synth.MODE_NAMES[mode]}-{'f32' if f32 else 'bf16'}-x{mult:g}"


@pytest.mark.parametrize("case", CASES, ids=_id)
def test_parity_against_oracle(case):
    BH, N, d, dv, mode, out_f32, mult, p_mask = case
    c = synth.random_case(1000 + N + d + dv + 7 * mode, BH, N, d, dv, mode, mult, p_mask)
    O, L = run_gpu(c, out_f32=out_f32)
    O_ref, L_ref, _ = oracle.attention(c["Q"], c["K"], c["V"], mode, c["C"], c["scale"])
    compare(O, L, O_ref, L_ref, out_bf16=not out_f32, label=_id(case))


def test_scale_other_than_inverse_sqrt_d():
    c = synth.random_case(7, 1, 300, 64, 64, NONE)
    c["scale"] = 0.3
    O, L = run_gpu(c)
    O_ref, L_ref, _ = oracle.attention(c["Q"], c["K"], c["V"], NONE, None, 0.3)
    compare(O, L, O_ref, L_ref)


def test_deterministic_bitwise():
    c = synth.random_case(8, 2, 700, 128, 128, CAUSAL)
    dev = device_inputs(c)
    O1, L1 = run_gpu(c, dev_inputs=dev)
    O2, L2 = run_gpu(c, dev_inputs=dev)
    assert np.array_equal(O1, O2) and np.array_equal(L1, L2)


def test_concurrent_streams():
    import torch

    ca = synth.random_case(9, 3, 640, 128, 128, CAUSAL)
    cb = synth.random_case(10, 1, 512, 64, 128, DENSE, p_mask=0.3)
    ref_a = run_gpu(ca)
    ref_b = run_gpu(cb)
    import exact_tiled_attention_13_gb300 as eta

    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    outs = []
    for c, s in ((ca, s1), (cb, s2)):
        Q, K, V, C = device_inputs(c)
        torch.cuda.synchronize()
        O = torch.empty(Q.shape[0], Q.shape[1], V.shape[2], dtype=torch.float32, device="cuda")
        L = torch.empty(Q.shape[0], Q.shape[1], dtype=torch.float32, device="cuda")
        with torch.cuda.stream(s):
            for _ in range(3):
                eta.attn_fwd(Q, K, V, c["mode"], C, c["scale"], O, L, stream=s)
        outs.append((O, L, (Q, K, V, C)))
    torch.cuda.synchronize()
    for (O, L, _), ref in zip(outs, (ref_a, ref_b)):
        assert np.array_equal(O.cpu().numpy().astype(np.float64), ref[0])
        assert np.array_equal(L.cpu().numpy().astype(np.float64), ref[1])


def test_single_allowed_key_returns_that_value():
    N = 300
    c = synth.random_case(11, 1, N, 64, 128, DENSE)
    rng = np.random.default_rng(11)
    keep = rng.integers(0, N, size=N)
    C = np.full((1, N, N), -np.inf, dtype=np.float32)
    C[0, np.arange(N), keep] = c["C"][0, np.arange(N), keep]
    c["C"] = C
    O, L = run_gpu(c)
    V = synth.bf16_to_f32(c["V"][0]).astype(np.float64)
    assert np.array_equal(O[0], V[keep])
    _, L_ref, _ = oracle.attention(c["Q"], c["K"], c["V"], DENSE, C, c["scale"])
    assert np.max(np.abs(L - L_ref)) <= 1e-3


def test_whole_masked_tiles():
    N = 512
    c = synth.random_case(12, 2, N, 64, 128, DENSE, p_mask=0.0)
    C = c["C"].copy()
    C[:, :, 0:128] = -np.inf      # first K/V tile forbidden for every row
    C[:, :, 384:512] = -np.inf    # last tile too
    C[1, 5, :] = -np.inf
    C[1, 5, 300] = 0.25           # a row with exactly one allowed key in the third tile
    c["C"] = C
    O, L = run_gpu(c)
    O_ref, L_ref, _ = oracle.attention(c["Q"], c["K"], c["V"], DENSE, C, c["scale"])
    compare(O, L, O_ref, L_ref)


def test_rows_without_allowed_key_are_zero():
    # Outside the pages' assumption: the defined result is O_i = 0, LSE_i = -inf, no NaN.
    N = 256
    c = synth.random_case(13, 1, N, 128, 128, DENSE)
    C = c["C"].copy()
    C[0, 3, :] = -np.inf
    C[0, 200, :] = -np.inf
    c["C"] = C
    O, L = run_gpu(c)
    assert np.all(O[0, 3] == 0.0) and np.all(O[0, 200] == 0.0)
    assert np.isneginf(L[0, 3]) and np.isneginf(L[0, 200])
    O_ref, L_ref, _ = oracle.attention(c["Q"], c["K"], c["V"], DENSE, C, c["scale"])
    compare(O, L, O_ref, L_ref)


def test_outputs_depend_on_every_input():
    base = synth.random_case(14, 1, 384, 128, 128, CAUSAL)
    O0, L0 = run_gpu(base)

    def changed(field, index, value):
        c = dict(base)
        arr = c[field].copy()
        arr[index] = synth.bf16_bits(np.array([value], dtype=np.float32))[0]
        c[field] = arr
        return run_gpu(c)

    # A key at position 200 is seen by rows >= 200 only.
    O1, L1 = changed("K", (0, 200, 5), 8.0)
    assert np.array_equal(O1[0, :200], O0[0, :200]) and np.array_equal(L1[0, :200], L0[0, :200])
    assert np.all(np.any(O1[0, 200:] != O0[0, 200:], axis=1))
    # A value row at position 10 changes rows >= 10 only.
    O2, _ = changed("V", (0, 10, 3), 9.0)
    assert np.array_equal(O2[0, :10], O0[0, :10])
    assert np.all(O2[0, 10:, 3] != O0[0, 10:, 3])
    # A query row changes only its own output row.
    O3, L3 = changed("Q", (0, 77, 0), -6.0)
    rows = np.any(O3[0] != O0[0], axis=1)
    assert rows[77] and rows.sum() == 1
    # A bias entry changes only its own row.
    cd = synth.random_case(15, 1, 256, 64, 128, DENSE, p_mask=0.2)
    Od, _ = run_gpu(cd)
    C2 = cd["C"].copy()
    j = int(np.flatnonzero(np.isfinite(C2[0, 40]))[0])
    C2[0, 40, j] += 3.0
    Od2, _ = run_gpu(dict(cd, C=C2))
    rows = np.any(Od2[0] != Od[0], axis=1)
    assert rows[40] and rows.sum() == 1


def test_lse_optional_and_output_dtypes_agree():
    c = synth.random_case(16, 2, 333, 128, 128, NONE)
    O_f, L_f = run_gpu(c, out_f32=True)
    O_n, L_n = run_gpu(c, out_f32=True, with_lse=False)
    assert L_n is None and np.array_equal(O_f, O_n)
    O_b, _ = run_gpu(c, out_f32=False)
    # bf16 output is the fp32 result rounded once (round to nearest even).
    expect = synth.bf16_to_f32(synth.bf16_bits(O_f.astype(np.float32))).astype(np.float64)
    assert np.array_equal(O_b, expect)


def test_zero_length_is_a_noop():
    import torch

    import exact_tiled_attention_13_gb300 as eta

    Q = torch.empty(2, 0, 64, dtype=torch.bfloat16, device="cuda")
    V = torch.empty(2, 0, 64, dtype=torch.bfloat16, device="cuda")
    O = torch.empty(2, 0, 64, dtype=torch.float32, device="cuda")
    eta.attn_fwd(Q, Q.clone(), V, eta.ATTN_MASK_NONE, None, 0.125, O)
    torch.cuda.synchronize()
    assert eta.attn_device_status(None)[0] == eta.ATTN_OK


def test_rejects_host_memory():
    import torch

    import exact_tiled_attention_13_gb300 as eta

    Q = torch.zeros(1, 128, 64, dtype=torch.bfloat16)  # CPU tensor
    O = torch.zeros(1, 128, 64, dtype=torch.float32)
    with pytest.raises(eta.AttnError) as ei:
        eta.attn_fwd(Q, Q.clone(), Q.clone(), eta.ATTN_MASK_NONE, None, 0.125, O, stream=0)
    assert ei.value.code == eta.ATTN_ERR_INVALID_ARG
