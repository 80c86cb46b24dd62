"""The seeded input generator (no GPU): published test vectors, rounding, recipes."""
import json
import os

import numpy as np

import synth
from exact_tiled_attention_13_gb300 import accounting

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_splitmix64_reference_vector():
    # SplitMix64 from state 0: the first outputs of the published reference generator.
    out = synth.splitmix64(0, 0, 2)
    assert int(out[0]) == 0xE220A8397B1DCDAF
    assert int(out[1]) == 0x6E789E6AA1B965F4


def test_stream_is_counter_based():
    a = synth.splitmix64(12345, 0, 100)
    b = synth.splitmix64(12345, 40, 60)
    assert np.array_equal(a[40:], b)


def test_uniform_range_and_normal_moments():
    u = synth.uniform01(7, 0, 200000)
    assert u.min() > 0.0 and u.max() <= 1.0
    z = synth.normal_f32(8, 400001).astype(np.float64)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1.0) < 0.01
    assert np.array_equal(z[:1000], synth.normal_f32(8, 1000).astype(np.float64))


def test_bf16_round_to_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -8 + 2 ** -20, -2.5, 0.0,
                  -(1.0 + 2 ** -8)], dtype=np.float32)
    bits = synth.bf16_bits(x)
    assert [int(b) for b in bits] == [0x3F80, 0x3F80, 0x3F82, 0x3F81, 0xC020, 0x0000, 0xBF80]
    back = synth.bf16_to_f32(bits)
    assert back[2] == 1.0 + 4 * 2 ** -8
    # Rounding error stays within half a bf16 ulp.
    z = synth.normal_f32(9, 10000)
    r = synth.bf16_to_f32(synth.bf16_bits(z))
    assert np.all(np.abs(r - z) <= np.abs(z) * 2.0 ** -8)


def test_workload_recipes():
    w = synth.WORKLOADS[3]
    assert (w.BH, w.N, w.d, w.dv, w.mode, w.out_dtype) == (64, 8192, 128, 128, synth.MODE_CAUSAL,
                                                            "bf16")
    w4 = synth.WORKLOADS[4]
    assert (w4.BH, w4.N, w4.d, w4.dv, w4.mode) == (8, 4096, 64, 128, synth.MODE_DENSE)
    assert w4.scale == 0.125
    small = synth.Workload("t", 1, 2, 64, 16, 8, synth.MODE_NONE, "f32", qk_mult=4.0)
    a = synth.make_inputs(small, 5)
    b = synth.make_inputs(small, 5)
    assert np.array_equal(a["Q"], b["Q"]) and not np.array_equal(a["Q"], a["K"])
    q = synth.bf16_to_f32(a["Q"])
    # qk_mult 4 is a power of two: every value is 4 x a bf16 value.
    assert np.array_equal(synth.bf16_bits(q / 4.0), synth.bf16_bits(synth.bf16_to_f32(
        synth.bf16_bits(synth.normal_f32(synth.seed_for(5, "Q"), q.size)))).reshape(q.shape))


def test_dense_bias_key_padding():
    C = synth.dense_bias(1, 2, 3, 200, 0.3)
    masked = np.isneginf(C)
    # One draw per (head, key): a masked key is masked in every row.
    assert np.array_equal(masked, np.broadcast_to(masked[:, :1, :], masked.shape))
    frac = masked[:, 0, :].mean()
    assert 0.2 < frac < 0.4
    # Every key masked: key 0 comes back with its bias value.
    C1 = synth.dense_bias(1, 2, 2, 5, 1.0)
    assert np.isfinite(C1[:, :, 0]).all() and np.isneginf(C1[:, :, 1:]).all()


def test_byte_accounting_matches_pages():
    with open(os.path.join(GOLDEN, "byte_accounting.json")) as f:
        g = json.load(f)
    L, d = g["L"], g["d"]
    per_tensor = L * d * accounting.BF16
    assert per_tensor == g["qkvo_MiB_each"] * accounting.MiB
    inter = accounting.materialized_intermediate_bytes(L, accounting.F32)
    assert inter["S"] == g["S_MiB"] * accounting.MiB and inter["P"] == g["P_MiB"] * accounting.MiB
    assert inter["roundtrip"] == g["SP_roundtrip_GiB"] * accounting.GiB
    req = accounting.required_bytes(1, L, d, d, accounting.BF16, lse=False)
    assert req == 4 * per_tensor
    assert inter["roundtrip"] // req == g["ratio_to_required"]


def test_flop_count():
    # 4 N^2 d for d = dv, halved when causal.
    assert accounting.flops(1, 8192, 128, 128, False) == 4 * 8192 ** 2 * 128
    assert accounting.flops(64, 8192, 128, 128, True) == 64 * 2 * 8192 ** 2 * 128
    assert abs(accounting.flops(8, 4096, 64, 128, False) / 1e9 - 51.54) < 0.01
