"""Shared helpers of the GPU tests: move seeded inputs to the device, run the CUDA path
through the C ABI, and compare with the oracle at the stated tolerances.

Tolerances (fp32 output): max |O - O_ref| <= 1e-2, mean |O - O_ref| <= 1e-3,
max |LSE - LSE_ref| <= 1e-3. For bf16 output the rounding of O itself adds up to half
a bf16 ulp, 2^-9 |O_ref|, to each element bound and to the mean bound.
"""
from __future__ import annotations

import numpy as np

TOL_MAX = 1e-2
TOL_MEAN = 1e-3
TOL_LSE = 1e-3
BF16_HALF_ULP = 2.0 ** -9


def torch_mod():
    import torch

    return torch


def bf16_device(bits, device="cuda"):
    torch = torch_mod()
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.to(device).view(torch.bfloat16)


def device_inputs(case, device="cuda"):
    torch = torch_mod()
    Q = bf16_device(case["Q"], device)
    K = bf16_device(case["K"], device)
    V = bf16_device(case["V"], device)
    C = None if case["C"] is None else torch.from_numpy(np.ascontiguousarray(case["C"])).to(device)
    return Q, K, V, C


def run_gpu(case, out_f32=True, stream=None, with_lse=True, fill=float("nan"), dev_inputs=None):
    """Runs the CUDA path; returns (O, LSE) as fp64 numpy arrays (LSE None if skipped)."""
    import exact_tiled_attention_13_gb300 as eta

    torch = torch_mod()
    Q, K, V, C = dev_inputs if dev_inputs is not None else device_inputs(case)
    BH, N, _ = Q.shape
    dv = V.shape[2]
    O = torch.full((BH, N, dv), fill, dtype=torch.float32 if out_f32 else torch.bfloat16,
                   device=Q.device)
    LSE = torch.full((BH, N), fill, dtype=torch.float32, device=Q.device) if with_lse else None
    if case.get("ckey") is None:
        eta.attn_fwd(Q, K, V, case["mode"], C, case["scale"], O, LSE, stream=stream)
    else:
        ckey = torch.from_numpy(np.ascontiguousarray(case["ckey"])).to(Q.device)
        eta.attn_fwd_ex(Q, K, V, case["mode"], C, ckey, case["scale"], O, LSE, stream=stream)
    torch.cuda.synchronize()
    code, word = eta.attn_device_status(None)
    assert code == eta.ATTN_OK, f"device watchdog tripped: {word:#x}"
    O_np = O.float().cpu().numpy().astype(np.float64)
    L_np = LSE.cpu().numpy().astype(np.float64) if with_lse else None
    return O_np, L_np


def compare(O, L, O_ref, L_ref, out_bf16=False, label=""):
    """Asserts the tolerances; returns the error statistics."""
    assert O.shape == O_ref.shape, (O.shape, O_ref.shape)
    assert np.isfinite(O).all(), f"{label}: non-finite O"
    err = np.abs(O - O_ref)
    slack = BF16_HALF_ULP * np.abs(O_ref) if out_bf16 else 0.0
    stats = {"max_abs_O": float(err.max()) if err.size else 0.0,
             "mean_abs_O": float(err.mean()) if err.size else 0.0}
    assert np.all(err <= TOL_MAX + slack), (
        f"{label}: max |dO| {stats['max_abs_O']:.3e} at {np.unravel_index(err.argmax(), err.shape)}")
    mean_bound = TOL_MEAN + (float(np.mean(slack)) if out_bf16 else 0.0)
    assert stats["mean_abs_O"] <= mean_bound, f"{label}: mean |dO| {stats['mean_abs_O']:.3e}"
    if L is not None:
        fin = np.isfinite(L_ref)
        assert np.array_equal(np.isfinite(L), fin), f"{label}: LSE finiteness differs"
        assert np.array_equal(L[~fin], L_ref[~fin]), f"{label}: LSE infinities differ"
        lerr = np.abs(L[fin] - L_ref[fin])
        stats["max_abs_LSE"] = float(lerr.max()) if lerr.size else 0.0
        assert stats["max_abs_LSE"] <= TOL_LSE, f"{label}: max |dLSE| {stats['max_abs_LSE']:.3e}"
    return stats


def sample_rows(BH, N, per_head_edge=64, stride=97, heads=None):
    """Flat row ids: the first and last rows of selected heads plus a strided sweep."""
    heads = range(BH) if heads is None else heads
    rows = []
    for bh in heads:
        base = bh * N
        rows.extend(range(base, base + min(per_head_edge, N)))
        rows.extend(range(base + max(0, N - per_head_edge), base + N))
        rows.extend(range(base + (bh * 13) % stride, base + N, stride))
    return np.unique(np.array(rows, dtype=np.int64))
