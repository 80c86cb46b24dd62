"""The synthetic benchmark workloads at full size, launched exactly as bench.py launches
them (exact_tiled_attention_13_gb300.workload.DeviceWorkload), against the oracle on
sampled rows (the oracle computes rows one by one), plus properties that hold at any
size (every output written and finite)."""
import numpy as np
import pytest

import oracle
import synth
from gpu_helpers import compare, sample_rows

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("wid", sorted(synth.WORKLOADS))
def test_workload_sampled_parity(wid):
    import torch

    import exact_tiled_attention_13_gb300 as eta
    from exact_tiled_attention_13_gb300.workload import DeviceWorkload

    wl = DeviceWorkload(wid)
    w, c = wl.w, wl.host
    if w.backward:
        return _check_backward(wl)
    wl.O.fill_(float("nan"))
    wl.LSE.fill_(float("nan"))
    wl.launch()
    torch.cuda.synchronize()
    code, word = eta.attn_device_status(None)
    assert code == eta.ATTN_OK, f"device watchdog tripped: {word:#x}"
    O = wl.O.float().cpu().numpy().astype(np.float64)
    L = wl.LSE.cpu().numpy().astype(np.float64)
    assert np.isfinite(O).all() and np.isfinite(L).all(), "unwritten (NaN) or non-finite output"
    if w.BH * w.N <= 4096:
        rows = np.arange(w.BH * w.N, dtype=np.int64)
    else:
        heads = sorted({0, w.BH // 2, w.BH - 1})
        rows = sample_rows(w.BH, w.N, per_head_edge=48, stride=257, heads=heads)
    O_ref, L_ref, _ = oracle.attention_ex(c["Q"], c["K"], c["V"], w.mode, c["C"], c["ckey"],
                                          w.scale, rows=rows)
    stats = compare(O.reshape(-1, w.dv)[rows], L.reshape(-1)[rows], O_ref, L_ref,
                    out_bf16=w.out_dtype != "f32", label=w.name)
    print(w.name, len(rows), "rows", stats)


def _check_backward(wl):
    """Backward workloads: dQ on sampled rows and dK, dV on sampled keys of three heads
    against the oracle's gradients, at the tolerance of tests/test_gpu_bwd.py."""
    import torch

    import exact_tiled_attention_13_gb300 as eta
    from test_gpu_bwd import compare_grad

    w, c = wl.w, wl.host
    for t in (wl.dQ, wl.dK, wl.dV):
        t.fill_(float("nan"))
    wl.launch()
    torch.cuda.synchronize()
    code, word = eta.attn_device_status(None)
    assert code == eta.ATTN_OK, f"device watchdog tripped: {word:#x}"
    dQ, dK, dV = (t.cpu().numpy().astype(np.float64) for t in (wl.dQ, wl.dK, wl.dV))
    assert np.isfinite(dQ).all() and np.isfinite(dK).all() and np.isfinite(dV).all()
    heads = sorted({0, w.BH // 2, w.BH - 1})
    qr = np.unique(np.r_[np.arange(48), np.arange(w.N - 48, w.N), np.arange(7, w.N, 97)])
    kr = np.unique(np.r_[np.arange(48), np.arange(w.Nkv - 48, w.Nkv), np.arange(5, w.Nkv, 89)])
    rQ, rK, rV, _ = oracle.attention_bwd(c["Q"], c["K"], c["V"], c["dO"], w.mode, c["C"],
                                         c["ckey"], w.scale, heads=heads, qrows=qr, krows=kr)
    stats = {}
    for name, G, R, idx in (("dQ", dQ, rQ, qr), ("dK", dK, rK, kr), ("dV", dV, rV, kr)):
        stats[name] = compare_grad(G[heads][:, idx], R, f"{w.name} {name}")
    print(w.name, stats)
