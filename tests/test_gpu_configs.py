"""The synthetic benchmark workloads at full size, launched exactly as bench.py
launches them, against the oracle on sampled rows (the oracle computes rows one by
one), plus properties that hold at any size (every output written and finite)."""
import numpy as np
import pytest

import oracle
import synth
from gpu_helpers import compare, run_gpu, sample_rows

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("wid", sorted(synth.WORKLOADS))
def test_workload_sampled_parity(wid):
    w = synth.WORKLOADS[wid]
    c = synth.make_inputs(w, wid)
    out_f32 = w.out_dtype == "f32"
    O, L = run_gpu(c, out_f32=out_f32)
    assert np.isfinite(O).all() and np.isfinite(L).all(), "unwritten (NaN) or non-finite output"
    if w.BH * w.N <= 4096:
        rows = np.arange(w.BH * w.N, dtype=np.int64)
    else:
        heads = sorted({0, w.BH // 2, w.BH - 1})
        rows = sample_rows(w.BH, w.N, per_head_edge=48, stride=257, heads=heads)
    O_ref, L_ref, _ = oracle.attention_ex(c["Q"], c["K"], c["V"], w.mode, c["C"], c["ckey"],
                                          w.scale, rows=rows)
    stats = compare(O.reshape(-1, w.dv)[rows], L.reshape(-1)[rows], O_ref, L_ref,
                    out_bf16=not out_f32, label=w.name)
    print(w.name, len(rows), "rows", stats)
