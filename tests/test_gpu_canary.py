"""Writes stay inside the output buffers, and exact ties in the scores.

Each output (O, LSE, the split workspace, dQ, dK, dV) is placed inside a larger buffer
whose margins hold a sentinel; after the call the margins must be untouched and the
inside fully written. Ties: keys repeated so several keys share a row's maximum score,
and Q = 0 so every allowed key ties.
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_helpers import compare, device_inputs

pytestmark = pytest.mark.gpu

PAD = 64  # sentinel elements on each side (256 bytes for fp32, 128 for bf16)


def guarded(shape, dtype, sentinel):
    """A tensor of `shape` inside a sentinel-filled buffer; returns (inner view, buffer)."""
    import torch

    n = int(np.prod(shape))
    buf = torch.full((n + 2 * PAD,), sentinel, dtype=dtype, device="cuda")
    return buf[PAD:PAD + n].view(*shape), buf


def margins_intact(buf, sentinel):
    import torch

    head, tail = buf[:PAD], buf[-PAD:]
    ref = torch.full_like(head, sentinel)
    return torch.equal(head, ref) and torch.equal(tail, ref)


@pytest.mark.parametrize("out_f32", [True, False])
def test_forward_writes_stay_inside(out_f32):
    import torch

    import exact_tiled_attention_13_gb300 as eta

    BH, Nq, Nk, d, dv = 3, 333, 517, 128, 64
    c = synth.random_case_ex(901, BH, Nq, Nk, d, dv, synth.MODE_CAUSAL)
    Q, K, V, _ = device_inputs(c)
    dt = torch.float32 if out_f32 else torch.bfloat16
    sentinel = 12345.0
    O, obuf = guarded((BH, Nq, dv), dt, sentinel)
    L, lbuf = guarded((BH, Nq), torch.float32, sentinel)
    eta.attn_fwd_ex(Q, K, V, synth.MODE_CAUSAL, None, None, c["scale"], O, L)
    torch.cuda.synchronize()
    assert margins_intact(obuf, sentinel) and margins_intact(lbuf, sentinel)
    assert not (O.float() == sentinel).any() and not (L == sentinel).any(), "unwritten outputs"


def test_split_forward_writes_stay_inside():
    import torch

    import exact_tiled_attention_13_gb300 as eta

    BH, Nq, Nk, d, dv = 2, 70, 1500, 64, 128
    c = synth.random_case_ex(902, BH, Nq, Nk, d, dv, synth.MODE_CAUSAL)
    Q, K, V, _ = device_inputs(c)
    code, splits, nbytes = eta.attn_fwd_splitkv_plan(synth.MODE_CAUSAL, BH, Nq, Nk, d, dv, 6)
    assert code == eta.ATTN_OK and splits > 1
    sentinel = 7.0
    ws, wbuf = guarded((nbytes // 4,), torch.float32, sentinel)
    O, obuf = guarded((BH, Nq, dv), torch.float32, sentinel)
    L, lbuf = guarded((BH, Nq), torch.float32, sentinel)
    eta.attn_fwd_splitkv(Q, K, V, synth.MODE_CAUSAL, None, None, c["scale"], O, L, workspace=ws,
                         n_splits=6)
    torch.cuda.synchronize()
    for buf in (wbuf, obuf, lbuf):
        assert margins_intact(buf, sentinel)
    O_ref, L_ref, _ = oracle.attention_ex(c["Q"], c["K"], c["V"], synth.MODE_CAUSAL, None, None,
                                          c["scale"])
    compare(O.cpu().numpy().astype(np.float64), L.cpu().numpy().astype(np.float64), O_ref, L_ref,
            label="split in guarded buffers")


def test_backward_writes_stay_inside():
    import torch

    import exact_tiled_attention_13_gb300 as eta

    BH, Nq, Nk, d, dv = 2, 200, 333, 64, 128
    c = synth.random_case_ex(903, BH, Nq, Nk, d, dv, synth.MODE_CAUSAL)
    Q, K, V, _ = device_inputs(c)
    dO = torch.randn(BH, Nq, dv, device="cuda").to(torch.bfloat16)
    O = torch.empty(BH, Nq, dv, device="cuda")
    L = torch.empty(BH, Nq, device="cuda")
    eta.attn_fwd_ex(Q, K, V, synth.MODE_CAUSAL, None, None, c["scale"], O, L)
    sentinel = -3.5
    dQ, qbuf = guarded((BH, Nq, d), torch.float32, sentinel)
    dK, kbuf = guarded((BH, Nk, d), torch.float32, sentinel)
    dV, vbuf = guarded((BH, Nk, dv), torch.float32, sentinel)
    code, nbytes = eta.attn_bwd_workspace_bytes(BH, Nq)
    ws, wbuf = guarded((nbytes // 4,), torch.float32, sentinel)
    eta.attn_bwd(Q, K, V, O, dO, L, synth.MODE_CAUSAL, None, None, c["scale"], dQ, dK, dV, ws)
    torch.cuda.synchronize()
    for buf in (qbuf, kbuf, vbuf, wbuf):
        assert margins_intact(buf, sentinel)
    for t in (dQ, dK, dV):
        assert torch.isfinite(t).all() and not (t == sentinel).any()


def test_exact_ties_in_scores():
    """Keys repeated in groups of four: a row's maximum is shared by (at least) four keys.
    With Q = 0 every allowed key ties, and O_i is the mean of the allowed values."""
    import torch

    import exact_tiled_attention_13_gb300 as eta

    BH, N, d, dv = 2, 300, 64, 64
    c = synth.random_case(904, BH, N, d, dv, synth.MODE_CAUSAL)
    K = c["K"].copy()
    K[:, 1::4] = K[:, 0::4][:, :K[:, 1::4].shape[1]]
    K[:, 2::4] = K[:, 0::4][:, :K[:, 2::4].shape[1]]
    K[:, 3::4] = K[:, 0::4][:, :K[:, 3::4].shape[1]]
    for Qbits in (c["Q"], np.zeros_like(c["Q"])):
        case = dict(c, K=K, Q=Qbits)
        Q, Kd, V, _ = device_inputs(case)
        O = torch.empty(BH, N, dv, device="cuda")
        L = torch.empty(BH, N, device="cuda")
        eta.attn_fwd(Q, Kd, V, synth.MODE_CAUSAL, None, c["scale"], O, L)
        torch.cuda.synchronize()
        O_ref, L_ref, _ = oracle.attention(Qbits, K, c["V"], synth.MODE_CAUSAL, None, c["scale"])
        compare(O.cpu().numpy().astype(np.float64), L.cpu().numpy().astype(np.float64), O_ref,
                L_ref, label="ties")
