"""attn_fwd_host and attn_bwd_host on the GPU: host tensors streamed through a device
staging buffer in chunks of heads. Every head runs the same kernels as attn_fwd_ex and
attn_bwd, so the host outputs must equal theirs bit for bit; those calls themselves are
checked against the oracle elsewhere."""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

NONE, CAUSAL, DENSE, KEY = synth.MODE_NONE, synth.MODE_CAUSAL, synth.MODE_DENSE, synth.MODE_KEY

# (BH, Nq, Nk, d, dv, mode, out_f32, p_mask, heads_per_chunk, with_lse)
CASES = [
    (5, 300, 300, 128, 128, CAUSAL, False, 0.0, 2, True),   # ragged last chunk
    (3, 200, 333, 64, 128, DENSE, True, 0.3, 1, True),
    (4, 256, 512, 128, 64, KEY, True, 0.3, 0, True),
    (2, 129, 129, 64, 64, NONE, True, 0.0, 0, False),       # no LSE
    (9, 64, 1000, 128, 128, CAUSAL | KEY, False, 0.2, 4, True),
    (1, 400, 200, 64, 64, CAUSAL, True, 0.0, 0, True),      # rows with no allowed key
]


def _id(c):
    BH, Nq, Nk, d, dv, mode, f32, pm, hpc, lse = c
    return (f"bh{BH}-nq{Nq}-nk{Nk}-d{d}-dv{dv}-{synth.MODE_NAMES[mode]}-{'f32' if f32 else 'bf16'}"
            f"-h{hpc}{'' if lse else '-nolse'}")


def host_tensors(c, pin=True):
    import torch

    def bits(a):
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
        return t.pin_memory() if pin else t.clone()

    def f32(a):
        if a is None:
            return None
        t = torch.from_numpy(np.ascontiguousarray(a))
        return t.pin_memory() if pin else t.clone()

    return bits(c["Q"]), bits(c["K"]), bits(c["V"]), f32(c["C"]), f32(c["ckey"])


def run_both(c, out_f32, hpc, with_lse, pin=True):
    """(O, LSE) from attn_fwd_host and from attn_fwd_ex on the same data, as numpy arrays."""
    import torch

    import exact_tiled_attention_13_gb300 as eta

    Q, K, V, C, ck = host_tensors(c, pin)
    BH, Nq, d = Q.shape
    Nk, dv = K.shape[1], V.shape[2]
    odt = torch.float32 if out_f32 else torch.bfloat16
    O_h = torch.full((BH, Nq, dv), float("nan"), dtype=odt)
    L_h = torch.full((BH, Nq), float("nan")) if with_lse else None
    if pin:
        O_h = O_h.pin_memory()
        L_h = None if L_h is None else L_h.pin_memory()
    staging = eta.host_staging(c["mode"], BH, Nq, Nk, d, dv, 1 if out_f32 else 0, hpc)
    eta.attn_fwd_host(Q, K, V, c["mode"], C, ck, c["scale"], O_h, L_h, staging, hpc)
    torch.cuda.current_stream().synchronize()

    cuda = [None if t is None else t.cuda() for t in (Q, K, V, C, ck)]
    O_d = torch.empty((BH, Nq, dv), dtype=odt, device="cuda")
    L_d = torch.empty((BH, Nq), device="cuda") if with_lse else None
    eta.attn_fwd_ex(cuda[0], cuda[1], cuda[2], c["mode"], cuda[3], cuda[4], c["scale"], O_d, L_d)
    torch.cuda.synchronize()
    code, word = eta.attn_device_status(None)
    assert code == eta.ATTN_OK, f"watchdog {word:#x}"
    as_np = lambda t: None if t is None else t.float().cpu().numpy()
    return as_np(O_h), as_np(L_h), as_np(O_d), as_np(L_d)


@pytest.mark.parametrize("case", CASES, ids=_id)
def test_host_stream_equals_device_call(case):
    BH, Nq, Nk, d, dv, mode, f32, pm, hpc, lse = case
    c = synth.random_case_ex(9100 + BH + Nq + Nk, BH, Nq, Nk, d, dv, mode, 1.0, pm)
    O_h, L_h, O_d, L_d = run_both(c, f32, hpc, lse)
    assert np.array_equal(O_h, O_d, equal_nan=False), "O differs from attn_fwd_ex"
    if lse:
        assert np.array_equal(L_h, L_d), "LSE differs from attn_fwd_ex"


def test_pageable_host_memory_gives_the_same_result():
    c = synth.random_case_ex(9201, 3, 128, 256, 64, 64, CAUSAL, 1.0, 0.0)
    O_h, L_h, O_d, L_d = run_both(c, True, 1, True, pin=False)
    assert np.array_equal(O_h, O_d) and np.array_equal(L_h, L_d)


def test_consecutive_calls_share_staging_in_stream_order():
    import torch

    import exact_tiled_attention_13_gb300 as eta

    cases = [synth.random_case_ex(9300 + k, 6, 256, 256, 128, 128, CAUSAL, 1.0, 0.0) for k in range(2)]
    staging = eta.host_staging(CAUSAL, 6, 256, 256, 128, 128, 0, 2)
    outs = []
    for c in cases:
        Q, K, V, _, _ = host_tensors(c)
        O_h = torch.empty((6, 256, 128), dtype=torch.bfloat16).pin_memory()
        eta.attn_fwd_host(Q, K, V, CAUSAL, None, None, c["scale"], O_h, None, staging, 2)
        outs.append(O_h)
    torch.cuda.current_stream().synchronize()
    for c, O_h in zip(cases, outs):
        Q, K, V, _, _ = host_tensors(c)
        O_d = torch.empty((6, 256, 128), dtype=torch.bfloat16, device="cuda")
        eta.attn_fwd_ex(Q.cuda(), K.cuda(), V.cuda(), CAUSAL, None, None, c["scale"], O_d, None)
        torch.cuda.synchronize()
        assert torch.equal(O_h, O_d.cpu())


def test_device_pointer_where_host_belongs_is_rejected():
    import torch

    import exact_tiled_attention_13_gb300 as eta

    Qd = torch.zeros(1, 128, 64, dtype=torch.bfloat16, device="cuda")
    K = torch.zeros(1, 128, 64, dtype=torch.bfloat16).pin_memory()
    O = torch.zeros(1, 128, 64).pin_memory()
    staging = eta.host_staging(0, 1, 128, 128, 64, 64, 1)
    code = eta.attn_fwd_host_raw(Qd.data_ptr(), K.data_ptr(), K.data_ptr(), 0, None, None, 1, 128, 128,
                                 64, 64, 0.125, O.data_ptr(), 1, None, staging.data_ptr(),
                                 staging.numel(), 0, torch.cuda.current_stream().cuda_stream)
    assert code == eta.ATTN_ERR_INVALID_ARG


# (BH, Nq, Nk, d, dv, mode, o_f32, p_mask, heads_per_chunk)
BWD_CASES = [
    (5, 256, 256, 128, 128, CAUSAL, False, 0.0, 2),
    (3, 200, 333, 64, 128, CAUSAL | DENSE, True, 0.2, 1),
    (4, 130, 257, 128, 64, KEY, True, 0.3, 0),
    (2, 333, 200, 64, 64, CAUSAL, True, 0.0, 1),   # rows with no allowed key
]


@pytest.mark.parametrize("case", BWD_CASES, ids=lambda c: f"bh{c[0]}-nq{c[1]}-nk{c[2]}-d{c[3]}-dv{c[4]}-"
                         f"{synth.MODE_NAMES[c[5]]}-h{c[8]}")
def test_bwd_host_stream_equals_device_call(case):
    import torch

    import exact_tiled_attention_13_gb300 as eta

    BH, Nq, Nk, d, dv, mode, o_f32, pm, hpc = case
    c = synth.random_case_ex(9400 + BH + Nq + Nk, BH, Nq, Nk, d, dv, mode, 1.0, pm)
    Q, K, V, C, ck = host_tensors(c)
    dO = torch.from_numpy(synth.bf16_tensor(9500 + Nq, (BH, Nq, dv)).view(np.int16)).view(torch.bfloat16).pin_memory()
    cuda = lambda t: None if t is None else t.cuda()
    # Forward on the device for O and LSE.
    odt = torch.float32 if o_f32 else torch.bfloat16
    O_d = torch.empty((BH, Nq, dv), dtype=odt, device="cuda")
    L_d = torch.empty((BH, Nq), device="cuda")
    eta.attn_fwd_ex(cuda(Q), cuda(K), cuda(V), mode, cuda(C), cuda(ck), c["scale"], O_d, L_d)
    O_h, L_h = O_d.cpu().pin_memory(), L_d.cpu().pin_memory()
    grads_h = [torch.full(s, float("nan")).pin_memory() for s in ((BH, Nq, d), (BH, Nk, d), (BH, Nk, dv))]
    staging = eta.bwd_host_staging(mode, BH, Nq, Nk, d, dv, 1 if o_f32 else 0, hpc)
    eta.attn_bwd_host(Q, K, V, O_h, dO, L_h, mode, C, ck, c["scale"], *grads_h, staging, hpc)
    torch.cuda.current_stream().synchronize()
    grads_d = [torch.empty(g.shape, device="cuda") for g in grads_h]
    ws = eta.bwd_workspace(BH, Nq)
    eta.attn_bwd(cuda(Q), cuda(K), cuda(V), O_d, cuda(dO), L_d, mode, cuda(C), cuda(ck), c["scale"], *grads_d, ws)
    torch.cuda.synchronize()
    code, word = eta.attn_device_status(None)
    assert code == eta.ATTN_OK, f"watchdog {word:#x}"
    for name, gh, gd in zip(("dQ", "dK", "dV"), grads_h, grads_d):
        assert torch.equal(gh, gd.cpu()), f"{name} differs from attn_bwd"
