"""attn_bwd on the GPU against the oracle's gradients.

The forward pass (attn_fwd_ex) produces O and LSE on the GPU; attn_bwd turns them and a
seeded dO into dQ, dK, dV, which are compared with the fp64 oracle (the chain rule on
the definition, S and P recomputed from the inputs).

Tolerance, per gradient tensor G against the oracle's G_ref:
    ||G - G_ref||_F <= 1e-2 ||G_ref||_F   and   max |G - G_ref| <= 2e-2 max |G_ref|.
The kernels round P and dS to bf16 before the tensor-core products (relative 2^-9, about
2e-3 per element, independent from element to element, so the normwise error of each
sum stays near 2e-3) and take D_i = dO_i . O_i from the stored forward output; the
bounds leave a margin of about five over that, while a wrong mask, scale, transpose or a
dropped D changes the gradients by tens of percent or more.
"""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu

NONE, CAUSAL, DENSE, KEY = synth.MODE_NONE, synth.MODE_CAUSAL, synth.MODE_DENSE, synth.MODE_KEY
REL_FRO = 1e-2
REL_MAX = 2e-2

# (BH, Nq, Nk, d, dv, mode, O dtype fp32?, p_mask)
CASES = [
    (2, 256, 256, 128, 128, NONE, True, 0.0),
    (1, 300, 300, 64, 64, CAUSAL, False, 0.0),
    (2, 200, 333, 128, 64, CAUSAL, True, 0.0),
    (1, 333, 200, 64, 128, CAUSAL, True, 0.0),
    (2, 256, 384, 64, 128, KEY, True, 0.3),
    (1, 130, 257, 128, 128, CAUSAL | KEY, False, 0.2),
    (1, 192, 192, 64, 64, DENSE, True, 0.3),
    (1, 255, 260, 128, 128, CAUSAL | DENSE, True, 0.2),
    (1, 1, 129, 64, 64, NONE, True, 0.0),
    (1, 1024, 1024, 128, 128, CAUSAL, False, 0.0),
    (3, 77, 1000, 128, 128, NONE, True, 0.0),
]


def _id(c):
    BH, Nq, Nk, d, dv, mode, f32, pm = c
    return f"bh{BH}-nq{Nq}-nk{Nk}-d{d}-dv{dv}-{synth.MODE_NAMES[mode]}-{'f32' if f32 else 'bf16'}O"


def bwd_case(seed, BH, Nq, Nk, d, dv, mode, p_mask):
    c = synth.random_case_ex(seed, BH, Nq, Nk, d, dv, mode, 1.0, p_mask)
    c["dO"] = synth.bf16_tensor(seed + 17, (BH, Nq, dv))
    return c


def run_gpu_bwd(c, o_f32=True):
    """Forward then backward on the GPU; returns (dQ, dK, dV) as fp64 numpy arrays."""
    import torch

    import exact_tiled_attention_13_gb300 as eta

    def bits(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)

    Q, K, V, dO = bits(c["Q"]), bits(c["K"]), bits(c["V"]), bits(c["dO"])
    C = None if c["C"] is None else torch.from_numpy(c["C"]).cuda()
    ck = None if c["ckey"] is None else torch.from_numpy(c["ckey"]).cuda()
    BH, Nq, d = Q.shape
    Nk, dv = K.shape[1], V.shape[2]
    O = torch.empty(BH, Nq, dv, device="cuda", dtype=torch.float32 if o_f32 else torch.bfloat16)
    L = torch.empty(BH, Nq, device="cuda")
    eta.attn_fwd_ex(Q, K, V, c["mode"], C, ck, c["scale"], O, L)
    nan = float("nan")
    dQ = torch.full((BH, Nq, d), nan, device="cuda")
    dK = torch.full((BH, Nk, d), nan, device="cuda")
    dV = torch.full((BH, Nk, dv), nan, device="cuda")
    ws = eta.bwd_workspace(BH, Nq)
    eta.attn_bwd(Q, K, V, O, dO, L, c["mode"], C, ck, c["scale"], dQ, dK, dV, ws)
    torch.cuda.synchronize()
    code, word = eta.attn_device_status(None)
    assert code == eta.ATTN_OK, f"watchdog {word:#x}"
    return tuple(t.cpu().numpy().astype(np.float64) for t in (dQ, dK, dV))


def compare_grad(G, G_ref, label):
    assert G.shape == G_ref.shape, (G.shape, G_ref.shape)
    assert np.isfinite(G).all(), f"{label}: non-finite or unwritten entries"
    err = G - G_ref
    ref_fro = np.linalg.norm(G_ref)
    ref_max = np.abs(G_ref).max()
    if ref_max == 0.0:
        assert np.abs(G).max() <= 1e-6, f"{label}: expected zeros"
        return {}
    rel_fro = np.linalg.norm(err) / ref_fro
    rel_max = np.abs(err).max() / ref_max
    assert rel_fro <= REL_FRO, f"{label}: normwise relative error {rel_fro:.3e}"
    assert rel_max <= REL_MAX, (f"{label}: max error {rel_max:.3e} of max |G| at "
                                f"{np.unravel_index(np.abs(err).argmax(), err.shape)}")
    return {"rel_fro": rel_fro, "rel_max": rel_max}


@pytest.mark.parametrize("case", CASES, ids=_id)
def test_bwd_parity(case):
    BH, Nq, Nk, d, dv, mode, o_f32, p_mask = case
    c = bwd_case(7000 + Nq + 3 * Nk + mode, BH, Nq, Nk, d, dv, mode, p_mask)
    dQ, dK, dV = run_gpu_bwd(c, o_f32)
    rQ, rK, rV, _ = oracle.attention_bwd(c["Q"], c["K"], c["V"], c["dO"], mode, c["C"], c["ckey"],
                                         c["scale"])
    stats = {name: compare_grad(G, R, f"{_id(case)} {name}")
             for name, G, R in (("dQ", dQ, rQ), ("dK", dK, rK), ("dV", dV, rV))}
    print(_id(case), stats)


def test_bwd_is_deterministic():
    c = bwd_case(8001, 2, 500, 700, 128, 128, CAUSAL, 0.0)
    a = run_gpu_bwd(c)
    b = run_gpu_bwd(c)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_bwd_no_queries_zeroes_key_gradients():
    import torch

    import exact_tiled_attention_13_gb300 as eta
    from exact_tiled_attention_13_gb300 import _lib

    K = torch.randn(2, 300, 64, device="cuda").to(torch.bfloat16)
    V = torch.randn(2, 300, 64, device="cuda").to(torch.bfloat16)
    dK = torch.full((2, 300, 64), 7.0, device="cuda")
    dV = torch.full((2, 300, 64), 7.0, device="cuda")
    code = _lib.attn_bwd_raw(None, K.data_ptr(), V.data_ptr(), None, 1, None, None, 0, None, None,
                             2, 0, 300, 64, 64, 0.125, None, dK.data_ptr(), dV.data_ptr(), None, 0,
                             torch.cuda.current_stream().cuda_stream)
    assert code == eta.ATTN_OK
    torch.cuda.synchronize()
    assert dK.abs().max().item() == 0.0 and dV.abs().max().item() == 0.0
