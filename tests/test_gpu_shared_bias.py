"""A dense bias shared by every head (ATTN_BIAS_SHARED): one fp32 [Nq, Nk] array C that
each head adds, S_h = scale Q_h K_h^T + C ("Compilers and kernels", section "FlashAttention
rewrites the algorithm around IO": C is any additive bias; the same C for all heads is the
broadcast form). Checked against the oracle with C written out for every head, and bit for
bit against the same call with a replicated [BH, Nq, Nk] C, which runs the same kernels."""
import numpy as np
import pytest

import oracle
import synth
from gpu_helpers import compare

pytestmark = pytest.mark.gpu

CAUSAL, DENSE = synth.MODE_CAUSAL, synth.MODE_DENSE

# (BH, Nq, Nk, d, dv, mode, out fp32?, p_mask)
CASES = [
    (3, 300, 300, 64, 128, DENSE, True, 0.3),        # bias through the TMA ring (Nk % 4 == 0)
    (2, 257, 301, 128, 128, DENSE, True, 0.2),       # bias read directly (Nk % 4 != 0)
    (2, 200, 333, 128, 64, CAUSAL | DENSE, False, 0.0),
    (4, 512, 512, 64, 64, CAUSAL | DENSE, True, 0.3),
]


def _id(c):
    BH, Nq, Nk, d, dv, mode, f32, pm = c
    return f"bh{BH}-nq{Nq}-nk{Nk}-d{d}-dv{dv}-{synth.MODE_NAMES[mode]}-{'f32' if f32 else 'bf16'}O"


def shared_case(seed, BH, Nq, Nk, d, dv, mode, p_mask):
    """A seeded case whose bias is head 0's, used by every head."""
    c = synth.random_case_ex(seed, BH, Nq, Nk, d, dv, mode, 1.0, p_mask)
    c["C_shared"] = np.ascontiguousarray(c["C"][0])
    c["C"] = np.ascontiguousarray(np.broadcast_to(c["C_shared"], (BH, Nq, Nk)))
    return c


def _bits(a):
    import torch

    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)


def _forward(c, C, mode, out_f32):
    import torch

    import exact_tiled_attention_13_gb300 as eta

    Q, K, V = _bits(c["Q"]), _bits(c["K"]), _bits(c["V"])
    BH, Nq, _ = Q.shape
    dv = V.shape[2]
    O = torch.full((BH, Nq, dv), float("nan"), device="cuda",
                   dtype=torch.float32 if out_f32 else torch.bfloat16)
    L = torch.full((BH, Nq), float("nan"), device="cuda")
    eta.attn_fwd_ex(Q, K, V, mode, torch.from_numpy(C).cuda(), None, c["scale"], O, L)
    torch.cuda.synchronize()
    code, word = eta.attn_device_status(None)
    assert code == eta.ATTN_OK, f"watchdog {word:#x}"
    return O.cpu(), L.cpu()


@pytest.mark.parametrize("case", CASES, ids=_id)
def test_shared_bias_forward(case):
    BH, Nq, Nk, d, dv, mode, out_f32, p_mask = case
    c = shared_case(9100 + Nq + Nk + mode, BH, Nq, Nk, d, dv, mode, p_mask)
    O, L = _forward(c, c["C_shared"], mode | synth.MODE_SHARED, out_f32)
    O_ref, L_ref, _ = oracle.attention_ex(c["Q"], c["K"], c["V"], mode, c["C"], None, c["scale"])
    compare(O.float().numpy().astype(np.float64), L.numpy().astype(np.float64), O_ref, L_ref,
            out_bf16=not out_f32, label=_id(case))
    # The same kernels with the bias written out for every head: identical bits.
    O2, L2 = _forward(c, c["C"], mode, out_f32)
    import torch

    as_int = torch.int32 if out_f32 else torch.int16
    assert torch.equal(O.view(as_int), O2.view(as_int))
    assert np.array_equal(L.numpy().view(np.int32), L2.numpy().view(np.int32))


def test_shared_bias_split_forward():
    import torch

    import exact_tiled_attention_13_gb300 as eta

    mode = CAUSAL | DENSE
    c = shared_case(9200, 2, 40, 2000, 128, 128, mode, 0.2)
    Q, K, V = _bits(c["Q"]), _bits(c["K"]), _bits(c["V"])
    O = torch.full((2, 40, 128), float("nan"), device="cuda")
    L = torch.full((2, 40), float("nan"), device="cuda")
    smode = mode | synth.MODE_SHARED
    ws = eta.splitkv_workspace(smode, 2, 40, 2000, 128, 128, 5)
    eta.attn_fwd_splitkv(Q, K, V, smode, torch.from_numpy(c["C_shared"]).cuda(), None, c["scale"], O, L,
                         workspace=ws, n_splits=5)
    torch.cuda.synchronize()
    O_ref, L_ref, _ = oracle.attention_ex(c["Q"], c["K"], c["V"], mode, c["C"], None, c["scale"])
    compare(O.cpu().numpy().astype(np.float64), L.cpu().numpy().astype(np.float64), O_ref, L_ref,
            label="split")


def test_shared_bias_backward():
    import torch

    import exact_tiled_attention_13_gb300 as eta
    from test_gpu_bwd import compare_grad

    mode = CAUSAL | DENSE
    c = shared_case(9300, 3, 250, 320, 128, 128, mode, 0.2)
    dO_bits = synth.bf16_tensor(9317, (3, 250, 128))
    Q, K, V, dO = _bits(c["Q"]), _bits(c["K"]), _bits(c["V"]), _bits(dO_bits)
    grads = {}
    for label, C, m in (("shared", c["C_shared"], mode | synth.MODE_SHARED), ("full", c["C"], mode)):
        Cd = torch.from_numpy(C).cuda()
        O = torch.empty(3, 250, 128, device="cuda")
        L = torch.empty(3, 250, device="cuda")
        eta.attn_fwd_ex(Q, K, V, m, Cd, None, c["scale"], O, L)
        g = [torch.full(t.shape, float("nan"), device="cuda") for t in (Q, K, V)]
        eta.attn_bwd(Q, K, V, O, dO, L, m, Cd, None, c["scale"], *g, eta.bwd_workspace(3, 250))
        torch.cuda.synchronize()
        grads[label] = [t.cpu().numpy() for t in g]
    refs = oracle.attention_bwd(c["Q"], c["K"], c["V"], dO_bits, mode, c["C"], None, c["scale"])[:3]
    for name, G, R in zip(("dQ", "dK", "dV"), grads["shared"], refs):
        compare_grad(G.astype(np.float64), R, f"shared bias {name}")
    for G, H in zip(grads["shared"], grads["full"]):
        assert np.array_equal(G.view(np.int32), H.view(np.int32))


def test_shared_bias_autograd():
    import torch

    import exact_tiled_attention_13_gb300 as eta

    c = shared_case(9400, 2, 192, 192, 64, 64, CAUSAL | DENSE, 0.0)
    q, k, v = (_bits(c[n]).requires_grad_() for n in ("Q", "K", "V"))
    bias2 = torch.from_numpy(c["C_shared"]).cuda()
    out = eta.attention(q, k, v, causal=True, bias=bias2)
    out.float().sum().backward()
    g = [t.grad.clone() for t in (q, k, v)]
    for t in (q, k, v):
        t.grad = None
    out2 = eta.attention(q, k, v, causal=True, bias=torch.from_numpy(c["C"]).cuda())
    out2.float().sum().backward()
    assert torch.equal(out, out2)
    for a, t in zip(g, (q, k, v)):
        assert torch.equal(a, t.grad)
