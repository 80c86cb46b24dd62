"""attention(): autograd through attn_fwd_ex and attn_bwd. The forward output and the
gradients must equal those of the C-ABI calls on the same data (the same kernels), and
the gradients must be close to the fp64 oracle's."""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("causal,key", [(True, False), (False, True)])
def test_attention_autograd_matches_the_c_abi_and_the_oracle(causal, key):
    import torch

    import exact_tiled_attention_13_gb300 as eta

    mode = (synth.MODE_CAUSAL if causal else 0) | (synth.MODE_KEY if key else 0)
    c = synth.random_case_ex(9600 + mode, 3, 200, 300, 64, 128, mode, 1.0, 0.2 if key else 0.0)
    bits = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)
    q, k, v = (bits(c[n]).requires_grad_(True) for n in ("Q", "K", "V"))
    ck = None if c["ckey"] is None else torch.from_numpy(c["ckey"]).cuda()
    dO_np = synth.bf16_tensor(9700 + mode, (3, 200, 128))
    dO = bits(dO_np)

    O = eta.attention(q, k, v, causal=causal, key_bias=ck, scale=c["scale"])
    O.backward(dO)
    torch.cuda.synchronize()

    # The same through the C ABI.
    O2 = torch.empty((3, 200, 128), dtype=torch.bfloat16, device="cuda")
    L2 = torch.empty((3, 200), device="cuda")
    eta.attn_fwd_ex(q.detach(), k.detach(), v.detach(), mode, None, ck, c["scale"], O2, L2)
    grads = [torch.empty(t.shape, device="cuda") for t in (q, k, v)]
    eta.attn_bwd(q.detach(), k.detach(), v.detach(), O2, dO, L2, mode, None, ck, c["scale"], *grads,
                 eta.bwd_workspace(3, 200))
    torch.cuda.synchronize()
    assert torch.equal(O, O2)
    for g_auto, g_abi in zip((q.grad, k.grad, v.grad), grads):
        assert torch.equal(g_auto, g_abi.to(torch.bfloat16))

    # And near the oracle's gradients (bf16-rounded fp32 gradients: relative 2^-8 more).
    refs = oracle.attention_bwd(c["Q"], c["K"], c["V"], dO_np, mode, None, c["ckey"], c["scale"])
    for g, ref in zip((q.grad, k.grad, v.grad), refs[:3]):
        g = g.float().cpu().numpy().astype(np.float64)
        assert np.linalg.norm(g - ref) <= 1.5e-2 * np.linalg.norm(ref)
