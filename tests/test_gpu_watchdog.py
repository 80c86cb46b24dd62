"""Failure detection on the GPU without a fault: a wait is made to run out (the first K
tile is never copied), the kernel reports it in the watchdog word and returns, and the
context stays usable for the next, correct call."""
import numpy as np
import pytest

import oracle
import synth
from gpu_helpers import compare, run_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("mode", [synth.MODE_CAUSAL, synth.MODE_DENSE])
def test_wait_timeout_is_reported_and_context_survives(mode):
    import torch

    import exact_tiled_attention_13_gb300 as eta

    c = synth.random_case(77, 2, 384, 128 if mode != synth.MODE_DENSE else 64, 128, mode,
                          p_mask=0.3)
    Q = torch.from_numpy(c["Q"].view(np.int16)).cuda().view(torch.bfloat16)
    K = torch.from_numpy(c["K"].view(np.int16)).cuda().view(torch.bfloat16)
    V = torch.from_numpy(c["V"].view(np.int16)).cuda().view(torch.bfloat16)
    C = None if c["C"] is None else torch.from_numpy(c["C"]).cuda()
    O = torch.zeros(2, 384, 128, dtype=torch.float32, device="cuda")
    prev = eta.attn_set_wait_timeout_ns(50_000_000)  # 50 ms
    try:
        assert eta.attn_set_fault_injection(eta.ATTN_FAULT_SKIP_FIRST_K) == eta.ATTN_OK
        eta.attn_fwd(Q, K, V, mode, C, c["scale"], O)
        code, word = eta.attn_device_status(None)
        assert code == eta.ATTN_ERR_DEVICE_TIMEOUT
        assert word & 0x80000000
        # The MMA warp waits on the missing K tile, the softmax warps on the S tile that
        # never comes, the load warps on slots that are never released; whichever wait
        # runs out first records its role (1 softmax, 2 MMA, 3 Q/K/V load, 4 bias load)
        # and barrier index.
        role = (word >> 24) & 0xF
        assert role in (1, 2, 3, 4), f"unexpected role in watchdog word {word:#x}"
        assert ((word >> 8) & 0xFFFF) < 64
        # The word was cleared by the read.
        assert eta.attn_device_status(None) == (eta.ATTN_OK, 0)
    finally:
        eta.attn_set_fault_injection(eta.ATTN_FAULT_NONE)
        eta.attn_set_wait_timeout_ns(prev)
    # Same context, next call: correct results.
    O2, L2 = run_gpu(c, out_f32=True)
    O_ref, L_ref, _ = oracle.attention(c["Q"], c["K"], c["V"], mode, c["C"], c["scale"])
    compare(O2, L2, O_ref, L_ref)
