"""attn_fwd_ex on the GPU against the oracle: queries and keys of their own lengths,
the causal mask aligned at the last key (both signs of Nk - Nq), the per-key bias
vector (aligned and ragged), and the causal mask combined with a bias."""
import numpy as np
import pytest

import oracle
import synth
from gpu_helpers import compare

pytestmark = pytest.mark.gpu

NONE, CAUSAL, DENSE, KEY = synth.MODE_NONE, synth.MODE_CAUSAL, synth.MODE_DENSE, synth.MODE_KEY

# (BH, Nq, Nk, d, dv, mode, out_f32, p_mask)
CASES = [
    (2, 100, 300, 64, 64, CAUSAL, True, 0.0),
    (1, 300, 100, 128, 128, CAUSAL, True, 0.0),
    (2, 256, 640, 128, 128, CAUSAL, False, 0.0),
    (1, 1, 1000, 128, 128, NONE, True, 0.0),
    (3, 1, 700, 64, 128, CAUSAL, True, 0.0),
    (1, 7, 513, 64, 128, CAUSAL | KEY, True, 0.3),
    (2, 384, 384, 128, 128, KEY, True, 0.3),
    (1, 129, 257, 64, 64, KEY, False, 0.5),
    (1, 200, 200, 64, 128, CAUSAL | DENSE, True, 0.3),
    (1, 130, 131, 128, 64, CAUSAL | DENSE, True, 0.2),
    (2, 512, 256, 128, 128, NONE, True, 0.0),
    (1, 1000, 2000, 128, 128, CAUSAL | KEY, False, 0.3),
    (1, 640, 384, 64, 64, CAUSAL | KEY, True, 0.2),
    # Dense bias with 128 value columns (Nk % 4 == 0): the CTA-pair kernel's bias rings,
    # ragged query and key tails, Nq != Nk with the causal offset, several units per pair.
    (2, 300, 520, 128, 128, DENSE, False, 0.3),
    (1, 96, 1024, 64, 128, CAUSAL | DENSE, True, 0.3),
    (3, 1000, 1000, 128, 128, DENSE, True, 0.1),
    (2, 777, 388, 64, 128, CAUSAL | DENSE, False, 0.3),
    # No bias, 128 value columns (the CTA-pair kernel): causal with Nq > Nk (units whose rows
    # see no key), unmasked with ragged query and key tails, d = 64.
    (2, 900, 300, 128, 128, CAUSAL, False, 0.0),
    (1, 513, 1000, 64, 128, NONE, True, 0.0),
    (3, 130, 1030, 128, 128, NONE, False, 0.0),
    # Per-key bias at d = 64 with 128 value columns (the CTA-pair kernel, bias folded into the
    # score product): ragged tails, Nk not a multiple of 4, causal with Nq > Nk, heavy padding.
    (2, 300, 520, 64, 128, KEY, False, 0.3),
    (1, 1000, 1000, 64, 128, CAUSAL | KEY, True, 0.3),
    (3, 130, 1030, 64, 128, KEY, True, 0.0),
    (2, 900, 300, 64, 128, CAUSAL | KEY, False, 0.2),
    (1, 600, 2048, 64, 128, KEY, True, 0.9),
]


def _id(c):
    BH, Nq, Nk, d, dv, mode, f32, pm = c
    return f"bh{BH}-nq{Nq}-nk{Nk}-d{d}-dv{dv}-{synth.MODE_NAMES[mode]}-{'f32' if f32 else 'bf16'}"


def run_ex(c, out_f32=True):
    import torch

    import exact_tiled_attention_13_gb300 as eta

    def dev_bits(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)

    Q, K, V = dev_bits(c["Q"]), dev_bits(c["K"]), dev_bits(c["V"])
    C = None if c["C"] is None else torch.from_numpy(c["C"]).cuda()
    ck = None if c["ckey"] is None else torch.from_numpy(c["ckey"]).cuda()
    BH, Nq = Q.shape[:2]
    dv = V.shape[2]
    O = torch.full((BH, Nq, dv), float("nan"), device="cuda",
                   dtype=torch.float32 if out_f32 else torch.bfloat16)
    L = torch.full((BH, Nq), float("nan"), device="cuda", dtype=torch.float32)
    eta.attn_fwd_ex(Q, K, V, c["mode"], C, ck, c["scale"], O, L)
    torch.cuda.synchronize()
    code, word = eta.attn_device_status(None)
    assert code == eta.ATTN_OK, f"watchdog {word:#x}"
    return O.float().cpu().numpy().astype(np.float64), L.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("case", CASES, ids=_id)
def test_ex_parity(case):
    BH, Nq, Nk, d, dv, mode, out_f32, p_mask = case
    c = synth.random_case_ex(3000 + Nq + Nk + mode, BH, Nq, Nk, d, dv, mode, 1.0, p_mask)
    O, L = run_ex(c, out_f32)
    O_ref, L_ref, _ = oracle.attention_ex(c["Q"], c["K"], c["V"], mode, c["C"], c["ckey"],
                                          c["scale"])
    compare(O, L, O_ref, L_ref, out_bf16=not out_f32, label=_id(case))


def test_square_ex_matches_attn_fwd_bitwise():
    import torch

    import exact_tiled_attention_13_gb300 as eta
    from gpu_helpers import device_inputs

    c = synth.random_case(31, 2, 500, 128, 128, CAUSAL)
    Q, K, V, _ = device_inputs(c)
    O1 = torch.empty(2, 500, 128, device="cuda")
    O2 = torch.empty(2, 500, 128, device="cuda")
    eta.attn_fwd(Q, K, V, CAUSAL, None, c["scale"], O1)
    eta.attn_fwd_ex(Q, K, V, CAUSAL, None, None, c["scale"], O2)
    torch.cuda.synchronize()
    assert torch.equal(O1, O2)


def test_key_bias_heads_with_no_allowed_key():
    """Every key of head 0 padded out (-inf): its rows get O = 0 and LSE = -inf; head 1,
    padded except for its last key, attends to that key alone. At d = 64 with 128 value
    columns the bias enters the score product as 1 x (-inf) (never 0 x inf)."""
    for d, dv in ((64, 128), (64, 64), (128, 128)):
        c = synth.random_case_ex(4242 + d + dv, 3, 300, 700, d, dv, KEY, 1.0, 0.0)
        c["ckey"][0, :] = -np.inf
        c["ckey"][1, :-1] = -np.inf
        O, L = run_ex(c, True)
        O_ref, L_ref, _ = oracle.attention_ex(c["Q"], c["K"], c["V"], KEY, None, c["ckey"],
                                              c["scale"])
        assert np.all(O[0] == 0.0) and np.all(L[0] == -np.inf)
        compare(O, L, O_ref, L_ref, label=f"padded heads d{d} dv{dv}")


@pytest.mark.parametrize("BH,Nq,Nk,mode", [(1, 1, 700, KEY), (5, 64, 256, CAUSAL | KEY)],
                         ids=["one-query", "causal-short"])
def test_key_bias_pair_without_lse(BH, Nq, Nk, mode):
    """Per-key bias on the CTA-pair path (d = 64, d_v = 128) with LSE = NULL: O alone is
    written, and it equals the oracle's."""
    import torch

    import exact_tiled_attention_13_gb300 as eta

    c = synth.random_case_ex(4700 + Nq + Nk, BH, Nq, Nk, 64, 128, mode, 1.0, 0.3)

    def bits(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)

    O = torch.full((BH, Nq, 128), float("nan"), device="cuda")
    eta.attn_fwd_ex(bits(c["Q"]), bits(c["K"]), bits(c["V"]), mode, None,
                    torch.from_numpy(c["ckey"]).cuda(), c["scale"], O, None)
    torch.cuda.synchronize()
    code, word = eta.attn_device_status(None)
    assert code == eta.ATTN_OK, f"watchdog {word:#x}"
    O_ref, L_ref, _ = oracle.attention_ex(c["Q"], c["K"], c["V"], mode, None, c["ckey"], c["scale"])
    compare(O.cpu().numpy().astype(np.float64), L_ref, O_ref, L_ref, label=f"no LSE {BH}x{Nq}x{Nk}")
