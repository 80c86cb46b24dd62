"""attn_fwd_splitkv on the GPU: each head's keys cut into ranges of whole tiles run as
separate blocks, then merged. The result is the same function, so it is compared with
the oracle's plain definition; the partials themselves are internal."""
import numpy as np
import pytest

import oracle
import synth
from gpu_helpers import TOL_MAX, compare

pytestmark = pytest.mark.gpu

NONE, CAUSAL, DENSE, KEY = synth.MODE_NONE, synth.MODE_CAUSAL, synth.MODE_DENSE, synth.MODE_KEY

# (BH, Nq, Nk, d, dv, mode, out_f32, p_mask, n_splits)   n_splits 0: the library's choice
CASES = [
    (1, 1, 4096, 128, 128, NONE, True, 0.0, 0),
    (2, 64, 3000, 64, 128, CAUSAL, False, 0.0, 5),
    (4, 128, 2048, 128, 64, KEY, True, 0.3, 7),
    (1, 200, 1500, 64, 64, CAUSAL | DENSE, True, 0.3, 3),
    (1, 300, 1000, 128, 128, CAUSAL, True, 0.0, 4),
    (1, 1000, 500, 128, 128, CAUSAL, True, 0.0, 3),
    (3, 17, 129, 128, 128, NONE, True, 0.0, 2),
    (2, 5, 700, 64, 64, CAUSAL | KEY, False, 0.2, 50),
    (1, 256, 1024, 128, 128, DENSE, False, 0.0, 8),
    (8, 128, 8192, 128, 128, CAUSAL, False, 0.0, 0),
    # More than 32 ranges: the merge takes the ranges' weights 32 at a time.
    (1, 70, 8192, 64, 64, NONE, True, 0.0, 64),
    (2, 130, 5000, 128, 128, CAUSAL, False, 0.0, 40),
]


def _id(c):
    BH, Nq, Nk, d, dv, mode, f32, pm, ns = c
    return (f"bh{BH}-nq{Nq}-nk{Nk}-d{d}-dv{dv}-{synth.MODE_NAMES[mode]}-"
            f"{'f32' if f32 else 'bf16'}-s{ns}")


def _dev(c):
    import torch

    def bits(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)

    C = None if c["C"] is None else torch.from_numpy(c["C"]).cuda()
    ck = None if c["ckey"] is None else torch.from_numpy(c["ckey"]).cuda()
    return bits(c["Q"]), bits(c["K"]), bits(c["V"]), C, ck


def run_split(c, n_splits, out_f32=True, workspace="plan"):
    import torch

    import exact_tiled_attention_13_gb300 as eta

    Q, K, V, C, ck = _dev(c)
    BH, Nq, d = Q.shape
    Nk, dv = K.shape[1], V.shape[2]
    if workspace == "plan":
        workspace = eta.splitkv_workspace(c["mode"], BH, Nq, Nk, d, dv, n_splits)
    O = torch.full((BH, Nq, dv), float("nan"), device="cuda",
                   dtype=torch.float32 if out_f32 else torch.bfloat16)
    L = torch.full((BH, Nq), float("nan"), device="cuda", dtype=torch.float32)
    eta.attn_fwd_splitkv(Q, K, V, c["mode"], C, ck, c["scale"], O, L, workspace=workspace,
                         n_splits=n_splits)
    torch.cuda.synchronize()
    code, word = eta.attn_device_status(None)
    assert code == eta.ATTN_OK, f"watchdog {word:#x}"
    return O, L


@pytest.mark.parametrize("case", CASES, ids=_id)
def test_splitkv_parity(case):
    import exact_tiled_attention_13_gb300 as eta

    BH, Nq, Nk, d, dv, mode, out_f32, p_mask, n_splits = case
    c = synth.random_case_ex(5000 + Nq + Nk + mode, BH, Nq, Nk, d, dv, mode, 1.0, p_mask)
    code, splits, _ = eta.attn_fwd_splitkv_plan(mode, BH, Nq, Nk, d, dv, n_splits)
    assert code == eta.ATTN_OK
    if n_splits > 1 and Nk > 128:
        assert splits > 1, "the case should exercise the merge"
    O, L = run_split(c, n_splits, out_f32)
    O_ref, L_ref, _ = oracle.attention_ex(c["Q"], c["K"], c["V"], mode, c["C"], c["ckey"],
                                          c["scale"])
    compare(O.float().cpu().numpy().astype(np.float64), L.cpu().numpy().astype(np.float64),
            O_ref, L_ref, out_bf16=not out_f32, label=_id(case))


def test_splitkv_is_deterministic_and_one_range_is_the_plain_call():
    import torch

    import exact_tiled_attention_13_gb300 as eta

    c = synth.random_case_ex(77, 2, 96, 2000, 128, 128, CAUSAL)
    O1, L1 = run_split(c, 6)
    O2, L2 = run_split(c, 6)
    assert torch.equal(O1, O2) and torch.equal(L1, L2)
    # One range: the kernel writes O itself, bit for bit what attn_fwd_ex writes.
    O3, L3 = run_split(c, 1, workspace=None)
    Q, K, V, _, _ = _dev(c)
    O4 = torch.empty_like(O3)
    L4 = torch.empty_like(L3)
    eta.attn_fwd_ex(Q, K, V, CAUSAL, None, None, c["scale"], O4, L4)
    torch.cuda.synchronize()
    assert torch.equal(O3, O4) and torch.equal(L3, L4)
    # Different range counts: the same function, different rounding.
    assert (O1 - O3).abs().max().item() <= TOL_MAX


def test_splitkv_range_without_allowed_keys():
    """Every key of the first two ranges is padded out (-inf): their partials carry weight
    zero in the merge, and rows still see the keys of the other ranges."""
    c = synth.random_case_ex(91, 2, 40, 1024, 64, 64, KEY, 1.0, 0.0)
    c["ckey"][:, :256] = -np.inf
    O, L = run_split(c, 8)
    O_ref, L_ref, _ = oracle.attention_ex(c["Q"], c["K"], c["V"], KEY, None, c["ckey"], c["scale"])
    compare(O.cpu().numpy().astype(np.float64), L.cpu().numpy().astype(np.float64), O_ref, L_ref,
            label="empty ranges")


def test_splitkv_workspace_checks():
    import torch

    import exact_tiled_attention_13_gb300 as eta

    c = synth.random_case_ex(5, 1, 64, 1024, 64, 64, NONE)
    Q, K, V, _, _ = _dev(c)
    code, splits, nbytes = eta.attn_fwd_splitkv_plan(NONE, 1, 64, 1024, 64, 64, 4)
    assert code == eta.ATTN_OK and splits == 4 and nbytes > 0
    O = torch.empty(1, 64, 64, device="cuda")
    small = torch.empty(nbytes - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(eta.AttnError) as e:
        eta.attn_fwd_splitkv(Q, K, V, NONE, None, None, c["scale"], O, workspace=small, n_splits=4)
    assert e.value.code == eta.ATTN_ERR_INVALID_ARG
    with pytest.raises(eta.AttnError) as e:
        eta.attn_fwd_splitkv(Q, K, V, NONE, None, None, c["scale"], O, workspace=None, n_splits=4)
    assert e.value.code == eta.ATTN_ERR_INVALID_ARG
    # A workspace that overlaps the output is rejected.
    big = torch.empty(nbytes + O.numel() * 4, dtype=torch.uint8, device="cuda")
    O_in = big[:O.numel() * 4].view(torch.float32).view(1, 64, 64)
    with pytest.raises(eta.AttnError) as e:
        eta.attn_fwd_splitkv(Q, K, V, NONE, None, None, c["scale"], O_in, workspace=big, n_splits=4)
    assert e.value.code == eta.ATTN_ERR_INVALID_ARG
