"""Rows whose exponent reference moves on almost every key tile.

The kernels move a row's exponent reference only when a tile's maximum exceeds it by more
than 2^8, and then rescale o. With N(0,1) inputs that happens on a row's first tiles and
rarely after, so these cases make the scores grow by about ten units per key tile in the
order the kernels visit the tiles (from the last key tile down): the reference then moves,
and o is rescaled, on nearly every tile. Covered: the split pass (one query tile per CTA,
two S buffers in tensor memory), the dense bias at d_v = 64 (the same kernel shape, bias
through TMA or direct loads), the per-key bias on the CTA-pair kernel (folded into the
score product) and on the single-CTA kernel, and the CTA-pair kernel without a bias.
Results are compared with the oracle's plain definition."""
import numpy as np
import pytest

import oracle
import synth
from gpu_helpers import compare

pytestmark = pytest.mark.gpu

NONE, CAUSAL, DENSE, KEY = synth.MODE_NONE, synth.MODE_CAUSAL, synth.MODE_DENSE, synth.MODE_KEY


def tiles_after(Nk):
    """For each key, how many key tiles the kernels visit after its own (0 for the last)."""
    j = np.arange(Nk)
    return ((Nk - 1) // 128 - j // 128).astype(np.float64)


def growing_keys(c, per_tile):
    """Column 0 of every query set to 1 and column 0 of key j to per_tile x sqrt(d) x
    tiles_after(j): every score of a tile is per_tile (natural units) above the tile visited
    next, on top of the random q.k of the other columns."""
    d = c["Q"].shape[2]
    Q = synth.bf16_to_f32(c["Q"]).copy()
    K = synth.bf16_to_f32(c["K"]).copy()
    Q[:, :, 0] = 1.0
    K[:, :, 0] = (per_tile * np.sqrt(d) * tiles_after(K.shape[1])).astype(np.float32)[None, :]
    c["Q"], c["K"] = synth.bf16_bits(Q), synth.bf16_bits(K)
    return c


def move_fraction(c, ranges=1):
    """Fraction of (row, key tile) visits after a row's first visible tile on which the
    kernels' lazy rule moves the exponent reference (tile maximum more than 8 above it in
    log2 units), replayed in float64 over the case's scores, each key range visited from
    its last tile down. The cases below need at least 80 % of the visits to move."""
    Q = synth.bf16_to_f32(c["Q"]).astype(np.float64)
    K = synth.bf16_to_f32(c["K"]).astype(np.float64)
    BH, Nq, _ = Q.shape
    Nk = K.shape[1]
    S = np.einsum("bqd,bkd->bqk", Q, K) * c["scale"]
    if c["C"] is not None:
        S = S + c["C"]
    if c["ckey"] is not None:
        S = S + c["ckey"][:, None, :]
    if c["mode"] & CAUSAL:
        allowed = np.arange(Nk)[None, :] <= np.arange(Nq)[:, None] + (Nk - Nq)
        S = np.where(allowed[None], S, -np.inf)
    ntiles = (Nk + 127) // 128
    per = -(-ntiles // ranges)
    moves = visits = 0
    for r0 in range(0, ntiles, per):
        m = np.full((BH, Nq), -np.inf)
        for t in range(min(r0 + per, ntiles) - 1, r0 - 1, -1):
            b = S[:, :, 128 * t:128 * (t + 1)].max(axis=2) * np.log2(np.e)
            seen = np.isfinite(m) & np.isfinite(b)
            visits += int(seen.sum())
            moves += int((seen & (b > m + 8.0)).sum())
            m = np.where(b > m + 8.0, b, m)
    return moves / max(visits, 1)


def run(c, out_f32=True, n_splits=None):
    import torch

    import exact_tiled_attention_13_gb300 as eta

    def bits(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)

    Q, K, V = bits(c["Q"]), bits(c["K"]), bits(c["V"])
    C = None if c["C"] is None else torch.from_numpy(np.ascontiguousarray(c["C"])).cuda()
    ck = None if c["ckey"] is None else torch.from_numpy(np.ascontiguousarray(c["ckey"])).cuda()
    BH, Nq, d = Q.shape
    Nk, dv = K.shape[1], V.shape[2]
    O = torch.full((BH, Nq, dv), float("nan"), device="cuda",
                   dtype=torch.float32 if out_f32 else torch.bfloat16)
    L = torch.full((BH, Nq), float("nan"), device="cuda", dtype=torch.float32)
    if n_splits is None:
        eta.attn_fwd_ex(Q, K, V, c["mode"], C, ck, c["scale"], O, L)
    else:
        ws = eta.splitkv_workspace(c["mode"], BH, Nq, Nk, d, dv, n_splits)
        eta.attn_fwd_splitkv(Q, K, V, c["mode"], C, ck, c["scale"], O, L, workspace=ws,
                             n_splits=n_splits)
    torch.cuda.synchronize()
    code, word = eta.attn_device_status(None)
    assert code == eta.ATTN_OK, f"watchdog {word:#x}"
    return O.float().cpu().numpy().astype(np.float64), L.cpu().numpy().astype(np.float64)


def check(c, label, out_f32=True, n_splits=None):
    O, L = run(c, out_f32, n_splits)
    O_ref, L_ref, _ = oracle.attention_ex(c["Q"], c["K"], c["V"], c["mode"], c["C"], c["ckey"],
                                          c["scale"])
    compare(O, L, O_ref, L_ref, out_bf16=not out_f32, label=label)


@pytest.mark.parametrize("mode", [NONE, CAUSAL], ids=["nomask", "causal"])
def test_split_pass_reference_moves(mode):
    # 32 key tiles in 4 ranges of 8; the scores grow by about 12 (natural units) a tile.
    c = growing_keys(synth.random_case_ex(6100 + mode, 2, 128, 4096, 128, 128, mode), 12.0)
    assert move_fraction(c, ranges=4) > 0.8
    check(c, f"split {synth.MODE_NAMES[mode]}", out_f32=False, n_splits=4)


@pytest.mark.parametrize("Nk", [1024, 1030], ids=["bias-tma", "bias-direct"])
def test_dense_bias_dv64_reference_moves(Nk):
    c = synth.random_case_ex(6200 + Nk, 1, 256, Nk, 64, 64, DENSE)
    c["C"] = (c["C"].astype(np.float64) + 10.0 * tiles_after(Nk)[None, None, :]).astype(np.float32)
    assert move_fraction(c) > 0.8
    check(c, f"dense bias Nk={Nk}")


@pytest.mark.parametrize("d", [64, 128], ids=["pair-d64", "single-d128"])
def test_key_bias_reference_moves(d):
    c = synth.random_case_ex(6300 + d, 2, 300, 1500, d, 128, KEY, 1.0, 0.2)
    finite = np.isfinite(c["ckey"])
    grow = (c["ckey"].astype(np.float64) + 10.0 * tiles_after(1500)[None, :]).astype(np.float32)
    c["ckey"] = np.where(finite, grow, c["ckey"]).astype(np.float32)
    assert move_fraction(c) > 0.8
    check(c, f"key bias d={d}", out_f32=False)


def test_pair_kernel_reference_moves():
    c = growing_keys(synth.random_case_ex(6400, 1, 512, 2048, 128, 128, CAUSAL), 12.0)
    assert move_fraction(c) > 0.8
    check(c, "pair causal")
