"""attn_fwd_splitkv_static: the split forward pass with its partials in the library's
fixed array instead of a caller workspace. Called through the C ABI (raw pointers) and
checked against attn_fwd_splitkv with a caller workspace, on two calls in a row that
both use the shared array. Both run the same kernels on the same key ranges, so the
outputs must agree bit for bit: a tolerance would hide a partial overwrite of the shared
array. Named to run after the other test files."""
import numpy as np
import pytest

import synth

CAUSAL, KEY = synth.MODE_CAUSAL, synth.MODE_KEY


def test_static_scratch_rejects_plans_beyond_the_array():
    from exact_tiled_attention_13_gb300 import _lib

    # 64 ranges x 8 heads x 1024 queries x 129 x 4 bytes = 270 MB > 32 MiB; an explicit
    # range count is planned without the device, so the limit is reported on the CPU too.
    code = _lib.attn_fwd_splitkv_static_raw(0x1000, 0x2000, 0x3000, CAUSAL, None, None, 8, 1024,
                                            65536, 128, 128, 0.088, 64, 0x4000, 0, None, None)
    assert code == _lib.ATTN_ERR_SCRATCH_LIMIT
    assert "scratch" in _lib.strerror(code)


def _bits(a):
    import torch

    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)


def _static_call(c, n_splits, out_f32):
    """One attn_fwd_splitkv_static call through the raw C entry point."""
    import torch

    from exact_tiled_attention_13_gb300 import _lib

    Q, K, V = _bits(c["Q"]), _bits(c["K"]), _bits(c["V"])
    ck = None if c["ckey"] is None else torch.from_numpy(c["ckey"]).cuda()
    BH, Nq, d = Q.shape
    Nk, dv = K.shape[1], V.shape[2]
    O = torch.full((BH, Nq, dv), float("nan"), device="cuda",
                   dtype=torch.float32 if out_f32 else torch.bfloat16)
    L = torch.full((BH, Nq), float("nan"), device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    code = _lib.attn_fwd_splitkv_static_raw(
        Q.data_ptr(), K.data_ptr(), V.data_ptr(), c["mode"], None,
        None if ck is None else ck.data_ptr(), BH, Nq, Nk, d, dv, c["scale"], n_splits,
        O.data_ptr(), _lib.ATTN_OUT_F32 if out_f32 else _lib.ATTN_OUT_BF16, L.data_ptr(), stream)
    assert code == _lib.ATTN_OK, _lib.strerror(code)
    return (Q, K, V, ck), O, L


def _workspace_call(dev, c, n_splits, out_f32):
    import torch

    import exact_tiled_attention_13_gb300 as eta

    Q, K, V, ck = dev
    BH, Nq, d = Q.shape
    Nk, dv = K.shape[1], V.shape[2]
    ws = eta.splitkv_workspace(c["mode"], BH, Nq, Nk, d, dv, n_splits)
    O = torch.empty((BH, Nq, dv), device="cuda", dtype=torch.float32 if out_f32 else torch.bfloat16)
    L = torch.empty((BH, Nq), device="cuda")
    eta.attn_fwd_splitkv(Q, K, V, c["mode"], None, ck, c["scale"], O, L, workspace=ws,
                         n_splits=n_splits)
    return O, L


@pytest.mark.gpu
def test_static_scratch_matches_workspace_call_twice_in_a_row():
    import torch

    import exact_tiled_attention_13_gb300 as eta

    a = synth.random_case_ex(401, 8, 128, 8192, 128, 128, CAUSAL)
    b = synth.random_case_ex(402, 2, 3, 5000, 64, 128, KEY, 1.0, 0.3)
    # Two calls in a row on the shared array, the second before the first is checked.
    dev_a, Oa, La = _static_call(a, 0, False)
    dev_b, Ob, Lb = _static_call(b, 7, True)
    torch.cuda.synchronize()
    code, word = eta.attn_device_status(None)
    assert code == eta.ATTN_OK, f"watchdog {word:#x}"
    Oa_ref, La_ref = _workspace_call(dev_a, a, 0, False)
    Ob_ref, Lb_ref = _workspace_call(dev_b, b, 7, True)
    torch.cuda.synchronize()
    for O, L, O_ref, L_ref, name in ((Oa, La, Oa_ref, La_ref, "first call"),
                                     (Ob, Lb, Ob_ref, Lb_ref, "second call")):
        o, o_ref = O.cpu(), O_ref.cpu()
        lse, lse_ref = L.cpu().numpy(), L_ref.cpu().numpy()
        assert np.isfinite(o.float().numpy()).all(), name
        # Bit for bit: the same kernels on the same ranges, whichever memory holds the partials.
        assert np.array_equal(o.view(torch.int16 if o.dtype == torch.bfloat16 else torch.int32).numpy(),
                              o_ref.view(torch.int16 if o_ref.dtype == torch.bfloat16 else torch.int32).numpy()), name
        assert np.array_equal(lse.view(np.int32), lse_ref.view(np.int32)), name
