"""The C-ABI library without a GPU: it builds for sm_103a, loads, exports every symbol
include/attn.h declares, and rejects bad arguments before touching a device."""
import ctypes
import os
import re
import subprocess

import pytest

import exact_tiled_attention_13_gb300 as eta
from exact_tiled_attention_13_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")


def _header_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^ATTN_API\s+[\w\s\*]*?\b(attn_\w+)\s*\(", text, re.M)))


def _header_defines():
    text = open(HEADER).read()
    return {k: int(v) for k, v in re.findall(r"#define\s+(ATTN_\w+)\s+\(?(-?\d+)\)?", text)}


def _gpu_present():
    try:
        import torch

        return torch.cuda.is_available()
    except Exception:
        return False


def test_every_declared_symbol_is_exported():
    lib = eta.load()
    names = _header_functions()
    assert names == sorted(_lib.SIGNATURES), names
    for name in names:
        assert hasattr(lib, name)
    out = subprocess.run(["nm", "-D", "--defined-only", eta.library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT\s+(attn_\w+)$", out, re.M))
    assert exported == set(names)


def test_library_is_in_tree_and_for_sm103a():
    path = eta.library_path()
    assert path.startswith(os.path.join(ROOT, "exact_tiled_attention_13_gb300", "_build"))
    from exact_tiled_attention_13_gb300 import _build

    assert _build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_header_constants_match_binding():
    defs = _header_defines()
    for name, value in defs.items():
        assert getattr(_lib, name) == value, name


def test_strerror_and_version():
    for code in range(-7, 1):
        assert eta.attn_strerror(code)
    assert "unknown" in eta.attn_strerror(-99)
    assert eta.attn_version() == _lib.ATTN_ABI_VERSION == 107


def test_timeout_setting_roundtrip():
    prev = eta.attn_set_wait_timeout_ns(12345)
    assert eta.attn_set_wait_timeout_ns(0) == 12345
    assert eta.attn_set_wait_timeout_ns(prev) == 2_000_000_000


# Fake, 16-byte aligned "device" addresses: validation must reject bad calls before it
# ever dereferences or registers them.
QP, KP, VP, OP, LP, CP = 0x100000, 0x200000, 0x300000, 0x400000, 0x500000, 0x600000
GOOD = dict(Q=QP, K=KP, V=VP, mode=0, C=None, BH=2, N=64, d=64, d_v=64, scale=0.125, O=OP,
            out_dtype=1, LSE=LP, stream=None)


def call(**over):
    a = dict(GOOD)
    a.update(over)
    return eta.attn_fwd_raw(a["Q"], a["K"], a["V"], a["mode"], a["C"], a["BH"], a["N"], a["d"],
                            a["d_v"], a["scale"], a["O"], a["out_dtype"], a["LSE"], a["stream"])


@pytest.mark.parametrize("over", [
    dict(Q=None), dict(K=None), dict(V=None), dict(O=None),
    dict(Q=QP + 8), dict(V=VP + 2), dict(O=OP + 4), dict(LSE=LP + 2),
    dict(mode=3), dict(mode=-1), dict(out_dtype=2),
    dict(BH=0), dict(N=-1),
    dict(scale=0.0), dict(scale=-0.5), dict(scale=float("nan")), dict(scale=float("inf")),
    dict(mode=2, C=None), dict(mode=0, C=CP), dict(mode=1, C=CP), dict(mode=2, C=CP + 8),
    dict(O=QP), dict(O=KP + 64), dict(LSE=VP), dict(LSE=OP + 128),
], ids=lambda d: ",".join(f"{k}={v}" for k, v in d.items()))
def test_invalid_arguments(over):
    assert call(**over) == eta.ATTN_ERR_INVALID_ARG


@pytest.mark.parametrize("d,dv", [(32, 64), (96, 64), (64, 256), (256, 128)])
def test_unsupported_widths(d, dv):
    assert call(d=d, d_v=dv) == _lib.ATTN_ERR_UNSUPPORTED


def test_zero_length_is_noop():
    assert call(N=0) == eta.ATTN_OK
    assert call(N=0, Q=None, K=None, V=None, O=None, LSE=None) == eta.ATTN_OK
    assert call(N=0, mode=7) == eta.ATTN_ERR_INVALID_ARG


@pytest.mark.skipif(_gpu_present(), reason="a GPU is present")
def test_valid_call_without_gpu_reports_no_device():
    assert call() == eta.ATTN_ERR_NO_DEVICE
    code, word = eta.attn_device_status(None)
    assert code == eta.ATTN_ERR_NO_DEVICE and word == 0


def test_fault_injection_setting():
    assert eta.attn_set_fault_injection(eta.ATTN_FAULT_SKIP_FIRST_K) == eta.ATTN_OK
    assert eta.attn_set_fault_injection(eta.ATTN_FAULT_NONE) == eta.ATTN_OK
    assert eta.attn_set_fault_injection(7) == eta.ATTN_ERR_INVALID_ARG


KP = 0x700000
GOOD_EX = dict(Q=QP, K=KP, V=VP, mode=0, C=None, ckey=None, BH=2, Nq=48, Nk=64, d=64, d_v=64,
               scale=0.125, O=OP, out_dtype=1, LSE=LP, stream=None)


def call_ex(**over):
    a = dict(GOOD_EX)
    a.update(over)
    return eta.attn_fwd_ex_raw(a["Q"], a["K"], a["V"], a["mode"], a["C"], a["ckey"], a["BH"],
                               a["Nq"], a["Nk"], a["d"], a["d_v"], a["scale"], a["O"],
                               a["out_dtype"], a["LSE"], a["stream"])


@pytest.mark.parametrize("over", [
    dict(mode=8), dict(mode=6, C=CP, ckey=KP), dict(mode=4, ckey=None), dict(mode=0, ckey=KP),
    dict(mode=5, ckey=KP + 2), dict(Nk=0), dict(Nq=-1), dict(Nk=-3), dict(mode=2, C=None),
    dict(O=KP), dict(LSE=KP + 128),
], ids=lambda d: ",".join(f"{k}={v}" for k, v in d.items()))
def test_invalid_arguments_ex(over):
    assert call_ex(**over) == eta.ATTN_ERR_INVALID_ARG


def test_ex_zero_queries_is_noop_and_key_mode_needs_ex():
    assert call_ex(Nq=0, Q=None, K=None, V=None, O=None, LSE=None) == eta.ATTN_OK
    # attn_fwd has no per-key vector argument.
    assert call(mode=4) == eta.ATTN_ERR_INVALID_ARG


@pytest.mark.skipif(_gpu_present(), reason="a GPU is present")
def test_valid_ex_call_without_gpu_reports_no_device():
    assert call_ex() == eta.ATTN_ERR_NO_DEVICE
    assert call_ex(mode=5, ckey=KP) == eta.ATTN_ERR_NO_DEVICE


# ---------------------------------------------------------------- split forward pass
WP = 0x900000


def call_split(n_splits=3, workspace=WP, workspace_bytes=1 << 30, **over):
    a = dict(GOOD_EX)
    a.update(over)
    return eta.attn_fwd_splitkv_raw(a["Q"], a["K"], a["V"], a["mode"], a["C"], a["ckey"], a["BH"],
                                    a["Nq"], a["Nk"], a["d"], a["d_v"], a["scale"], n_splits,
                                    workspace, workspace_bytes, a["O"], a["out_dtype"], a["LSE"],
                                    a["stream"])


@pytest.mark.parametrize("nk,req,splits", [
    (64, 1, 1), (64, 5, 1), (1000, 1, 1), (1000, 3, 3), (1000, 5, 4), (1000, 8, 8),
    (1000, 100, 8), (65536, 19, 19), (65536, 7, 7), (129, 2, 2), (129, 3, 2),
])
def test_splitkv_plan_rounds_to_whole_tiles(nk, req, splits):
    code, s, nbytes = eta.attn_fwd_splitkv_plan(1, 4, 100, nk, 128, 64, req)
    assert code == eta.ATTN_OK
    assert s == splits
    # ceil(tiles / ceil(tiles / req)) ranges; fp32 partial O and LSE per range and row.
    tiles = -(-nk // 128)
    assert s == -(-tiles // -(-tiles // min(req, tiles)))
    assert nbytes == (0 if s == 1 else s * 4 * 100 * (64 + 1) * 4)


def test_splitkv_plan_rejects_what_the_call_rejects():
    assert eta.attn_fwd_splitkv_plan(8, 1, 1, 1, 64, 64, 2)[0] == eta.ATTN_ERR_INVALID_ARG
    assert eta.attn_fwd_splitkv_plan(0, 1, 1, 0, 64, 64, 2)[0] == eta.ATTN_ERR_INVALID_ARG
    assert eta.attn_fwd_splitkv_plan(0, 1, 1, 1, 96, 64, 2)[0] == eta.ATTN_ERR_UNSUPPORTED
    assert eta.attn_fwd_splitkv_plan(0, 1, 1, 1, 64, 64, -1)[0] == eta.ATTN_ERR_INVALID_ARG
    assert eta.attn_fwd_splitkv_plan(0, 1, 0, 5, 64, 64, 2)[:2] == (eta.ATTN_OK, 1)


@pytest.mark.skipif(_gpu_present(), reason="a GPU is present")
def test_splitkv_automatic_plan_needs_a_device():
    assert eta.attn_fwd_splitkv_plan(0, 1, 1, 4096, 64, 64, 0)[0] == eta.ATTN_ERR_NO_DEVICE


@pytest.mark.parametrize("over", [
    dict(n_splits=-1), dict(mode=8), dict(Nk=0), dict(O=KP), dict(mode=4, ckey=None),
], ids=lambda d: ",".join(f"{k}={v}" for k, v in d.items()))
def test_invalid_arguments_splitkv(over):
    assert call_split(**over) == eta.ATTN_ERR_INVALID_ARG


def test_splitkv_zero_queries_is_noop():
    assert call_split(Nq=0, Q=None, K=None, V=None, O=None, LSE=None, workspace=None) == eta.ATTN_OK


@pytest.mark.skipif(_gpu_present(), reason="a GPU is present")
def test_valid_splitkv_call_without_gpu_reports_no_device():
    assert call_split(Nk=1000) == eta.ATTN_ERR_NO_DEVICE


def test_shared_bias_needs_the_dense_bias():
    # ATTN_BIAS_SHARED (one [Nq][Nk] bias for every head) qualifies ATTN_BIAS_DENSE only.
    assert call_ex(mode=_lib.ATTN_BIAS_SHARED, C=CP) == eta.ATTN_ERR_INVALID_ARG
    assert call_ex(mode=_lib.ATTN_BIAS_SHARED | _lib.ATTN_BIAS_KEY, ckey=KP) == eta.ATTN_ERR_INVALID_ARG
    assert call_ex(mode=_lib.ATTN_BIAS_SHARED | _lib.ATTN_BIAS_DENSE, C=None) == eta.ATTN_ERR_INVALID_ARG
    code, _ = eta.attn_fwd_host_staging_bytes(_lib.ATTN_BIAS_SHARED | _lib.ATTN_BIAS_DENSE, 2, 64, 64,
                                              64, 64, 1, 0)
    assert code == eta.ATTN_ERR_INVALID_ARG  # the host-streaming calls slice C per head


@pytest.mark.skipif(_gpu_present(), reason="a GPU is present")
def test_shared_bias_is_one_array_for_the_overlap_checks():
    # A shared C of Nq x Nk fp32 ends before O here; read as [BH][Nq][Nk] it would overlap O.
    a = dict(GOOD_EX)
    c_bytes = a["Nq"] * a["Nk"] * 4
    o = 0x7000000
    shared = call_ex(mode=_lib.ATTN_BIAS_SHARED | _lib.ATTN_BIAS_DENSE, C=o - c_bytes, O=o)
    full = call_ex(mode=_lib.ATTN_BIAS_DENSE, C=o - c_bytes, O=o)
    assert shared == eta.ATTN_ERR_NO_DEVICE and full == eta.ATTN_ERR_INVALID_ARG


@pytest.mark.skipif(_gpu_present(), reason="a GPU is present")
def test_static_splitkv_reports_the_device_like_the_workspace_call():
    # A plan that fits the fixed array: the device is examined before the array's address is
    # looked up, so the code is the one attn_fwd_splitkv returns, not a generic CUDA failure.
    code = _lib.attn_fwd_splitkv_static_raw(QP, KP, VP, 0, None, None, 2, 48, 1000, 64, 64,
                                            0.125, 4, OP, 1, LP, None)
    assert code == eta.ATTN_ERR_NO_DEVICE
    assert code == call_split(Nk=1000)


# ---------------------------------------------------------------- backward pass
def call_bwd(**over):
    a = dict(Q=QP, K=KP, V=VP, O=OP, o_dtype=1, dO=0xA00000, LSE=LP, mode=0, C=None, ckey=None,
             BH=2, Nq=48, Nk=64, d=64, d_v=64, scale=0.125, dQ=0xB00000, dK=0xC00000,
             dV=0xD00000, workspace=0xE00000, workspace_bytes=1 << 20, stream=None)
    a.update(over)
    return eta.attn_bwd_raw(*a.values())


def test_bwd_workspace_bytes():
    assert eta.attn_bwd_workspace_bytes(3, 200) == (eta.ATTN_OK, 2 * 3 * 256 * 4)
    assert eta.attn_bwd_workspace_bytes(1, 0) == (eta.ATTN_OK, 0)
    assert eta.attn_bwd_workspace_bytes(0, 5)[0] == eta.ATTN_ERR_INVALID_ARG


@pytest.mark.parametrize("over", [
    dict(mode=8), dict(mode=6, C=CP, ckey=KP), dict(Nk=0), dict(LSE=None), dict(dO=None),
    dict(workspace=None), dict(workspace_bytes=16), dict(dQ=QP), dict(dK=0xC00000 + 8),
    dict(dV=0xC00000), dict(workspace=0xA00000), dict(mode=2, C=None), dict(o_dtype=3),
], ids=lambda d: ",".join(f"{k}={v}" for k, v in d.items()))
def test_invalid_arguments_bwd(over):
    assert call_bwd(**over) == eta.ATTN_ERR_INVALID_ARG


def test_bwd_unsupported_width_and_empty():
    assert call_bwd(d=96) == eta.ATTN_ERR_UNSUPPORTED
    assert call_bwd(Nq=0, Nk=0, Q=None, K=None, V=None, O=None, dO=None, LSE=None, dQ=None,
                    dK=None, dV=None, workspace=None) == eta.ATTN_OK


@pytest.mark.skipif(_gpu_present(), reason="a GPU is present")
def test_valid_bwd_call_without_gpu_reports_no_device():
    assert call_bwd() == eta.ATTN_ERR_NO_DEVICE
    assert call_bwd(Nq=0, Q=None, O=None, dO=None, LSE=None, dQ=None, workspace=None) == eta.ATTN_ERR_NO_DEVICE


# ---------------------------------------------------------------- host-streamed forward
def test_host_staging_bytes():
    MiB = 1 << 20
    # 64 heads of 8192 x 128 (bf16 O): chunks of 8 heads (32 blocks a head);
    # a slot holds Q, K, V, O (16 MiB each at 8 heads) and LSE (256 KiB); two slots.
    code, nbytes = eta.attn_fwd_host_staging_bytes(1, 64, 8192, 8192, 128, 128, 0)
    assert code == eta.ATTN_OK and nbytes == 2 * (4 * 16 * MiB + 256 * 1024)
    # 8 heads of 4096 (16 blocks a head): one chunk of all 8 heads, one slot.
    code, nbytes = eta.attn_fwd_host_staging_bytes(4, 8, 4096, 4096, 64, 128, 1)
    parts = [8 * 4096 * 64 * 2, 8 * 4096 * 64 * 2, 8 * 4096 * 128 * 2, 0, 8 * 4096 * 4, 8 * 4096 * 128 * 4, 8 * 4096 * 4]
    assert code == eta.ATTN_OK and nbytes == sum(parts)
    # 16 heads of 16384 (64 blocks a head): chunks of 2 heads (128 blocks).
    code, nbytes = eta.attn_fwd_host_staging_bytes(0, 16, 16384, 16384, 128, 128, 1)
    assert code == eta.ATTN_OK and nbytes == 2 * 2 * 16384 * (3 * 128 * 2 + 128 * 4 + 4)
    # 64 heads of 2048 (8 blocks a head): chunks of 16 heads.
    code, nbytes = eta.attn_fwd_host_staging_bytes(1, 64, 2048, 2048, 128, 128, 0)
    assert code == eta.ATTN_OK and nbytes == 2 * 16 * 2048 * (4 * 128 * 2 + 4)
    # One chunk (every head at once): one slot, each part rounded up to 256 bytes: Q 384,
    # K 640, V 640, O 768 (fp32), LSE 12 bytes.
    code, nbytes = eta.attn_fwd_host_staging_bytes(0, 1, 3, 5, 64, 64, 1)
    assert code == eta.ATTN_OK and nbytes == 512 + 768 + 768 + 768 + 256
    # Dense bias and fp32 O, chunks of 3 heads of BH = 7: C is 3 x 10 x 20 x 4 bytes.
    code, nbytes = eta.attn_fwd_host_staging_bytes(2, 7, 10, 20, 64, 128, 1, 3)
    parts = [3 * 10 * 64 * 2, 3 * 20 * 64 * 2, 3 * 20 * 128 * 2, 3 * 10 * 20 * 4, 0, 3 * 10 * 128 * 4, 3 * 10 * 4]
    assert code == eta.ATTN_OK and nbytes == 2 * sum((x + 255) // 256 * 256 for x in parts)
    for bad in (dict(mode=8), dict(mode=6), dict(BH=0), dict(out_dtype=2), dict(heads_per_chunk=-1)):
        a = dict(mode=0, BH=2, Nq=4, Nk=4, d=64, d_v=64, out_dtype=0, heads_per_chunk=0)
        a.update(bad)
        assert eta.attn_fwd_host_staging_bytes(*a.values())[0] == eta.ATTN_ERR_INVALID_ARG
    assert eta.attn_fwd_host_staging_bytes(0, 2, 4, 4, 96, 64, 0)[0] == eta.ATTN_ERR_UNSUPPORTED


def call_host(**over):
    a = dict(Q=QP, K=KP, V=VP, mode=0, C=None, ckey=None, BH=2, Nq=48, Nk=64, d=64, d_v=64,
             scale=0.125, O=OP, out_dtype=1, LSE=LP, staging=0xF00000, staging_bytes=1 << 24,
             heads_per_chunk=0, stream=None)
    a.update(over)
    return eta.attn_fwd_host_raw(*a.values())


@pytest.mark.parametrize("over", [
    dict(mode=8), dict(Nk=0), dict(Q=None), dict(O=None), dict(staging=None), dict(staging_bytes=16),
    dict(staging=0xF00010), dict(mode=2), dict(mode=0, C=CP), dict(mode=4), dict(scale=0.0),
    dict(heads_per_chunk=-2), dict(O=QP + 64),
], ids=lambda d: ",".join(f"{k}={v}" for k, v in d.items()))
def test_invalid_arguments_host(over):
    assert call_host(**over) == eta.ATTN_ERR_INVALID_ARG


def test_host_zero_queries_is_noop_and_widths():
    assert call_host(Nq=0, Q=None, O=None, LSE=None, staging=None) == eta.ATTN_OK
    assert call_host(d=96) == eta.ATTN_ERR_UNSUPPORTED


def test_bwd_host_staging_bytes():
    # 64 heads of 2048 (16 query and 16 key tiles): chunks of 8 heads, two slots; per head
    # Q, K, V, O (bf16), dO 512 KiB each, LSE 8 KiB, dQ, dK, dV 1 MiB each, workspace 16 KiB.
    code, nbytes = eta.attn_bwd_host_staging_bytes(1, 64, 2048, 2048, 128, 128, 0)
    per_head = 5 * 512 * 1024 + 8 * 1024 + 3 * 1024 * 1024 + 16 * 1024
    assert code == eta.ATTN_OK and nbytes == 2 * 8 * per_head
    for bad in (dict(mode=8), dict(BH=0), dict(o_dtype=2), dict(heads_per_chunk=-1), dict(Nq=-1)):
        a = dict(mode=0, BH=2, Nq=4, Nk=4, d=64, d_v=64, o_dtype=0, heads_per_chunk=0)
        a.update(bad)
        assert eta.attn_bwd_host_staging_bytes(*a.values())[0] == eta.ATTN_ERR_INVALID_ARG
    assert eta.attn_bwd_host_staging_bytes(0, 2, 4, 4, 64, 96, 0)[0] == eta.ATTN_ERR_UNSUPPORTED


def call_bwd_host(**over):
    a = dict(Q=QP, K=KP, V=VP, O=OP, o_dtype=1, dO=0xA00000, LSE=LP, mode=0, C=None, ckey=None,
             BH=2, Nq=48, Nk=64, d=64, d_v=64, scale=0.125, dQ=0xB00000, dK=0xC00000,
             dV=0xD00000, staging=0xF00000, staging_bytes=1 << 24, heads_per_chunk=0, stream=None)
    a.update(over)
    return eta.attn_bwd_host_raw(*a.values())


@pytest.mark.parametrize("over", [
    dict(mode=8), dict(Nk=0), dict(K=None), dict(dV=None), dict(LSE=None), dict(dQ=None),
    dict(staging=None), dict(staging_bytes=16), dict(staging=0xF00040), dict(mode=2), dict(mode=4),
    dict(scale=-1.0), dict(dQ=QP + 16),
], ids=lambda d: ",".join(f"{k}={v}" for k, v in d.items()))
def test_invalid_arguments_bwd_host(over):
    assert call_bwd_host(**over) == eta.ATTN_ERR_INVALID_ARG


def test_bwd_host_empty_and_widths():
    assert call_bwd_host(Nq=0, Nk=0) == eta.ATTN_OK
    assert call_bwd_host(d=96) == eta.ATTN_ERR_UNSUPPORTED
