"""Exact tiled attention forward pass for NVIDIA GB300 (sm_103a).

O = softmax(Q K^T * scale + C) V with an additive bias or mask C, evaluated tile by
tile with the online-softmax recurrence in a hand-written CUDA kernel (TMA, tcgen05
tensor cores, tensor memory) behind the C ABI of include/attn.h. This module only
checks tensor shapes and passes device pointers to that ABI; every step of the
computation runs in the library's kernel.
"""
from __future__ import annotations

from ._lib import (ATTN_BIAS_DENSE, ATTN_BIAS_KEY, ATTN_BIAS_SHARED, ATTN_ERR_CUDA, ATTN_ERR_DEVICE_TIMEOUT, ATTN_ERR_INVALID_ARG,
                   ATTN_ERR_LAUNCH, ATTN_ERR_NO_DEVICE, ATTN_ERR_UNSUPPORTED,
                   ATTN_ERR_UNSUPPORTED_DEVICE, ATTN_FAULT_NONE, ATTN_FAULT_SKIP_FIRST_K,
                   ATTN_MASK_CAUSAL, ATTN_MASK_NONE, ATTN_OK, ATTN_OUT_BF16, ATTN_OUT_F32,
                   AttnError, attn_bwd_host_raw, attn_bwd_host_staging_bytes, attn_bwd_raw,
                   attn_bwd_workspace_bytes, attn_device_status,
                   attn_fwd_ex_raw, attn_fwd_host_raw, attn_fwd_host_staging_bytes, attn_fwd_raw,
                   attn_fwd_splitkv_plan, attn_fwd_splitkv_raw, attn_set_fault_injection,
                   attn_set_wait_timeout_ns, attn_version, library_path, load, strerror)

__all__ = [
    "attention", "attn_fwd", "attn_fwd_raw", "attn_fwd_ex", "attn_fwd_ex_raw", "attn_fwd_splitkv",
    "attn_fwd_splitkv_raw", "attn_fwd_splitkv_plan", "splitkv_workspace", "attn_fwd_host",
    "attn_fwd_host_raw", "attn_fwd_host_staging_bytes", "host_staging", "attn_bwd_host",
    "attn_bwd_host_raw", "attn_bwd_host_staging_bytes", "bwd_host_staging", "attn_bwd",
    "attn_bwd_raw", "attn_bwd_workspace_bytes", "bwd_workspace", "attn_strerror", "attn_device_status", "attn_set_wait_timeout_ns",
    "attn_set_fault_injection", "attn_version", "AttnError", "load", "library_path", "ATTN_MASK_NONE", "ATTN_MASK_CAUSAL",
    "ATTN_BIAS_DENSE", "ATTN_BIAS_KEY", "ATTN_BIAS_SHARED", "ATTN_OUT_BF16", "ATTN_OUT_F32",
]

attn_strerror = strerror


def _stream_handle(stream):
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def attn_fwd(Q, K, V, mode, C, scale, O, LSE=None, stream=None):
    """Launch O = softmax(Q K^T * scale + C) V (and LSE) through the C ABI.

    Q, K: bf16 CUDA tensors [BH, N, d]; V: bf16 [BH, N, d_v]; C: fp32 [BH, N, N] for
    mode ATTN_BIAS_DENSE ([N, N] with ATTN_BIAS_SHARED), else None; O: bf16 or fp32 [BH, N, d_v]; LSE: fp32 [BH, N] or
    None. All contiguous. `stream`: torch.cuda.Stream, a raw handle, or None for the
    current stream. Raises AttnError with the library's code on failure.
    """
    import torch

    for name, t in (("Q", Q), ("K", K), ("V", V), ("O", O)):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if Q.dtype != torch.bfloat16 or K.dtype != torch.bfloat16 or V.dtype != torch.bfloat16:
        raise ValueError("Q, K and V must be bf16")
    if Q.dim() != 3 or K.shape != Q.shape or V.dim() != 3 or V.shape[:2] != Q.shape[:2]:
        raise ValueError("expected Q, K [BH, N, d] and V [BH, N, d_v]")
    BH, N, d = Q.shape
    dv = V.shape[2]
    if tuple(O.shape) != (BH, N, dv) or O.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("O must be bf16 or fp32 [BH, N, d_v]")
    out_dtype = ATTN_OUT_F32 if O.dtype == torch.float32 else ATTN_OUT_BF16
    c_ptr = None
    if C is not None:
        c_shape = (N, N) if mode & ATTN_BIAS_SHARED else (BH, N, N)
        if C.dtype != torch.float32 or tuple(C.shape) != c_shape or not C.is_contiguous():
            raise ValueError(f"C must be a contiguous fp32 {list(c_shape)} tensor")
        c_ptr = C.data_ptr()
    lse_ptr = None
    if LSE is not None:
        if LSE.dtype != torch.float32 or tuple(LSE.shape) != (BH, N) or not LSE.is_contiguous():
            raise ValueError("LSE must be a contiguous fp32 [BH, N] tensor")
        lse_ptr = LSE.data_ptr()
    code = attn_fwd_raw(Q.data_ptr(), K.data_ptr(), V.data_ptr(), mode, c_ptr, BH, N, d, dv, scale,
                        O.data_ptr(), out_dtype, lse_ptr, _stream_handle(stream))
    if code != ATTN_OK:
        raise AttnError(code, "attn_fwd")
    return O, LSE


def _marshal_ex(Q, K, V, C, ckey, O, LSE, mode=0):
    """Shape/dtype checks of the Nq x Nk entry points; returns the integers they take."""
    import torch

    for name, t in (("Q", Q), ("K", K), ("V", V), ("O", O)):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if Q.dtype != torch.bfloat16 or K.dtype != torch.bfloat16 or V.dtype != torch.bfloat16:
        raise ValueError("Q, K and V must be bf16")
    if Q.dim() != 3 or K.dim() != 3 or V.dim() != 3:
        raise ValueError("expected Q [BH, Nq, d], K [BH, Nk, d], V [BH, Nk, d_v]")
    BH, Nq, d = Q.shape
    Nk, dv = K.shape[1], V.shape[2]
    if tuple(K.shape) != (BH, Nk, d) or tuple(V.shape[:2]) != (BH, Nk):
        raise ValueError("inconsistent Q, K, V shapes")
    if tuple(O.shape) != (BH, Nq, dv) or O.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("O must be bf16 or fp32 [BH, Nq, d_v]")
    out_dtype = ATTN_OUT_F32 if O.dtype == torch.float32 else ATTN_OUT_BF16
    c_ptr = k_ptr = lse_ptr = None
    if C is not None:
        c_shape = (Nq, Nk) if mode & ATTN_BIAS_SHARED else (BH, Nq, Nk)
        if C.dtype != torch.float32 or tuple(C.shape) != c_shape or not C.is_contiguous():
            raise ValueError(f"C must be a contiguous fp32 {list(c_shape)} tensor")
        c_ptr = C.data_ptr()
    if ckey is not None:
        if ckey.dtype != torch.float32 or tuple(ckey.shape) != (BH, Nk) or not ckey.is_contiguous():
            raise ValueError("ckey must be a contiguous fp32 [BH, Nk] tensor")
        k_ptr = ckey.data_ptr()
    if LSE is not None:
        if LSE.dtype != torch.float32 or tuple(LSE.shape) != (BH, Nq) or not LSE.is_contiguous():
            raise ValueError("LSE must be a contiguous fp32 [BH, Nq] tensor")
        lse_ptr = LSE.data_ptr()
    return BH, Nq, Nk, d, dv, out_dtype, c_ptr, k_ptr, lse_ptr


def attn_fwd_ex(Q, K, V, mode, C, ckey, scale, O, LSE=None, stream=None):
    """attn_fwd with Nq queries and Nk keys and the per-key bias term, through the C ABI.

    Q: bf16 [BH, Nq, d]; K: bf16 [BH, Nk, d]; V: bf16 [BH, Nk, d_v]; mode: bit set of
    ATTN_MASK_CAUSAL, ATTN_BIAS_DENSE, ATTN_BIAS_KEY, ATTN_BIAS_SHARED; C: fp32 [BH, Nq, Nk]
    ([Nq, Nk] with ATTN_BIAS_SHARED: one bias for every head) or None;
    ckey: fp32 [BH, Nk] or None; O: bf16/fp32 [BH, Nq, d_v]; LSE: fp32 [BH, Nq] or None.
    """
    BH, Nq, Nk, d, dv, out_dtype, c_ptr, k_ptr, lse_ptr = _marshal_ex(Q, K, V, C, ckey, O, LSE, mode)
    code = attn_fwd_ex_raw(Q.data_ptr(), K.data_ptr(), V.data_ptr(), mode, c_ptr, k_ptr, BH, Nq, Nk,
                           d, dv, scale, O.data_ptr(), out_dtype, lse_ptr, _stream_handle(stream))
    if code != ATTN_OK:
        raise AttnError(code, "attn_fwd_ex")
    return O, LSE


def splitkv_workspace(mode, BH, Nq, Nk, d, d_v, n_splits=0, device="cuda"):
    """A workspace tensor (uint8) of the size attn_fwd_splitkv_plan reports, or None when
    the plan has one key range. The caller keeps it for as long as the launches using
    it may run."""
    import torch

    code, splits, nbytes = attn_fwd_splitkv_plan(mode, BH, Nq, Nk, d, d_v, n_splits)
    if code != ATTN_OK:
        raise AttnError(code, "attn_fwd_splitkv_plan")
    return None if nbytes == 0 else torch.empty(nbytes, dtype=torch.uint8, device=device)


def attn_fwd_splitkv(Q, K, V, mode, C, ckey, scale, O, LSE=None, workspace=None, n_splits=0,
                     stream=None):
    """attn_fwd_ex with each head's keys split into ranges run as separate blocks and merged
    by a second kernel (include/attn.h, attn_fwd_splitkv). `workspace`: a contiguous CUDA
    tensor of at least the planned bytes (see splitkv_workspace), or None when the plan
    has one range; n_splits = 0 lets the library choose."""
    BH, Nq, Nk, d, dv, out_dtype, c_ptr, k_ptr, lse_ptr = _marshal_ex(Q, K, V, C, ckey, O, LSE, mode)
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        if not workspace.is_contiguous():
            raise ValueError("workspace must be contiguous")
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    code = attn_fwd_splitkv_raw(Q.data_ptr(), K.data_ptr(), V.data_ptr(), mode, c_ptr, k_ptr, BH,
                                Nq, Nk, d, dv, scale, n_splits, ws_ptr, ws_bytes, O.data_ptr(),
                                out_dtype, lse_ptr, _stream_handle(stream))
    if code != ATTN_OK:
        raise AttnError(code, "attn_fwd_splitkv")
    return O, LSE


def host_staging(mode, BH, Nq, Nk, d, d_v, out_dtype, heads_per_chunk=0, device="cuda"):
    """A device staging tensor (uint8) of the size attn_fwd_host needs."""
    import torch

    code, nbytes = attn_fwd_host_staging_bytes(mode, BH, Nq, Nk, d, d_v, out_dtype, heads_per_chunk)
    if code != ATTN_OK:
        raise AttnError(code, "attn_fwd_host_staging_bytes")
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def attn_fwd_host(Q, K, V, mode, C, ckey, scale, O, LSE=None, staging=None, heads_per_chunk=0,
                  stream=None):
    """attn_fwd_ex on host (CPU) tensors, streamed through the GPU in chunks of heads
    (include/attn.h, attn_fwd_host). Q, K, V, C, ckey, O, LSE: contiguous CPU tensors with
    the shapes and dtypes of attn_fwd_ex (page-locked for the copies to overlap); staging:
    a CUDA tensor of at least attn_fwd_host_staging_bytes (see host_staging). The call is
    asynchronous on `stream`."""
    BH, Nq, Nk, d, dv, out_dtype, c_ptr, k_ptr, lse_ptr = _marshal_ex(Q, K, V, C, ckey, O, LSE, mode)
    if staging is None or not staging.is_cuda or not staging.is_contiguous():
        raise ValueError("staging must be a contiguous CUDA tensor (see host_staging)")
    code = attn_fwd_host_raw(Q.data_ptr(), K.data_ptr(), V.data_ptr(), mode, c_ptr, k_ptr, BH, Nq, Nk,
                             d, dv, scale, O.data_ptr(), out_dtype, lse_ptr, staging.data_ptr(),
                             staging.numel() * staging.element_size(), heads_per_chunk,
                             _stream_handle(stream))
    if code != ATTN_OK:
        raise AttnError(code, "attn_fwd_host")
    return O, LSE


def bwd_workspace(BH, Nq, device="cuda"):
    """A workspace tensor (uint8) of the size attn_bwd needs."""
    import torch

    code, nbytes = attn_bwd_workspace_bytes(BH, Nq)
    if code != ATTN_OK:
        raise AttnError(code, "attn_bwd_workspace_bytes")
    return torch.empty(max(nbytes, 16), dtype=torch.uint8, device=device)


def attn_bwd(Q, K, V, O, dO, LSE, mode, C, ckey, scale, dQ, dK, dV, workspace, stream=None):
    """Gradients dQ, dK, dV (fp32, written in place) of the forward pass that produced O and
    LSE from Q, K, V, mode, C, ckey and scale, for the loss gradient dO (bf16, shaped like
    O), through the C ABI (include/attn.h, attn_bwd). `workspace`: see bwd_workspace."""
    import torch

    BH, Nq, Nk, d, dv, o_dtype, c_ptr, k_ptr, lse_ptr = _marshal_ex(Q, K, V, C, ckey, O, LSE, mode)
    if LSE is None:
        raise ValueError("the backward pass needs the forward LSE")
    if dO.dtype != torch.bfloat16 or tuple(dO.shape) != (BH, Nq, dv) or not dO.is_contiguous():
        raise ValueError("dO must be a contiguous bf16 [BH, Nq, d_v] tensor")
    for name, t, shape in (("dQ", dQ, (BH, Nq, d)), ("dK", dK, (BH, Nk, d)), ("dV", dV, (BH, Nk, dv))):
        if t.dtype != torch.float32 or tuple(t.shape) != shape or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous fp32 {list(shape)} tensor")
    if not workspace.is_contiguous():
        raise ValueError("workspace must be contiguous")
    code = attn_bwd_raw(Q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(), o_dtype,
                        dO.data_ptr(), lse_ptr, mode, c_ptr, k_ptr, BH, Nq, Nk, d, dv, scale,
                        dQ.data_ptr(), dK.data_ptr(), dV.data_ptr(), workspace.data_ptr(),
                        workspace.numel() * workspace.element_size(), _stream_handle(stream))
    if code != ATTN_OK:
        raise AttnError(code, "attn_bwd")
    return dQ, dK, dV


def bwd_host_staging(mode, BH, Nq, Nk, d, d_v, o_dtype, heads_per_chunk=0, device="cuda"):
    """A device staging tensor (uint8) of the size attn_bwd_host needs."""
    import torch

    code, nbytes = attn_bwd_host_staging_bytes(mode, BH, Nq, Nk, d, d_v, o_dtype, heads_per_chunk)
    if code != ATTN_OK:
        raise AttnError(code, "attn_bwd_host_staging_bytes")
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def attn_bwd_host(Q, K, V, O, dO, LSE, mode, C, ckey, scale, dQ, dK, dV, staging, heads_per_chunk=0,
                  stream=None):
    """attn_bwd on host (CPU) tensors, streamed through the GPU in chunks of heads
    (include/attn.h, attn_bwd_host); the arguments of attn_bwd, all on the CPU, plus a CUDA
    staging tensor (see bwd_host_staging). Asynchronous on `stream`."""
    import torch

    for name, t in (("Q", Q), ("K", K), ("V", V), ("O", O), ("dO", dO), ("LSE", LSE), ("dQ", dQ),
                    ("dK", dK), ("dV", dV)):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CPU tensor")
    if staging is None or not staging.is_cuda or not staging.is_contiguous():
        raise ValueError("staging must be a contiguous CUDA tensor (see bwd_host_staging)")
    BH, Nq, d = Q.shape
    Nk, dv = K.shape[1], V.shape[2]
    o_dtype = ATTN_OUT_F32 if O.dtype == torch.float32 else ATTN_OUT_BF16
    code = attn_bwd_host_raw(Q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(), o_dtype,
                             dO.data_ptr(), LSE.data_ptr(), mode,
                             None if C is None else C.data_ptr(), None if ckey is None else ckey.data_ptr(),
                             BH, Nq, Nk, d, dv, scale, dQ.data_ptr(), dK.data_ptr(), dV.data_ptr(),
                             staging.data_ptr(), staging.numel() * staging.element_size(), heads_per_chunk,
                             _stream_handle(stream))
    if code != ATTN_OK:
        raise AttnError(code, "attn_bwd_host")
    return dQ, dK, dV


def attention(q, k, v, causal=False, bias=None, key_bias=None, scale=None):
    """Differentiable attention on the library's kernels (see autograd.attention)."""
    from .autograd import attention as _attention

    return _attention(q, k, v, causal, bias, key_bias, scale)
