"""GB300-native FlashAttention-2 forward pass (sm_103a).

Python binding of ``libfa2.so`` (C ABI in ``include/fa2.h``).  This module
only marshals arguments: every step of the attention pass runs in the
library's CUDA kernels.  PyTorch provides device memory and streams.  There
is no fallback: if the library is missing or the device is unusable, calls
raise.
"""
from __future__ import annotations

import ctypes
import os

from .build import LIB_PATH

FA2_OK = 0
FA2_ERR_NULL = 1
FA2_ERR_ALIGN = 2
FA2_ERR_SHAPE = 3
FA2_ERR_HEADDIM = 4
FA2_ERR_LAUNCH = 5
FA2_ERR_TIMEOUT = 6
FA2_ERR_SCALE = 7
FA2_ERR_MEMORY = 8
FA2_ERR_DEVICE = 9
FA2_ERR_SCRATCH = 10
FA2_ERR_DTYPE = 11

FA2_DTYPE_BF16 = 0
FA2_DTYPE_FP16 = 1
FA2_DTYPE_FP32 = 2

# Every function the C header declares, with its ctypes signature.
_P, _I, _F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
_FORWARD_ARGS = [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P]
_Z, _LL = ctypes.c_size_t, ctypes.c_longlong
SIGNATURES = {
    "fa2_forward": (_I, _FORWARD_ARGS),
    "fa2_forward_simt": (_I, _FORWARD_ARGS),
    "fa2_forward_typed": (_I, _FORWARD_ARGS[:-1] + [_I, _I, _P]),
    "fa2_splitkv_workspace_bytes": (_Z, [_I, _I, _I, _I, _I]),
    "fa2_forward_splitkv": (_I, _FORWARD_ARGS[:-1] + [_I, _P, _Z, _P]),
    "fa2_splitkv_recommended_splits": (_I, [_I, _I, _I, _I, _I]),
    "fa2_forward_host": (_I, [_P] * 10 + [_I, _I, _I, _I, _I, _I, _F, _I, _P]),
    "fa2_merge": (_I, [_P, _P, _I, _LL, _I, _P, _P, _P]),
    "fa2_forward_splitkv_static": (_I, _FORWARD_ARGS[:-1] + [_I, _P]),
    "fa2_backward_workspace_bytes": (_Z, [_I, _I, _I]),
    "fa2_backward": (_I, [_P] * 9 + [_I] * 6 + [ctypes.c_float, _P, _Z, _P]),
    "fa2_backward_typed": (_I, [_P] * 9 + [_I] * 6 + [ctypes.c_float, _I, _P, _Z, _P]),
    "fa2_status_string": (ctypes.c_char_p, [_I]),
    "fa2_device_status": (_I, [_P, _I]),
    "fa2_check_wait_timeout": (_I, [ctypes.c_ulonglong, _P]),
}

_lib = None


class FA2Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {fa2_status_string(status)} (status {status})")


def library() -> ctypes.CDLL:
    """Load libfa2.so (built in-tree by ``exact_attention_17_gb300.build``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; run `python -m exact_attention_17_gb300.build`")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def fa2_forward(Q, K, V, O, LSE, B, H, Nq, Nk, d, causal, scale, stream) -> int:
    """Raw C call: pointers (ints) and sizes, returns the status code."""
    return library().fa2_forward(Q, K, V, O, LSE, B, H, Nq, Nk, d, int(bool(causal)), scale, stream)


def fa2_forward_typed(Q, K, V, O, LSE, B, H, Nq, Nk, d, causal, scale, qkv_dtype, o_dtype,
                      stream) -> int:
    """Raw C call with element types (FA2_DTYPE_*) for Q/K/V and for O."""
    return library().fa2_forward_typed(Q, K, V, O, LSE, B, H, Nq, Nk, d, int(bool(causal)), scale,
                                       qkv_dtype, o_dtype, stream)


def fa2_forward_simt(Q, K, V, O, LSE, B, H, Nq, Nk, d, causal, scale, stream) -> int:
    """Raw C call of the CUDA-core cross-check implementation."""
    return library().fa2_forward_simt(Q, K, V, O, LSE, B, H, Nq, Nk, d, int(bool(causal)), scale,
                                      stream)


def fa2_splitkv_workspace_bytes(B, H, Nq, d, num_splits) -> int:
    return library().fa2_splitkv_workspace_bytes(B, H, Nq, d, num_splits)


def fa2_forward_splitkv(Q, K, V, O, LSE, B, H, Nq, Nk, d, causal, scale, num_splits, workspace,
                        workspace_size, stream) -> int:
    """Raw C call of the split-KV forward (caller-provided device workspace)."""
    return library().fa2_forward_splitkv(Q, K, V, O, LSE, B, H, Nq, Nk, d, int(bool(causal)), scale,
                                         num_splits, workspace, workspace_size, stream)


def fa2_forward_splitkv_static(Q, K, V, O, LSE, B, H, Nq, Nk, d, causal, scale, num_splits,
                               stream) -> int:
    """Raw C call of the split-KV forward that allocates nothing: its scratch
    is the library's own 32 MiB device array (see include/fa2.h)."""
    return library().fa2_forward_splitkv_static(Q, K, V, O, LSE, B, H, Nq, Nk, d,
                                                int(bool(causal)), scale, num_splits, stream)


def fa2_splitkv_recommended_splits(B, H, Nq, Nk, sm_count=0) -> int:
    """Split count that fills the GPU for fa2_forward_splitkv (see fa2.h)."""
    return library().fa2_splitkv_recommended_splits(B, H, Nq, Nk, sm_count)


def fa2_forward_host(Qh, Kh, Vh, Oh, LSEh, Qd, Kd, Vd, Od, LSEd, B, H, Nq, Nk, d, causal, scale,
                     chunks, stream) -> int:
    """Raw C call of the forward pass from host memory, pipelined over groups of heads."""
    return library().fa2_forward_host(Qh, Kh, Vh, Oh, LSEh, Qd, Kd, Vd, Od, LSEd, B, H, Nq, Nk, d,
                                      int(bool(causal)), scale, chunks, stream)


def fa2_merge(O_parts, LSE_parts, num_parts, rows, d, O, LSE, stream) -> int:
    """Raw C call of the merge of partial attention results."""
    return library().fa2_merge(O_parts, LSE_parts, num_parts, rows, d, O, LSE, stream)


def fa2_backward_workspace_bytes(B, H, Nq) -> int:
    return library().fa2_backward_workspace_bytes(B, H, Nq)


def fa2_backward(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, Nq, Nk, d, causal, scale, workspace,
                 workspace_size, stream) -> int:
    """Raw C call of the backward pass (caller-provided device workspace)."""
    return library().fa2_backward(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, Nq, Nk, d,
                                  int(bool(causal)), scale, workspace, workspace_size, stream)


def fa2_backward_typed(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, Nq, Nk, d, causal, scale, qkv_dtype,
                       workspace, workspace_size, stream) -> int:
    """Raw C call of the backward pass with bf16 or fp16 Q, K, V and dO."""
    return library().fa2_backward_typed(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, Nq, Nk, d,
                                        int(bool(causal)), scale, qkv_dtype, workspace, workspace_size,
                                        stream)


def fa2_status_string(status: int) -> str:
    return library().fa2_status_string(status).decode()


def fa2_device_status(stream=None, reset: bool = False) -> int:
    return library().fa2_device_status(stream, int(bool(reset)))


def fa2_check_wait_timeout(timeout_ns: int, stream=None) -> int:
    """Raw C call: one bounded wait on a barrier nothing completes (see fa2.h)."""
    return library().fa2_check_wait_timeout(int(timeout_ns), stream)


def _stream_handle(stream):
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    handle = getattr(stream, "cuda_stream", None)
    return stream if handle is None else handle


_DTYPE_CODES = None


def _dtype_codes():
    global _DTYPE_CODES
    if _DTYPE_CODES is None:
        import torch

        _DTYPE_CODES = {torch.bfloat16: FA2_DTYPE_BF16, torch.float16: FA2_DTYPE_FP16,
                        torch.float32: FA2_DTYPE_FP32}
    return _DTYPE_CODES


class _on_device:
    """Make `device` current for the call, only when it is not already (the
    switch costs microseconds a small problem does not have)."""

    def __init__(self, device):
        import torch

        self.ctx = None if device.index == torch.cuda.current_device() else torch.cuda.device(device)

    def __enter__(self):
        if self.ctx is not None:
            self.ctx.__enter__()

    def __exit__(self, *exc):
        if self.ctx is not None:
            self.ctx.__exit__(*exc)


def forward(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None,
            stream=None, impl: str = "tc", num_splits=1, workspace=None, out_dtype=None):
    """Attention forward on torch CUDA tensors.

    q: [B,H,Nq,d]; k, v: [B,H,Nk,d]; all bf16 or all fp16, contiguous, on one
    device.  Returns (O [B,H,Nq,d], LSE fp32 [B,H,Nq]); O is fp32 unless
    ``out_dtype`` is the input dtype (then O is stored in that 16-bit type).  ``scale`` defaults to
    1/sqrt(d) rounded to float32.  ``impl="simt"`` runs the CUDA-core
    cross-check implementation instead of the tensor-core one.
    ``num_splits > 1`` runs the split-KV forward over that many key ranges;
    its workspace (a uint8 CUDA tensor) is allocated here unless given.
    ``num_splits="auto"`` takes the count fa2_splitkv_recommended_splits gives
    for the problem on q's device (1 when the grid already fills the GPU).
    """
    import torch

    codes = _dtype_codes()
    in_dtype = q.dtype
    if in_dtype is not torch.bfloat16 and in_dtype is not torch.float16:
        raise ValueError("q must be bf16 or fp16")
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype is not in_dtype or not t.is_cuda or t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous 4-D CUDA tensor of q's dtype")
    out_dtype = torch.float32 if out_dtype is None else out_dtype
    if out_dtype is not torch.float32 and out_dtype is not in_dtype:
        raise ValueError("out_dtype must be fp32 or the input dtype")
    typed = in_dtype is not torch.bfloat16 or out_dtype is not torch.float32
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if k.shape != (B, H, Nk, d) or v.shape != (B, H, Nk, d):
        raise ValueError("k and v must be [B, H, Nk, d] matching q")
    if scale is None:
        scale = float(torch.tensor(d, dtype=torch.float64).rsqrt().float())
    device = q.device
    if out is None:
        out = torch.empty((B, H, Nq, d), dtype=out_dtype, device=device)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=device)
    if (out.dtype is not out_dtype or out.shape != (B, H, Nq, d) or not out.is_contiguous()
            or out.device != device):
        raise ValueError(f"out must be a contiguous {out_dtype} tensor of shape {(B, H, Nq, d)} on {device}")
    if lse.dtype is not torch.float32 or lse.shape != (B, H, Nq) or not lse.is_contiguous() or lse.device != device:
        raise ValueError(f"lse must be a contiguous fp32 tensor of shape {(B, H, Nq)} on {device}")
    with _on_device(device):
        if num_splits == "auto":
            num_splits = fa2_splitkv_recommended_splits(B, H, Nq, Nk, 0)
        args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                B, H, Nq, Nk, d, causal, float(scale))
        sh = _stream_handle(stream)
        if typed:
            if impl != "tc" or num_splits > 1:
                raise ValueError("fp16 inputs and 16-bit outputs run on the single-pass tensor-core path")
            rc = fa2_forward_typed(*args, codes[in_dtype], codes[out_dtype], sh)
            name = "fa2_forward_typed"
        elif num_splits > 1:
            if impl != "tc":
                raise ValueError("split-KV runs on the tensor-core path only")
            need = fa2_splitkv_workspace_bytes(B, H, Nq, d, num_splits)
            if workspace is None:
                workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=device)
            rc = fa2_forward_splitkv(*args, num_splits, workspace.data_ptr(), workspace.numel(), sh)
            name = "fa2_forward_splitkv"
        elif impl == "tc":
            rc = fa2_forward(*args, sh)
            name = "fa2_forward"
        elif impl == "simt":
            rc = fa2_forward_simt(*args, sh)
            name = "fa2_forward_simt"
        else:
            raise ValueError(f"unknown impl {impl!r}")
    if rc != FA2_OK:
        raise FA2Error(rc, name)
    return out, lse


def forward_host(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None,
                 device_buffers=None, chunks: int = 4, stream=None):
    """Attention forward with inputs and outputs in host memory (fa2_forward_host).

    q: [B,H,Nq,d], k, v: [B,H,Nk,d] contiguous bf16 CPU tensors (pinned
    memory lets the copies overlap the computation).  Returns (O, LSE) as
    fp32 CPU tensors (``out``/``lse`` if given; pinned when allocated here).
    ``device_buffers`` = (q_dev, k_dev, v_dev, o_dev, lse_dev) CUDA tensors of
    the full sizes, allocated on the current device unless given.  The call
    is asynchronous on ``stream``: synchronise it before reading the result.
    """
    import torch

    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != torch.bfloat16 or t.is_cuda or t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous 4-D bf16 CPU tensor")
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if tuple(k.shape) != (B, H, Nk, d) or tuple(v.shape) != (B, H, Nk, d):
        raise ValueError("k and v must be [B, H, Nk, d] matching q")
    if scale is None:
        scale = float(torch.tensor(d, dtype=torch.float64).rsqrt().float())
    if out is None:
        out = torch.empty((B, H, Nq, d), dtype=torch.float32).pin_memory()
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32).pin_memory()
    for name, t, shape in (("out", out, (B, H, Nq, d)), ("lse", lse, (B, H, Nq))):
        if t.dtype != torch.float32 or tuple(t.shape) != shape or not t.is_contiguous() or t.is_cuda:
            raise ValueError(f"{name} must be a contiguous fp32 CPU tensor of shape {shape}")
    if device_buffers is None:
        dev = torch.device("cuda", torch.cuda.current_device())
        device_buffers = (torch.empty_like(q, device=dev), torch.empty_like(k, device=dev),
                          torch.empty_like(v, device=dev), torch.empty(out.shape, device=dev),
                          torch.empty(lse.shape, device=dev))
    qd, kd, vd, od, ld = device_buffers
    for name, t, ref in (("q_dev", qd, q), ("k_dev", kd, k), ("v_dev", vd, v), ("o_dev", od, out),
                         ("lse_dev", ld, lse)):
        if (not t.is_cuda or t.dtype != ref.dtype or tuple(t.shape) != tuple(ref.shape)
                or not t.is_contiguous() or t.device != qd.device):
            raise ValueError(f"{name} must be a contiguous CUDA tensor like {name[:-4]} on one device")
    with torch.cuda.device(qd.device):
        rc = fa2_forward_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                              qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), od.data_ptr(), ld.data_ptr(),
                              B, H, Nq, Nk, d, causal, float(scale), int(chunks), _stream_handle(stream))
    if rc != FA2_OK:
        raise FA2Error(rc, "fa2_forward_host")
    return out, lse


def merge(o_parts, lse_parts, out=None, lse=None, stream=None):
    """Merge partial results over disjoint key subsets (fa2_merge).

    o_parts fp32 [P, ..., d], lse_parts fp32 [P, ...] (contiguous CUDA
    tensors); returns (O [..., d], LSE [...]).
    """
    import torch

    if o_parts.dtype != torch.float32 or lse_parts.dtype != torch.float32:
        raise ValueError("parts must be fp32")
    if not (o_parts.is_cuda and lse_parts.is_contiguous() and o_parts.is_contiguous()):
        raise ValueError("parts must be contiguous CUDA tensors")
    P, d = o_parts.shape[0], o_parts.shape[-1]
    if tuple(lse_parts.shape) != tuple(o_parts.shape[:-1]):
        raise ValueError("lse_parts must match o_parts without the last dimension")
    rows = lse_parts.numel() // P if P else 0
    if out is None:
        out = torch.empty(o_parts.shape[1:], dtype=torch.float32, device=o_parts.device)
    if lse is None:
        lse = torch.empty(lse_parts.shape[1:], dtype=torch.float32, device=o_parts.device)
    with torch.cuda.device(o_parts.device):
        rc = fa2_merge(o_parts.data_ptr(), lse_parts.data_ptr(), P, rows, d, out.data_ptr(),
                       lse.data_ptr(), _stream_handle(stream))
    if rc != FA2_OK:
        raise FA2Error(rc, "fa2_merge")
    return out, lse


def backward(q, k, v, o, lse, do, causal: bool = False, scale: float | None = None, dq=None,
             dk=None, dv=None, workspace=None, stream=None):
    """Attention backward on torch CUDA tensors (fa2_backward_typed).

    q, do: [B,H,Nq,d]; k, v: [B,H,Nk,d], all bf16 or all fp16; o fp32
    [B,H,Nq,d] and lse fp32 [B,H,Nq] as returned by ``forward`` for the same
    inputs.  Returns fp32 (dQ, dK, dV).  The workspace (a uint8 CUDA tensor)
    is allocated here unless given.
    """
    import torch

    in_dt = q.dtype
    if in_dt not in (torch.bfloat16, torch.float16):
        raise ValueError("q, k, v and do must be bf16 or fp16")
    for name, t, dt in (("q", q, in_dt), ("k", k, in_dt), ("v", v, in_dt),
                        ("do", do, in_dt), ("o", o, torch.float32), ("lse", lse, torch.float32)):
        if t.dtype != dt or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous {dt} CUDA tensor")
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if (tuple(k.shape) != (B, H, Nk, d) or tuple(v.shape) != (B, H, Nk, d)
            or tuple(o.shape) != (B, H, Nq, d) or tuple(do.shape) != (B, H, Nq, d)
            or tuple(lse.shape) != (B, H, Nq)):
        raise ValueError("shapes must be q, o, do [B,H,Nq,d], k, v [B,H,Nk,d], lse [B,H,Nq]")
    if scale is None:
        scale = float(torch.tensor(d, dtype=torch.float64).rsqrt().float())
    outs = []
    for name, t, shape in (("dq", dq, (B, H, Nq, d)), ("dk", dk, (B, H, Nk, d)), ("dv", dv, (B, H, Nk, d))):
        if t is None:
            t = torch.empty(shape, dtype=torch.float32, device=q.device)
        if t.dtype != torch.float32 or tuple(t.shape) != shape or not t.is_contiguous() or t.device != q.device:
            raise ValueError(f"{name} must be a contiguous fp32 tensor of shape {shape} on {q.device}")
        outs.append(t)
    dq, dk, dv = outs
    need = fa2_backward_workspace_bytes(B, H, Nq)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    with torch.cuda.device(q.device):
        rc = fa2_backward_typed(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
                                lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, Nq, Nk,
                                d, causal, float(scale),
                                FA2_DTYPE_FP16 if in_dt == torch.float16 else FA2_DTYPE_BF16,
                                workspace.data_ptr(), workspace.numel(), _stream_handle(stream))
    if rc != FA2_OK:
        raise FA2Error(rc, "fa2_backward_typed")
    return dq, dk, dv
