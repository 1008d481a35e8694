"""Python binding of libkda (ctypes).  Argument marshalling only.

Every step of the recurrence runs in the CUDA kernels behind the C ABI in
``include/kda.h``.  PyTorch supplies device memory and the stream; nothing
here computes any part of the method, and there is no CPU fallback: if the
library is missing or a call fails, an exception is raised.

The names follow the C ABI: ``prefill`` / ``prefill_into`` wrap
``kda_prefill`` / ``kda_prefill_ex``, ``decode_step`` wraps
``kda_decode_step``, ``workspace_size`` wraps ``kda_prefill_workspace_size``
(``kda_prefill_workspace_size_tokens`` when given the token count),
``device_status`` wraps ``kda_prefill_device_status`` and ``backward`` /
``backward_into`` / ``backward_workspace_size`` wrap ``kda_backward`` and
``kda_backward_workspace_size``; ``attnres_layer`` wraps the Blocked Attention
Residuals call of ``include/attnres.h``.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libkda.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_DEVICE_INPUT, ERR_DEVICE_TIMEOUT = 0, 1, 2, 3, 4, 5
ERR_DEVICE_RANGE = 6
BF16, FP32 = 0, 1
KERNEL_AUTO, KERNEL_CHUNK_SIMT, KERNEL_CHUNK_TC, KERNEL_CHUNK_TC_SPLIT = 0, 1, 2, 3
_KERNELS = {"auto": KERNEL_AUTO, "simt": KERNEL_CHUNK_SIMT, "tc": KERNEL_CHUNK_TC,
            "tc_split": KERNEL_CHUNK_TC_SPLIT}
GATE_CHANNEL_F32, GATE_HEAD_F32, GATE_CHANNEL_LOG_BF16 = 0, 1, 2
# gate layout -> (code, dtype, alpha tensor rank)
_GATES = {"channel": (GATE_CHANNEL_F32, torch.float32, 3),
          "head": (GATE_HEAD_F32, torch.float32, 2),
          "log_bf16": (GATE_CHANNEL_LOG_BF16, torch.bfloat16, 3)}

_lib = None


class KdaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


def load(path: str | None = None):
    """Load libkda.so (built by ``gated_delta_rule_45_gb300.build``); raise if absent."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"libkda.so not found at {p}: build it with "
                           "`python -m gated_delta_rule_45_gb300.build` (needs nvcc)")
    lib = ctypes.CDLL(p)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    lib.kda_prefill_workspace_size.restype = sz
    lib.kda_prefill_workspace_size.argtypes = [i32, i32, i32, i32, i32]
    lib.kda_prefill_workspace_size_tokens.restype = sz
    lib.kda_prefill_workspace_size_tokens.argtypes = [i32, i64, i32, i32, i32, i32]
    prefill_args = [vp, vp, vp, vp, vp, vp, vp, i32, i64, i32, i32, i32, ctypes.c_int, i32,
                    vp, vp, vp, sz]
    lib.kda_prefill.restype = ctypes.c_int
    lib.kda_prefill.argtypes = prefill_args + [vp]
    lib.kda_prefill_ex.restype = ctypes.c_int
    lib.kda_prefill_ex.argtypes = prefill_args + [ctypes.c_int, vp]
    lib.kda_prefill_gates.restype = ctypes.c_int
    lib.kda_prefill_gates.argtypes = [vp, vp, vp, vp, ctypes.c_int] + prefill_args[4:] + \
        [ctypes.c_int, vp]
    lib.kda_prefill_noalloc.restype = ctypes.c_int
    lib.kda_prefill_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i64, i32, i32, i32,
                                        ctypes.c_int, i32, vp, vp, vp]
    lib.kda_prefill_supported.restype = ctypes.c_int
    lib.kda_prefill_supported.argtypes = [ctypes.c_int, i32, i32, i32, ctypes.c_int, i32]
    lib.kda_segment_combine.restype = ctypes.c_int
    lib.kda_segment_combine.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, vp, vp]
    lib.kda_check_wait_timeout.restype = ctypes.c_int
    lib.kda_check_wait_timeout.argtypes = [vp, sz, ctypes.c_uint64, vp]
    lib.kda_prefill_device_status.restype = ctypes.c_int
    lib.kda_prefill_device_status.argtypes = [vp, vp]
    lib.kda_decode_step.restype = ctypes.c_int
    lib.kda_decode_step.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, ctypes.c_int,
                                    vp, vp]
    lib.kda_decode_step_gates.restype = ctypes.c_int
    lib.kda_decode_step_gates.argtypes = [vp, vp, vp, vp, ctypes.c_int, vp, vp, i32, i32, i32,
                                          i32, ctypes.c_int, vp, vp]
    lib.kda_backward_workspace_size.restype = sz
    lib.kda_backward_workspace_size.argtypes = [i32, i64, i32, i32, i32, i32]
    lib.kda_backward.restype = ctypes.c_int
    lib.kda_backward.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i64, i32, i32, i32,
                                 ctypes.c_int, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.kda_prefill_additive.restype = ctypes.c_int
    lib.kda_prefill_additive.argtypes = prefill_args + [ctypes.c_int, vp]
    lib.kda_decode_step_additive.restype = ctypes.c_int
    lib.kda_decode_step_additive.argtypes = lib.kda_decode_step.argtypes
    lib.kda_backward_gates_workspace_size.restype = sz
    lib.kda_backward_gates_workspace_size.argtypes = [i32, i64, i32, i32, i32, i32, ctypes.c_int]
    lib.kda_backward_gates.restype = ctypes.c_int
    lib.kda_backward_gates.argtypes = [vp, vp, vp, vp, ctypes.c_int, vp, vp, vp, i32, i64, i32,
                                       i32, i32, ctypes.c_int, i32, vp, vp, vp, vp, vp, vp, vp,
                                       vp, vp, sz, vp]
    lib.attnres_layer.restype = ctypes.c_int
    lib.attnres_layer.argtypes = [vp, i32, vp, vp, vp, vp, vp, ctypes.c_float, i64, i32,
                                  ctypes.c_int, vp, vp]
    lib.kda_status_string.restype = ctypes.c_char_p
    lib.kda_status_string.argtypes = [ctypes.c_int]
    lib.kda_version.restype = i32
    lib.kda_version.argtypes = []
    if path is None:
        _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().kda_status_string(int(status)).decode()


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_ptr(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return FP32
    raise TypeError(f"the storage dtype must be bfloat16 or float32, got {t.dtype}")


# Types are checked before placement, for every entry point: the C ABI reads
# alpha, beta, states and gradients as fp32 and cu_seqlens as int32, so a
# tensor of another type would be misread rather than rejected.
def _check_qkv(q, *others):
    """q and the tensors stored like it (k, v, o, dO) share one dtype, bf16 or fp32."""
    _dtype_code(q)
    for t in others:
        if t is not None and t.dtype != q.dtype:
            raise TypeError("q, k, v and the tensors stored like them must share one dtype")


def _check_f32(what: str, *ts):
    for t in ts:
        if t is not None and t.dtype != torch.float32:
            raise TypeError(f"{what} must be float32")


def _check_int32(cu_seqlens):
    if cu_seqlens.dtype != torch.int32:
        raise TypeError("cu_seqlens must be int32")


def _check_cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("all tensors must be contiguous CUDA tensors")


def supported(kernel: str, H: int, d_k: int, d_v: int, dtype: torch.dtype, chunk: int) -> bool:
    """Whether kda_prefill_ex with this kernel choice accepts the shape (host-only query)."""
    code = BF16 if dtype == torch.bfloat16 else FP32
    return load().kda_prefill_supported(_KERNELS[kernel], H, d_k, d_v, code, chunk) == OK


def workspace_size(num_seqs: int, H: int = 1, d_k: int = 128, d_v: int = 128,
                   chunk: int = 64, total_tokens: int | None = None) -> int:
    """Prefill workspace bytes: kda_prefill_workspace_size_tokens when the
    token count is given (room for the sequence-axis split where it applies),
    else kda_prefill_workspace_size (no split)."""
    if total_tokens is None:
        return int(load().kda_prefill_workspace_size(num_seqs, H, d_k, d_v, chunk))
    return int(load().kda_prefill_workspace_size_tokens(num_seqs, total_tokens, H, d_k, d_v,
                                                        chunk))


def prefill_into(q, k, v, alpha, beta, S0, cu_seqlens, o, S_T, workspace, *, chunk: int = 64,
                 kernel: str = "auto", stream=None) -> None:
    """Enqueue kda_prefill_ex on `stream` (default: current stream) into preallocated outputs.

    q, k: [T, H, d_k]; v, o: [T, H, d_v] (bf16 or fp32, all the same); alpha:
    [T, H, d_v] fp32; beta: [T, H] fp32; S0: [N, H, d_v, d_k] fp32 or None;
    cu_seqlens: int32 [N+1] on the device; S_T: [N, H, d_v, d_k] fp32 (may be S0);
    workspace: a uint8 device tensor of at least ``workspace_size(N)`` bytes.
    """
    _check_int32(cu_seqlens)
    _check_f32("alpha, beta and the states", alpha, beta, S0, S_T)
    _check_qkv(q, k, v, o)
    _check_cuda(q, k, v, alpha, beta, S0, cu_seqlens, o, S_T, workspace)
    T, H, d_k = q.shape
    d_v = v.shape[2]
    N = cu_seqlens.numel() - 1
    dt = _dtype_code(q)
    st = load().kda_prefill_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(S0),
                               _ptr(cu_seqlens), N, T, H, d_k, d_v, dt, chunk, _ptr(o),
                               _ptr(S_T), _ptr(workspace), workspace.numel(), _KERNELS[kernel],
                               _stream_ptr(stream))
    if st != OK:
        raise KdaError(st, "kda_prefill")


def prefill_gates_into(q, k, v, alpha, beta, S0, cu_seqlens, o, S_T, workspace, *,
                       gate: str = "channel", chunk: int = 64, kernel: str = "auto",
                       stream=None) -> None:
    """Enqueue kda_prefill_gates: as prefill_into with the forget gate in layout `gate`:
    "channel" alpha [T, H, d_v] fp32, "head" alpha [T, H] fp32 (one gate per head),
    "log_bf16" log alpha [T, H, d_v] bf16."""
    code, adt, arank = _GATES[gate]
    if alpha.dtype != adt or alpha.dim() != arank:
        raise TypeError(f"gate layout {gate!r} wants a rank-{arank} {adt} tensor")
    _check_int32(cu_seqlens)
    _check_f32("beta and the states", beta, S0, S_T)
    _check_qkv(q, k, v, o)
    _check_cuda(q, k, v, alpha, beta, S0, cu_seqlens, o, S_T, workspace)
    T, H, d_k = q.shape
    d_v = v.shape[2]
    N = cu_seqlens.numel() - 1
    dt = _dtype_code(q)
    st = load().kda_prefill_gates(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), code, _ptr(beta),
                                  _ptr(S0), _ptr(cu_seqlens), N, T, H, d_k, d_v, dt, chunk,
                                  _ptr(o), _ptr(S_T), _ptr(workspace), workspace.numel(),
                                  _KERNELS[kernel], _stream_ptr(stream))
    if st != OK:
        raise KdaError(st, "kda_prefill_gates")


def prefill_gates(q, k, v, alpha, beta, S0, cu_seqlens, *, gate: str = "channel",
                  chunk: int = 64, kernel: str = "auto", stream=None,
                  check_device_status: bool = False):
    """Allocate outputs with PyTorch and run kda_prefill_gates; returns (o, S_T)."""
    T, H, d_k = q.shape
    d_v = v.shape[2]
    N = cu_seqlens.numel() - 1
    o = torch.empty((T, H, d_v), dtype=q.dtype, device=q.device)
    S_T = torch.empty((N, H, d_v, d_k), dtype=torch.float32, device=q.device)
    ws = torch.empty(workspace_size(N, H, d_k, d_v, chunk, T), dtype=torch.uint8,
                     device=q.device)
    prefill_gates_into(q, k, v, alpha, beta, S0, cu_seqlens, o, S_T, ws, gate=gate, chunk=chunk,
                       kernel=kernel, stream=stream)
    if check_device_status:
        device_status(ws, stream=stream)
    return o, S_T


def prefill(q, k, v, alpha, beta, S0, cu_seqlens, *, chunk: int = 64, kernel: str = "auto",
            stream=None, check_device_status: bool = False):
    """Allocate outputs with PyTorch and run kda_prefill; returns (o, S_T)."""
    T, H, d_k = q.shape
    d_v = v.shape[2]
    N = cu_seqlens.numel() - 1
    o = torch.empty((T, H, d_v), dtype=q.dtype, device=q.device)
    S_T = torch.empty((N, H, d_v, d_k), dtype=torch.float32, device=q.device)
    ws = torch.empty(workspace_size(N, H, d_k, d_v, chunk, T), dtype=torch.uint8,
                     device=q.device)
    prefill_into(q, k, v, alpha, beta, S0, cu_seqlens, o, S_T, ws, chunk=chunk, kernel=kernel,
                 stream=stream)
    if check_device_status:
        device_status(ws, stream=stream)
    return o, S_T


NOALLOC_MAX_SEQS = 65536


def prefill_noalloc_into(q, k, v, alpha, beta, S0, cu_seqlens, o, S_T, *, chunk: int = 64,
                         stream=None) -> None:
    """Enqueue kda_prefill_noalloc: like ``prefill_into`` but the scratch lives in
    the library (for callers that cannot allocate).  Calls must not overlap on
    the GPU; at most NOALLOC_MAX_SEQS sequences."""
    _check_int32(cu_seqlens)
    _check_f32("alpha, beta and the states", alpha, beta, S0, S_T)
    _check_qkv(q, k, v, o)
    _check_cuda(q, k, v, alpha, beta, S0, cu_seqlens, o, S_T)
    T, H, d_k = q.shape
    d_v = v.shape[2]
    N = cu_seqlens.numel() - 1
    if N > NOALLOC_MAX_SEQS:
        raise ValueError(f"kda_prefill_noalloc takes at most {NOALLOC_MAX_SEQS} sequences, "
                         f"got {N}")
    st = load().kda_prefill_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta),
                                    _ptr(S0), _ptr(cu_seqlens), N, T, H, d_k, d_v,
                                    _dtype_code(q), chunk, _ptr(o), _ptr(S_T),
                                    _stream_ptr(stream))
    if st != OK:
        raise KdaError(st, "kda_prefill_noalloc")


def segment_combine(S_in, g, P, R, S_out=None, *, stream=None):
    """Enqueue kda_segment_combine: S_out = diag(g) S_in P + R per (sequence, head);
    S_in, R [N, H, d_v, d_k], g [N, H, d_v], P [N, H, d_k, d_k], fp32.  Returns S_out."""
    _check_f32("segment maps", S_in, g, P, R)
    _check_cuda(S_in, g, P, R)
    N, H, d_v, d_k = S_in.shape
    if S_out is None:
        S_out = torch.empty_like(S_in)
    st = load().kda_segment_combine(_ptr(S_in), _ptr(g), _ptr(P), _ptr(R), N, H, d_k, d_v,
                                    _ptr(S_out), _stream_ptr(stream))
    if st != OK:
        raise KdaError(st, "kda_segment_combine")
    return S_out


def check_wait_timeout(workspace, timeout_ns: int, *, stream=None) -> None:
    """Enqueue kda_check_wait_timeout: the prefill's device-side timeout path
    run on purpose; afterwards the workspace's status reads
    ERR_DEVICE_TIMEOUT."""
    _check_cuda(workspace)
    st = load().kda_check_wait_timeout(_ptr(workspace), workspace.numel() * workspace.element_size(),
                                       int(timeout_ns), _stream_ptr(stream))
    if st != OK:
        raise KdaError(st, "kda_check_wait_timeout")


def device_status(workspace, stream=None) -> None:
    """Synchronise `stream` and raise KdaError if the device rejected the last prefill's input."""
    st = load().kda_prefill_device_status(_ptr(workspace), _stream_ptr(stream))
    if st != OK:
        raise KdaError(st, "kda_prefill (device check)")


def decode_step(q, k, v, alpha, beta, S, o=None, *, stream=None):
    """Enqueue kda_decode_step: S [B, H, d_v, d_k] fp32 updated in place; returns o [B, H, d_v]."""
    B, H, d_k = q.shape
    d_v = v.shape[2]
    if o is None:
        o = torch.empty((B, H, d_v), dtype=q.dtype, device=q.device)
    _check_f32("S, alpha and beta", S, alpha, beta)
    _check_qkv(q, k, v, o)
    _check_cuda(q, k, v, alpha, beta, S, o)
    dt = _dtype_code(q)
    st = load().kda_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(S),
                                B, H, d_k, d_v, dt, _ptr(o), _stream_ptr(stream))
    if st != OK:
        raise KdaError(st, "kda_decode_step")
    return o


def decode_step_gates(q, k, v, alpha, beta, S, o=None, *, gate: str = "channel", stream=None):
    """kda_decode_step_gates: decode_step with the forget gate in layout `gate`
    ("channel" alpha [B, H, d_v] fp32, "head" alpha [B, H] fp32, "log_bf16" log
    alpha [B, H, d_v] bf16); S updated in place; returns o [B, H, d_v]."""
    code, adt, arank = _GATES[gate]
    B, H, d_k = q.shape
    d_v = v.shape[2]
    if o is None:
        o = torch.empty((B, H, d_v), dtype=q.dtype, device=q.device)
    if alpha.dtype != adt or alpha.dim() != arank:
        raise TypeError(f"gate layout {gate!r} wants a rank-{arank} {adt} tensor")
    _check_f32("S and beta", S, beta)
    _check_qkv(q, k, v, o)
    _check_cuda(q, k, v, alpha, beta, S, o)
    dt = _dtype_code(q)
    st = load().kda_decode_step_gates(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), code, _ptr(beta),
                                      _ptr(S), B, H, d_k, d_v, dt, _ptr(o), _stream_ptr(stream))
    if st != OK:
        raise KdaError(st, "kda_decode_step_gates")
    return o


def prefill_additive_into(q, k, v, alpha, beta, S0, cu_seqlens, o, S_T, workspace, *,
                          chunk: int = 64, kernel: str = "auto", stream=None) -> None:
    """Enqueue kda_prefill_additive into preallocated outputs (as prefill_into)."""
    T, H, d_k = q.shape
    d_v = v.shape[2]
    N = cu_seqlens.numel() - 1
    _check_int32(cu_seqlens)
    _check_f32("alpha, beta and the states", alpha, beta, S0, S_T)
    _check_qkv(q, k, v, o)
    _check_cuda(q, k, v, alpha, beta, S0, cu_seqlens, o, S_T, workspace)
    st = load().kda_prefill_additive(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta),
                                     _ptr(S0), _ptr(cu_seqlens), N, T, H, d_k, d_v,
                                     _dtype_code(q), chunk, _ptr(o), _ptr(S_T), _ptr(workspace),
                                     workspace.numel(), _KERNELS[kernel], _stream_ptr(stream))
    if st != OK:
        raise KdaError(st, "kda_prefill_additive")


def prefill_additive(q, k, v, alpha, beta, S0, cu_seqlens, *, chunk: int = 64,
                     kernel: str = "auto", stream=None, check_device_status: bool = False):
    """kda_prefill_additive: the additive update of linear attention (no predict
    step; naive linear attention when alpha = beta = 1).  Returns (o, S_T)."""
    T, H, d_k = q.shape
    d_v = v.shape[2]
    N = cu_seqlens.numel() - 1
    o = torch.empty((T, H, d_v), dtype=q.dtype, device=q.device)
    S_T = torch.empty((N, H, d_v, d_k), dtype=torch.float32, device=q.device)
    ws = torch.empty(workspace_size(N, H, d_k, d_v, chunk, T), dtype=torch.uint8,
                     device=q.device)
    prefill_additive_into(q, k, v, alpha, beta, S0, cu_seqlens, o, S_T, ws, chunk=chunk,
                          kernel=kernel, stream=stream)
    if check_device_status:
        device_status(ws, stream=stream)
    return o, S_T


def decode_step_additive(q, k, v, alpha, beta, S, o=None, *, stream=None):
    """kda_decode_step_additive: one step of the additive update, S in place; returns o."""
    B, H, d_k = q.shape
    d_v = v.shape[2]
    if o is None:
        o = torch.empty((B, H, d_v), dtype=q.dtype, device=q.device)
    _check_f32("S, alpha and beta", S, alpha, beta)
    _check_qkv(q, k, v, o)
    _check_cuda(q, k, v, alpha, beta, S, o)
    st = load().kda_decode_step_additive(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta),
                                         _ptr(S), B, H, d_k, d_v, _dtype_code(q), _ptr(o),
                                         _stream_ptr(stream))
    if st != OK:
        raise KdaError(st, "kda_decode_step_additive")
    return o


def backward_workspace_size(num_seqs: int, total_tokens: int, H: int, d_k: int = 128,
                            d_v: int = 128, chunk: int = 64) -> int:
    """kda_backward_workspace_size: bytes of workspace (0: shape not supported)."""
    return int(load().kda_backward_workspace_size(num_seqs, total_tokens, H, d_k, d_v, chunk))


def backward_into(q, k, v, alpha, beta, S0, cu_seqlens, dO, dS_T, grads, workspace, *,
                  chunk: int = 64, stream=None) -> None:
    """Enqueue kda_backward into preallocated fp32 gradients.

    Inputs as ``prefill_into`` (bf16 q, k, v); dO: [T, H, d_v] bf16; dS_T:
    [N, H, d_v, d_k] fp32 or None; grads: dict with "dq", "dk" [T, H, d_k],
    "dv", "dalpha" [T, H, d_v], "dbeta" [T, H] and optionally "dS0"
    [N, H, d_v, d_k], all fp32; workspace: uint8 device tensor of at least
    ``backward_workspace_size`` bytes.
    """
    dS0 = grads.get("dS0")
    _check_int32(cu_seqlens)
    _check_qkv(q, k, v, dO)
    _check_f32("alpha, beta, states and gradients", alpha, beta, S0, dS_T, grads["dq"],
               grads["dk"], grads["dv"], grads["dalpha"], grads["dbeta"], dS0)
    _check_cuda(q, k, v, alpha, beta, S0, cu_seqlens, dO, dS_T, grads["dq"], grads["dk"],
                grads["dv"], grads["dalpha"], grads["dbeta"], dS0, workspace)
    T, H, d_k = q.shape
    d_v = v.shape[2]
    N = cu_seqlens.numel() - 1
    st = load().kda_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(S0),
                             _ptr(cu_seqlens), N, T, H, d_k, d_v, _dtype_code(q), chunk,
                             _ptr(dO), _ptr(dS_T), _ptr(grads["dq"]), _ptr(grads["dk"]),
                             _ptr(grads["dv"]), _ptr(grads["dalpha"]), _ptr(grads["dbeta"]),
                             _ptr(dS0), _ptr(workspace), workspace.numel(), _stream_ptr(stream))
    if st != OK:
        raise KdaError(st, "kda_backward")


def backward(q, k, v, alpha, beta, S0, cu_seqlens, dO, dS_T=None, *, chunk: int = 64,
             stream=None, check_device_status: bool = False):
    """Allocate fp32 gradients with PyTorch and run kda_backward; returns a dict
    with dq, dk, dv, dalpha, dbeta and dS0 (tokens past cu_seqlens[-1] zero)."""
    T, H, d_k = q.shape
    d_v = v.shape[2]
    N = cu_seqlens.numel() - 1
    dev = q.device
    grads = {"dq": torch.zeros((T, H, d_k), dtype=torch.float32, device=dev),
             "dk": torch.zeros((T, H, d_k), dtype=torch.float32, device=dev),
             "dv": torch.zeros((T, H, d_v), dtype=torch.float32, device=dev),
             "dalpha": torch.zeros((T, H, d_v), dtype=torch.float32, device=dev),
             "dbeta": torch.zeros((T, H), dtype=torch.float32, device=dev),
             "dS0": torch.zeros((N, H, d_v, d_k), dtype=torch.float32, device=dev)}
    nbytes = backward_workspace_size(N, T, H, d_k, d_v, chunk)
    if nbytes == 0:
        raise KdaError(ERR_UNSUPPORTED, "kda_backward")
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    backward_into(q, k, v, alpha, beta, S0, cu_seqlens, dO, dS_T, grads, ws, chunk=chunk,
                  stream=stream)
    if check_device_status:
        device_status(ws, stream=stream)
    return grads


def backward_gates(q, k, v, alpha, beta, S0, cu_seqlens, dO, dS_T=None, *, gate: str = "channel",
                   chunk: int = 64, stream=None, check_device_status: bool = False):
    """kda_backward_gates: ``backward`` with the forget gate in layout `gate`
    ("channel", "head" [T, H] fp32, "log_bf16" log alpha [T, H, d_v] bf16).
    Returns the gradients; "dgate" is the gradient with respect to the gate in
    its own layout ([T, H] for "head", d/d log alpha for "log_bf16")."""
    code, adt, arank = _GATES[gate]
    T, H, d_k = q.shape
    d_v = v.shape[2]
    N = cu_seqlens.numel() - 1
    if alpha.dtype != adt or alpha.dim() != arank:
        raise TypeError(f"gate layout {gate!r} wants a rank-{arank} {adt} tensor")
    _check_int32(cu_seqlens)
    _check_f32("beta and the states", beta, S0, dS_T)
    _check_qkv(q, k, v, dO)
    _check_cuda(q, k, v, alpha, beta, S0, cu_seqlens, dO, dS_T)
    dev = q.device
    gshape = (T, H) if gate == "head" else (T, H, d_v)
    grads = {"dq": torch.zeros((T, H, d_k), dtype=torch.float32, device=dev),
             "dk": torch.zeros((T, H, d_k), dtype=torch.float32, device=dev),
             "dv": torch.zeros((T, H, d_v), dtype=torch.float32, device=dev),
             "dgate": torch.zeros(gshape, dtype=torch.float32, device=dev),
             "dbeta": torch.zeros((T, H), dtype=torch.float32, device=dev),
             "dS0": torch.zeros((N, H, d_v, d_k), dtype=torch.float32, device=dev)}
    lib = load()
    nbytes = int(lib.kda_backward_gates_workspace_size(N, T, H, d_k, d_v, chunk, code))
    if nbytes == 0:
        raise KdaError(ERR_UNSUPPORTED, "kda_backward_gates")
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    st = lib.kda_backward_gates(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), code, _ptr(beta),
                                _ptr(S0), _ptr(cu_seqlens), N, T, H, d_k, d_v, _dtype_code(q),
                                chunk, _ptr(dO), _ptr(dS_T), _ptr(grads["dq"]), _ptr(grads["dk"]),
                                _ptr(grads["dv"]), _ptr(grads["dgate"]), _ptr(grads["dbeta"]),
                                _ptr(grads["dS0"]), _ptr(ws), ws.numel(), _stream_ptr(stream))
    if st != OK:
        raise KdaError(st, "kda_backward_gates")
    if check_device_status:
        device_status(ws, stream=stream)
    return grads


def attnres_layer(blocks, q, *, partial=None, h_last=None, partial_out=None, block_out=None,
                  scale=None, h=None, stream=None):
    """Enqueue attnres_layer: one layer's input under Blocked Attention Residuals.

    blocks: [nb, T, d] (bf16 or fp32; nb may be 0 when partial or h_last is
    given); q: [d] fp32; partial: [T, d] fp32 or None; h_last: [T, d] like
    blocks or None; partial_out: [T, d] fp32 or None (may be partial);
    block_out: [T, d] like blocks or None; scale: default 1/sqrt(d).
    Returns h [T, d] (allocated when not given)."""
    nb, T, d = blocks.shape
    if h is None:
        h = torch.empty((T, d), dtype=blocks.dtype, device=blocks.device)
    _dtype_code(blocks)
    _check_f32("q", q)
    _check_f32("the running sum", partial, partial_out)
    for t in (h_last, block_out, h):
        if t is not None and t.dtype != blocks.dtype:
            raise TypeError("h_last, block_out and h share the dtype of blocks")
    _check_cuda(blocks, q, partial, h_last, partial_out, block_out, h)
    if scale is None:
        scale = 1.0 / float(d) ** 0.5
    st = load().attnres_layer(_ptr(blocks) if nb > 0 else None, nb, _ptr(partial), _ptr(h_last),
                              _ptr(partial_out), _ptr(block_out), _ptr(q), float(scale), T, d,
                              _dtype_code(blocks), _ptr(h), _stream_ptr(stream))
    if st != OK:
        raise KdaError(st, "attnres_layer")
    return h
