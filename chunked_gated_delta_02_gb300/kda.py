"""Python binding of the KDA chunked forward C ABI (argument marshalling only).

``fwd`` mirrors the KDA forward call of the cuLA / FLA API (cuLA README mirror,
"Quick Start"; FlashKDA page, "flash-linear-attention 백엔드로 사용"), with the
in-kernel options fixed on: q/k L2 norm, gate activation with a lower bound and
beta sigmoid. The variants of kda_fwd_ex are chosen from the arguments: a
[B,T,H] gate (one decay per token and head, the gated delta rule), fp32 beta
logits, a bf16 state and the [N,H,K,V] state layout. All compute runs in
libkda.so on the caller's current CUDA stream; torch only provides device memory.
"""
from __future__ import annotations

import ctypes
from typing import Optional, Tuple

import torch

from ._lib import check, lib

__all__ = ["fwd", "fwd_noalloc", "workspace_size", "debug_chunk_matrices", "device_status", "max_chunks",
           "NOALLOC_MAX_SCRATCH", "GATE_PER_HEAD", "BETA_F32", "STATE_BF16", "STATE_KV", "EXP2_POLY",
           "CP_OFF", "CP_SEGMENTS", "plan"]

# Size of the library's fixed scratch array used by fwd_noalloc (KDA_NOALLOC_MAX_SCRATCH).
NOALLOC_MAX_SCRATCH = 16 * 1024 * 1024

# Variant flags of kda_fwd_ex (include/kda.h).
GATE_PER_HEAD, BETA_F32, STATE_BF16, STATE_KV, EXP2_POLY = 0x1, 0x2, 0x4, 0x8, 0x10
# Context parallelism (include/kda.h): off, or forced with n segments per sequence.
CP_OFF = 0x20


def CP_SEGMENTS(n: int) -> int:
    return (int(n) & 0xFF) << 8


def _cp_flags(context_parallel) -> int:
    """None: chosen by the library; False: off; an int n >= 2: n segments per sequence."""
    if context_parallel is None or context_parallel is True:
        return 0
    if context_parallel is False:
        return CP_OFF
    n = int(context_parallel)
    if not 2 <= n <= 64:
        raise ValueError("context_parallel must be None, False, True or a segment count in [2, 64]")
    return CP_SEGMENTS(n)


class _StageEvents(ctypes.Structure):
    _fields_ = [("prep_start", ctypes.c_void_p), ("prep_done", ctypes.c_void_p),
                ("recur_done", ctypes.c_void_p)]


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_ptr(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need(t, name, dtype, shape=None, device=None):
    """Type, dtype, contiguity, shape and device of one tensor argument. The device is compared
    with the reference device (q's) here; that q itself is on a GPU is checked last, so that
    every argument is refused for its own fault."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} must be on {device} (the device of q), got {t.device}")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _on_gpu(q):
    if q.device.type != "cuda":
        raise ValueError("q must be a CUDA tensor (there is no CPU path)")


def _check_inputs(q, k, v, g, beta, A_log, dt_bias, cu_seqlens):
    """Checks the token tensors and the gate parameters of a forward call. Returns
    (B, T, H, K, V, N, flags) with the variant flags the arguments select."""
    if not isinstance(q, torch.Tensor) or q.dim() != 4:
        raise ValueError("q must be a 4-D torch.Tensor [B,T,H,K]")
    if not isinstance(v, torch.Tensor) or v.dim() != 4:
        raise ValueError("v must be a 4-D torch.Tensor [B,T,H,V]")
    B, T, H, K = q.shape
    V = v.shape[-1]
    dev = q.device
    flags = 0
    _need(q, "q", torch.bfloat16, None, dev)
    _need(k, "k", torch.bfloat16, (B, T, H, K), dev)
    if isinstance(g, torch.Tensor) and g.dim() == 3:
        flags |= GATE_PER_HEAD
        _need(g, "g", torch.bfloat16, (B, T, H), dev)
    else:
        _need(g, "g", torch.bfloat16, (B, T, H, K), dev)
    _need(v, "v", torch.bfloat16, (B, T, H, V), dev)
    if isinstance(beta, torch.Tensor) and beta.dtype == torch.float32:
        flags |= BETA_F32
        _need(beta, "beta", torch.float32, (B, T, H), dev)
    else:
        _need(beta, "beta", torch.bfloat16, (B, T, H), dev)
    _need(A_log, "A_log", torch.float32, (H,), dev)
    if dt_bias is not None:
        _need(dt_bias, "dt_bias", torch.float32, None, dev)
        want = H if flags & GATE_PER_HEAD else H * K
        if dt_bias.numel() != want:
            raise ValueError(f"dt_bias must hold {want} values")
    if cu_seqlens is not None:
        _need(cu_seqlens, "cu_seqlens", torch.int32, None, dev)
        if cu_seqlens.dim() != 1 or cu_seqlens.numel() < 1:
            raise ValueError("cu_seqlens must be a 1-D tensor of N + 1 offsets")
        N = cu_seqlens.numel() - 1
    else:
        N = B
    return B, T, H, K, V, N, flags


def workspace_size(B: int, T: int, H: int, K: int, V: int, num_seqs: int, varlen: bool = False,
                   flags: int = 0) -> int:
    """Scratch bytes of a forward call (kda_fwd_workspace_size_ex): `flags` as passed to the call
    (only the context-parallel flags matter), `varlen` whether it passes cu_seqlens."""
    return int(lib().kda_fwd_workspace_size_ex(B, T, H, K, V, num_seqs, int(bool(varlen)), flags))


def plan(B: int, T: int, H: int, K: int, V: int, num_seqs: int, varlen: bool = False, context_parallel=None):
    """(segments per sequence, V columns per recurrence CTA) that a forward call with these sizes
    would use on the current device; 0 segments is the plain recurrence (kda_fwd_plan)."""
    n, bv = ctypes.c_int(0), ctypes.c_int(0)
    rc = lib().kda_fwd_plan(B, T, H, K, V, num_seqs, int(bool(varlen)), _cp_flags(context_parallel),
                            ctypes.byref(n), ctypes.byref(bv))
    check("kda_fwd_plan", rc)
    return int(n.value), int(bv.value)


def max_chunks(B: int, T: int, num_seqs: int) -> int:
    return int(lib().kda_max_chunks(B, T, num_seqs))


def fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor, beta: torch.Tensor,
        A_log: torch.Tensor, dt_bias: Optional[torch.Tensor] = None, lower_bound: float = -5.0,
        scale: Optional[float] = None, initial_state: Optional[torch.Tensor] = None,
        output_final_state: bool = False, cu_seqlens: Optional[torch.Tensor] = None,
        workspace: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
        final_state: Optional[torch.Tensor] = None,
        events=None, state_layout: str = "vk",
        state_dtype: Optional[torch.dtype] = None,
        exp2_poly: bool = False, context_parallel=None) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """KDA chunked forward on the GPU.

    q, k: bf16 [B,T,H,K]; v: bf16 [B,T,H,V]; g: bf16 [B,T,H,K], or [B,T,H] for one
    decay per token and head (then dt_bias is [H]); beta: bf16 or fp32 [B,T,H]
    logits; A_log: fp32 [H]; dt_bias: fp32 [H,K] (or [H*K]) or None;
    initial_state: [N,H,V,K] (state_layout "vk") or [N,H,K,V] ("kv"), fp32 or
    bf16, or None; cu_seqlens: int32 [N+1] or None (then B must be 1).
    state_dtype: dtype of the returned final state when there is no
    initial_state (default fp32; with an initial_state, its dtype).
    exp2_poly: evaluate the per-token decays with the FMA-pipe polynomial
    instead of the SFU exponential (an implementation option, KDA_EXP2_POLY).
    context_parallel: None (the library decides), False (off) or a segment count
    n in [2, 64] (forced): intracard context parallelism of long fixed-length
    sequences (KDA_CP_OFF / KDA_CP_SEGMENTS(n)); ignored with cu_seqlens.
    Returns (o bf16 [B,T,H,V], final_state in the state layout and dtype, or None).
    events: optional (prep_start, prep_done, recur_done) torch.cuda.Event triple
    recorded on the current stream at the kernel boundaries (profiling only; a None
    entry is not recorded). Without prep_done the recurrence kernel's launch
    overlaps the end of the prep kernel, as without events; with it the two run
    one after the other, so that the event splits their times.
    """
    B, T, H, K, V, N, flags = _check_inputs(q, k, v, g, beta, A_log, dt_bias, cu_seqlens)
    if exp2_poly:
        flags |= EXP2_POLY
    flags |= _cp_flags(context_parallel)
    if state_layout not in ("vk", "kv"):
        raise ValueError("state_layout must be 'vk' ([N,H,V,K]) or 'kv' ([N,H,K,V])")
    sshape = (N, H, V, K) if state_layout == "vk" else (N, H, K, V)
    if state_layout == "kv":
        flags |= STATE_KV
    sdt = initial_state.dtype if initial_state is not None else (state_dtype or torch.float32)
    if sdt not in (torch.float32, torch.bfloat16):
        raise TypeError("the state must be float32 or bfloat16")
    if sdt == torch.bfloat16:
        flags |= STATE_BF16
    dev = q.device
    if initial_state is not None:
        _need(initial_state, "initial_state", sdt, sshape, dev)
    if scale is None:
        scale = K ** -0.5
    if out is not None:
        _need(out, "out", torch.bfloat16, (B, T, H, V), dev)
    if output_final_state and final_state is not None:
        _need(final_state, "final_state", sdt, sshape, dev)
    if workspace is not None:
        _need(workspace, "workspace", workspace.dtype, None, dev)
    _on_gpu(q)
    o = out if out is not None else torch.empty(B, T, H, V, dtype=torch.bfloat16, device=dev)
    fs = None
    if output_final_state:
        fs = final_state if final_state is not None else torch.empty(*sshape, dtype=sdt, device=dev)
    need = workspace_size(B, T, H, K, V, N, cu_seqlens is not None, flags)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    elif workspace.numel() * workspace.element_size() < need:
        raise ValueError(f"workspace too small: need {need} bytes")
    ev = None
    if events is not None:
        ev = ctypes.byref(_StageEvents(*[ctypes.c_void_p(e.cuda_event if e is not None else 0)
                                         for e in events]))
    with torch.cuda.device(dev):
        rc = lib().kda_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(A_log),
                              _ptr(dt_bias), float(lower_bound), float(scale),
                              _ptr(initial_state), _ptr(fs), _ptr(cu_seqlens), B, T, H, K, V, N, flags,
                              _ptr(o), _ptr(workspace), workspace.numel() * workspace.element_size(),
                              _stream_ptr(), ev)
    check("kda_fwd", rc)
    return o, fs


def fwd_noalloc(q, k, v, g, beta, A_log, dt_bias=None, lower_bound=-5.0, scale=None, initial_state=None,
                final_state=None, cu_seqlens=None, out=None):
    """KDA forward through kda_fwd_noalloc: the library allocates nothing.

    For callers that cannot allocate device memory (a runtime that owns the
    whole pool, or a path where cudaMalloc is not allowed): the scratch is a
    fixed array inside libkda.so, so the problem must satisfy
    workspace_size(...) <= NOALLOC_MAX_SCRATCH. The caller passes the output
    buffers (`out`, bf16 [B,T,H,V]; `final_state`, fp32 [N,H,V,K] or None).
    Calls that overlap on the GPU share the array and race: keep them ordered.
    Returns (out, final_state).
    """
    B, T, H, K, V, N, flags = _check_inputs(q, k, v, g, beta, A_log, dt_bias, cu_seqlens)
    if flags:
        raise TypeError("fwd_noalloc takes the default variant only: g [B,T,H,K] and bf16 beta")
    dev = q.device
    sshape = (N, H, V, K)
    if initial_state is not None:
        _need(initial_state, "initial_state", torch.float32, sshape, dev)
    if final_state is not None:
        _need(final_state, "final_state", torch.float32, sshape, dev)
    if out is None:
        raise ValueError("fwd_noalloc needs the caller's output buffer `out`")
    _need(out, "out", torch.bfloat16, (B, T, H, V), dev)
    _on_gpu(q)
    need = workspace_size(B, T, H, K, V, N, cu_seqlens is not None, CP_OFF)
    if need > NOALLOC_MAX_SCRATCH:
        raise ValueError(f"problem needs {need} bytes of scratch, more than the fixed {NOALLOC_MAX_SCRATCH}")
    if scale is None:
        scale = K ** -0.5
    with torch.cuda.device(q.device):
        rc = lib().kda_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(A_log), _ptr(dt_bias),
                                   float(lower_bound), float(scale), _ptr(initial_state), _ptr(final_state),
                                   _ptr(cu_seqlens), B, T, H, K, V, N, _ptr(out), _stream_ptr())
    check("kda_fwd_noalloc", rc)
    return out, final_state


def debug_chunk_matrices(q, k, g, beta, A_log, dt_bias=None, lower_bound=-5.0, cu_seqlens=None):
    """The prep kernel's per-(chunk, head) hand-off matrices, fp16 [max_chunks, H, 128, 64] (row-major)."""
    B, T, H, K = q.shape
    N = B if cu_seqlens is None else cu_seqlens.numel() - 1
    mc = max_chunks(B, T, N)
    mats = torch.zeros(max(mc, 1), H, 128, 64, dtype=torch.float16, device=q.device)
    ws = torch.empty(max(workspace_size(B, T, H, K, K, N), 1), dtype=torch.uint8, device=q.device)
    with torch.cuda.device(q.device):
        rc = lib().kda_debug_chunk_matrices(_ptr(q), _ptr(k), _ptr(g), _ptr(beta), _ptr(A_log),
                                            _ptr(dt_bias), float(lower_bound), _ptr(cu_seqlens), B, T,
                                            H, K, N, _ptr(mats), _ptr(ws), ws.numel(), _stream_ptr())
    check("kda_debug_chunk_matrices", rc)
    # undo the 128-byte swizzle of the stored blocks: chunk c of row r sits at r*8 + (c ^ (r % 8))
    r = torch.arange(128, device=mats.device).view(128, 1)
    c = torch.arange(8, device=mats.device).view(1, 8)
    src = (c ^ (r % 8)).view(1, 1, 128, 8, 1).expand(mats.shape[0], H, 128, 8, 8)
    blocks = mats[:mc].view(mc, H, 128, 8, 8)
    return torch.gather(blocks, 3, src[:mc]).view(mc, H, 128, 64)


def device_status(stream=None) -> int:
    """Synchronise and read+clear the device data-error word (0 = none)."""
    code = ctypes.c_int(0)
    rc = lib().kda_get_device_status(_stream_ptr(stream), ctypes.byref(code))
    if rc not in (0, 5):
        check("kda_get_device_status", rc)
    return int(code.value)
