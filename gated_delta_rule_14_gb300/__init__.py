"""KLA gated delta-rule recurrence on NVIDIA GB300 (sm_103a): thin Python binding.

The recurrence (Gist.science, "Riepilogo Tecnico: Attenzione Lineare Kaczmarz (KLA)"):
for each sequence and head, a d_k x d_v state S is carried over tokens with
``S~ = alpha (.) S``, ``e = v - S~^T k``, ``beta = eta / (||k||^2 + eps)``,
``S = S~ + beta k e^T`` and the read ``o = S^T q`` after the write. ``alpha`` is a
scalar per token and head, or one value per key channel. ``beta_mode="raw"`` takes
``beta = eta`` instead (the write strength of DeltaNet / Gated DeltaNet), and
``q_scale`` reads with a scaled query, ``o = S^T (s q)`` (GeekNews, "Revisando las
variantes de atencion lineal de la familia DeltaNet", sections "Gated DeltaNet" and
"Kimi Delta Attention").

``chunk_fwd`` runs the chunkwise prefill, ``decode_step`` one fused single-token
step and ``chunk_bwd`` the backward pass (gradients of a loss given dL/do and
dL/dS_T). Both call the C ABI of ``include/kla.h`` through ctypes; torch
only supplies device memory and the current CUDA stream. Every step of the
computation runs in this package's CUDA kernels; if the library is missing the
calls raise.
"""
from __future__ import annotations

from typing import Optional, Tuple

import torch

from . import _native
from ._native import KlaError  # noqa: F401

__all__ = ["chunk_fwd", "chunk_fwd_host", "chunk_bwd", "decode_step", "workspace_size", "bwd_workspace_size",
           "device_status", "KlaError"]


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return _native.KLA_DTYPE_BF16
    if t.dtype == torch.float32:
        return _native.KLA_DTYPE_F32
    raise TypeError(f"q/k/v must be bfloat16 or float32, got {t.dtype}")


def _check_dev(name: str, t: torch.Tensor, dtype=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor (got {t.device})")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _stream_ptr(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


_BETA_MODES = {"kla": _native.KLA_BETA_KACZMARZ, "raw": _native.KLA_BETA_RAW}


def _beta_code(beta_mode: str) -> int:
    if beta_mode not in _BETA_MODES:
        raise ValueError(f"beta_mode must be 'kla' or 'raw', got {beta_mode!r}")
    return _BETA_MODES[beta_mode]


def workspace_size(B: int, T: int, H: int, d_k: int, d_v: int, chunk: int = 64,
                   dtype: torch.dtype = torch.bfloat16, per_channel_gate: bool = False) -> int:
    """Device scratch bytes ``chunk_fwd`` needs for these sizes (0 when none)."""
    code = _native.KLA_DTYPE_BF16 if dtype == torch.bfloat16 else _native.KLA_DTYPE_F32
    gate = _native.KLA_GATE_CHANNEL if per_channel_gate else _native.KLA_GATE_SCALAR
    return int(_native.lib().kla_chunk_fwd_workspace_size(B, T, H, d_k, d_v, chunk, code, gate))


def chunk_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, alpha: torch.Tensor, eta: torch.Tensor,
              eps: float = 1e-6, S0: Optional[torch.Tensor] = None, *, chunk: int = 64,
              out: Optional[torch.Tensor] = None, final_state: bool = True,
              S_T: Optional[torch.Tensor] = None,
              workspace: Optional[torch.Tensor] = None, beta_mode: str = "kla",
              q_scale: float = 1.0) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Chunkwise KLA prefill.

    q, k: [B,T,H,d_k]; v: [B,T,H,d_v] (bf16 or fp32, same dtype); alpha: fp32 [B,T,H]
    (scalar gate) or [B,T,H,d_k] (per-key-channel gate); eta: fp32 [B,T,H];
    S0: fp32 [B,H,d_k,d_v] or None (zeros). Returns (o [B,T,H,d_v] in q's dtype,
    S_T fp32 [B,H,d_k,d_v] or None). ``S_T`` may be passed (it may be ``S0`` itself).
    ``beta_mode``: "kla" (beta = eta / (||k||^2 + eps)) or "raw" (beta = eta);
    ``q_scale``: o = S^T (q_scale q).
    """
    bcode = _beta_code(beta_mode)
    for n, t in (("q", q), ("k", k), ("v", v)):
        _check_dev(n, t)
    dcode = _dtype_code(q)
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k and v must share one dtype")
    if q.dim() != 4:
        raise ValueError("q must be [B, T, H, d_k]")
    B, T, H, d_k = q.shape
    d_v = v.shape[-1]
    if k.shape != q.shape or v.shape[:3] != q.shape[:3]:
        raise ValueError("q, k, v shapes disagree")
    _check_dev("alpha", alpha, torch.float32)
    _check_dev("eta", eta, torch.float32)
    if tuple(alpha.shape) == (B, T, H):
        gate = _native.KLA_GATE_SCALAR
    elif tuple(alpha.shape) == (B, T, H, d_k):
        gate = _native.KLA_GATE_CHANNEL
    else:
        raise ValueError(f"alpha must be [B,T,H] or [B,T,H,d_k], got {tuple(alpha.shape)}")
    if tuple(eta.shape) != (B, T, H):
        raise ValueError("eta must be [B, T, H]")
    if S0 is not None:
        _check_dev("S0", S0, torch.float32)
        if tuple(S0.shape) != (B, H, d_k, d_v):
            raise ValueError("S0 must be [B, H, d_k, d_v]")
    if out is None:
        out = torch.empty((B, T, H, d_v), dtype=q.dtype, device=q.device)
    else:
        _check_dev("out", out, q.dtype)
    if S_T is None and final_state:
        S_T = torch.empty((B, H, d_k, d_v), dtype=torch.float32, device=q.device)
    elif S_T is not None:
        _check_dev("S_T", S_T, torch.float32)
    ws_need = _native.lib().kla_chunk_fwd_workspace_size(B, T, H, d_k, d_v, chunk, dcode, gate)
    if ws_need and workspace is None:
        workspace = torch.empty(ws_need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = _native.lib().kla_chunk_fwd_ex(
        _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(eta), float(eps), _ptr(S0), _ptr(out), _ptr(S_T),
        B, T, H, d_k, d_v, int(chunk), dcode, gate, bcode, float(q_scale), _ptr(workspace), ws_bytes,
        _stream_ptr(q.device))
    _native.check(st, "kla_chunk_fwd_ex")
    return out, S_T


def chunk_fwd_host(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, alpha: torch.Tensor, eta: torch.Tensor,
                   eps: float = 1e-6, S0: Optional[torch.Tensor] = None, *, chunk: int = 64,
                   parts: Optional[int] = None, out: Optional[torch.Tensor] = None, S_T: Optional[torch.Tensor] = None,
                   final_state: bool = True, device=None, buffers: Optional[dict] = None, beta_mode: str = "kla",
                   q_scale: float = 1.0) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Chunkwise prefill of HOST tensors (pin them for overlap): the work runs in ``parts`` parts
    whose host->device copies, prefills and device->host copies overlap (kla_chunk_fwd_host):
    time slices of whole chunks for bf16 with the scalar gate and d = 128 (up to 64 parts, at most
    one per chunk), ranges of whole sequences otherwise (up to min(B, 64) parts).

    Same shapes as ``chunk_fwd``; ``out`` / ``S_T`` are host tensors (pinned ones are allocated
    when None). ``buffers`` (from ``host_buffers``) holds the device tensors, reused across calls.
    Returns (o, S_T) on the host; they are complete once the current stream of ``device`` has
    been synchronised.
    """
    bcode = _beta_code(beta_mode)
    dev = torch.device("cuda") if device is None else torch.device(device)
    for n, t in (("q", q), ("k", k), ("v", v), ("alpha", alpha), ("eta", eta)):
        if t.device.type != "cpu" or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous host tensor")
    dcode = _dtype_code(q)
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k and v must share one dtype")
    if q.dim() != 4 or k.shape != q.shape or v.dim() != 4 or v.shape[:3] != q.shape[:3]:
        raise ValueError("q, k must be [B, T, H, d_k] and v [B, T, H, d_v]")
    B, T, H, d_k = q.shape
    d_v = v.shape[-1]
    if alpha.dtype != torch.float32 or eta.dtype != torch.float32:
        raise TypeError("alpha and eta must be float32")
    if tuple(alpha.shape) == (B, T, H):
        gate = _native.KLA_GATE_SCALAR
    elif tuple(alpha.shape) == (B, T, H, d_k):
        gate = _native.KLA_GATE_CHANNEL
    else:
        raise ValueError(f"alpha must be [B,T,H] or [B,T,H,d_k], got {tuple(alpha.shape)}")
    if tuple(eta.shape) != (B, T, H):
        raise ValueError("eta must be [B, T, H]")
    if S0 is not None and (S0.device.type != "cpu" or S0.dtype != torch.float32 or
                           tuple(S0.shape) != (B, H, d_k, d_v) or not S0.is_contiguous()):
        raise ValueError("S0 must be a contiguous float32 host tensor [B, H, d_k, d_v]")
    if buffers is None:
        buffers = host_buffers(q, v, alpha, device=dev, with_S0=S0 is not None, with_S_T=final_state or S_T is not None)
    if out is None:
        out = torch.empty((B, T, H, d_v), dtype=q.dtype, pin_memory=True)
    if S_T is None and final_state:
        S_T = torch.empty((B, H, d_k, d_v), dtype=torch.float32, pin_memory=True)
    parts = parts or min(B, 8)
    st = _native.lib().kla_chunk_fwd_host(
        _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(eta), _ptr(S0), _ptr(out), _ptr(S_T),
        _ptr(buffers["q"]), _ptr(buffers["k"]), _ptr(buffers["v"]), _ptr(buffers["alpha"]), _ptr(buffers["eta"]),
        _ptr(buffers.get("S0") if S0 is not None else None), _ptr(buffers["o"]),
        _ptr(buffers.get("S_T") if S_T is not None else None), float(eps),
        B, T, H, d_k, d_v, int(chunk), dcode, gate, bcode, float(q_scale), int(parts), _stream_ptr(dev))
    _native.check(st, "kla_chunk_fwd_host")
    return out, S_T


def host_buffers(q: torch.Tensor, v: torch.Tensor, alpha: torch.Tensor, *, device=None, with_S0: bool = False,
                 with_S_T: bool = True) -> dict:
    """Device tensors for ``chunk_fwd_host`` calls on host tensors shaped like q, v and alpha."""
    dev = torch.device("cuda") if device is None else torch.device(device)
    B, T, H, d_k = q.shape
    d_v = v.shape[-1]
    b = {"q": torch.empty(q.shape, dtype=q.dtype, device=dev), "k": torch.empty(q.shape, dtype=q.dtype, device=dev),
         "v": torch.empty(v.shape, dtype=v.dtype, device=dev),
         "alpha": torch.empty(alpha.shape, dtype=torch.float32, device=dev),
         "eta": torch.empty((B, T, H), dtype=torch.float32, device=dev),
         "o": torch.empty((B, T, H, d_v), dtype=q.dtype, device=dev)}
    if with_S0:
        b["S0"] = torch.empty((B, H, d_k, d_v), dtype=torch.float32, device=dev)
    if with_S_T:
        b["S_T"] = torch.empty((B, H, d_k, d_v), dtype=torch.float32, device=dev)
    return b


def bwd_workspace_size(B: int, T: int, H: int, d_k: int, d_v: int, dtype: Optional[torch.dtype] = None,
                       per_channel_gate: bool = False) -> int:
    """Device scratch bytes ``chunk_bwd`` needs for these sizes: enough for either backward path,
    or, given the input dtype (and the gate), the need of the path that 16-byte aligned inputs
    take."""
    if dtype is None:
        return int(_native.lib().kla_chunk_bwd_workspace_size(B, T, H, d_k, d_v))
    dcode = _native.KLA_DTYPE_BF16 if dtype == torch.bfloat16 else _native.KLA_DTYPE_F32
    gcode = _native.KLA_GATE_CHANNEL if per_channel_gate else _native.KLA_GATE_SCALAR
    return int(_native.lib().kla_chunk_bwd_workspace_size_ex(B, T, H, d_k, d_v, dcode, gcode))


def chunk_bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, alpha: torch.Tensor, eta: torch.Tensor,
              dO: torch.Tensor, eps: float = 1e-6, S0: Optional[torch.Tensor] = None,
              dS_T: Optional[torch.Tensor] = None, *, beta_mode: str = "kla", q_scale: float = 1.0,
              want_dS0: bool = True, workspace: Optional[torch.Tensor] = None):
    """Backward pass of ``chunk_fwd`` run with the same inputs and options.

    dO: [B,T,H,d_v] in q's dtype (dL/do); dS_T: fp32 [B,H,d_k,d_v] or None (dL/dS_T = 0).
    Returns a dict of fp32 gradients: dq, dk [B,T,H,d_k]; dv [B,T,H,d_v]; dalpha (alpha's shape);
    deta [B,T,H]; dS0 [B,H,d_k,d_v] (None unless ``want_dS0``).
    """
    bcode = _beta_code(beta_mode)
    for n, t in (("q", q), ("k", k), ("v", v), ("dO", dO)):
        _check_dev(n, t)
    dcode = _dtype_code(q)
    if k.dtype != q.dtype or v.dtype != q.dtype or dO.dtype != q.dtype:
        raise TypeError("q, k, v and dO must share one dtype")
    B, T, H, d_k = q.shape
    d_v = v.shape[-1]
    if k.shape != q.shape or v.shape[:3] != q.shape[:3] or dO.shape != v.shape:
        raise ValueError("q, k, v, dO shapes disagree")
    _check_dev("alpha", alpha, torch.float32)
    _check_dev("eta", eta, torch.float32)
    if tuple(alpha.shape) == (B, T, H):
        gate = _native.KLA_GATE_SCALAR
    elif tuple(alpha.shape) == (B, T, H, d_k):
        gate = _native.KLA_GATE_CHANNEL
    else:
        raise ValueError(f"alpha must be [B,T,H] or [B,T,H,d_k], got {tuple(alpha.shape)}")
    if tuple(eta.shape) != (B, T, H):
        raise ValueError("eta must be [B, T, H]")
    for n, t in (("S0", S0), ("dS_T", dS_T)):
        if t is not None:
            _check_dev(n, t, torch.float32)
            if tuple(t.shape) != (B, H, d_k, d_v):
                raise ValueError(f"{n} must be [B, H, d_k, d_v]")
    f32 = dict(dtype=torch.float32, device=q.device)
    g = {"dq": torch.empty((B, T, H, d_k), **f32), "dk": torch.empty((B, T, H, d_k), **f32),
         "dv": torch.empty((B, T, H, d_v), **f32), "dalpha": torch.empty(alpha.shape, **f32),
         "deta": torch.empty((B, T, H), **f32),
         "dS0": torch.empty((B, H, d_k, d_v), **f32) if want_dS0 else None}
    aligned = all(t.data_ptr() % 16 == 0 for t in (q, k, v, dO))
    need = (bwd_workspace_size(B, T, H, d_k, d_v, q.dtype, gate == _native.KLA_GATE_CHANNEL) if aligned
            else bwd_workspace_size(B, T, H, d_k, d_v))
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = _native.lib().kla_chunk_bwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(eta), float(eps), _ptr(S0), _ptr(dO), _ptr(dS_T),
        _ptr(g["dq"]), _ptr(g["dk"]), _ptr(g["dv"]), _ptr(g["dalpha"]), _ptr(g["deta"]), _ptr(g["dS0"]),
        B, T, H, d_k, d_v, dcode, gate, bcode, float(q_scale), _ptr(workspace), ws_bytes, _stream_ptr(q.device))
    _native.check(st, "kla_chunk_bwd")
    return g


def decode_step(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, alpha: torch.Tensor, eta: torch.Tensor,
                S: torch.Tensor, eps: float = 1e-6, *, out: Optional[torch.Tensor] = None,
                beta_mode: str = "kla", q_scale: float = 1.0) -> torch.Tensor:
    """One fused KLA token step for B sequences; ``S`` (fp32 [B,H,d_k,d_v]) is updated in place.

    q, k: [B,H,d_k]; v: [B,H,d_v]; alpha: fp32 [B,H] or [B,H,d_k]; eta: fp32 [B,H].
    Returns o [B,H,d_v] in q's dtype. ``beta_mode`` and ``q_scale`` as in ``chunk_fwd``.
    """
    bcode = _beta_code(beta_mode)
    for n, t in (("q", q), ("k", k), ("v", v)):
        _check_dev(n, t)
    dcode = _dtype_code(q)
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k and v must share one dtype")
    B, H, d_k = q.shape
    d_v = v.shape[-1]
    _check_dev("alpha", alpha, torch.float32)
    _check_dev("eta", eta, torch.float32)
    _check_dev("S", S, torch.float32)
    if tuple(alpha.shape) == (B, H):
        gate = _native.KLA_GATE_SCALAR
    elif tuple(alpha.shape) == (B, H, d_k):
        gate = _native.KLA_GATE_CHANNEL
    else:
        raise ValueError("alpha must be [B,H] or [B,H,d_k]")
    if tuple(S.shape) != (B, H, d_k, d_v) or tuple(eta.shape) != (B, H) or tuple(k.shape) != (B, H, d_k):
        raise ValueError("shape mismatch")
    if out is None:
        out = torch.empty((B, H, d_v), dtype=q.dtype, device=q.device)
    else:
        _check_dev("out", out, q.dtype)
    st = _native.lib().kla_decode_step_ex(
        _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(eta), float(eps), _ptr(S), _ptr(out),
        B, H, d_k, d_v, dcode, gate, bcode, float(q_scale), _stream_ptr(q.device))
    _native.check(st, "kla_decode_step_ex")
    return out


def device_status(device=None) -> None:
    """Synchronise the current stream and raise if a bounded device wait or range check fired."""
    dev = torch.device("cuda") if device is None else torch.device(device)
    _native.check(_native.lib().kla_device_status(_stream_ptr(dev)), "kla_device_status")
