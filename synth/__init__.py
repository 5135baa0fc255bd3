"""Seeded synthetic inputs for the KLA gated delta-rule recurrence.

This module only draws random numbers and rounds them to the storage types the
recurrence consumes. It holds none of the recurrence's arithmetic: both the fp64
oracle and the CUDA path receive exactly the arrays produced here.

Generator: NumPy ``Generator(PCG64)`` seeded with ``SeedSequence(seed)``; one
independent child stream per tensor, spawned in the fixed order
q, k, v, alpha, eta, S0. Normals are drawn in float32 (NumPy's ziggurat),
the gate/relaxation transforms are evaluated in float64 and rounded once to
float32, and q/k/v are rounded to bfloat16 with round-to-nearest-even when the
workload stores them in bf16.

Workloads (shapes and distributions of the five standard cases):

=========  =====================================================================
tiny       B1 H1 T64 d16, fp32 q/k/v ~ N(0,1), scalar alpha = sigmoid(N(3,1)),
           eta = sigmoid(N(0,1)), eps 1e-6, S0 = 0, chunk 16
gdn4k      B8 H16 T4096 d128, bf16 q/k/v ~ N(0,1), scalar
           alpha = exp(-softplus(N(-4,1))), eta = sigmoid(N(0,1)), chunk 64
kda8k      B4 H16 T8192 d128, bf16, per-key-channel
           log alpha = -softplus(N(-4,1.5)), eta = sigmoid(N(0,1)), chunk 64
long131k   B1 H16 T131072 d128, bf16, scalar alpha = exp(-softplus(N(-5,1))),
           chunk 64 (2048 chunks)
decode     batch 64, H16, d128, 1024 single-token steps, bf16 q/k/v ~ N(0,1),
           scalar alpha = sigmoid(N(3,1)), eta = sigmoid(N(0,1)),
           S drawn i.i.d. N(0, 0.02^2) in fp32 (stand-in for a 32K-token state)
=========  =====================================================================

Any workload can be redrawn with ``key_norm="l2"``: keys scaled to unit L2 norm
(in float64, before the storage rounding), as DeltaNet normalises them; the raw
write strength beta = eta is only stable with such keys.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

__all__ = [
    "Workload", "WORKLOADS", "make_prefill", "make_decode", "f32_to_bf16_bits",
    "bf16_bits_to_f32", "PrefillInputs", "DecodeInputs", "custom_prefill",
]


# --------------------------------------------------------------------------- bf16
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round to nearest, ties to even); return the bit patterns."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float32."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# ---------------------------------------------------------------------- workloads
@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    H: int
    d_k: int
    d_v: int
    chunk: int
    dtype: str          # "f32" or "bf16": storage type of q, k, v and o
    gate: str           # "scalar" or "channel"
    alpha_mu: float
    alpha_sigma: float
    alpha_form: str     # "sigmoid" (alpha = sigmoid(x)) or "expnegsoftplus" (alpha = exp(-softplus(x)))
    eps: float = 1e-6
    s0_sigma: float = 0.0   # 0 => S0 = 0
    steps: int = 0          # decode workloads: number of single-token steps
    key_norm: str = "none"  # "l2": every key scaled to unit L2 norm before storage (DeltaNet keys)


WORKLOADS = {
    "tiny": Workload("tiny", 1, 64, 1, 16, 16, 16, "f32", "scalar", 3.0, 1.0, "sigmoid"),
    "gdn4k": Workload("gdn4k", 8, 4096, 16, 128, 128, 64, "bf16", "scalar", -4.0, 1.0, "expnegsoftplus"),
    "kda8k": Workload("kda8k", 4, 8192, 16, 128, 128, 64, "bf16", "channel", -4.0, 1.5, "expnegsoftplus"),
    "long131k": Workload("long131k", 1, 131072, 16, 128, 128, 64, "bf16", "scalar", -5.0, 1.0, "expnegsoftplus"),
    "decode": Workload("decode", 64, 1, 16, 128, 128, 0, "bf16", "scalar", 3.0, 1.0, "sigmoid",
                       s0_sigma=0.02, steps=1024),
}


@dataclasses.dataclass
class PrefillInputs:
    """Host arrays in the library's layouts.

    q, k: [B,T,H,d_k]; v: [B,T,H,d_v] -- uint16 bf16 bit patterns or float32.
    alpha: float32 [B,T,H] (scalar gate) or [B,T,H,d_k] (per-key-channel gate).
    eta: float32 [B,T,H].  S0: float32 [B,H,d_k,d_v] or None (zeros).
    """
    wl: Workload
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    alpha: np.ndarray
    eta: np.ndarray
    S0: Optional[np.ndarray]

    def as_f64(self, name: str) -> np.ndarray:
        a = getattr(self, name)
        if a is None:
            return None
        if a.dtype == np.uint16:
            return bf16_bits_to_f32(a).astype(np.float64)
        return a.astype(np.float64)


@dataclasses.dataclass
class DecodeInputs:
    """Decode workload: per step q, k, v [steps,B,H,d] (bf16 bits), alpha/eta [steps,B,H], S [B,H,d_k,d_v]."""
    wl: Workload
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    alpha: np.ndarray
    eta: np.ndarray
    S: np.ndarray


def _streams(seed: int, n: int):
    return [np.random.Generator(np.random.PCG64(s)) for s in np.random.SeedSequence(seed).spawn(n)]


def _normal(rng, shape, mu=0.0, sigma=1.0):
    z = rng.standard_normal(shape, dtype=np.float32)
    if mu == 0.0 and sigma == 1.0:
        return z
    return (z.astype(np.float64) * sigma + mu)


def _gate(rng, shape, wl: Workload) -> np.ndarray:
    x = _normal(rng, shape, wl.alpha_mu, wl.alpha_sigma).astype(np.float64)
    if wl.alpha_form == "sigmoid":
        a = 1.0 / (1.0 + np.exp(-x))
    elif wl.alpha_form == "expnegsoftplus":
        a = np.exp(-np.logaddexp(0.0, x))
    else:
        raise ValueError(wl.alpha_form)
    return a.astype(np.float32)


def _keys(rng, shape, wl: Workload) -> np.ndarray:
    k = _normal(rng, shape)
    if wl.key_norm == "l2":
        k = k.astype(np.float64)
        k = k / np.sqrt(np.sum(k * k, axis=-1, keepdims=True))
    elif wl.key_norm != "none":
        raise ValueError(wl.key_norm)
    return k


def _sigmoid01(rng, shape) -> np.ndarray:
    x = rng.standard_normal(shape, dtype=np.float32).astype(np.float64)
    return (1.0 / (1.0 + np.exp(-x))).astype(np.float32)


def _store(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return f32_to_bf16_bits(x.astype(np.float32))
    return np.ascontiguousarray(x, dtype=np.float32)


def custom_prefill(wl: Workload, seed: int = 0) -> PrefillInputs:
    """Draw one prefill problem with the shapes and distributions of ``wl``."""
    rq, rk, rv, ra, re, rs = _streams(seed, 6)
    B, T, H, dk, dv = wl.B, wl.T, wl.H, wl.d_k, wl.d_v
    q = _store(_normal(rq, (B, T, H, dk)), wl.dtype)
    k = _store(_keys(rk, (B, T, H, dk), wl), wl.dtype)
    v = _store(_normal(rv, (B, T, H, dv)), wl.dtype)
    ashape = (B, T, H) if wl.gate == "scalar" else (B, T, H, dk)
    alpha = _gate(ra, ashape, wl)
    eta = _sigmoid01(re, (B, T, H))
    S0 = None
    if wl.s0_sigma > 0:
        S0 = (_normal(rs, (B, H, dk, dv)).astype(np.float64) * wl.s0_sigma).astype(np.float32)
    return PrefillInputs(wl, q, k, v, alpha, eta, S0)


def make_prefill(name: str, seed: int = 0, **override) -> PrefillInputs:
    """Inputs of a named workload; keyword overrides change shapes (e.g. B=1, T=256) keeping distributions."""
    wl = dataclasses.replace(WORKLOADS[name], **override)
    return custom_prefill(wl, seed)


def make_decode(seed: int = 0, **override) -> DecodeInputs:
    """Decode inputs: ``steps`` single-token problems for ``B`` sequences and the starting state."""
    wl = dataclasses.replace(WORKLOADS["decode"], **override)
    rq, rk, rv, ra, re, rs = _streams(seed, 6)
    n, B, H, dk, dv = wl.steps, wl.B, wl.H, wl.d_k, wl.d_v
    q = _store(_normal(rq, (n, B, H, dk)), wl.dtype)
    k = _store(_keys(rk, (n, B, H, dk), wl), wl.dtype)
    v = _store(_normal(rv, (n, B, H, dv)), wl.dtype)
    ashape = (n, B, H) if wl.gate == "scalar" else (n, B, H, dk)
    alpha = _gate(ra, ashape, wl)
    eta = _sigmoid01(re, (n, B, H))
    S = (_normal(rs, (B, H, dk, dv)).astype(np.float64) * wl.s0_sigma).astype(np.float32)
    return DecodeInputs(wl, q, k, v, alpha, eta, S)
