"""fp64 CPU oracle of the KLA gated delta-rule recurrence -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The CUDA library never imports, links or
calls it, and it imports nothing from the CUDA library.

Two independent restatements of what the recurrence computes:

* ``recurrent`` -- the plain sequential fp64 recurrence (C, ``kla_oracle.c``),
  token by token: forget, predict, residual, step size (the KLA step, or the raw
  write strength of DeltaNet / Gated DeltaNet), write, read (with an optional
  query scale).
  This is the definition the GPU results are compared against.
* ``Oracle.backward`` -- the reverse-mode derivative of ``recurrent`` (C), the chain
  rule through the same six steps in reverse order (the pages give no backward
  algebra), pinned by finite differences of ``recurrent``.
* ``chunkwise`` -- an fp64 NumPy restatement of the chunk algebra (cumulative
  log-decay, provisional error, unit-triangular correction, end-of-chunk state
  and in-chunk outputs) from GeekNews "Revisando las variantes de atencion
  lineal de la familia DeltaNet", section "KDA por chunks". Used only to pin
  that algebra against the recurrence (they must agree to rounding).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from .chunkwise import chunkwise  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kla_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_lock = threading.Lock()
_cache: dict = {}


def build(mutant: int = 0, out_dir: str | None = None) -> str:
    """Compile ``kla_oracle.c`` with gcc (plain C99, IEEE fp64, no fast-math).

    ``mutant`` > 0 plants one of the deliberate mistakes the tests use to show
    that the pins catch it; the oracle itself is ``mutant=0``.
    """
    out_dir = out_dir or _BUILD
    os.makedirs(out_dir, exist_ok=True)
    name = "libkla_oracle.so" if mutant == 0 else f"libkla_oracle_mutant{mutant}.so"
    out = os.path.join(out_dir, name)
    if (not os.path.exists(out)) or os.path.getmtime(out) < os.path.getmtime(_SRC):
        tmp = out + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-pthread", "-fno-fast-math",
               "-ffp-contract=off", f"-DKLA_ORACLE_MUTANT={mutant}", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)
    return out


class Oracle:
    """ctypes handle on one build of the C oracle."""

    def __init__(self, path: str):
        self.path = path
        self.lib = ctypes.CDLL(path)
        f = self.lib.kla_oracle_recurrent_ex
        dp = ctypes.POINTER(ctypes.c_double)
        f.argtypes = [dp, dp, dp, dp, ctypes.c_int, dp, ctypes.c_double, dp, dp, dp,
                      ctypes.c_long, ctypes.c_long, ctypes.c_long, ctypes.c_long, ctypes.c_long,
                      ctypes.c_int, ctypes.c_double, ctypes.c_int]
        f.restype = ctypes.c_int
        self._f = f

    def recurrent(self, q, k, v, alpha, eta, eps, S0=None, nthreads: int = 1, beta_mode: str = "kla",
                  q_scale: float = 1.0):
        """Run the fp64 recurrence.

        q, k: [B,T,H,d_k]; v: [B,T,H,d_v]; alpha: [B,T,H] (scalar gate) or
        [B,T,H,d_k] (per-key-channel gate); eta: [B,T,H]; S0: [B,H,d_k,d_v] or None.
        beta_mode "kla": beta = eta / (||k||^2 + eps); "raw": beta = eta (DeltaNet /
        Gated DeltaNet write strength). The read is o_t = S_t^T (q_scale * q_t).
        Returns (o [B,T,H,d_v], S_T [B,H,d_k,d_v]) as float64.
        """
        modes = {"kla": 0, "raw": 1}
        if beta_mode not in modes:
            raise ValueError(f"beta_mode {beta_mode!r}")
        q = np.ascontiguousarray(q, dtype=np.float64)
        k = np.ascontiguousarray(k, dtype=np.float64)
        v = np.ascontiguousarray(v, dtype=np.float64)
        alpha = np.ascontiguousarray(alpha, dtype=np.float64)
        eta = np.ascontiguousarray(eta, dtype=np.float64)
        B, T, H, dk = q.shape
        dv = v.shape[-1]
        assert k.shape == (B, T, H, dk) and v.shape == (B, T, H, dv)
        assert eta.shape == (B, T, H)
        if alpha.shape == (B, T, H):
            per_channel = 0
        elif alpha.shape == (B, T, H, dk):
            per_channel = 1
        else:
            raise ValueError(f"alpha shape {alpha.shape}")
        if S0 is not None:
            S0 = np.ascontiguousarray(S0, dtype=np.float64)
            assert S0.shape == (B, H, dk, dv)
        o = np.zeros((B, T, H, dv), dtype=np.float64)
        ST = np.zeros((B, H, dk, dv), dtype=np.float64)
        dp = ctypes.POINTER(ctypes.c_double)

        def P(a):
            return None if a is None else a.ctypes.data_as(dp)

        rc = self._f(P(q), P(k), P(v), P(alpha), per_channel, P(eta), float(eps), P(S0), P(o), P(ST),
                     B, T, H, dk, dv, modes[beta_mode], float(q_scale), int(nthreads))
        if rc != 0:
            raise RuntimeError(f"kla_oracle_recurrent failed with {rc}")
        return o, ST


    def backward(self, q, k, v, alpha, eta, eps, S0, dO, dS_T=None, nthreads: int = 1, beta_mode: str = "kla",
                 q_scale: float = 1.0):
        """Reverse-mode derivative of ``recurrent`` for a loss with dL/do = dO [B,T,H,d_v] and
        dL/dS_T = dS_T [B,H,d_k,d_v] (None: 0). Returns a dict of float64 arrays: dq, dk, dv,
        dalpha (shaped like alpha), deta, dS0. Keeps every chain's states: small cases only."""
        modes = {"kla": 0, "raw": 1}
        if beta_mode not in modes:
            raise ValueError(f"beta_mode {beta_mode!r}")
        c = lambda a: None if a is None else np.ascontiguousarray(a, dtype=np.float64)  # noqa: E731
        q, k, v, alpha, eta, S0, dO, dS_T = (c(x) for x in (q, k, v, alpha, eta, S0, dO, dS_T))
        B, T, H, dk = q.shape
        dv = v.shape[-1]
        per_channel = 1 if alpha.shape == (B, T, H, dk) else 0
        if not per_channel and alpha.shape != (B, T, H):
            raise ValueError(f"alpha shape {alpha.shape}")
        assert dO.shape == (B, T, H, dv)
        out = {"dq": np.zeros_like(q), "dk": np.zeros_like(k), "dv": np.zeros_like(v),
               "dalpha": np.zeros_like(alpha), "deta": np.zeros_like(eta), "dS0": np.zeros((B, H, dk, dv))}
        dp = ctypes.POINTER(ctypes.c_double)

        def P(a):
            return None if a is None else a.ctypes.data_as(dp)
        f = self.lib.kla_oracle_backward
        f.argtypes = [dp, dp, dp, dp, ctypes.c_int, dp, ctypes.c_double, dp, dp, dp, dp, dp, dp, dp, dp, dp,
                      ctypes.c_long, ctypes.c_long, ctypes.c_long, ctypes.c_long, ctypes.c_long,
                      ctypes.c_int, ctypes.c_double, ctypes.c_int]
        f.restype = ctypes.c_int
        rc = f(P(q), P(k), P(v), P(alpha), per_channel, P(eta), float(eps), P(S0), P(dO), P(dS_T),
               P(out["dq"]), P(out["dk"]), P(out["dv"]), P(out["dalpha"]), P(out["deta"]), P(out["dS0"]),
               B, T, H, dk, dv, modes[beta_mode], float(q_scale), int(nthreads))
        if rc != 0:
            raise RuntimeError(f"kla_oracle_backward failed with {rc}")
        return out


def load(mutant: int = 0) -> Oracle:
    """Build (if needed) and load the oracle library; cached per mutant id."""
    with _lock:
        if mutant not in _cache:
            _cache[mutant] = Oracle(build(mutant))
        return _cache[mutant]


def recurrent(*args, **kw):
    """``load().recurrent(...)``: the fp64 sequential recurrence."""
    return load().recurrent(*args, **kw)


def rel_l2(x, ref) -> float:
    """||x - ref||_2 / ||ref||_2 over the whole tensor, accumulated in fp64."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.sqrt(np.sum(ref * ref))
    num = np.sqrt(np.sum((x - ref) ** 2))
    return float(num / den) if den > 0 else float(num)
