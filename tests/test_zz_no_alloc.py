"""kla_chunk_fwd_noalloc: the prefill entry point for callers that cannot allocate device memory.

Such callers (a runtime whose memory manager owns every byte of device memory, or code that
must not allocate while its stream has work in flight) cannot hand kla_chunk_fwd a workspace.
The no-allocation variant takes its scratch from a fixed array inside the library. It runs the
same kernels with the same segment plan as kla_chunk_fwd, so its results must equal
kla_chunk_fwd's bit for bit, call after call, whatever an earlier call left in the array; they
must also meet the oracle's tolerance. Invalid arguments get kla_chunk_fwd's errors, and only
valid sizes whose scratch exceeds the array are refused (before anything runs).

This file is collected last so that a run stopping at the first failure has already run every
other test; it also passes on its own in a fresh process.
"""
import ctypes
import math

import numpy as np
import pytest

import oracle
import synth
from gpu_util import DEV, oracle_chains, to_dev

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 24 << 20   # KLA_NOALLOC_SCRATCH_BYTES in include/kla.h
TOL_BF16 = 1e-2            # rel-L2 against the fp64 oracle for bf16 inputs with the fp32 state


def _noalloc():
    import gated_delta_rule_14_gb300 as kla
    lib = kla._native.lib()
    f = lib.kla_chunk_fwd_noalloc
    vp, i = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [vp, vp, vp, vp, vp, ctypes.c_float, vp, vp, vp, i, i, i, i, i, i, i, i, vp]
    f.restype = ctypes.c_int
    return f


def _call_noalloc(inp, S0):
    import torch

    import gated_delta_rule_14_gb300 as kla
    wl = inp.wl
    q, k, v, a, e = (to_dev(getattr(inp, n)) for n in ("q", "k", "v", "alpha", "eta"))
    o = torch.empty((wl.B, wl.T, wl.H, wl.d_v), dtype=torch.bfloat16, device=DEV)
    ST = torch.empty((wl.B, wl.H, wl.d_k, wl.d_v), dtype=torch.float32, device=DEV)
    gate = 1 if inp.alpha.ndim == 4 else 0
    st = _noalloc()(q.data_ptr(), k.data_ptr(), v.data_ptr(), a.data_ptr(), e.data_ptr(), wl.eps,
                    None if S0 is None else S0.data_ptr(), o.data_ptr(), ST.data_ptr(),
                    wl.B, wl.T, wl.H, wl.d_k, wl.d_v, wl.chunk, 1, gate,
                    torch.cuda.current_stream(DEV).cuda_stream)
    assert st == 0, st
    kla.device_status(DEV)
    return o.float().cpu().numpy(), ST.cpu().numpy()


def _call_reference_entry(inp, S0):
    import gated_delta_rule_14_gb300 as kla
    o, ST = kla.chunk_fwd(to_dev(inp.q), to_dev(inp.k), to_dev(inp.v), to_dev(inp.alpha), to_dev(inp.eta),
                          inp.wl.eps, S0, chunk=inp.wl.chunk)
    kla.device_status(DEV)
    return o.float().cpu().numpy(), ST.cpu().numpy()


@pytest.mark.parametrize("name,over", [
    ("long131k", dict(B=1, T=64 * 200 + 17, H=2, s0_sigma=0.05)),   # split into segments: uses the scratch
    ("kda8k", dict(B=1, T=64 * 120, H=1)),                          # per-channel gate, segments
    ("gdn4k", dict(B=2, T=300, H=3)),                                # no segments: no scratch
    ("kda8k", dict(B=2, T=200, H=2, starve=True)),                   # per-channel rerun marks in the scratch
])
def test_matches_kla_chunk_fwd_bit_for_bit(name, over):
    import gated_delta_rule_14_gb300 as kla
    over = dict(over)
    starve = over.pop("starve", False)
    inp = synth.make_prefill(name, seed=11, **over)
    if starve:   # gates out of the tensor-core path's range in one chain: it is rerun exactly
        inp.alpha[1, 70:110, 0, 9] = 1e-3
    wl = inp.wl
    need = kla.workspace_size(wl.B, wl.T, wl.H, wl.d_k, wl.d_v, wl.chunk, per_channel_gate=(wl.gate == "channel"))
    assert need <= SCRATCH_BYTES
    S0 = None if inp.S0 is None else to_dev(inp.S0)
    o_ref, s_ref = _call_reference_entry(inp, S0)
    # unrelated inputs of the same shapes (so the same segment plan) fill the scratch with other
    # values between the two checked calls: a pass that read a scratch element before writing it
    # would then give a different result
    other = synth.make_prefill(name, seed=12, **dict(over, s0_sigma=0.3))
    S0_other = to_dev(other.S0)
    o_fp, s_fp = oracle_chains(inp)
    for i in range(2):
        if i == 1:
            _call_noalloc(other, S0_other)
        o, s = _call_noalloc(inp, S0)
        assert np.array_equal(o, o_ref), f"call {i}: o differs from kla_chunk_fwd"
        assert np.array_equal(s, s_ref), f"call {i}: S_T differs from kla_chunk_fwd"
        o_g = np.stack([o[b, :, h] for b in range(wl.B) for h in range(wl.H)])
        s_g = np.stack([s[b, h] for b in range(wl.B) for h in range(wl.H)])
        eo, es = oracle.rel_l2(o_g, o_fp), oracle.rel_l2(s_g, s_fp)
        assert eo <= TOL_BF16 and es <= TOL_BF16, f"call {i}: rel-L2 o={eo:.3e} S={es:.3e}"


def _oversized():
    """B, T, H of a valid prefill whose segment scratch exceeds the fixed array on this device."""
    import gated_delta_rule_14_gb300 as kla
    B, H, T = 1, 8, 64 * 400
    need = kla.workspace_size(B, T, H, 128, 128, 64)
    if need <= SCRATCH_BYTES:
        pytest.skip(f"this device plans only {need} bytes of scratch for B={B} H={H} T={T}")
    return B, T, H


def test_refuses_sizes_beyond_the_scratch():
    import torch
    B, T, H = _oversized()
    z = torch.zeros((B, T, H, 128), dtype=torch.bfloat16, device=DEV)
    g = torch.ones((B, T, H), dtype=torch.float32, device=DEV)
    o = torch.empty_like(z)
    st = _noalloc()(z.data_ptr(), z.data_ptr(), z.data_ptr(), g.data_ptr(), g.data_ptr(), 1e-6, None,
                    o.data_ptr(), None, B, T, H, 128, 128, 64, 1, 0, torch.cuda.current_stream(DEV).cuda_stream)
    assert st == 2   # KLA_ERR_UNSUPPORTED


def test_argument_errors_come_before_the_size_refusal():
    """An oversized call with a bad argument gets kla_chunk_fwd's error for that argument."""
    import torch
    B, T, H = _oversized()
    z = torch.zeros((B, T, H, 128), dtype=torch.bfloat16, device=DEV)
    g = torch.ones((B, T, H), dtype=torch.float32, device=DEV)
    o = torch.empty_like(z)
    s = torch.cuda.current_stream(DEV).cuda_stream
    f = _noalloc()
    args = [z.data_ptr(), z.data_ptr(), z.data_ptr(), g.data_ptr(), g.data_ptr(), 1e-6, None, o.data_ptr(), None,
            B, T, H, 128, 128, 64, 1, 0, s]
    bad_eps = list(args)
    bad_eps[5] = math.nan
    assert f(*bad_eps) == 1                      # NaN stabiliser: KLA_ERR_INVALID_ARG
    bad_q = list(args)
    bad_q[0] = None
    assert f(*bad_q) == 1                        # null q
    bad_align = list(args)
    bad_align[1] = z.data_ptr() + 2
    assert f(*bad_align) == 1                    # k not 16-byte aligned
    bad_chunk = list(args)
    bad_chunk[14] = 48
    assert f(*bad_chunk) == 2                    # unsupported chunk, as kla_chunk_fwd reports it
