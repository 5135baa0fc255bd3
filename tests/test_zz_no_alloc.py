"""kla_chunk_fwd_noalloc: the prefill entry point for callers that cannot allocate device memory.

Such callers (a runtime whose memory manager owns every byte of device memory, or code that
must not allocate while its stream has work in flight) cannot hand kla_chunk_fwd a workspace.
The no-allocation variant takes its scratch from a fixed array inside the library; its results
must match kla_chunk_fwd on the same inputs, call after call, and sizes whose scratch exceeds
that array are refused before anything runs.

This file is collected last so that a run stopping at the first failure has already run every
other test; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest

import oracle
import synth
from gpu_util import DEV, to_dev

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 24 << 20   # KLA_NOALLOC_SCRATCH_BYTES in include/kla.h


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
])
def test_matches_kla_chunk_fwd_twice(name, over):
    import gated_delta_rule_14_gb300 as kla
    inp = synth.make_prefill(name, seed=11, **over)
    wl = inp.wl
    need = kla.workspace_size(wl.B, wl.T, wl.H, wl.d_k, wl.d_v, wl.chunk, per_channel_gate=(wl.gate == "channel"))
    assert need <= SCRATCH_BYTES
    S0 = None if inp.S0 is None else to_dev(inp.S0)
    o_ref, s_ref = _call_reference_entry(inp, S0)
    for _ in range(2):   # the second call starts from the first call's scratch contents
        o, s = _call_noalloc(inp, S0)
        assert np.isfinite(o).all() and np.isfinite(s).all()
        assert oracle.rel_l2(o, o_ref) <= 1e-2 and oracle.rel_l2(s, s_ref) <= 1e-2


def test_refuses_sizes_beyond_the_scratch():
    import torch

    import gated_delta_rule_14_gb300 as kla
    # few chains and a long sequence: the segment plan (it depends on the SM count) may need
    # more scratch than the fixed array; such calls must be refused before anything runs
    B, H, T = 1, 8, 64 * 400
    need = kla.workspace_size(B, T, H, 128, 128, 64)
    if need <= SCRATCH_BYTES:
        pytest.skip(f"this device plans only {need} bytes of scratch for B={B} H={H} T={T}")
    z = torch.zeros((B, T, H, 128), dtype=torch.bfloat16, device=DEV)
    g = torch.ones((B, T, H), dtype=torch.float32, device=DEV)
    o = torch.empty_like(z)
    st = _noalloc()(z.data_ptr(), z.data_ptr(), z.data_ptr(), g.data_ptr(), g.data_ptr(), 1e-6, None,
                    o.data_ptr(), None, B, T, H, 128, 128, 64, 1, 0, torch.cuda.current_stream(DEV).cuda_stream)
    assert st == 2   # KLA_ERR_UNSUPPORTED
