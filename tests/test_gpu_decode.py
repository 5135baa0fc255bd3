"""Fused decode step on the GPU against the fp64 oracle (the steps of one head are the
tokens of one recurrence chain)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import DEV, decode_oracle, to_dev

pytestmark = pytest.mark.gpu


def run_decode(d):
    import gated_delta_rule_14_gb300 as kla
    S = to_dev(d.S).clone()
    q, k, v, a, e = (to_dev(x) for x in (d.q, d.k, d.v, d.alpha, d.eta))
    outs = torch.empty(q.shape[:3] + (d.S.shape[-1],), dtype=q.dtype, device=DEV)
    for i in range(q.shape[0]):
        kla.decode_step(q[i], k[i], v[i], a[i], e[i], S, d.wl.eps, out=outs[i])
    kla.device_status(DEV)
    return outs.float().cpu().numpy(), S.cpu().numpy()


@pytest.mark.parametrize("dtype,d,gate", [("bf16", 128, "scalar"), ("f32", 16, "scalar"), ("f32", 64, "channel"),
                                          ("bf16", 128, "channel"), ("bf16", 32, "scalar")])
def test_decode_small(dtype, d, gate):
    dd = synth.make_decode(seed=d, B=3, H=2, steps=12, d_k=d, d_v=d, dtype=dtype, gate=gate)
    o, S = run_decode(dd)
    o_ref, s_ref = decode_oracle(dd)
    heads = [(b, h) for b in range(3) for h in range(2)]
    o_g = np.stack([o[:, b, h] for b, h in heads])
    s_g = np.stack([S[b, h] for b, h in heads])
    tol = 1e-5 if dtype == "f32" else 1e-2
    assert oracle.rel_l2(o_g, o_ref) <= tol and oracle.rel_l2(s_g, s_ref) <= tol


def test_decode_full_config_whole_tensor():
    """The decode workload at full size (64 sequences x 16 heads, 1024 steps) against the oracle
    over every head: relative L2 over all outputs of all steps and over the whole final state."""
    dd = synth.make_decode(seed=0)
    o, S = run_decode(dd)
    assert np.isfinite(o).all() and np.isfinite(S).all()
    heads = [(b, h) for b in range(dd.wl.B) for h in range(dd.wl.H)]
    o_ref, s_ref = decode_oracle(dd, heads)
    o_g = np.stack([o[:, b, h] for b, h in heads])
    s_g = np.stack([S[b, h] for b, h in heads])
    eo, es = oracle.rel_l2(o_g, o_ref), oracle.rel_l2(s_g, s_ref)
    assert eo <= 1e-2 and es <= 1e-2, f"rel-L2 o={eo:.3e} S={es:.3e}"


def test_decode_equals_one_token_prefill():
    """A decode step is a one-token prefill: both match the oracle (the decode state in fp32
    arithmetic to 1e-5; the prefill, which may use bf16 tensor-core operands, to 1e-2)."""
    import gated_delta_rule_14_gb300 as kla
    dd = synth.make_decode(seed=4, B=2, H=3, steps=1)
    S = to_dev(dd.S)
    q, k, v, a, e = (to_dev(x)[0] for x in (dd.q, dd.k, dd.v, dd.alpha, dd.eta))
    o_p, S_p = kla.chunk_fwd(q[:, None], k[:, None], v[:, None], a[:, None], e[:, None], dd.wl.eps, S)
    S_d = S.clone()
    o_d = kla.decode_step(q, k, v, a, e, S_d, dd.wl.eps)
    kla.device_status(DEV)
    heads = [(b, h) for b in range(2) for h in range(3)]
    o_ref, s_ref = decode_oracle(dd, heads)
    o_d_g = np.stack([o_d.float().cpu().numpy()[b, h] for b, h in heads])[:, None]
    o_p_g = np.stack([o_p[:, 0].float().cpu().numpy()[b, h] for b, h in heads])[:, None]
    s_d_g = np.stack([S_d.cpu().numpy()[b, h] for b, h in heads])
    s_p_g = np.stack([S_p.cpu().numpy()[b, h] for b, h in heads])
    assert oracle.rel_l2(s_d_g, s_ref) <= 1e-5
    assert oracle.rel_l2(s_p_g, s_ref) <= 1e-2
    assert oracle.rel_l2(o_d_g, o_ref) <= 1e-2 and oracle.rel_l2(o_p_g, o_ref) <= 1e-2


def test_decode_unaligned_vectors_take_the_per_tile_kernel():
    """Vectors aligned only to their element size (allowed by kla_decode_step) cannot be copied
    in 16-byte units: those calls run the one-CTA-per-tile kernel; the result must be the same
    as the pipelined kernel's (same arithmetic in the same order) and match the oracle."""
    import gated_delta_rule_14_gb300 as kla
    dd = synth.make_decode(seed=8, B=4, H=2, steps=3)
    heads = [(b, h) for b in range(4) for h in range(2)]
    o_ref, s_ref = decode_oracle(dd, heads)
    outs = {}
    for shift in (0, 1):   # element offset of q, k, v inside a larger buffer
        S = to_dev(dd.S).clone()
        q, k, v, a, e = (to_dev(x) for x in (dd.q, dd.k, dd.v, dd.alpha, dd.eta))
        o = []
        for i in range(3):
            vec = []
            for x in (q[i], k[i], v[i]):
                buf = torch.empty(x.numel() + 8, dtype=x.dtype, device=DEV)
                y = buf[shift:shift + x.numel()].view(x.shape)
                y.copy_(x)
                vec.append(y)
            o.append(kla.decode_step(vec[0], vec[1], vec[2], a[i], e[i], S, dd.wl.eps))
        kla.device_status(DEV)
        outs[shift] = (torch.stack(o).float().cpu().numpy(), S.cpu().numpy())
    assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1])
    o, S = outs[1]
    o_g = np.stack([o[:, b, h] for b, h in heads])
    s_g = np.stack([S[b, h] for b, h in heads])
    assert oracle.rel_l2(o_g, o_ref) <= 1e-2 and oracle.rel_l2(s_g, s_ref) <= 1e-5
