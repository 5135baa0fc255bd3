"""The raw-beta step (beta = eta, the write strength of DeltaNet / Gated DeltaNet) and the query
scale of the read (o = S^T (s q), s = d_k^{-1/2} in Kimi Delta Attention) on every path, against
the fp64 oracle run in the same mode. Raw-beta inputs use unit-norm keys, as DeltaNet does: with
beta ||k||^2 above 2 the transition has an eigenvalue below -1 and the state grows without bound."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import DEV, decode_oracle, gather_chains, oracle_chains, run_prefill, sample_chains, to_dev

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-5, "bf16": 1e-2}


def check(inp, o, S, chains=None, **mode):
    o_ref, s_ref = oracle_chains(inp, chains, **mode)
    if chains is None:
        chains = [(b, h) for b in range(inp.wl.B) for h in range(inp.wl.H)]
    o_g, s_g = gather_chains(o, S, chains)
    tol = TOL[inp.wl.dtype]
    eo, es = oracle.rel_l2(o_g, o_ref), oracle.rel_l2(s_g, s_ref)
    assert np.isfinite(o).all() and np.isfinite(S).all()
    assert eo <= tol and es <= tol, f"rel-L2 o={eo:.3e} S={es:.3e} tol={tol}"


# (name, overrides, chunk) -- one case per kernel: tensor-core (scalar, per-channel), fp32 CUDA-core,
# short sequence (bf16, fp32), sequence-parallel segments
CASES = [
    ("gdn4k", dict(B=2, T=300, H=3, s0_sigma=0.05), None),
    ("kda8k", dict(B=1, T=200, H=2, s0_sigma=0.05), None),
    ("gdn4k", dict(B=2, T=97, H=2, d_k=64, d_v=32, chunk=32, dtype="f32", s0_sigma=0.1), None),
    ("decode", dict(B=4, T=5, H=3, chunk=64, s0_sigma=0.02), None),
    ("kda8k", dict(B=2, T=7, H=2, d_k=32, d_v=64, dtype="f32", s0_sigma=0.1), None),
    ("long131k", dict(B=1, T=64 * 120 + 9, H=2, s0_sigma=0.05), None),
]


@pytest.mark.parametrize("beta_mode,q_scale", [("raw", 1.0), ("raw", 128 ** -0.5), ("kla", 128 ** -0.5)])
@pytest.mark.parametrize("name,over,chunk", CASES, ids=lambda x: str(x)[:40])
def test_modes_against_oracle(name, over, chunk, beta_mode, q_scale):
    key_norm = "l2" if beta_mode == "raw" else "none"
    inp = synth.make_prefill(name, seed=len(name) + over["T"], key_norm=key_norm, **over)
    o, S = run_prefill(inp, chunk=chunk, beta_mode=beta_mode, q_scale=q_scale)
    chains = None if inp.wl.B * inp.wl.H <= 8 else sample_chains(inp.wl.B, inp.wl.H, 8, seed=2)
    check(inp, o, S, chains, beta_mode=beta_mode, q_scale=q_scale)


def test_scale_only_scales_the_outputs():
    import gated_delta_rule_14_gb300 as kla
    inp = synth.make_prefill("gdn4k", seed=3, B=1, T=130, H=2, s0_sigma=0.05)
    args = [to_dev(x) for x in (inp.q, inp.k, inp.v, inp.alpha, inp.eta)]
    S0 = to_dev(inp.S0)
    o1, s1 = kla.chunk_fwd(*args, inp.wl.eps, S0)
    o2, s2 = kla.chunk_fwd(*args, inp.wl.eps, S0, q_scale=0.25)
    kla.device_status(DEV)
    assert bool((s1 == s2).all())
    # a power-of-two scale commutes with the rounding to bf16
    assert bool((o2.float() == 0.25 * o1.float()).all())


@pytest.mark.parametrize("beta_mode,q_scale", [("raw", 1.0), ("raw", 0.125), ("kla", 0.5)])
def test_decode_modes(beta_mode, q_scale):
    import gated_delta_rule_14_gb300 as kla
    d = synth.make_decode(seed=4, steps=6, B=3, H=2, key_norm="l2" if beta_mode == "raw" else "none")
    q, k, v, a, e = (to_dev(x) for x in (d.q, d.k, d.v, d.alpha, d.eta))
    S = to_dev(d.S)
    outs = [kla.decode_step(q[i], k[i], v[i], a[i], e[i], S, d.wl.eps, beta_mode=beta_mode, q_scale=q_scale)
            for i in range(d.wl.steps)]
    kla.device_status(DEV)
    o_ref, s_ref = decode_oracle(d, beta_mode=beta_mode, q_scale=q_scale)
    heads = [(b, h) for b in range(3) for h in range(2)]
    o_g = np.stack([np.stack([outs[i][b, h].float().cpu().numpy() for i in range(d.wl.steps)]) for b, h in heads])
    s_g = np.stack([S[b, h].cpu().numpy() for b, h in heads])
    assert oracle.rel_l2(o_g, o_ref) <= 1e-2 and oracle.rel_l2(s_g, s_ref) <= 1e-5


def test_raw_mode_is_kla_with_rescaled_eta_on_the_gpu():
    # the same relation the oracle is pinned to, between the two modes of the tensor-core path
    import gated_delta_rule_14_gb300 as kla
    inp = synth.make_prefill("gdn4k", seed=6, B=1, T=128, H=2, s0_sigma=0.05)
    args = [to_dev(x) for x in (inp.q, inp.k, inp.v, inp.alpha)]
    k = args[1].float()
    eta = to_dev(inp.eta)
    eta_raw = (eta.double() / ((k.double() ** 2).sum(-1) + inp.wl.eps)).float().contiguous()
    S0 = to_dev(inp.S0)
    o1, s1 = kla.chunk_fwd(*args, eta, inp.wl.eps, S0)
    o2, s2 = kla.chunk_fwd(*args, eta_raw, inp.wl.eps, S0, beta_mode="raw")
    kla.device_status(DEV)
    assert oracle.rel_l2(o2.float().cpu().numpy(), o1.float().cpu().numpy()) <= 1e-2
    assert oracle.rel_l2(s2.cpu().numpy(), s1.cpu().numpy()) <= 1e-3
