"""Short sequences (T <= 16: multi-token decode, speculative verification) against the fp64
oracle. kla_chunk_fwd runs these either on a kernel that keeps each state tile in registers and
walks the tokens one by one (whose result must equal T single-token decode steps as well), or,
for bf16 with a scalar gate, d_k = d_v = 128 and T >= 5, on the chunk form of the recurrence
with the call's tokens as one chunk (warp-level tensor cores, one CTA per head)."""
import ctypes
import dataclasses

import numpy as np
import pytest

import oracle
import synth
from gpu_util import DEV, gather_chains, oracle_chains, run_prefill, sample_chains, to_dev

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-5, "bf16": 1e-2}

CASES = [
    # (dtype, d_k, d_v, T, gate, s0)
    ("f32", 16, 16, 1, "scalar", 0.1),
    ("f32", 16, 32, 2, "channel", 0.1),
    ("f32", 32, 16, 3, "scalar", 0.0),
    ("f32", 64, 128, 4, "channel", 0.05),
    ("f32", 128, 64, 8, "scalar", 0.05),
    ("f32", 128, 128, 16, "channel", 0.05),
    ("bf16", 128, 128, 2, "scalar", 0.02),
    ("bf16", 128, 128, 4, "scalar", 0.0),
    ("bf16", 128, 128, 15, "channel", 0.05),
    ("bf16", 128, 128, 16, "scalar", 0.05),
    ("bf16", 64, 64, 7, "channel", 0.1),
    ("bf16", 128, 128, 1, "channel", 0.05),
    ("f32", 128, 64, 1, "scalar", 0.0),
]


def check(inp, o, S, chains=None):
    o_ref, s_ref = oracle_chains(inp, chains)
    if chains is None:
        chains = [(b, h) for b in range(inp.wl.B) for h in range(inp.wl.H)]
    o_g, s_g = gather_chains(o, S, chains)
    tol = TOL[inp.wl.dtype]
    eo, es = oracle.rel_l2(o_g, o_ref), oracle.rel_l2(s_g, s_ref)
    assert np.isfinite(o).all() and np.isfinite(S).all()
    assert eo <= tol and es <= tol, f"rel-L2 o={eo:.3e} S={es:.3e} tol={tol}"


@pytest.mark.parametrize("dtype,dk,dv,T,gate,s0", CASES, ids=lambda x: str(x))
def test_short_shapes(dtype, dk, dv, T, gate, s0):
    base = "kda8k" if gate == "channel" else "decode"
    inp = synth.make_prefill(base, seed=100 + T * 3 + dk, B=3, T=T, H=2, d_k=dk, d_v=dv, chunk=64,
                             dtype=dtype, s0_sigma=s0)
    o, S = run_prefill(inp)
    check(inp, o, S)


@pytest.mark.parametrize("T", [16, 17])
def test_both_sides_of_the_short_limit(T):
    # T = 16 runs the register-resident short kernel, T = 17 the chunkwise tensor-core path
    inp = synth.make_prefill("gdn4k", seed=T, B=2, T=T, H=3, s0_sigma=0.05)
    o, S = run_prefill(inp)
    check(inp, o, S)


def test_equals_repeated_decode_steps():
    """T tokens in one call equal T calls of the single-token step (both fp32 arithmetic in the
    same order per token; only the fused read of the output differs)."""
    import torch

    import gated_delta_rule_14_gb300 as kla
    inp = synth.make_prefill("decode", seed=21, B=4, T=6, H=4, chunk=64, dtype="f32", s0_sigma=0.02)
    q, k, v, a, e, S0 = (to_dev(x) for x in (inp.q, inp.k, inp.v, inp.alpha, inp.eta, inp.S0))
    o, ST = kla.chunk_fwd(q, k, v, a, e, inp.wl.eps, S0)
    S = S0.clone()
    outs = []
    for t in range(inp.wl.T):
        outs.append(kla.decode_step(q[:, t].contiguous(), k[:, t].contiguous(), v[:, t].contiguous(),
                                    a[:, t].contiguous(), e[:, t].contiguous(), S, inp.wl.eps))
    kla.device_status(DEV)
    o_dec = torch.stack(outs, dim=1)
    assert oracle.rel_l2(o.cpu().numpy(), o_dec.cpu().numpy()) <= 1e-6
    assert oracle.rel_l2(ST.cpu().numpy(), S.cpu().numpy()) <= 1e-6


@pytest.mark.parametrize("T,j", [(4, 2), (8, 5), (16, 9)])
def test_speculative_verify_then_accept_prefix(T, j):
    """Verification pattern: run T draft tokens from the committed state without touching it,
    accept a prefix of j tokens, then advance the committed state by those j tokens in place.
    Outputs of the prefix and the advanced state must match the oracle on the prefix alone. Each
    pair runs on one kernel (the token loop below 5 tokens, the chunk form with the same token
    padding from 5), where later tokens add exact zeros to the prefix, so the accepted outputs
    equal the draft's bit for bit."""
    import gated_delta_rule_14_gb300 as kla
    inp = synth.make_prefill("decode", seed=33, B=8, T=T, H=4, chunk=64, s0_sigma=0.02)
    q, k, v, a, e = (to_dev(x) for x in (inp.q, inp.k, inp.v, inp.alpha, inp.eta))
    S = to_dev(inp.S0).clone()
    S_before = S.clone()
    o_draft, _ = kla.chunk_fwd(q, k, v, a, e, inp.wl.eps, S)       # S_T into a new buffer
    kla.device_status(DEV)
    assert (S == S_before).all().item()
    o_acc, S_out = kla.chunk_fwd(q[:, :j].contiguous(), k[:, :j].contiguous(), v[:, :j].contiguous(),
                                 a[:, :j].contiguous(), e[:, :j].contiguous(), inp.wl.eps, S, S_T=S)
    kla.device_status(DEV)
    assert S_out.data_ptr() == S.data_ptr()
    # the accepted outputs are the first j draft outputs (causal: later tokens do not affect them)
    assert (o_acc == o_draft[:, :j]).all().item()
    pre = synth.PrefillInputs(dataclasses.replace(inp.wl, T=j), inp.q[:, :j], inp.k[:, :j], inp.v[:, :j],
                              inp.alpha[:, :j], inp.eta[:, :j], inp.S0)
    check(pre, o_acc.float().cpu().numpy().astype(np.float64), S.cpu().numpy().astype(np.float64))


def test_zero_initial_state_and_no_final_state():
    import torch

    import gated_delta_rule_14_gb300 as kla
    inp = synth.make_prefill("kda8k", seed=7, B=2, T=9, H=2)
    assert inp.S0 is None
    o, S = run_prefill(inp)
    check(inp, o, S)
    # S_T not requested through the C ABI: the outputs are still written
    o2 = torch.empty((2, 9, 2, 128), dtype=torch.bfloat16, device=DEV)
    lib = kla._native.lib()
    args = [to_dev(x) for x in (inp.q, inp.k, inp.v, inp.alpha, inp.eta)]
    st = lib.kla_chunk_fwd(*(x.data_ptr() for x in args), ctypes.c_float(inp.wl.eps), None, o2.data_ptr(),
                           None, 2, 9, 2, 128, 128, 64, 1, 1, None, 0,
                           torch.cuda.current_stream(DEV).cuda_stream)
    assert st == 0
    kla.device_status(DEV)
    assert np.array_equal(o2.float().cpu().numpy(), o.astype(np.float32))


def test_serving_batch_sampled():
    # speculative verification at the decode batch: 64 sequences x 16 heads, 4 tokens each
    inp = synth.make_prefill("decode", seed=2, T=4, chunk=64)
    o, S = run_prefill(inp)
    check(inp, o, S, sample_chains(inp.wl.B, inp.wl.H, 16, seed=3))


# The chunk-form kernel: both token paddings (T <= 8 packs K and Q into one 16-row tile, 9..16
# uses two), ragged T inside each, and a head count that does not divide the persistent grid.
@pytest.mark.parametrize("T", [5, 7, 8, 9, 13, 16])
def test_chunk_form_tokens(T):
    inp = synth.make_prefill("decode", seed=500 + T, B=5, T=T, H=3, chunk=64, s0_sigma=0.05)
    o, S = run_prefill(inp)
    check(inp, o, S)


def test_chunk_form_zero_state_and_no_final_state():
    import torch

    import gated_delta_rule_14_gb300 as kla
    inp = synth.make_prefill("decode", seed=9, B=2, T=11, H=3, chunk=64, s0_sigma=0.0)
    inp = dataclasses.replace(inp, S0=None)
    o, S = run_prefill(inp)
    check(inp, o, S)
    o2 = torch.empty((2, 11, 3, 128), dtype=torch.bfloat16, device=DEV)
    lib = kla._native.lib()
    args = [to_dev(x) for x in (inp.q, inp.k, inp.v, inp.alpha, inp.eta)]
    st = lib.kla_chunk_fwd(*(x.data_ptr() for x in args), ctypes.c_float(inp.wl.eps), None, o2.data_ptr(),
                           None, 2, 11, 3, 128, 128, 64, 1, 0, None, 0,
                           torch.cuda.current_stream(DEV).cuda_stream)
    assert st == 0
    kla.device_status(DEV)
    assert np.array_equal(o2.float().cpu().numpy(), o.astype(np.float32))


@pytest.mark.parametrize("T", [6, 12])
def test_chunk_form_degenerate_tokens(T):
    """Keys that are exactly zero with eps = 0 (beta = 0: the step writes nothing), gates of
    exactly 1 (no decay) and of exactly 0 (the state before the token is forgotten)."""
    inp = synth.make_prefill("decode", seed=40 + T, B=2, T=T, H=2, chunk=64, s0_sigma=0.05, eps=0.0)
    k, alpha = inp.k.copy(), inp.alpha.copy()
    k[0, [0, T - 1], 0] = 0
    k[1, 2, 1] = 0
    alpha[0, 1:4, 1] = 1.0
    alpha[1, 3, 0] = 0.0
    inp = dataclasses.replace(inp, k=k, alpha=alpha)
    o, S = run_prefill(inp)
    check(inp, o, S)


def test_chunk_form_serving_batch_sampled():
    # verification of 8 draft tokens at the decode batch: 64 sequences x 16 heads
    inp = synth.make_prefill("decode", seed=5, T=8, chunk=64)
    o, S = run_prefill(inp)
    check(inp, o, S, sample_chains(inp.wl.B, inp.wl.H, 16, seed=4))



# The chunk form with the per-key-channel gate (bf16, d_k = d_v = 128, 9 to 16 tokens): in-call
# products R and A formed exactly per channel, the decays inside scaled K, Q and K_end tiles.
# T = 8 runs the token loop beside it.
@pytest.mark.parametrize("T", [8, 9, 10, 13, 16])
def test_channel_chunk_form_tokens(T):
    inp = synth.make_prefill("kda8k", seed=700 + T, B=5, T=T, H=3, s0_sigma=0.05)
    o, S = run_prefill(inp)
    check(inp, o, S)


def test_channel_chunk_form_extreme_gates():
    """Per-channel gates of 1e-30 (the in-call decay far beyond e^-80 in some channels), exactly 0
    and exactly 1, and keys that are exactly zero with eps = 0: the in-call products take
    e^{G_i - G_m} <= 1 directly, so every gate in [0, 1] is exact."""
    inp = synth.make_prefill("kda8k", seed=71, B=2, T=14, H=2, s0_sigma=0.05, eps=0.0)
    k, alpha = inp.k.copy(), inp.alpha.copy()
    alpha[0, 2:12, 0, 5:40] = 1e-30
    alpha[1, 4, 1, :] = 0.0
    alpha[1, 6:10, 0, :] = 1.0
    k[0, [0, 13], 1] = 0
    k[1, 7, 0] = 0
    inp = dataclasses.replace(inp, k=k, alpha=alpha)
    o, S = run_prefill(inp)
    check(inp, o, S)


def test_channel_chunk_form_verify_then_accept_prefix():
    """Verification with the per-channel gate: the first j outputs of a 14-token draft equal a
    j-token call's bit for bit (both padded to 16 tokens; later tokens add exact zeros), and the
    state advanced in place by the accepted prefix matches the oracle."""
    import gated_delta_rule_14_gb300 as kla
    T, j = 14, 10
    inp = synth.make_prefill("kda8k", seed=72, B=6, T=T, H=4, s0_sigma=0.02)
    q, k, v, a, e = (to_dev(x) for x in (inp.q, inp.k, inp.v, inp.alpha, inp.eta))
    S = to_dev(inp.S0).clone()
    o_draft, _ = kla.chunk_fwd(q, k, v, a, e, inp.wl.eps, S)
    o_acc, _ = kla.chunk_fwd(q[:, :j].contiguous(), k[:, :j].contiguous(), v[:, :j].contiguous(),
                             a[:, :j].contiguous(), e[:, :j].contiguous(), inp.wl.eps, S, S_T=S)
    kla.device_status(DEV)
    assert (o_acc == o_draft[:, :j]).all().item()
    pre = synth.PrefillInputs(dataclasses.replace(inp.wl, T=j), inp.q[:, :j], inp.k[:, :j], inp.v[:, :j],
                              inp.alpha[:, :j], inp.eta[:, :j], inp.S0)
    check(pre, o_acc.float().cpu().numpy().astype(np.float64), S.cpu().numpy().astype(np.float64))


def test_channel_chunk_form_serving_batch_whole():
    """16 draft tokens with the per-channel gate at the decode batch (64 sequences x 16 heads),
    every head against the oracle."""
    inp = synth.make_prefill("kda8k", seed=73, B=64, T=16, H=16, s0_sigma=0.02)
    o, S = run_prefill(inp)
    check(inp, o, S)
