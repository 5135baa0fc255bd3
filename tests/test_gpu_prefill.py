"""Chunkwise prefill on the GPU against the fp64 oracle (relative L2 over the whole tensor:
<= 1e-5 for fp32 inputs, <= 1e-2 for bf16 inputs with the fp32 state)."""
import dataclasses

import numpy as np
import pytest

import oracle
import synth
from gpu_util import gather_chains, oracle_chains, oracle_whole, run_prefill, to_dev, worst_chain, DEV

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-5, "bf16": 1e-2}


def check(inp, o, S, chains=None):
    o_ref, s_ref = oracle_chains(inp, chains)
    if chains is None:
        chains = [(b, h) for b in range(inp.wl.B) for h in range(inp.wl.H)]
    o_g, s_g = gather_chains(o, S, chains)
    tol = TOL[inp.wl.dtype]
    eo, es = oracle.rel_l2(o_g, o_ref), oracle.rel_l2(s_g, s_ref)
    assert np.isfinite(o).all() and np.isfinite(S).all()
    assert eo <= tol and es <= tol, f"rel-L2 o={eo:.3e} S={es:.3e} tol={tol}"
    return eo, es


def test_tiny_config():
    inp = synth.make_prefill("tiny", seed=0)
    o, S = run_prefill(inp)
    check(inp, o, S)


CASES = [
    # (dtype, d_k, d_v, chunk, T, gate, s0)
    ("f32", 16, 16, 16, 1, "scalar", 0.0),
    ("f32", 16, 16, 16, 17, "channel", 0.1),
    ("f32", 32, 64, 32, 100, "scalar", 0.1),
    ("f32", 64, 32, 64, 130, "channel", 0.0),
    ("f32", 128, 128, 64, 75, "scalar", 0.05),
    ("f32", 128, 128, 16, 40, "channel", 0.05),
    ("bf16", 16, 16, 16, 33, "scalar", 0.1),
    ("bf16", 64, 64, 32, 97, "channel", 0.1),
    ("bf16", 128, 128, 64, 1, "scalar", 0.05),
    ("bf16", 128, 128, 64, 63, "scalar", 0.0),
    ("bf16", 128, 128, 64, 64, "scalar", 0.05),
    ("bf16", 128, 128, 64, 65, "scalar", 0.05),
    ("bf16", 128, 128, 64, 300, "scalar", 0.05),
    ("bf16", 128, 128, 64, 257, "channel", 0.05),
    ("bf16", 128, 128, 16, 50, "scalar", 0.0),
]


@pytest.mark.parametrize("dtype,dk,dv,C,T,gate,s0", CASES, ids=lambda x: str(x))
def test_small_shapes(dtype, dk, dv, C, T, gate, s0):
    base = "kda8k" if gate == "channel" else "gdn4k"
    inp = synth.make_prefill(base, seed=T * 7 + dk, B=2, T=T, H=3, d_k=dk, d_v=dv, chunk=C, dtype=dtype,
                             s0_sigma=s0)
    o, S = run_prefill(inp)
    check(inp, o, S)


def test_eta_one_eps_zero_exact_projection_and_extreme_gates():
    # unrelaxed KLA (eta = 1, eps = 0) and gates near 0 and 1
    inp = synth.make_prefill("gdn4k", seed=5, B=1, T=130, H=2, s0_sigma=0.05)
    inp.eta[...] = 1.0
    inp.alpha[0, :40] = 1.0
    inp.alpha[0, 40:50] = 1e-30
    inp = synth.PrefillInputs(dataclasses.replace(inp.wl, eps=0.0), inp.q, inp.k, inp.v, inp.alpha, inp.eta, inp.S0)
    o, S = run_prefill(inp)
    check(inp, o, S)


def test_continuation_two_calls_equal_one():
    import gated_delta_rule_14_gb300 as kla
    inp = synth.make_prefill("gdn4k", seed=9, B=2, T=200, H=2, s0_sigma=0.05)
    q, k, v, a, e, S0 = (to_dev(x) for x in (inp.q, inp.k, inp.v, inp.alpha, inp.eta, inp.S0))
    o_full, S_full = kla.chunk_fwd(q, k, v, a, e, inp.wl.eps, S0)
    T1 = 77
    o1, S1 = kla.chunk_fwd(q[:, :T1].contiguous(), k[:, :T1].contiguous(), v[:, :T1].contiguous(),
                           a[:, :T1].contiguous(), e[:, :T1].contiguous(), inp.wl.eps, S0)
    o2, S2 = kla.chunk_fwd(q[:, T1:].contiguous(), k[:, T1:].contiguous(), v[:, T1:].contiguous(),
                           a[:, T1:].contiguous(), e[:, T1:].contiguous(), inp.wl.eps, S1)
    kla.device_status(DEV)
    o_ref, s_ref = oracle_chains(inp)
    o_cat = np.concatenate([o1.float().cpu().numpy(), o2.float().cpu().numpy()], axis=1)
    o_g, s_g = gather_chains(o_cat, S2.cpu().numpy(), [(b, h) for b in range(2) for h in range(2)])
    assert oracle.rel_l2(o_g, o_ref) <= 1e-2 and oracle.rel_l2(s_g, s_ref) <= 1e-2
    assert oracle.rel_l2(S2.cpu().numpy(), S_full.cpu().numpy()) <= 1e-2


def test_state_in_place_and_empty_sequence():
    import torch

    import gated_delta_rule_14_gb300 as kla
    inp = synth.make_prefill("gdn4k", seed=10, B=1, T=70, H=2, s0_sigma=0.05)
    S = to_dev(inp.S0).clone()
    o, S_out = kla.chunk_fwd(to_dev(inp.q), to_dev(inp.k), to_dev(inp.v), to_dev(inp.alpha), to_dev(inp.eta),
                             inp.wl.eps, S, S_T=S)
    kla.device_status(DEV)
    assert S_out.data_ptr() == S.data_ptr()
    o_ref, s_ref = oracle_chains(inp)
    assert oracle.rel_l2(S.cpu().numpy()[0], s_ref) <= 1e-2
    # T = 0: the final state is the initial state, no output
    z = torch.empty((1, 0, 2, 128), dtype=torch.bfloat16, device=DEV)
    za = torch.empty((1, 0, 2), dtype=torch.float32, device=DEV)
    S0 = to_dev(inp.S0)
    o, ST = kla.chunk_fwd(z, z, z, za, za, 1e-6, S0)
    kla.device_status(DEV)
    assert o.shape == (1, 0, 2, 128) and torch.equal(ST, S0)
    o, ST = kla.chunk_fwd(z, z, z, za, za, 1e-6, None)
    assert torch.count_nonzero(ST).item() == 0


@pytest.mark.parametrize("name", ["gdn4k", "kda8k", "long131k"])
def test_full_config_whole_tensor(name):
    """The workloads at full size, in the launch configuration the benchmark times, against the
    oracle over every (sequence, head) chain: relative L2 over the whole o and S_T tensors."""
    inp = synth.make_prefill(name, seed=0)
    o, S = run_prefill(inp)
    assert np.isfinite(o).all() and np.isfinite(S).all()
    o_ref, s_ref = oracle_whole(inp)
    eo, es = oracle.rel_l2(o, o_ref), oracle.rel_l2(S, s_ref)
    tol = TOL[inp.wl.dtype]
    assert eo <= tol and es <= tol, f"rel-L2 o={eo:.3e} S={es:.3e} (worst chain {worst_chain(o, o_ref):.3e})"


@pytest.mark.parametrize("base", ["gdn4k", "kda8k"])
def test_more_chains_than_sms(base):
    """More (sequence, head) chains than a GB300 has SMs (192 against 152): the tensor-core
    prefill's CTAs, one per chain and each holding all of its SM's tensor memory, run in two
    waves, the second allocating what the first released. Every chain against the oracle."""
    inp = synth.make_prefill(base, seed=41, B=3, T=130, H=64, s0_sigma=0.05)
    o, S = run_prefill(inp)
    check(inp, o, S)


@pytest.mark.parametrize("gate", ["scalar", "channel"])
def test_zero_keys_eps_zero_unit_gates(gate):
    """Degenerate tokens on the tensor-core prefill: keys that are exactly zero with eps = 0 (the
    step is 0 by definition, so the token only decays the state), including the first and last
    token of a chunk and the ragged tail, and gates of exactly 1 (no decay) over part of a chunk
    and across a chunk boundary."""
    base = "kda8k" if gate == "channel" else "gdn4k"
    inp = synth.make_prefill(base, seed=31, B=1, T=150, H=2, s0_sigma=0.05, eps=0.0)
    k = inp.k.copy()
    k[:, [0, 5, 31, 32, 63, 64, 100, 149]] = 0        # bf16 zero bits
    alpha = inp.alpha.copy()
    alpha[:, 10:40] = 1.0
    alpha[:, 60:70] = 1.0
    inp = dataclasses.replace(inp, k=k, alpha=alpha)
    o, S = run_prefill(inp)
    check(inp, o, S)


def _starve(alpha, b, h, t0, n, ch, value=1e-3):
    """Per-channel gates of `value` for n tokens from t0 in key channel ch of chain (b, h): their
    product over half a chunk falls far below e^-80."""
    alpha[b, t0:t0 + n, h, ch] = value


def test_channel_gate_out_of_range_is_rerun_exactly():
    """Per-channel gates whose product over half a chunk falls below e^-80 leave the range of the
    tensor-core path's factorised products: the call marks those chains and reruns them on the
    fp32 token-by-token path in the same call, so the results are valid and no error is
    reported. The rerun chains' final states match the oracle to the fp32 bar, which the
    tensor-core path (bf16 operands) would not meet."""
    inp = synth.make_prefill("kda8k", seed=3, B=2, T=150, H=2, s0_sigma=0.05)
    _starve(inp.alpha, 0, 1, 0, 32, 5)               # first half of chunk 0
    _starve(inp.alpha, 1, 0, 70, 40, 100, 1e-30)     # across the halves of chunk 1, down to 1e-30
    o, S = run_prefill(inp)                          # device_status raises on any reported error
    check(inp, o, S)
    o_ref, s_ref = oracle_chains(inp, [(0, 1), (1, 0)])
    o_g, s_g = gather_chains(o, S, [(0, 1), (1, 0)])
    assert oracle.rel_l2(s_g, s_ref) <= 1e-5, "marked chains were not rerun on the fp32 path"
    # the same gates on the fp32 path throughout (chunk 32)
    o32, S32 = run_prefill(inp, chunk=32)
    check(inp, o32, S32)
    # unmarked chains keep the tensor-core results: a call without the starved chains agrees
    clean = synth.make_prefill("kda8k", seed=3, B=2, T=150, H=2, s0_sigma=0.05)
    o_c, S_c = run_prefill(clean)
    for b, h in [(0, 0), (1, 1)]:
        assert np.array_equal(o[b, :, h], o_c[b, :, h]) and np.array_equal(S[b, h], S_c[b, h])


def test_channel_gate_out_of_range_in_place_state():
    """S_T = S0 (in-place continuation) with a marked chain: the tensor-core kernel must leave that
    chain's state alone, because its exact rerun starts from S0."""
    import gated_delta_rule_14_gb300 as kla
    inp = synth.make_prefill("kda8k", seed=8, B=1, T=200, H=2, s0_sigma=0.05)
    _starve(inp.alpha, 0, 0, 100, 30, 17)
    S = to_dev(inp.S0).clone()
    o, S_out = kla.chunk_fwd(to_dev(inp.q), to_dev(inp.k), to_dev(inp.v), to_dev(inp.alpha), to_dev(inp.eta),
                             inp.wl.eps, S, S_T=S)
    kla.device_status(DEV)
    assert S_out.data_ptr() == S.data_ptr()
    check(inp, o.float().cpu().numpy().astype(np.float64), S.cpu().numpy().astype(np.float64))


def test_channel_gate_out_of_range_with_segments():
    """A long per-channel sequence split into segments (value runs, transitions, reruns), with
    starved gates in a middle segment and in the last one."""
    import gated_delta_rule_14_gb300 as kla
    T = 64 * 100 + 5
    inp = synth.make_prefill("kda8k", seed=21, B=1, T=T, H=1, s0_sigma=0.05)
    assert kla.workspace_size(1, T, 1, 128, 128, 64, per_channel_gate=True) > 4
    _starve(inp.alpha, 0, 0, 64 * 40 + 2, 33, 64)
    _starve(inp.alpha, 0, 0, T - 50, 40, 3)
    o, S = run_prefill(inp)
    check(inp, o, S)


@pytest.mark.parametrize("gate,T,H,s0", [("scalar", 64 * 200 + 17, 2, 0.05), ("scalar", 64 * 40, 1, 0.0),
                                         ("channel", 64 * 100 + 5, 1, 0.05)])
def test_long_sequence_segments(gate, T, H, s0):
    """Few chains and a long sequence: the tensor-core path splits each chain into segments that
    run in parallel (value runs, transition runs, a combine pass, then the rerun); the result must
    still match the sequential recurrence."""
    import gated_delta_rule_14_gb300 as kla
    base = "kda8k" if gate == "channel" else "long131k"
    inp = synth.make_prefill(base, seed=T % 97, B=1, T=T, H=H, s0_sigma=s0)
    assert kla.workspace_size(1, T, H, 128, 128, 64, per_channel_gate=(gate == "channel")) > 0
    o, S = run_prefill(inp)
    check(inp, o, S)


def test_long_sequence_segments_state_in_place():
    import gated_delta_rule_14_gb300 as kla
    inp = synth.make_prefill("long131k", seed=5, B=1, T=64 * 64, H=1, s0_sigma=0.05)
    S = to_dev(inp.S0).clone()
    o, S_out = kla.chunk_fwd(to_dev(inp.q), to_dev(inp.k), to_dev(inp.v), to_dev(inp.alpha), to_dev(inp.eta),
                             inp.wl.eps, S, S_T=S)
    kla.device_status(DEV)
    o_ref, s_ref = oracle_chains(inp)
    assert oracle.rel_l2(S.cpu().numpy()[0], s_ref) <= 1e-2
    assert oracle.rel_l2(o.float().cpu().numpy()[:, :, 0], o_ref) <= 1e-2


def test_channel_gate_alpha_not_16_byte_aligned():
    """The ABI needs only 4-byte alignment of alpha: a view of the per-channel gates starting 4 bytes
    past a 16-byte boundary gives the aligned call's results bit for bit and meets the oracle's bar."""
    import torch

    import gated_delta_rule_14_gb300 as kla
    inp = synth.make_prefill("kda8k", seed=41, B=2, T=200, H=2, s0_sigma=0.05)
    a = to_dev(inp.alpha)
    buf = torch.empty(a.numel() + 4, dtype=torch.float32, device=DEV)
    a_off = buf[1:1 + a.numel()].view(a.shape)
    a_off.copy_(a)
    assert a.data_ptr() % 16 == 0 and a_off.data_ptr() % 16 == 4
    args = (to_dev(inp.q), to_dev(inp.k), to_dev(inp.v))
    o1, s1 = kla.chunk_fwd(*args, a, to_dev(inp.eta), inp.wl.eps, to_dev(inp.S0))
    o2, s2 = kla.chunk_fwd(*args, a_off, to_dev(inp.eta), inp.wl.eps, to_dev(inp.S0))
    kla.device_status(DEV)
    assert torch.equal(o1, o2) and torch.equal(s1, s2)
    check(inp, o2.float().cpu().numpy().astype(np.float64), s2.cpu().numpy().astype(np.float64))
