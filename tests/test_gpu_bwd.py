"""Backward pass (kla_chunk_bwd) against the fp64 oracle's backward, which is itself pinned to
finite differences of the forward. Every gradient (q, k, v, alpha, eta, S0) is compared by
relative L2 over the whole tensor, and the oracle receives the same stored (fp32 or bf16-rounded)
inputs.

Two paths, two bars:
  * bf16 inputs with d_k = d_v = 128 and more than 16 tokens run the chunkwise tensor-core
    backward (scalar or per-channel gate), whose products take bf16 operands with fp32
    accumulation and fp32 carried states, like the forward's tensor-core path; they are held to
    the bf16 bar of the forward, 1e-2;
  * every other shape runs the token-by-token fp32 backward: 1e-5 for fp32 inputs, 1e-4 for bf16
    inputs (longer sums of larger terms)."""
import os

import numpy as np
import pytest

import oracle
import synth
from gpu_util import DEV, to_dev

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-5, "bf16": 1e-4}
TOL_CHUNK = 1e-2


def tol(wl):
    chunked = wl.dtype == "bf16" and wl.d_k == 128 and wl.d_v == 128 and wl.T > 16
    return TOL_CHUNK if chunked else TOL[wl.dtype]
NAMES = ("dq", "dk", "dv", "dalpha", "deta", "dS0")


def _grad_inputs(inp, seed, with_dst):
    rng = np.random.default_rng(seed)
    wl = inp.wl
    dO = rng.standard_normal((wl.B, wl.T, wl.H, wl.d_v)).astype(np.float32)
    if wl.dtype == "bf16":
        dO = synth.f32_to_bf16_bits(dO)
    dST = rng.standard_normal((wl.B, wl.H, wl.d_k, wl.d_v)).astype(np.float32) if with_dst else None
    return dO, dST


def _as64(a):
    if a is None:
        return None
    return synth.bf16_bits_to_f32(a).astype(np.float64) if a.dtype == np.uint16 else a.astype(np.float64)


def run_gpu(inp, dO, dST, **mode):
    import gated_delta_rule_14_gb300 as kla
    g = kla.chunk_bwd(to_dev(inp.q), to_dev(inp.k), to_dev(inp.v), to_dev(inp.alpha), to_dev(inp.eta), to_dev(dO),
                      inp.wl.eps, to_dev(inp.S0), to_dev(dST), **mode)
    kla.device_status(DEV)
    return {n: (None if g[n] is None else g[n].cpu().numpy().astype(np.float64)) for n in NAMES}


def run_oracle(inp, dO, dST, chains=None, **mode):
    """Oracle gradients on the listed (b, h) chains, each as its own B=1, H=1 problem."""
    wl = inp.wl
    chains = chains or [(b, h) for b in range(wl.B) for h in range(wl.H)]
    out = {n: [] for n in NAMES}
    for b, h in chains:
        f = lambda a: None if a is None else _as64(a)[b:b + 1, :, h:h + 1]  # noqa: E731
        s0 = None if inp.S0 is None else inp.S0[b:b + 1, h:h + 1].astype(np.float64)
        dst = None if dST is None else dST[b:b + 1, h:h + 1].astype(np.float64)
        g = oracle.load().backward(f(inp.q), f(inp.k), f(inp.v), f(inp.alpha), f(inp.eta), wl.eps, s0, f(dO), dst,
                                   **mode)
        for n in NAMES:
            out[n].append(g[n][0, :, 0] if n != "dS0" else g[n][0, 0])
    return {n: np.stack(v) for n, v in out.items()}


def pick(g, chains):
    return {n: (None if g[n] is None else
                np.stack([g[n][b, :, h] if n != "dS0" else g[n][b, h] for b, h in chains])) for n in NAMES}


def compare(got, ref, tol, skip=()):
    for n in NAMES:
        if n in skip:
            continue
        assert np.isfinite(got[n]).all(), n
        err = oracle.rel_l2(got[n], ref[n])
        assert err <= tol, f"{n}: rel-L2 {err:.3e} > {tol}"


CASES = [
    # (base, overrides, mode, with dL/dS_T)
    ("tiny", dict(B=2, T=1, H=2, s0_sigma=0.1), {}, True),
    ("tiny", dict(B=1, T=37, H=3, d_k=32, d_v=64, s0_sigma=0.1), {}, False),
    ("kda8k", dict(B=2, T=21, H=2, d_k=64, d_v=16, dtype="f32", s0_sigma=0.1), {}, True),
    ("gdn4k", dict(B=1, T=100, H=2, dtype="f32", s0_sigma=0.05, key_norm="l2"), dict(beta_mode="raw"), True),
    ("gdn4k", dict(B=2, T=130, H=2, s0_sigma=0.05), {}, True),
    ("kda8k", dict(B=1, T=64, H=2, s0_sigma=0.05), dict(q_scale=128 ** -0.5), False),
    ("gdn4k", dict(B=1, T=203, H=1, d_k=16, d_v=128, dtype="f32"), dict(q_scale=0.5), True),
    ("gdn4k", dict(B=1, T=1, H=3), {}, True),     # short: the token-by-token fp32 backward
    # chunkwise tensor-core path: shortest chunked length, exactly one chunk, ragged tails, raw
    # step, query scale
    ("gdn4k", dict(B=1, T=17, H=2), {}, True),
    ("gdn4k", dict(B=1, T=64, H=1), {}, False),
    ("gdn4k", dict(B=2, T=257, H=1, s0_sigma=0.05, key_norm="l2"), dict(beta_mode="raw", q_scale=0.5), True),
    ("gdn4k", dict(B=1, T=200, H=2, s0_sigma=0.02), dict(q_scale=128 ** -0.5), True),
    ("long131k", dict(T=320, H=2), {}, True),
    # chunkwise per-channel gate: shortest chunked length, ragged tails over several chunks, raw
    # step, query scale, initial state and dL/dS_T
    ("kda8k", dict(B=1, T=17, H=2), {}, True),
    ("kda8k", dict(B=2, T=200, H=2, s0_sigma=0.05), {}, True),
    ("kda8k", dict(B=1, T=257, H=2, s0_sigma=0.05, key_norm="l2"), dict(beta_mode="raw", q_scale=0.5), True),
    ("kda8k", dict(B=1, T=128, H=3), dict(q_scale=128 ** -0.5), False),
]


@pytest.mark.parametrize("base,over,mode,with_dst", CASES, ids=lambda x: str(x)[:36])
def test_backward_against_oracle(base, over, mode, with_dst):
    inp = synth.make_prefill(base, seed=over["T"] + 5, **over)
    dO, dST = _grad_inputs(inp, seed=over["T"], with_dst=with_dst)
    got = run_gpu(inp, dO, dST, **mode)
    ref = run_oracle(inp, dO, dST, **mode)
    chains = [(b, h) for b in range(inp.wl.B) for h in range(inp.wl.H)]
    compare(pick(got, chains), ref, tol(inp.wl))


@pytest.mark.parametrize("base", ["gdn4k", "kda8k"])
def test_more_chains_than_sms(base):
    """More chains than a GB300 has SMs (192 against 152): the tensor-core carries, one CTA per
    chain holding all of its SM's tensor memory, run in two waves (and the per-channel gate's two
    carries one after the other, as they no longer fit side by side). Every gradient of every
    chain against the oracle."""
    inp = synth.make_prefill(base, seed=43, B=3, T=130, H=64, s0_sigma=0.05)
    dO, dST = _grad_inputs(inp, seed=44, with_dst=True)
    got = run_gpu(inp, dO, dST)
    ref = run_oracle(inp, dO, dST)
    chains = [(b, h) for b in range(inp.wl.B) for h in range(inp.wl.H)]
    compare(pick(got, chains), ref, tol(inp.wl))


def test_backward_without_ds0_and_empty_sequence():
    import torch

    import gated_delta_rule_14_gb300 as kla
    inp = synth.make_prefill("gdn4k", seed=3, B=1, T=19, H=2, s0_sigma=0.05)
    dO, dST = _grad_inputs(inp, seed=4, with_dst=True)
    full = run_gpu(inp, dO, dST)
    g = kla.chunk_bwd(to_dev(inp.q), to_dev(inp.k), to_dev(inp.v), to_dev(inp.alpha), to_dev(inp.eta), to_dev(dO),
                      inp.wl.eps, to_dev(inp.S0), to_dev(dST), want_dS0=False)
    kla.device_status(DEV)
    assert g["dS0"] is None
    for n in ("dq", "dk", "dv", "dalpha", "deta"):
        assert np.array_equal(g[n].cpu().numpy().astype(np.float64), full[n]), n
    # T = 0: dL/dS0 = dL/dS_T
    z = torch.empty((1, 0, 2, 128), dtype=torch.bfloat16, device=DEV)
    za = torch.empty((1, 0, 2), dtype=torch.float32, device=DEV)
    dst = to_dev(dST)
    g = kla.chunk_bwd(z, z, z, za, za, z, 1e-6, to_dev(inp.S0), dst)
    kla.device_status(DEV)
    assert torch.equal(g["dS0"], dst)


def run_oracle_whole(inp, dO, dST, **mode):
    """Oracle gradients of the whole input in one call, chains split over the host cores. The
    oracle keeps every state of the chains it is working on ((T + 1) d_k d_v doubles each), so the
    thread count is capped to hold that under ~8 GB."""
    wl = inp.wl
    per_chain = (wl.T + 1) * wl.d_k * wl.d_v * 8
    threads = max(1, min(os.cpu_count() or 1, int(8e9 // per_chain)))
    g = oracle.load().backward(_as64(inp.q), _as64(inp.k), _as64(inp.v), _as64(inp.alpha), _as64(inp.eta), wl.eps,
                               None if inp.S0 is None else inp.S0.astype(np.float64), _as64(dO),
                               None if dST is None else dST.astype(np.float64), nthreads=threads, **mode)
    return {n: g[n] for n in NAMES}


@pytest.mark.parametrize("name", ["gdn4k", "kda8k"])
def test_full_config_whole_tensor(name):
    """The backward of the prefill workloads at full size on the chunkwise path (scalar gate on
    gdn4k, per-channel gate on kda8k), every gradient compared over the whole tensor."""
    inp = synth.make_prefill(name, seed=1)
    dO, dST = _grad_inputs(inp, seed=2, with_dst=True)
    got = run_gpu(inp, dO, dST)
    ref = run_oracle_whole(inp, dO, dST)
    compare(got, ref, tol(inp.wl))


def test_chunked_backward_is_deterministic():
    """The chunkwise path sums in a fixed order (no atomics): two calls agree bit for bit."""
    inp = synth.make_prefill("gdn4k", seed=11, B=2, T=150, H=2, s0_sigma=0.05)
    dO, dST = _grad_inputs(inp, seed=12, with_dst=True)
    a = run_gpu(inp, dO, dST)
    b = run_gpu(inp, dO, dST)
    for n in NAMES:
        assert np.array_equal(a[n], b[n]), n


def test_unaligned_inputs_take_the_token_path():
    """q, k, v, dO views that start 2 bytes past a 16-byte boundary are valid bf16 arguments; the
    chunkwise path needs 16-byte rows, so they run the token-by-token fp32 backward and meet its
    1e-4 bar."""
    import torch

    import gated_delta_rule_14_gb300 as kla
    inp = synth.make_prefill("gdn4k", seed=13, B=1, T=70, H=2, s0_sigma=0.05)
    dO, dST = _grad_inputs(inp, seed=14, with_dst=True)

    def shifted(a):
        t = to_dev(a)
        buf = torch.empty(t.numel() + 8, dtype=t.dtype, device=DEV)
        view = buf[1:1 + t.numel()].view(t.shape)
        view.copy_(t)
        assert view.data_ptr() % 16 == 2
        return view
    g = kla.chunk_bwd(shifted(inp.q), shifted(inp.k), shifted(inp.v), to_dev(inp.alpha), to_dev(inp.eta), shifted(dO),
                      inp.wl.eps, to_dev(inp.S0), to_dev(dST))
    kla.device_status(DEV)
    got = {n: g[n].cpu().numpy().astype(np.float64) for n in NAMES}
    ref = run_oracle(inp, dO, dST)
    chains = [(b, h) for b in range(inp.wl.B) for h in range(inp.wl.H)]
    compare(pick(got, chains), ref, TOL["bf16"])


@pytest.mark.parametrize("T,mode", [(4059, {}), (2048 + 31, dict(beta_mode="raw", q_scale=0.5)),
                                    (16384 - 5, {})])   # 256 chunks on two chains: 32 segments of 8
def test_long_chain_segmented_carries(T, mode):
    """Few chains and many chunks: the chunkwise backward splits both carries into segments run in
    parallel (value runs, transitions from the identity, start states combined, reruns; with two
    chains and 64 chunks the cost model picks 8 segments), with S0, dL/dS_T and a ragged tail."""
    over = dict(B=1, T=T, H=2, s0_sigma=0.05)
    if mode:
        over["key_norm"] = "l2"
    inp = synth.make_prefill("gdn4k", seed=T, **over)
    dO, dST = _grad_inputs(inp, seed=T + 1, with_dst=True)
    got = run_gpu(inp, dO, dST, **mode)
    ref = run_oracle(inp, dO, dST, **mode)
    compare(pick(got, [(0, 0), (0, 1)]), ref, TOL_CHUNK)


@pytest.mark.parametrize("mode", [{}, dict(beta_mode="raw")])
def test_chunked_backward_zero_keys_and_unit_gates(mode):
    """Degenerate tokens inside chunks: keys that are exactly zero with eps = 0 (beta = 0 by
    definition, no gradient flows through the step size) and gates of exactly 1 (no decay)."""
    import dataclasses
    # the raw step (beta = eta) needs unit keys: beta norm(k)^2 > 2 makes the recurrence diverge
    norm = dict(key_norm="l2") if mode else {}
    inp = synth.make_prefill("gdn4k", seed=77, B=1, T=150, H=2, s0_sigma=0.05, eps=0.0, **norm)
    k = inp.k.copy()
    k[:, [0, 5, 63, 64, 100, 149]] = 0                      # bf16 zero bits
    alpha = inp.alpha.copy()
    alpha[:, 10:40] = 1.0
    inp = dataclasses.replace(inp, k=k, alpha=alpha)
    dO, dST = _grad_inputs(inp, seed=78, with_dst=True)
    got = run_gpu(inp, dO, dST, **mode)
    ref = run_oracle(inp, dO, dST, **mode)
    compare(pick(got, [(0, 0), (0, 1)]), ref, TOL_CHUNK)


@pytest.mark.parametrize("mode", [{}, dict(beta_mode="raw")])
def test_channel_chunked_backward_zero_keys_and_unit_gates(mode):
    """Per-channel gate, degenerate tokens inside chunks: zero keys with eps = 0 (beta = 0, no
    gradient through the step size), gates of exactly 1 on every channel, and gates of 1 on half
    of the channels only."""
    import dataclasses
    norm = dict(key_norm="l2") if mode else {}
    inp = synth.make_prefill("kda8k", seed=79, B=1, T=150, H=2, s0_sigma=0.05, eps=0.0, **norm)
    k = inp.k.copy()
    k[:, [0, 5, 63, 64, 100, 149]] = 0
    alpha = inp.alpha.copy()
    alpha[:, 10:40] = 1.0
    alpha[:, 70:120, :, ::2] = 1.0
    inp = dataclasses.replace(inp, k=k, alpha=alpha)
    dO, dST = _grad_inputs(inp, seed=80, with_dst=True)
    got = run_gpu(inp, dO, dST, **mode)
    ref = run_oracle(inp, dO, dST, **mode)
    compare(pick(got, [(0, 0), (0, 1)]), ref, TOL_CHUNK)


def test_channel_chunked_backward_strong_decay():
    """Per-channel gates well below those of the kda8k workload (log alpha = -softplus(N(-2, 1.5)),
    inside the factorised range): the decay-crossing terms of d alpha cancel in pairs, and the
    kernel keeps them cancelling under bf16 rounding."""
    import dataclasses
    inp = synth.make_prefill("kda8k", seed=81, B=1, T=300, H=2, s0_sigma=0.05)
    rng = np.random.default_rng(82)
    x = rng.normal(-2.0, 1.5, inp.alpha.shape)
    alpha = np.exp(-np.logaddexp(0.0, x)).astype(np.float32)
    alpha = np.maximum(alpha, np.float32(0.12))   # half-chunk products stay above e^-78
    inp = dataclasses.replace(inp, alpha=alpha)
    dO, dST = _grad_inputs(inp, seed=83, with_dst=True)
    got = run_gpu(inp, dO, dST)
    ref = run_oracle(inp, dO, dST)
    compare(pick(got, [(0, 0), (0, 1)]), ref, TOL_CHUNK)


def test_channel_chunked_backward_is_deterministic():
    inp = synth.make_prefill("kda8k", seed=84, B=2, T=150, H=2, s0_sigma=0.05)
    dO, dST = _grad_inputs(inp, seed=85, with_dst=True)
    a = run_gpu(inp, dO, dST)
    b = run_gpu(inp, dO, dST)
    for n in NAMES:
        assert np.array_equal(a[n], b[n]), n


def test_channel_gate_out_of_range_chain_takes_the_exact_path():
    """A chain whose per-channel gates multiply below ~e^-78 over half a chunk is outside the range
    of the factorised in-chunk products: the chunkwise kernels skip it and the token-sequential
    fp32 backward reruns it in the same call, so it meets that path's 1e-4 bar while the other
    chains stay chunkwise."""
    inp = synth.make_prefill("kda8k", seed=86, B=2, T=200, H=2, s0_sigma=0.05)
    inp.alpha[1, 70:110, 0, 9] = 1e-3
    dO, dST = _grad_inputs(inp, seed=87, with_dst=True)
    got = run_gpu(inp, dO, dST)
    chains = [(0, 0), (0, 1), (1, 0), (1, 1)]
    ref = run_oracle(inp, dO, dST, chains=chains)
    compare(pick(got, chains), ref, TOL_CHUNK)
    compare(pick(got, [(1, 0)]), run_oracle(inp, dO, dST, chains=[(1, 0)]), TOL["bf16"])


@pytest.mark.parametrize("T,mode", [(4059, {}), (2048 + 31, dict(beta_mode="raw", q_scale=0.5)), (16384 - 5, {})])
def test_channel_long_chain_segmented_carries(T, mode):
    """Per-channel gate with few chains and many chunks: both carries split into segments run in
    parallel, reading the per-channel records (decayed keys, scaled queries, end decays); also
    with the raw step (unit keys) and a query scale."""
    over = dict(B=1, T=T, H=2, s0_sigma=0.05)
    if mode:
        over["key_norm"] = "l2"
    inp = synth.make_prefill("kda8k", seed=T + 3, **over)
    dO, dST = _grad_inputs(inp, seed=T + 4, with_dst=True)
    got = run_gpu(inp, dO, dST, **mode)
    ref = run_oracle(inp, dO, dST, **mode)
    compare(pick(got, [(0, 0), (0, 1)]), ref, TOL_CHUNK)
