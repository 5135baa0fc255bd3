"""Prefill of host tensors (kla_chunk_fwd_host): the work split into parts whose copies and
kernels overlap must give exactly what kla_chunk_fwd gives on device copies of the same inputs,
for any part count, with or without an initial and a final state. bf16 calls with the scalar gate
and d = 128 split along time (slices of whole chunks, the state carried in fp32 between them);
the others split the batch (whole sequences through the same kernels). The last part of a batch
of long sequences runs the sequence-parallel segments instead; it is checked against the
oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import DEV, oracle_chains, to_dev

pytestmark = pytest.mark.gpu


def host(a):
    a = np.ascontiguousarray(a)
    t = torch.from_numpy(a)
    if a.dtype == np.uint16:
        t = t.view(torch.int16).view(torch.bfloat16)
    return t.pin_memory()


@pytest.mark.parametrize("base,over,parts", [
    ("gdn4k", dict(B=4, T=300, H=2, s0_sigma=0.05), 1),
    ("gdn4k", dict(B=4, T=300, H=2, s0_sigma=0.05), 3),
    ("kda8k", dict(B=5, T=130, H=2), 5),
    ("gdn4k", dict(B=3, T=77, H=2, d_k=64, d_v=32, chunk=32, dtype="f32", s0_sigma=0.1), 2),
    ("decode", dict(B=6, T=4, H=2, chunk=64, s0_sigma=0.02), 4),
])
def test_host_prefill_matches_device_prefill(base, over, parts):
    import gated_delta_rule_14_gb300 as kla
    inp = synth.make_prefill(base, seed=over["B"] * 10 + parts, **over)
    args = [inp.q, inp.k, inp.v, inp.alpha, inp.eta]
    o_d, s_d = kla.chunk_fwd(*(to_dev(x) for x in args), inp.wl.eps, to_dev(inp.S0), chunk=inp.wl.chunk)
    S0 = None if inp.S0 is None else host(inp.S0)
    o_h, s_h = kla.chunk_fwd_host(*(host(x) for x in args), inp.wl.eps, S0, chunk=inp.wl.chunk, parts=parts,
                                  device=DEV)
    torch.cuda.synchronize(DEV)
    kla.device_status(DEV)
    assert torch.equal(o_h, o_d.cpu()) and torch.equal(s_h, s_d.cpu())
    o_ref, s_ref = oracle_chains(inp)
    chains = [(b, h) for b in range(inp.wl.B) for h in range(inp.wl.H)]
    o_g = np.stack([o_h.float().numpy()[b, :, h] for b, h in chains])
    s_g = np.stack([s_h.numpy()[b, h] for b, h in chains])
    tol = 1e-5 if inp.wl.dtype == "f32" else 1e-2
    assert oracle.rel_l2(o_g, o_ref) <= tol and oracle.rel_l2(s_g, s_ref) <= tol


def test_host_prefill_without_final_state_and_bad_parts():
    import gated_delta_rule_14_gb300 as kla
    inp = synth.make_prefill("gdn4k", seed=2, B=2, T=100, H=2)
    args = [host(x) for x in (inp.q, inp.k, inp.v, inp.alpha, inp.eta)]
    o_h, s_h = kla.chunk_fwd_host(*args, inp.wl.eps, final_state=False, parts=2, device=DEV)
    torch.cuda.synchronize(DEV)
    assert s_h is None
    o_d, _ = kla.chunk_fwd(*(to_dev(x) for x in (inp.q, inp.k, inp.v, inp.alpha, inp.eta)), inp.wl.eps)
    assert torch.equal(o_h, o_d.cpu())
    with pytest.raises(kla.KlaError):
        kla.chunk_fwd_host(*args, inp.wl.eps, parts=3, device=DEV)   # more parts than sequences


def test_host_prefill_segments_the_last_part():
    """Batch parts of one sequence of 4096 tokens (16 chains of 64 chunks, per-channel gate): the
    last part, the call's tail, runs the sequence-parallel segments on the library's fixed
    scratch. A second call (one part, so its prefill runs on another of the library's compute
    streams) is issued from another stream while the first may still run: the two share the
    scratch, ordered by the library's event. Both match the oracle on sampled chains; repeating
    the first call reproduces it bit for bit."""
    import gated_delta_rule_14_gb300 as kla
    lib = kla._native.lib()
    torch.cuda.set_device(DEV)
    assert lib.kla_chunk_fwd_workspace_size(1, 4096, 16, 128, 128, 64, 1, 1) > 4 * 16   # segments pay off here
    inp = synth.make_prefill("kda8k", seed=41, B=2, T=4096, H=16, s0_sigma=0.05)
    args = [host(x) for x in (inp.q, inp.k, inp.v, inp.alpha, inp.eta)]
    S0 = host(inp.S0)
    o1, s1 = kla.chunk_fwd_host(*args, inp.wl.eps, S0, parts=2, device=DEV)
    side = torch.cuda.Stream(DEV)
    with torch.cuda.stream(side):
        o2, s2 = kla.chunk_fwd_host(*args, inp.wl.eps, S0, parts=1, device=DEV)
    o3, s3 = kla.chunk_fwd_host(*args, inp.wl.eps, S0, parts=2, device=DEV)
    torch.cuda.synchronize(DEV)
    kla.device_status(DEV)
    assert torch.equal(o1, o3) and torch.equal(s1, s3)
    chains = [(0, 0), (0, 9), (0, 15), (1, 0), (1, 6), (1, 15)]
    o_ref, s_ref = oracle_chains(inp, chains)
    for o, st in ((o1, s1), (o2, s2)):
        o_g = np.stack([o.float().numpy()[b, :, h] for b, h in chains])
        s_g = np.stack([st.numpy()[b, h] for b, h in chains])
        assert oracle.rel_l2(o_g, o_ref) <= 1e-2 and oracle.rel_l2(s_g, s_ref) <= 1e-2


@pytest.mark.parametrize("parts", [1, 3])
def test_host_prefill_reruns_out_of_range_channel_gates(parts):
    """Per-channel gates outside the factorised range in a part other than the last and in the
    last part: both are rerun exactly inside the host call, as kla_chunk_fwd does."""
    import gated_delta_rule_14_gb300 as kla
    inp = synth.make_prefill("kda8k", seed=40 + parts, B=3, T=130, H=2)
    inp.alpha[0, 10:45, 1, 7] = 1e-3     # part 0 (of 3)
    inp.alpha[2, 64:100, 0, 90] = 1e-3   # the last part
    args = [inp.q, inp.k, inp.v, inp.alpha, inp.eta]
    o_d, s_d = kla.chunk_fwd(*(to_dev(x) for x in args), inp.wl.eps, None, chunk=inp.wl.chunk)
    o_h, s_h = kla.chunk_fwd_host(*(host(x) for x in args), inp.wl.eps, None, chunk=inp.wl.chunk, parts=parts,
                                  device=DEV)
    torch.cuda.synchronize(DEV)
    kla.device_status(DEV)   # raises if anything was only reported
    assert torch.equal(o_h, o_d.cpu()) and torch.equal(s_h, s_d.cpu())
    o_ref, s_ref = oracle_chains(inp)
    chains = [(b, h) for b in range(inp.wl.B) for h in range(inp.wl.H)]
    o_g = np.stack([o_h.float().numpy()[b, :, h] for b, h in chains])
    s_g = np.stack([s_h.numpy()[b, h] for b, h in chains])
    assert oracle.rel_l2(o_g, o_ref) <= 1e-2 and oracle.rel_l2(s_g, s_ref) <= 1e-2


@pytest.mark.parametrize("parts,final", [(5, True), (16, False), (1, False)])
def test_host_prefill_time_parts(parts, final):
    """Time parts (bf16, scalar gate, d = 128): slices of whole chunks of every sequence, the last
    one ragged; the state carried between slices in S_T, or, without a final state, in the
    library's fixed scratch (two calls back to back share it). Equal bit for bit to kla_chunk_fwd
    on device copies, whose kernel keeps the state in fp32 as the slices do."""
    import gated_delta_rule_14_gb300 as kla
    inp = synth.make_prefill("gdn4k", seed=60 + parts, B=3, T=1100, H=2, s0_sigma=0.05)
    dev_args = [to_dev(x) for x in (inp.q, inp.k, inp.v, inp.alpha, inp.eta)]
    o_d, s_d = kla.chunk_fwd(*dev_args, inp.wl.eps, to_dev(inp.S0))
    args = [host(x) for x in (inp.q, inp.k, inp.v, inp.alpha, inp.eta)]
    outs = [kla.chunk_fwd_host(*args, inp.wl.eps, host(inp.S0), parts=parts, final_state=final, device=DEV)
            for _ in range(2)]
    torch.cuda.synchronize(DEV)
    kla.device_status(DEV)
    for o_h, s_h in outs:
        assert torch.equal(o_h, o_d.cpu())
        assert (s_h is None) if not final else torch.equal(s_h, s_d.cpu())
