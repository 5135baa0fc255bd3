"""Helpers shared by the GPU parity tests: move seeded host inputs to the device, call the
library, and run the fp64 oracle on all or on a sample of the (sequence, head) chains."""
import os

import numpy as np
import torch

import oracle
import synth

DEV = torch.device("cuda:0")


def to_dev(a, bf16=None):
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    t = torch.from_numpy(a)
    if a.dtype == np.uint16:
        t = t.view(torch.int16).view(torch.bfloat16)
    return t.to(DEV)


def run_prefill(inp, chunk=None, **kw):
    import gated_delta_rule_14_gb300 as kla
    o, ST = kla.chunk_fwd(to_dev(inp.q), to_dev(inp.k), to_dev(inp.v), to_dev(inp.alpha), to_dev(inp.eta),
                          inp.wl.eps, to_dev(inp.S0), chunk=chunk or inp.wl.chunk, **kw)
    kla.device_status(DEV)
    return o.float().cpu().numpy().astype(np.float64), ST.cpu().numpy().astype(np.float64)


def oracle_chains(inp, chains=None, **mode):
    """fp64 oracle on the listed (b, h) chains (all when None); returns o [n,T,dv], S [n,dk,dv].
    ``mode``: beta_mode / q_scale passed to the oracle."""
    B, T, H = inp.wl.B, inp.wl.T, inp.wl.H
    if chains is None:
        chains = [(b, h) for b in range(B) for h in range(H)]

    def pick(name):
        a = inp.as_f64(name)
        if a is None:
            return None
        if name == "S0":
            return np.stack([a[b, h] for b, h in chains])[:, None]
        return np.stack([a[b, :, h] for b, h in chains])[:, :, None]
    o, S = oracle.recurrent(pick("q"), pick("k"), pick("v"), pick("alpha"), pick("eta"), inp.wl.eps, pick("S0"),
                            nthreads=os.cpu_count() or 1, **mode)
    return o[:, :, 0], S[:, 0]


def oracle_whole(inp, **mode):
    """fp64 oracle over the whole input (every chain, all host cores): o [B,T,H,dv], S_T [B,H,dk,dv]."""
    return oracle.recurrent(inp.as_f64("q"), inp.as_f64("k"), inp.as_f64("v"), inp.as_f64("alpha"),
                            inp.as_f64("eta"), inp.wl.eps, inp.as_f64("S0"), nthreads=os.cpu_count() or 1, **mode)


def worst_chain(o, o_ref):
    """Largest per-(sequence, head) relative L2 error of o [B,T,H,dv]: a diagnostic beside the
    whole-tensor figure."""
    B, H = o.shape[0], o.shape[2]
    return max(oracle.rel_l2(o[b, :, h], o_ref[b, :, h]) for b in range(B) for h in range(H))


def gather_chains(o, S, chains):
    return (np.stack([o[b, :, h] for b, h in chains]), np.stack([S[b, h] for b, h in chains]))


def sample_chains(B, H, n, seed=0):
    rng = np.random.default_rng(seed)
    idx = rng.choice(B * H, size=min(n, B * H), replace=False)
    return [(int(i) // H, int(i) % H) for i in sorted(idx)]


def decode_oracle(d, heads=None, **mode):
    """Oracle over all decode steps: the steps of one head are the tokens of one chain."""
    n, B, H = d.alpha.shape[:3]
    heads = heads or [(b, h) for b in range(B) for h in range(H)]
    f = lambda a: synth.bf16_bits_to_f32(a).astype(np.float64) if a.dtype == np.uint16 else a.astype(np.float64)  # noqa
    q, k, v = f(d.q), f(d.k), f(d.v)
    al, et = d.alpha.astype(np.float64), d.eta.astype(np.float64)
    Q = np.stack([q[:, b, h] for b, h in heads])[:, :, None]
    K = np.stack([k[:, b, h] for b, h in heads])[:, :, None]
    V = np.stack([v[:, b, h] for b, h in heads])[:, :, None]
    Al = np.stack([al[:, b, h] for b, h in heads])[:, :, None]
    Et = np.stack([et[:, b, h] for b, h in heads])[:, :, None]
    S0 = np.stack([d.S[b, h] for b, h in heads]).astype(np.float64)[:, None]
    o, S = oracle.recurrent(Q, K, V, Al, Et, d.wl.eps, S0, nthreads=os.cpu_count() or 1, **mode)
    return o[:, :, 0], S[:, 0]
