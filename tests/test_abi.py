"""The C-ABI library loads, exports every symbol include/kla.h declares, and rejects bad
arguments on the host before launching anything (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from gated_delta_rule_14_gb300 import _native, build
    build.build()
    return _native.lib()


def declared_functions():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if h.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", h)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(kla_[a-z_0-9]+)\s*\(", txt, flags=re.M)
    return sorted(set(names))


def test_header_declares_entry_points():
    names = declared_functions()
    for required in ("kla_chunk_fwd", "kla_decode_step", "kla_chunk_fwd_workspace_size", "kla_status_string",
                     "kla_device_status", "kla_abi_version", "kla_chunk_fwd_ex", "kla_decode_step_ex",
                     "kla_chunk_bwd", "kla_chunk_bwd_workspace_size", "kla_chunk_bwd_workspace_size_ex",
                     "kla_chunk_fwd_host",
                     "kla_selftest_wait_timeout"):
        assert required in names, names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings_and_version(lib):
    for code, token in [(0, "KLA_OK"), (1, "INVALID_ARG"), (2, "UNSUPPORTED"), (3, "CUDA"), (4, "TIMEOUT")]:
        assert token in lib.kla_status_string(code).decode()
    assert "UNKNOWN" in lib.kla_status_string(99).decode()
    assert lib.kla_abi_version() == 102


# Fake, never dereferenced device addresses: every case below must be rejected on the host.
A = 0x7f0000000000


def chunk(lib, **kw):
    args = dict(q=A, k=A + 0x10000000, v=A + 0x20000000, alpha=A + 0x30000000, eta=A + 0x38000000, eps=1e-6,
                S0=None, o=A + 0x40000000, S_T=None, B=1, T=64, H=1, d_k=16, d_v=16, chunk=16, dtype=0, gate=0,
                ws=None, ws_bytes=0, stream=None)
    args.update(kw)
    return lib.kla_chunk_fwd(args["q"], args["k"], args["v"], args["alpha"], args["eta"], args["eps"],
                             args["S0"], args["o"], args["S_T"], args["B"], args["T"], args["H"], args["d_k"],
                             args["d_v"], args["chunk"], args["dtype"], args["gate"], args["ws"], args["ws_bytes"],
                             args["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), 1), (dict(o=None), 1), (dict(q=None, T=0), 0), (dict(alpha=None), 1), (dict(eta=None), 1),
    (dict(T=-1), 1), (dict(B=0), 1), (dict(H=0), 1), (dict(dtype=7), 1), (dict(gate=3), 1),
    (dict(q=A + 8), 1), (dict(o=A + 0x40000004), 1), (dict(S0=A + 0x50000002), 1),
    (dict(d_k=48), 2), (dict(d_v=256), 2), (dict(chunk=128), 2), (dict(chunk=8), 2),
    (dict(eps=float("nan")), 1),
    (dict(S_T=A + 0x10000000), 1),                     # final state overlapping k
    (dict(S0=A + 0x50000000, S_T=A + 0x50000200), 1),  # partial overlap of S0 and S_T
])
def test_chunk_fwd_rejects_on_host(lib, kw, code):
    assert chunk(lib, **kw) == code


def test_decode_rejects_on_host(lib):
    f = lib.kla_decode_step
    ok = dict(q=A, k=A + 0x1000000, v=A + 0x2000000, alpha=A + 0x3000000, eta=A + 0x3800000, S=A + 0x4000000,
              o=A + 0x5000000)

    def call(**kw):
        a = dict(ok)
        a.update(kw)
        return f(a["q"], a["k"], a["v"], a["alpha"], a["eta"], 1e-6, a["S"], a["o"], 2, 2, 16, 16, 1, 0, None)
    assert call(S=None) == 1
    assert call(S=A + 0x4000004) == 1
    assert call(q=A + 1) == 1                # bf16 vector not aligned to its element
    assert call(v=None) == 1
    assert call(S=A) == 1                    # state overlaps q
    assert f(A, A + 0x1000000, A + 0x2000000, A + 0x3000000, A + 0x3800000, 1e-6, A + 0x4000000, A + 0x5000000,
             2, 2, 24, 16, 1, 0, None) == 2


def test_workspace_size_is_a_host_call(lib):
    assert lib.kla_chunk_fwd_workspace_size(8, 4096, 16, 128, 128, 64, 1, 0) >= 0


@pytest.mark.parametrize("mode,scale,code", [
    (2, 1.0, 1), (-1, 1.0, 1), (0, float("nan"), 1), (1, float("inf"), 1), (0, float("-inf"), 1),
])
def test_ex_entry_points_reject_bad_options_on_host(lib, mode, scale, code):
    f = lib.kla_chunk_fwd_ex
    assert f(A, A + 0x10000000, A + 0x20000000, A + 0x30000000, A + 0x38000000, 1e-6, None, A + 0x40000000,
             None, 1, 64, 1, 16, 16, 16, 0, 0, mode, scale, None, 0, None) == code
    g = lib.kla_decode_step_ex
    assert g(A, A + 0x1000000, A + 0x2000000, A + 0x3000000, A + 0x3800000, 1e-6, A + 0x4000000, A + 0x5000000,
             2, 2, 16, 16, 1, 0, mode, scale, None) == code


def test_ex_entry_points_accept_the_options_before_checking_pointers(lib):
    # valid options do not mask an argument error that comes after them
    f = lib.kla_chunk_fwd_ex
    assert f(None, A, A, A, A, 1e-6, None, A, None, 1, 64, 1, 16, 16, 16, 0, 0, 1, 0.25, None, 0, None) == 1
    assert f(A, A + 0x10000000, A + 0x20000000, A + 0x30000000, A + 0x38000000, 1e-6, None, A + 0x40000000,
             None, 1, 64, 1, 48, 16, 16, 0, 0, 1, 0.0, None, 0, None) == 2


def bwd(lib, **kw):
    args = dict(q=A, k=A + 0x10000000, v=A + 0x20000000, alpha=A + 0x30000000, eta=A + 0x38000000, S0=None,
                dO=A + 0x40000000, dST=None, dq=A + 0x50000000, dk=A + 0x58000000, dv=A + 0x60000000,
                dalpha=A + 0x68000000, deta=A + 0x6c000000, dS0=None, B=1, T=64, H=1, d_k=16, d_v=16, dtype=0,
                gate=0, mode=0, scale=1.0, ws=A + 0x70000000, ws_bytes=1 << 26, stream=None)
    args.update(kw)
    a = args
    return lib.kla_chunk_bwd(a["q"], a["k"], a["v"], a["alpha"], a["eta"], 1e-6, a["S0"], a["dO"], a["dST"], a["dq"],
                             a["dk"], a["dv"], a["dalpha"], a["deta"], a["dS0"], a["B"], a["T"], a["H"], a["d_k"],
                             a["d_v"], a["dtype"], a["gate"], a["mode"], a["scale"], a["ws"], a["ws_bytes"],
                             a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(dq=None), 1), (dict(dO=None), 1), (dict(ws=None), 1), (dict(ws_bytes=16), 1), (dict(ws=A + 0x70000008), 1),
    (dict(dv=A + 0x60000004), 1), (dict(dq=A + 0x20000000), 1),      # dq overlaps v
    (dict(dk=A + 0x50000100), 1),                                   # dk overlaps dq
    (dict(dS0=A + 0x70000000), 1),                                  # dS0 overlaps the workspace
    (dict(mode=3), 1), (dict(scale=float("nan")), 1), (dict(d_k=24), 2), (dict(T=-1), 1),
])
def test_bwd_rejects_on_host(lib, kw, code):
    assert bwd(lib, **kw) == code


def test_bwd_workspace_size(lib):
    # state every 8 tokens plus every residual, fp32
    seq = (2 * 3 * 3 * 16 * 32 + 2 * 20 * 3 * 32) * 4
    assert lib.kla_chunk_bwd_workspace_size(2, 20, 3, 16, 32) == seq
    assert lib.kla_chunk_bwd_workspace_size(2, 0, 3, 16, 32) == 0
    lib.kla_chunk_bwd_workspace_size_ex.restype = ctypes.c_size_t
    ex = lib.kla_chunk_bwd_workspace_size_ex
    assert ex(2, 20, 3, 16, 32, 1, 0) == seq                       # not the chunkwise shape
    # bf16, scalar gate, d = 128: per 64-token chunk of every chain, G / beta / norm (fp32) and
    # W, U (then dE), E, A, T, S_c, dS_{c+1} (bf16); no segments without a device to plan on
    per_chunk = 3 * 64 * 4 + 2 * (3 * 64 * 128 + 2 * 64 * 64 + 2 * 128 * 128)
    assert ex(2, 200, 3, 128, 128, 1, 0) == 2 * 3 * 4 * per_chunk
    assert ex(2, 200, 3, 128, 128, 0, 0) == (2 * 3 * 25 * 128 * 128 + 2 * 200 * 3 * 128) * 4  # fp32: token path
    assert ex(2, 16, 3, 128, 128, 1, 0) == (2 * 3 * 2 * 128 * 128 + 2 * 16 * 3 * 128) * 4   # T <= 16: token path
    # bf16, per-channel gate, d = 128: one mark per chain (256-byte aligned), then room for the larger
    # of the chunkwise records (those above plus dE of its own, K e^{G_end - G}, s Q e^{G} and
    # e^{G_end}) and the token path's checkpoints, which rerun the chains outside the factorised range
    seq_ws = (2 * 3 * 25 * 128 * 128 + 2 * 200 * 3 * 128) * 4
    rec_ch = 2 * 3 * 4 * (per_chunk + 3 * 2 * 64 * 128 + 4 * 128)
    assert ex(2, 200, 3, 128, 128, 1, 1) == 256 + max(rec_ch, seq_ws)
    assert ex(2, 200, 3, 128, 128, 0, 1) == seq_ws                  # fp32 per-channel: token path
    assert lib.kla_chunk_bwd_workspace_size(2, 200, 3, 128, 128) >= ex(2, 200, 3, 128, 128, 1, 0)
    assert lib.kla_chunk_bwd_workspace_size(2, 200, 3, 128, 128) >= ex(2, 200, 3, 128, 128, 1, 1)


def test_host_prefill_rejects_on_host(lib):
    f = lib.kla_chunk_fwd_host
    H_ = 0x10000   # fake host and device addresses, never touched: every case fails validation first

    def call(**kw):
        a = dict(q=H_, k=H_, v=H_, al=H_, et=H_, s0h=None, oh=H_, sth=None, qd=A, kd=A, vd=A, ald=A, etd=A, s0d=None,
                 od=A, std=None, B=2, T=8, H=1, parts=2)
        a.update(kw)
        return f(a["q"], a["k"], a["v"], a["al"], a["et"], a["s0h"], a["oh"], a["sth"], a["qd"], a["kd"], a["vd"],
                 a["ald"], a["etd"], a["s0d"], a["od"], a["std"], 1e-6, a["B"], a["T"], a["H"], 16, 16, 16, 0, 0, 0,
                 1.0, a["parts"], None)
    assert call(parts=3) == 1          # more parts than sequences
    assert call(parts=0) == 1
    assert call(q=None) == 1
    assert call(od=None) == 1
    assert call(s0h=H_) == 1           # host S0 without a device buffer for it
    assert call(std=A) == 1            # device S_T without a host one
    assert call(T=0) == 1


def test_selftest_rejects_limits_on_host(lib):
    lib.kla_selftest_wait_timeout.argtypes = [ctypes.c_uint, ctypes.c_void_p]
    assert lib.kla_selftest_wait_timeout(0, None) == 1
    assert lib.kla_selftest_wait_timeout(100001, None) == 1
