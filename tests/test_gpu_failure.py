"""Failure detection without a GPU fault: a bounded wait that gives up is reported by
kla_device_status as KLA_ERR_TIMEOUT, the flag is cleared by that read, and the context keeps
working (a prefill right after matches the oracle)."""
import pytest

import oracle
import synth
from gpu_util import DEV, oracle_chains, run_prefill

pytestmark = pytest.mark.gpu


def test_bounded_wait_timeout_is_reported_and_recovered():
    import torch

    import gated_delta_rule_14_gb300 as kla
    lib = kla._native.lib()
    stream = torch.cuda.current_stream(DEV).cuda_stream
    kla.device_status(DEV)                                        # start from a clear flag
    assert lib.kla_selftest_wait_timeout(200, stream) == 0        # gives up after <= 4 ms
    assert lib.kla_device_status(stream) == kla._native.KLA_ERR_TIMEOUT
    assert lib.kla_device_status(stream) == kla._native.KLA_OK    # cleared by the read
    inp = synth.make_prefill("gdn4k", seed=12, B=1, T=130, H=2, s0_sigma=0.05)
    o, S = run_prefill(inp)
    o_ref, s_ref = oracle_chains(inp)
    assert oracle.rel_l2(o[0].transpose(1, 0, 2), o_ref) <= 1e-2
    assert oracle.rel_l2(S[0], s_ref) <= 1e-2
