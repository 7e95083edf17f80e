"""Failure detection without a GPU fault: a bounded device-side wait runs out on purpose (a
barrier nothing completes), the kernel records DR_ERR_TIMEOUT and returns, the host reads
the status, and the context keeps working."""
import pytest
import torch

import oracle
from gated_delta_rule_15_gb300 import inputs
from parity import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dr():
    import gated_delta_rule_15_gb300.dr as m
    return m


def test_expired_wait_is_reported_and_cleared(dr):
    assert dr.device_status() == dr.DR_OK
    assert dr.selftest_bounded_wait(2_000_000) == dr.DR_OK   # about a millisecond
    assert dr.device_status() == dr.DR_ERR_TIMEOUT
    assert dr.device_status() == dr.DR_OK                    # read once, then cleared


def test_context_usable_after_an_expired_wait(dr):
    assert dr.selftest_bounded_wait(1_000_000) == dr.DR_OK
    assert dr.device_status() == dr.DR_ERR_TIMEOUT
    d = inputs.chunk_inputs(1, 130, 2, 128, 128, gate="scalar", dtype="bf16", init_state=True,
                            seed=1)
    g = {k: (None if v is None else v.cuda()) for k, v in d.items()}
    out, fin = dr.chunk_fwd(g["q"], g["k"], g["v"], g["log_alpha"], g["beta"], g["init_state"])
    torch.cuda.synchronize()
    assert dr.device_status() == dr.DR_OK
    o_ref, f_ref = oracle.forward(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"],
                                  d["init_state"])
    assert_close(out, o_ref, "bf16", "out")
    assert_close(fin, f_ref, "bf16", "final_state")
