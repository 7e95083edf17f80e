"""dr_chunk_fwd_host (host buffers in, host buffers out, the sequence split into time pieces
whose copies and kernels overlap, the state carried on the device) against the device entry
point.  The pieces are whole chunks and every kernel carries the state between chunks in
fp32, as it is carried between pieces, so the results are the same bit for bit."""
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


@pytest.mark.parametrize("pieces", [1, 3, 8])
@pytest.mark.parametrize("gate,dtype,dk,init", [("scalar", "bf16", 128, False),
                                                ("channel", "bf16", 128, True),
                                                ("scalar", "f32", 64, True),
                                                ("none", "bf16", 128, True)])
def test_host_path_equals_device_path(dr, pieces, gate, dtype, dk, init):
    d = inputs.chunk_inputs(5, 150, 3, dk, dk, gate=gate, dtype=dtype, init_state=init, seed=4)
    g = {k: (None if v is None else v.cuda()) for k, v in d.items()}
    out_d, fin_d = dr.chunk_fwd(g["q"], g["k"], g["v"], g["log_alpha"], g["beta"], g["init_state"])
    host = {k: (None if v is None else v.pin_memory()) for k, v in d.items()}
    out_h, fin_h = dr.HostChunkRunner(host, pieces=pieces)(host)
    assert dr.device_status() == 0
    # whole chunks per piece, the state carried in fp32 as inside one call: the same bits
    assert torch.equal(out_h, out_d.cpu()) and torch.equal(fin_h, fin_d.cpu())
    o_ref, f_ref = oracle.forward(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"],
                                  d["init_state"])
    assert_close(out_h, o_ref, dtype, "out")
    assert_close(fin_h, f_ref, dtype, "final_state")


def test_host_path_runs_repeatedly(dr):
    d = inputs.chunk_inputs(4, 130, 2, 128, 128, gate="scalar", dtype="bf16", seed=6)
    host = {k: (None if v is None else v.pin_memory()) for k, v in d.items()}
    runner = dr.HostChunkRunner(host, pieces=2)
    first = [t.clone() for t in runner(host)]
    for _ in range(3):
        again = runner(host)
        assert all(torch.equal(a, b) for a, b in zip(first, again))
