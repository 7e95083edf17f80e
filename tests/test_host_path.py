"""dr_chunk_fwd_host (host buffers in, host buffers out, the batch split into pieces whose
copies and kernels overlap) against the device entry point: the same results bit for bit,
since every (b, h) chain runs the same kernel code whichever piece holds it."""
import pytest
import torch

from gated_delta_rule_15_gb300 import inputs

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
    assert torch.equal(out_h, out_d.cpu()) and torch.equal(fin_h, fin_d.cpu())


def test_host_path_runs_repeatedly(dr):
    d = inputs.chunk_inputs(4, 130, 2, 128, 128, gate="scalar", dtype="bf16", seed=6)
    host = {k: (None if v is None else v.pin_memory()) for k, v in d.items()}
    runner = dr.HostChunkRunner(host, pieces=2)
    first = [t.clone() for t in runner(host)]
    for _ in range(3):
        again = runner(host)
        assert all(torch.equal(a, b) for a, b in zip(first, again))
