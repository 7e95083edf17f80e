"""dr_chunk_fwd_noalloc against dr_chunk_fwd, on the GPU, through the C ABI.

The allocation-free entry point serves callers that cannot allocate device memory (a host
framework that owns all device memory through its own pool, plugin callbacks that must not
allocate, loops that cannot pay cudaMalloc's implicit synchronisation).  It must give the
workspace entry point's results, call after call, although its static scratch keeps the
previous call's contents.  This file is collected last on purpose.
"""
import pytest
import torch

from gated_delta_rule_15_gb300 import inputs
from parity import assert_close

pytestmark = pytest.mark.gpu


def _run_both(dr, d, dtype):
    g = {k: (None if t is None else t.cuda()) for k, t in d.items()}
    ref_out, ref_fin = dr.chunk_fwd(g["q"], g["k"], g["v"], g["log_alpha"], g["beta"],
                                    g["init_state"])
    out = torch.full_like(ref_out, float("nan"))
    fin = torch.full_like(ref_fin, float("nan"))
    rc = dr.chunk_fwd_noalloc(g["q"], g["k"], g["v"], g["log_alpha"], g["beta"],
                              g["init_state"], out, fin)
    assert rc == dr.DR_OK, dr.strerror(rc)
    torch.cuda.synchronize()
    assert_close(out, ref_out.double().cpu().numpy(), dtype, "out")
    assert_close(fin, ref_fin.double().cpu().numpy(), dtype, "final_state")


def test_noalloc_matches_workspace_entry_two_calls_in_a_row():
    import gated_delta_rule_15_gb300.dr as dr
    # Two different problems back to back: the second runs on scratch left by the first.
    d1 = inputs.chunk_inputs(2, 300, 4, 128, 128, gate="channel", dtype="bf16",
                             init_state=True, seed=41)
    d2 = inputs.chunk_inputs(3, 190, 2, 128, 128, gate="scalar", dtype="f32",
                             init_state=False, seed=42)
    # Few long chains of the scalar gate take the segment-parallel form, whose segment
    # states also live in the scratch; it runs third, on what the two calls before left.
    d3 = inputs.chunk_inputs(1, 4096, 2, 128, 128, gate="scalar", dtype="bf16",
                             init_state=True, seed=43)
    desc3 = dr.chunk_desc(1, 4096, 2, 128, 128, dr.DR_BF16, dr.DR_BF16, dr.DR_GATE_SCALAR, 64)
    assert dr.workspace_bytes(desc3) > 0
    # The per-channel gate's segment states follow its per-chunk operands in the scratch.
    d4 = inputs.chunk_inputs(1, 4096, 2, 128, 128, gate="channel", dtype="bf16",
                             init_state=True, seed=44)
    desc4 = dr.chunk_desc(1, 4096, 2, 128, 128, dr.DR_BF16, dr.DR_BF16, dr.DR_GATE_CHANNEL, 64)
    assert dr.workspace_bytes(desc4) > 2 * 64 * 131584
    _run_both(dr, d1, "bf16")
    _run_both(dr, d2, "f32")
    _run_both(dr, d3, "bf16")
    _run_both(dr, d4, "bf16")


def test_noalloc_rejects_problems_beyond_its_scratch():
    import gated_delta_rule_15_gb300.dr as dr
    # The per-channel gate (bf16, d = 128, C = 64) needs 131,584 B of workspace per
    # (b, h, chunk): 600 chunks of one head exceed 64 MiB.
    T = 64 * 600
    desc = dr.chunk_desc(1, T, 1, 128, 128, dr.DR_BF16, dr.DR_BF16, dr.DR_GATE_CHANNEL, 64)
    assert dr.workspace_bytes(desc) > dr.NOALLOC_SCRATCH_BYTES
    q = torch.zeros((1, T, 1, 128), dtype=torch.bfloat16, device="cuda")
    la = torch.zeros((1, T, 1, 128), dtype=torch.float32, device="cuda")
    b = torch.zeros((1, T, 1), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((1, T, 1, 128), dtype=torch.bfloat16, device="cuda")
    rc = dr.chunk_fwd_noalloc(q, q, q, la, b, None, out, None)
    assert rc == dr.DR_ERR_WORKSPACE
