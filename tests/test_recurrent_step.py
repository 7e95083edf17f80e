"""GPU parity of dr_recurrent_step against the fp64 oracle (through the C ABI)."""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_15_gb300 import inputs
from parity import assert_close, plain_err, record

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dr():
    import gated_delta_rule_15_gb300.dr as m
    return m


def la_at(s, t):
    return None if s["log_alpha"] is None else s["log_alpha"][t]


@pytest.mark.parametrize("gate", ["none", "scalar", "channel"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 128), (128, 64), (64, 64)])
def test_steps_small(dr, gate, dtype, dk, dv):
    steps = 16
    s = inputs.decode_inputs(5, 3, dk, dv, steps, gate=gate, dtype=dtype, seed=2)
    st = s["state"].cuda()
    ref = s["state"]
    for t in range(steps):
        o = dr.recurrent_step(s["q"][t].cuda(), s["k"][t].cuda(), s["v"][t].cuda(),
                              None if la_at(s, t) is None else la_at(s, t).cuda(),
                              s["beta"][t].cuda(), st)
        o_ref, ref = oracle.step(s["q"][t], s["k"][t], s["v"][t], la_at(s, t),
                                 s["beta"][t], ref)
        assert_close(o, o_ref, dtype, f"out step {t}")
    assert_close(st, ref, dtype, "state")
    assert dr.device_status() == 0


def test_step_equals_chunk_forward(dr):
    """Decode after a prefill continues the prefill: chunk_fwd over T tokens, then one
    step, equals the oracle over T + 1 tokens."""
    d = inputs.chunk_inputs(2, 97, 2, 128, 128, gate="channel", dtype="f32",
                            init_state=True, seed=8)
    g = {k: (None if v is None else v.cuda()) for k, v in d.items()}
    sl = lambda t, a, b: t[:, a:b].contiguous()
    _, st = dr.chunk_fwd(sl(g["q"], 0, 96), sl(g["k"], 0, 96), sl(g["v"], 0, 96),
                         sl(g["log_alpha"], 0, 96), sl(g["beta"], 0, 96), g["init_state"])
    o = dr.recurrent_step(g["q"][:, 96].contiguous(), g["k"][:, 96].contiguous(),
                          g["v"][:, 96].contiguous(), g["log_alpha"][:, 96].contiguous(),
                          g["beta"][:, 96].contiguous(), st)
    torch.cuda.synchronize()
    o_ref, f_ref = oracle.forward(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"],
                                  d["init_state"])
    assert_close(o, o_ref[:, 96], "f32", "out")
    assert_close(st, f_ref, "f32", "state")


@pytest.mark.slow
@pytest.mark.parametrize("out_dtype", ["bf16", "f32"])
@pytest.mark.parametrize("name", ["decode_scalar_B256_H32_d128", "decode_channel_B256_H32_d128"])
def test_full_size_64_steps_sampled(dr, name, out_dtype):
    """B = 256, H = 32, 512 MiB state, 64 steps in place; the oracle follows a sample of
    chains through all 64 steps; every output of every step on the sampled chains and
    their final states are compared.  An fp32-stored output is held to the plain rule (no
    representation allowance); for the bf16 output the plain error is recorded beside the
    allowanced one."""
    w = inputs.DECODE_WORKLOADS[name]
    s = inputs.decode_workload_inputs(w)
    st = s["state"].cuda()
    g = {k: (None if v is None else v.cuda()) for k, v in s.items() if k != "state"}
    odt = torch.float32 if out_dtype == "f32" else None
    outs = []
    for t in range(w.steps):
        outs.append(dr.recurrent_step(g["q"][t], g["k"][t], g["v"][t],
                                      None if g["log_alpha"] is None else g["log_alpha"][t],
                                      g["beta"][t], st, out_dtype=odt))
    torch.cuda.synchronize()
    outs = torch.stack(outs).cpu()
    st_h = st.cpu()
    rng = np.random.default_rng(0)
    worst = {"out": 0.0, "out_plain": 0.0, "state": 0.0}
    for c in rng.choice(w.B * w.H, size=16, replace=False):
        b, h = int(c) // w.H, int(c) % w.H
        ref = s["state"][b:b + 1, h:h + 1]
        for t in range(w.steps):
            pick = lambda x: None if x is None else x[t, b:b + 1, h:h + 1]
            o_ref, ref = oracle.step(pick(s["q"]), pick(s["k"]), pick(s["v"]),
                                     pick(s["log_alpha"]), pick(s["beta"]), ref, nthreads=1)
            o_gpu = outs[t, b:b + 1, h:h + 1]
            worst["out"] = max(worst["out"], assert_close(o_gpu, o_ref, "bf16", f"out {(t, b, h)}"))
            worst["out_plain"] = max(worst["out_plain"], plain_err(o_gpu, o_ref))
        worst["state"] = max(worst["state"], assert_close(st_h[b:b + 1, h:h + 1], ref, "bf16", f"state {(b, h)}"))
    record(name, f"recurrent_step out={out_dtype}", **worst)


@pytest.mark.parametrize("gate", ["none", "scalar", "channel"])
def test_bf16_inputs_fp32_output_strict(dr, gate):
    """With an fp32-stored output there is no representation allowance."""
    steps = 8
    s = inputs.decode_inputs(5, 3, 128, 128, steps, gate=gate, dtype="bf16", seed=6)
    st = s["state"].cuda()
    ref = s["state"]
    for t in range(steps):
        o = dr.recurrent_step(s["q"][t].cuda(), s["k"][t].cuda(), s["v"][t].cuda(),
                              None if la_at(s, t) is None else la_at(s, t).cuda(),
                              s["beta"][t].cuda(), st, out_dtype=torch.float32)
        assert o.dtype == torch.float32
        o_ref, ref = oracle.step(s["q"][t], s["k"][t], s["v"][t], la_at(s, t),
                                 s["beta"][t], ref)
        assert_close(o, o_ref, "bf16", f"out step {t}")
    assert_close(st, ref, "bf16", "state")
