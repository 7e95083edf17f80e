"""GPU parity of the fused neighbours (dr_chunk_fwd_ex, dr_recurrent_step_ex: L2-normalised
q and k, beta from logits, SiLU output gate) against the oracle's forward_fused and
step_fused, through the C ABI, on every kernel path: the scalar-gate tensor-core kernel
(bf16, d = 128, C = 64, including its segment-parallel form), the per-channel pair, the
CUDA-core fallback (fp32 inputs, d = 64, C < 64) and the decode step."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_15_gb300 import inputs
from parity import assert_close, assert_close_gated, record

pytestmark = pytest.mark.gpu

# (qk_l2norm, beta_sigmoid, output gate)
FLAGS = [(True, False, False), (False, True, False), (False, False, True), (True, True, True)]
FLAG_IDS = ["l2", "sigmoid", "silu", "all"]


@pytest.fixture(scope="module")
def dr():
    import gated_delta_rule_15_gb300.dr as m
    return m


def problem(B, T, H, dk, dv, flags, **kw):
    """Inputs for the requested neighbours: the raw q, k (normalisation fused), beta
    logits (sigmoid fused) and z (gate fused) of one draw, the prepared values of the same
    draw otherwise (raw keys of norm ~ sqrt(dk), or logits used as beta, make the rule
    diverge)."""
    l2, sig, gz = flags
    raw = inputs.chunk_inputs(B, T, H, dk, dv, raw=True, **kw)
    d = inputs.chunk_inputs(B, T, H, dk, dv, **kw)
    if l2:
        d["q"], d["k"] = raw["q"], raw["k"]
    if sig:
        d["beta"] = raw["beta"]
    d["z"] = raw["z"] if gz else None
    return d


def run(dr, d, flags, **kw):
    l2, sig, _ = flags
    g = {k: (None if v is None else v.cuda()) for k, v in d.items()}
    out, fin = dr.chunk_fwd(g["q"], g["k"], g["v"], g["log_alpha"], g["beta"],
                            g["init_state"], qk_l2norm=l2, beta_sigmoid=sig, z=g["z"], **kw)
    torch.cuda.synchronize()
    assert dr.device_status() == 0
    return out, fin


def assert_out(out, o_ungated, z, dtype, what="out"):
    """The output against the oracle: directly, or through the gate's elementwise bound
    when the SiLU gate is fused."""
    if z is None:
        return assert_close(out, o_ungated, dtype, what)
    return assert_close_gated(out, o_ungated, oracle.silu(oracle.to_f64(z)), dtype, what)


def check(dr, d, flags, dtype, **kw):
    l2, sig, _ = flags
    out, fin = run(dr, d, flags, **kw)
    o_ref, f_ref = oracle.forward_fused(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"],
                                        d["init_state"], qk_l2norm=l2, beta_sigmoid=sig)
    if d["q"].shape[1]:
        assert_out(out, o_ref, d["z"], dtype)
    assert_close(fin, f_ref, dtype, "final_state")


@pytest.mark.parametrize("flags", FLAGS, ids=FLAG_IDS)
@pytest.mark.parametrize("gate", ["none", "scalar", "channel"])
def test_tensor_core_paths(dr, gate, flags):
    # bf16, d = 128: the fused scalar-gate kernel (none, scalar) or the per-channel pair;
    # T = 200: three chunks and a ragged tail of 8 tokens
    d = problem(2, 200, 3, 128, 128, flags, gate=gate, dtype="bf16", init_state=True, seed=21)
    check(dr, d, flags, "bf16")


@pytest.mark.parametrize("flags", FLAGS, ids=FLAG_IDS)
@pytest.mark.parametrize("gate", ["none", "scalar"])
def test_tensor_core_single_kernel(dr, gate, flags):
    """The scalar / no-gate configurations run the fused neighbours on the two-kernel path
    when the workspace holds its operands (dr_chunk_fwd_ex_workspace_bytes), and on the
    single kernel otherwise: that path too, with the least workspace."""
    d = problem(2, 200, 3, 128, 128, flags, gate=gate, dtype="bf16", init_state=True, seed=22)
    desc = dr.chunk_desc(2, 200, 3, 128, 128, dr.DR_BF16, dr.DR_BF16, inputs.GATE_CODE[gate], 64)
    fl = dr.fuse_flags(*flags[:2], flags[2] or None)
    assert dr.min_workspace_bytes(desc) == 0 and dr.ex_workspace_bytes(desc, fl) > 0
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    check(dr, d, flags, "bf16", workspace=ws)


@pytest.mark.parametrize("la_range", [(0.001, 0.1), (0.0, 3.0)])
def test_two_kernel_path_decay_forms_all_flags(dr, la_range):
    """The two-kernel path folds the row norms into the decay factors of P: around the
    chunk's middle token for spans up to 80 (log space), per pair beyond."""
    d = problem(2, 190, 2, 128, 128, FLAGS[-1], gate="scalar", dtype="bf16", init_state=True,
                seed=23, log_alpha_range=la_range)
    check(dr, d, FLAGS[-1], "bf16", out_dtype=torch.float32)


@pytest.mark.parametrize("flags", FLAGS, ids=FLAG_IDS)
@pytest.mark.parametrize("dtype,dk,dv,chunk", [("f32", 128, 128, 64), ("f32", 64, 64, 32),
                                               ("bf16", 64, 128, 64), ("bf16", 128, 128, 16)])
def test_cuda_core_path(dr, flags, dtype, dk, dv, chunk):
    d = problem(2, 150, 2, dk, dv, flags, gate="channel", dtype=dtype, init_state=True, seed=5)
    check(dr, d, flags, dtype, chunk=chunk)
    d = problem(1, 100, 2, dk, dv, flags, gate="scalar", dtype=dtype, init_state=True, seed=6)
    check(dr, d, flags, dtype, chunk=chunk)


@pytest.mark.parametrize("T", [1, 63, 64, 65, 130])
@pytest.mark.parametrize("gate", ["scalar", "channel"])
def test_edge_lengths_all_flags(dr, T, gate):
    d = problem(1, T, 2, 128, 128, FLAGS[-1], gate=gate, dtype="bf16", init_state=True, seed=T)
    check(dr, d, FLAGS[-1], "bf16")


@pytest.mark.parametrize("gate", ["scalar", "channel"])
def test_fp32_output(dr, gate):
    d = problem(2, 130, 2, 128, 128, FLAGS[-1], gate=gate, dtype="bf16", init_state=True, seed=9)
    check(dr, d, FLAGS[-1], "bf16", out_dtype=torch.float32)


@pytest.mark.parametrize("least", [False, True])
def test_segment_parallel_all_flags(dr, least):
    # two chains of 64 chunks: split into segments whose end states are chained; the
    # normalisation and sigmoid enter the segment transitions, the gate only the outputs
    # (the two-kernel path, or with the least workspace the single kernel)
    d = problem(1, 4096, 2, 128, 128, FLAGS[-1], gate="scalar", dtype="bf16", init_state=True,
                seed=12)
    kw = {}
    if least:
        desc = dr.chunk_desc(1, 4096, 2, 128, 128, dr.DR_BF16, dr.DR_BF16, dr.DR_GATE_SCALAR, 64)
        kw["workspace"] = torch.empty(dr.min_workspace_bytes(desc), dtype=torch.uint8, device="cuda")
    check(dr, d, FLAGS[-1], "bf16", **kw)


def test_strong_decay_all_flags(dr):
    d = problem(1, 200, 2, 128, 128, FLAGS[-1], gate="channel", dtype="bf16", init_state=True,
                seed=4, log_alpha_range=(0.0, 3.0))
    check(dr, d, FLAGS[-1], "bf16")


@pytest.mark.parametrize("gate", ["scalar", "channel"])
def test_zero_flags_match_plain_entry_point(dr, gate):
    """dr_chunk_fwd_ex with fuse = 0 is dr_chunk_fwd, bit for bit."""
    d = inputs.chunk_inputs(1, 130, 2, 128, 128, gate=gate, dtype="bf16", init_state=True, seed=2)
    g = {k: (None if v is None else v.cuda()) for k, v in d.items()}
    out1, fin1 = dr.chunk_fwd(g["q"], g["k"], g["v"], g["log_alpha"], g["beta"], g["init_state"])
    B, T, H, dk = g["q"].shape
    desc = dr.chunk_desc(B, T, H, dk, 128, dr.DR_BF16, dr.DR_BF16, inputs.GATE_CODE[gate])
    ws = torch.empty(max(dr.workspace_bytes(desc), 16), dtype=torch.uint8, device="cuda")
    out2, fin2 = torch.empty_like(out1), torch.empty_like(fin1)
    p = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None
    rc = dr.lib().dr_chunk_fwd_ex(ctypes.byref(desc), 0, p(g["q"]), p(g["k"]), p(g["v"]),
                                  p(g["log_alpha"]), p(g["beta"]), None, p(g["init_state"]),
                                  p(out2), p(fin2), p(ws), ws.numel(),
                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    torch.cuda.synchronize()
    assert torch.equal(out1, out2) and torch.equal(fin1, fin2)


def test_normalised_inputs_unchanged_by_l2_flag(dr):
    """Unit inputs: the fused normalisation changes the result only at rounding level."""
    d = inputs.chunk_inputs(2, 130, 2, 128, 128, gate="scalar", dtype="f32", init_state=True,
                            seed=3)
    d["z"] = None
    o1, f1 = run(dr, d, (False, False, False))
    o2, f2 = run(dr, d, (True, False, False))
    assert (o1 - o2).abs().max().item() < 1e-5
    assert (f1 - f2).abs().max().item() < 1e-5


@pytest.mark.parametrize("flags", FLAGS, ids=FLAG_IDS)
@pytest.mark.parametrize("gate", ["none", "scalar", "channel"])
@pytest.mark.parametrize("dtype,dk,dv", [("bf16", 128, 128), ("f32", 64, 128), ("f32", 128, 64)])
def test_decode_steps(dr, flags, gate, dtype, dk, dv):
    l2, sig, gz = flags
    steps = 8
    raw = inputs.decode_inputs(5, 3, dk, dv, steps, gate=gate, dtype=dtype, seed=4, raw=True)
    s = inputs.decode_inputs(5, 3, dk, dv, steps, gate=gate, dtype=dtype, seed=4)
    if l2:
        s["q"], s["k"] = raw["q"], raw["k"]
    beta = raw["beta"] if sig else s["beta"]
    z = raw["z"] if gz else None
    st = s["state"].cuda()
    ref = s["state"]
    for t in range(steps):
        la = None if s["log_alpha"] is None else s["log_alpha"][t]
        o = dr.recurrent_step(s["q"][t].cuda(), s["k"][t].cuda(), s["v"][t].cuda(),
                              None if la is None else la.cuda(), beta[t].cuda(), st,
                              qk_l2norm=l2, beta_sigmoid=sig,
                              z=None if z is None else z[t].cuda())
        o_ref, ref = oracle.step_fused(s["q"][t], s["k"][t], s["v"][t], la, beta[t], ref,
                                       qk_l2norm=l2, beta_sigmoid=sig)
        assert_out(o, o_ref, None if z is None else z[t], dtype, f"out step {t}")
    assert_close(st, ref, dtype, "state")
    assert dr.device_status() == 0


def test_decode_continues_fused_prefill(dr):
    """A fused prefill (chunk forward) followed by a fused step equals the oracle over
    T + 1 tokens with the same neighbours."""
    d = problem(2, 97, 2, 128, 128, FLAGS[-1], gate="channel", dtype="bf16", init_state=True,
                seed=8)
    g = {k: (None if v is None else v.cuda()) for k, v in d.items()}
    sl = lambda t, a, b: t[:, a:b].contiguous()
    kw = dict(qk_l2norm=True, beta_sigmoid=True)
    _, st = dr.chunk_fwd(*(sl(g[n], 0, 96) for n in ("q", "k", "v", "log_alpha", "beta")),
                         g["init_state"], z=sl(g["z"], 0, 96), **kw)
    o = dr.recurrent_step(*(g[n][:, 96].contiguous() for n in ("q", "k", "v", "log_alpha", "beta")),
                          st, z=g["z"][:, 96].contiguous(), **kw)
    torch.cuda.synchronize()
    o_ref, f_ref = oracle.forward_fused(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"],
                                        d["init_state"], **kw)
    assert_out(o, o_ref[:, 96], d["z"][:, 96], "bf16")
    assert_close(st, f_ref, "bf16", "state")


@pytest.mark.slow
@pytest.mark.parametrize("out_dtype", ["bf16", "f32"])
def test_full_size_sampled_chains_all_flags(dr, out_dtype):
    """Every neighbour fused on the headline workload at full size (B8 H16 T4096), in the
    configuration the benchmark times; the oracle recomputes a sample of whole chains.  An
    fp32-stored output gets no representation allowance."""
    w = inputs.WORKLOADS["gdn_bf16_B8_H16_T4096_d128"]
    d = problem(w.B, w.T, w.H, w.dk, w.dv, FLAGS[-1], gate=w.gate, dtype=w.dtype, seed=0)
    odt = torch.float32 if out_dtype == "f32" else None
    out, fin = run(dr, d, FLAGS[-1], out_dtype=odt)
    out, fin = out.cpu(), fin.cpu()
    rng = np.random.default_rng(1)
    worst = {"out_gated": 0.0, "state": 0.0}
    for c in rng.choice(w.B * w.H, size=3, replace=False):
        b, h = int(c) // w.H, int(c) % w.H
        pick = lambda t: None if t is None else t[b:b + 1, :, h:h + 1].contiguous()
        o_ref, f_ref = oracle.forward_fused(pick(d["q"]), pick(d["k"]), pick(d["v"]),
                                            pick(d["log_alpha"]), pick(d["beta"]), None,
                                            qk_l2norm=True, beta_sigmoid=True)
        worst["out_gated"] = max(worst["out_gated"], assert_out(out[b:b + 1, :, h:h + 1], o_ref, pick(d["z"]), "bf16",
                                                                f"out chain {(b, h)}"))
        worst["state"] = max(worst["state"], assert_close(fin[b:b + 1, h:h + 1], f_ref, "bf16", f"state chain {(b, h)}"))
    record("fused_all_gdn_bf16_B8_H16_T4096_d128", f"chunk_fwd_ex out={out_dtype}", **worst)
