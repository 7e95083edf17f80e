"""GPU parity of dr_chunk_bwd (the backward of the chunk forward) against the fp64 oracle's
reverse mode of the token loop, through the C ABI.

Tolerance (the pages fix none for gradients): fp32 inputs, max|g - g_ref| <=
1e-4 max(1, RMS(g_ref)) per gradient (the forward's absolute bound for unit-scale values,
scaled with gradients that sum many unit-scale terms); bf16 inputs, the forward's rule
(max-abs/RMS <= 2e-2, half a bf16 ulp allowed on bf16-stored gradients)."""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_15_gb300 import inputs
from parity import err, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dr():
    import gated_delta_rule_15_gb300.dr as m
    return m


def assert_grad(gpu, ref, dtype, what):
    if dtype == "f32":
        g, r = to_np(gpu), np.asarray(ref)
        assert g.shape == r.shape, what
        assert np.isfinite(g).all(), what
        scale = max(1.0, float(np.sqrt((r ** 2).mean()))) if r.size else 1.0
        e = float(np.abs(g - r).max()) / scale if r.size else 0.0
        assert e <= 1e-4, f"{what}: error {e:.3e} > 1e-4"
    else:
        e, tol = err(gpu, ref, "bf16")
        assert e <= tol, f"{what}: error {e:.3e} > {tol:.1e}"


def grads_problem(B, T, H, dk, dv, *, gate, dtype, seed, init_state=True, d_final=True,
                  log_alpha_range=(0.001, 0.1)):
    d = inputs.chunk_inputs(B, T, H, dk, dv, gate=gate, dtype=dtype, init_state=init_state,
                            seed=seed, log_alpha_range=log_alpha_range)
    g = torch.Generator().manual_seed(seed + 100)
    d["d_out"] = torch.randn((B, T, H, dv), generator=g).to(inputs.DTYPES[dtype])
    d["d_final"] = torch.randn((B, H, dk, dv), generator=g) if d_final else None
    return d


def check(dr, d, dtype, chunk=64):
    dev = {k: (None if v is None else v.cuda()) for k, v in d.items()}
    got = dr.chunk_bwd(dev["q"], dev["k"], dev["v"], dev["log_alpha"], dev["beta"],
                       dev["init_state"], dev["d_out"], dev["d_final"], chunk=chunk)
    torch.cuda.synchronize()
    assert dr.device_status() == 0
    ref = oracle.backward(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["init_state"],
                          d["d_out"], d["d_final"])
    for name, g, r in zip(("dq", "dk", "dv", "dlog_alpha", "dbeta", "dinit"), got, ref):
        if r is None:
            assert g is None, name
            continue
        assert_grad(g, r, "f32" if name in ("dlog_alpha", "dinit") and dtype == "f32" else dtype,
                    name)


@pytest.mark.parametrize("gate", ["none", "scalar", "channel"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 128), (128, 64), (64, 64)])
def test_small_shapes(dr, gate, dtype, dk, dv):
    # T = 150: two full chunks and a ragged tail; initial state and final-state gradient
    check(dr, grads_problem(2, 150, 3, dk, dv, gate=gate, dtype=dtype, seed=7), dtype)


@pytest.mark.parametrize("chunk", [16, 32, 64])
@pytest.mark.parametrize("gate", ["scalar", "channel"])
def test_chunk_sizes(dr, chunk, gate):
    check(dr, grads_problem(1, 100, 2, 128, 128, gate=gate, dtype="f32", seed=chunk), "f32",
          chunk=chunk)


@pytest.mark.parametrize("T", [1, 15, 63, 64, 65, 129])
def test_edge_lengths(dr, T):
    check(dr, grads_problem(1, T, 2, 128, 128, gate="channel", dtype="f32", seed=T), "f32")


def test_no_initial_state_no_final_gradient(dr):
    check(dr, grads_problem(2, 130, 2, 128, 128, gate="scalar", dtype="f32", seed=3,
                            init_state=False, d_final=False), "f32")


@pytest.mark.parametrize("gate", ["scalar", "channel"])
def test_strong_decay(dr, gate):
    """log alpha ~ -U(0, 5): every exponent the backward takes stays <= 0."""
    check(dr, grads_problem(1, 200, 2, 128, 128, gate=gate, dtype="f32", seed=9,
                            log_alpha_range=(0.0, 5.0)), "f32")


def test_zero_length_returns_final_gradient(dr):
    d = grads_problem(1, 0, 2, 64, 64, gate="scalar", dtype="f32", seed=1)
    dev = {k: (None if v is None else v.cuda()) for k, v in d.items()}
    got = dr.chunk_bwd(dev["q"], dev["k"], dev["v"], dev["log_alpha"], dev["beta"],
                       dev["init_state"], dev["d_out"], dev["d_final"])
    torch.cuda.synchronize()
    assert torch.equal(got[5].cpu(), d["d_final"])


def test_longer_sequence_bf16(dr):
    # 32 chunks: the reverse state-gradient pass carries dS through every chunk
    check(dr, grads_problem(1, 2048, 2, 128, 128, gate="scalar", dtype="bf16", seed=5), "bf16")


@pytest.mark.slow
@pytest.mark.parametrize("name,nsample", [("gdn_bf16_B8_H16_T4096_d128", 2),
                                          ("kda_bf16_B4_H32_T8192_d128", 1)])
def test_full_size_sampled_chains(dr, name, nsample):
    """The backward of the full workload, in the configuration the benchmark times; the
    oracle's reverse mode recomputes a sample of whole (b, h) chains.  bf16 inputs: every
    gradient under the bf16 rule, as in `check` (the chunk-start states come from the
    tensor-core forward, whose products round their operands to bf16)."""
    import numpy as np
    w = inputs.WORKLOADS[name]
    d = inputs.workload_inputs(w)
    g = torch.Generator().manual_seed(1)
    d_out = torch.randn((w.B, w.T, w.H, w.dv), generator=g).to(inputs.DTYPES[w.dtype])
    dev = {k: (None if v is None else v.cuda()) for k, v in d.items()}
    got = dr.chunk_bwd(dev["q"], dev["k"], dev["v"], dev["log_alpha"], dev["beta"],
                       dev["init_state"], d_out.cuda(), None, chunk=w.chunk)
    torch.cuda.synchronize()
    assert dr.device_status() == 0
    got = [None if t is None else t.cpu() for t in got]
    rng = np.random.default_rng(0)
    for c in rng.choice(w.B * w.H, size=nsample, replace=False):
        b, h = int(c) // w.H, int(c) % w.H
        pick = lambda t: None if t is None else t[b:b + 1, :, h:h + 1].contiguous()
        s0 = None if d["init_state"] is None else d["init_state"][b:b + 1, h:h + 1]
        ref = oracle.backward(pick(d["q"]), pick(d["k"]), pick(d["v"]), pick(d["log_alpha"]),
                              pick(d["beta"]), s0, pick(d_out), None)
        names = ("dq", "dk", "dv", "dlog_alpha", "dbeta")
        for name_, gt, r in zip(names, got, ref):
            if r is None:
                continue
            assert_grad(pick(gt), r, w.dtype, f"{name_} chain {(b, h)}")
        assert_grad(got[5][b:b + 1, h:h + 1], ref[5], w.dtype, f"dinit chain {(b, h)}")
