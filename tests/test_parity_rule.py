"""The parity measure itself (CPU): the bf16 representation allowance is exactly half an
ulp, and it is not granted to fp32-stored results."""
import numpy as np
import torch

from parity import err, half_ulp_bf16


def test_half_ulp_matches_rounding():
    x = (torch.randn(100000) * 10).double()   # fp32 values: one rounding to bf16
    xb = x.to(torch.bfloat16).double()
    d = (xb - x).abs().numpy()
    assert (d <= half_ulp_bf16(x.numpy()) * (1 + 1e-12)).all()
    # and the bound is attained within a factor of 2 somewhere
    assert (d > 0.5 * half_ulp_bf16(x.numpy())).any()


def test_rounded_exact_result_passes_and_perturbed_fails():
    r = np.random.default_rng(0).standard_normal((64, 64)) ** 3   # heavy tails
    g = torch.from_numpy(r).to(torch.bfloat16)
    e, tol = err(g, r, "bf16")
    assert e == 0.0
    rms = np.sqrt((r ** 2).mean())
    g2 = torch.from_numpy(r + 0.05 * rms).to(torch.bfloat16)
    e2, _ = err(g2, r, "bf16")
    assert e2 > tol
    e3, _ = err(torch.from_numpy(r).float(), r, "f32")     # fp32: no allowance
    assert e3 < 1e-4


def test_nonfinite_fails():
    e, _ = err(torch.tensor([1.0, float("nan")]), np.array([1.0, 1.0]), "f32")
    assert e == np.inf


def test_gated_rule_carries_the_bound_through_the_gate():
    """A deviation within the operation's bound, scaled by the gate, passes; a wrong gate
    (sigmoid for silu) or an ungated output fails."""
    import oracle
    from parity import err_gated
    rng = np.random.default_rng(1)
    o = rng.standard_normal((32, 128))
    z = rng.standard_normal((32, 128))
    gate = oracle.silu(z)
    rms = np.sqrt((o ** 2).mean())
    # within the bound: deviation 1e-2 RMS before the gate
    g = torch.from_numpy((o + 1e-2 * rms * rng.uniform(-1, 1, o.shape)) * gate).float()
    e, tol = err_gated(g, o, gate, "bf16")
    assert e <= tol
    e, _ = err_gated(torch.from_numpy(o * oracle.sigmoid(z)).float(), o, gate, "bf16")
    assert e > tol
    e, _ = err_gated(torch.from_numpy(o).float(), o, gate, "bf16")
    assert e > tol
