"""Error measures and tolerances of the parity tests (GPU result vs fp64 oracle).

fp32 inputs:  max |x_gpu - x_oracle| <= 1e-4 (absolute), for out and the final state.
bf16 inputs (fp32 state):  max |x_gpu - x_oracle| / RMS(x_oracle) <= 2e-2, separately for
out and the final state.

Reading for bf16-STORED results: the bound applies to the computed value; storing it in
bf16 adds a representation error of at most half a bf16 ulp of the value, which alone can
exceed 2e-2 * RMS when the outputs are heavy-tailed (max/RMS ~ 8).  So for a bf16 result
each element's deviation is first reduced by half a bf16 ulp of max(|x_gpu|, |x_oracle|)
(clamped at zero); fp32-stored results get no allowance.

Reading for the fused SiLU output gate (out = o * silu(z)): the bound is the operation's,
carried through the elementwise gate (err_gated).
"""
import numpy as np
import torch

TOL_F32_ABS = 1e-4
TOL_BF16_REL = 2e-2

# Measured errors of the full-size cases, printed at the end of the session (conftest) and
# written as JSON lines to $DR_ERROR_LOG when that is set.
ERROR_LOG = []


def record(case, what, **values):
    ERROR_LOG.append({"case": case, "what": what, **{k: float(v) for k, v in values.items()}})


def to_np(x):
    return x.detach().to("cpu", torch.float64).numpy() if isinstance(x, torch.Tensor) else x


def half_ulp_bf16(x):
    """Half the bf16 unit in the last place of |x| (bf16: 8 significant bits)."""
    _, e = np.frexp(np.abs(x))          # |x| = m 2^e, m in [0.5, 1)
    return np.ldexp(1.0, e - 9) * (x != 0) + np.ldexp(1.0, -133) * (x == 0)


def err(gpu, ref, dtype):
    """Returns (error, tolerance) under the rule for the input dtype."""
    stored_bf16 = isinstance(gpu, torch.Tensor) and gpu.dtype == torch.bfloat16
    g, r = to_np(gpu), np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    if not np.isfinite(g).all():
        return np.inf, 0.0
    if g.size == 0:
        return 0.0, (TOL_F32_ABS if dtype == "f32" else TOL_BF16_REL)
    dev = np.abs(g - r)
    if stored_bf16:
        dev = np.maximum(dev - half_ulp_bf16(np.maximum(np.abs(g), np.abs(r))), 0.0)
    if dtype == "f32":
        return dev.max(), TOL_F32_ABS
    rms = np.sqrt((r ** 2).mean())
    return dev.max() / max(rms, 1e-30), TOL_BF16_REL


def plain_err(gpu, ref):
    """max |x_gpu - x_oracle| / RMS(x_oracle) with no representation allowance."""
    g, r = to_np(gpu), np.asarray(ref, dtype=np.float64)
    if g.size == 0:
        return 0.0
    rms = np.sqrt((r ** 2).mean())
    return np.abs(g - r).max() / max(rms, 1e-30)


def assert_close(gpu, ref, dtype, what=""):
    e, tol = err(gpu, ref, dtype)
    assert e <= tol, f"{what}: error {e:.3e} > {tol:.1e}"
    return e


def err_gated(gpu, ref_ungated, gate, dtype):
    """Error of a gated output out = o * gate (gate = silu(z), fp64) against the oracle's
    ungated o.  The output gate is an elementwise scaling of the operation's result, so the
    operation's bound carries over element by element: |out_gpu - o_ref gate| <= tol *
    scale * |gate| (+ half a bf16 ulp of the stored value), scale = 1 (fp32 inputs) or
    RMS(o_ref) (bf16 inputs).  Returns (max of the scaled deviation, tolerance)."""
    stored_bf16 = isinstance(gpu, torch.Tensor) and gpu.dtype == torch.bfloat16
    g = to_np(gpu)
    o = np.asarray(ref_ungated, dtype=np.float64)
    gt = np.asarray(gate, dtype=np.float64)
    r = o * gt
    assert g.shape == r.shape, (g.shape, r.shape)
    if not np.isfinite(g).all():
        return np.inf, 0.0
    if g.size == 0:
        return 0.0, (TOL_F32_ABS if dtype == "f32" else TOL_BF16_REL)
    dev = np.abs(g - r)
    if stored_bf16:
        dev = np.maximum(dev - half_ulp_bf16(np.maximum(np.abs(g), np.abs(r))), 0.0)
    dev = dev / np.maximum(np.abs(gt), 1e-30)
    if dtype == "f32":
        return dev.max(), TOL_F32_ABS
    rms = np.sqrt((o ** 2).mean())
    return dev.max() / max(rms, 1e-30), TOL_BF16_REL


def assert_close_gated(gpu, ref_ungated, gate, dtype, what=""):
    e, tol = err_gated(gpu, ref_ungated, gate, dtype)
    assert e <= tol, f"{what}: gated error {e:.3e} > {tol:.1e}"
    return e
