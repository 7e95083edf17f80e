"""fp64 CPU oracle of the gated delta rule -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline legs of ``bench.py`` may
import this package.  The CUDA library and its Python binding never import it, and the
two share no code: the oracle is the plain token loop in ``dr_oracle.c`` (decay, predict,
write the residual, read), the recurrence

    S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T,   o_t = S_t^T q_t

as the page "NLP: linear attention summary" writes it for KDA (scalar alpha: Gated
DeltaNet, alpha = 1: DeltaNet), taken in the order of the teaching loop
``gated_delta_rule`` on the page "linear-attention gated-deltanet guide" (section 4).

Every input is first converted exactly to float64 (bf16 and fp32 values are exactly
representable), so the oracle sees the quantised values a GPU kernel sees.

Parity pins (tests/test_oracle.py) tie every function here to facts fixed by the pages
and by the mathematics; none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dr_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

GATE_NONE, GATE_SCALAR, GATE_CHANNEL = 0, 1, 2

_lib = None


def build(force: bool = False) -> str:
    """Compile ``dr_oracle.c`` with gcc into ``oracle/_build/liboracle.so``.

    fp64, ``-ffp-contract=off`` so that no multiply-add is fused on either host
    architecture.  The shared object is written to a temporary name and renamed, so
    concurrent builders never see a half-written file.
    """
    if not force and os.path.exists(_LIB_PATH) and \
            os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    os.makedirs(_BUILD_DIR, exist_ok=True)
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_BUILD_DIR)
    os.close(fd)
    cmd = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-pthread", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(cmd, check=True, capture_output=True, text=True)
        os.replace(tmp, _LIB_PATH)
    except subprocess.CalledProcessError as e:
        os.unlink(tmp)
        raise RuntimeError(f"oracle build failed:\n{e.stderr}") from e
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        dp = ctypes.POINTER(ctypes.c_double)
        i64 = ctypes.c_int64
        lib.oracle_forward.argtypes = [i64, i64, i64, i64, i64, ctypes.c_int,
                                       dp, dp, dp, dp, dp, dp, dp, dp,
                                       ctypes.c_int, i64]
        lib.oracle_forward.restype = ctypes.c_int
        lib.oracle_step.argtypes = [i64, i64, i64, i64, ctypes.c_int,
                                    dp, dp, dp, dp, dp, dp, dp, ctypes.c_int]
        lib.oracle_step.restype = ctypes.c_int
        _lib = lib
    return _lib


def to_f64(x) -> np.ndarray | None:
    """Exact conversion of a torch tensor (any float dtype, any device) or array to a
    contiguous float64 numpy array."""
    if x is None:
        return None
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return np.ascontiguousarray(x.detach().to("cpu", torch.float64).numpy())
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _gate_of(log_alpha, shape_bth, dk) -> int:
    if log_alpha is None:
        return GATE_NONE
    if tuple(log_alpha.shape) == tuple(shape_bth):
        return GATE_SCALAR
    if tuple(log_alpha.shape) == tuple(shape_bth) + (dk,):
        return GATE_CHANNEL
    raise ValueError(f"log_alpha shape {log_alpha.shape} fits neither {shape_bth} "
                     f"nor {tuple(shape_bth) + (dk,)}")


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def forward(q, k, v, log_alpha, beta, init_state=None, *, nthreads: int | None = None,
            col_block: int = 0):
    """Token-by-token fp64 forward.

    q, k [B,T,H,dk]; v [B,T,H,dv]; beta [B,T,H]; log_alpha None, [B,T,H] or [B,T,H,dk];
    init_state None or [B,H,dk,dv].  Returns (out [B,T,H,dv], final_state [B,H,dk,dv]),
    both float64 numpy arrays.
    """
    q, k, v, beta = to_f64(q), to_f64(k), to_f64(v), to_f64(beta)
    log_alpha, init_state = to_f64(log_alpha), to_f64(init_state)
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if k.shape != q.shape or v.shape[:3] != (B, T, H) or beta.shape != (B, T, H):
        raise ValueError("inconsistent shapes")
    if init_state is not None and init_state.shape != (B, H, dk, dv):
        raise ValueError("init_state must be [B,H,dk,dv]")
    gate = _gate_of(log_alpha, (B, T, H), dk)
    out = np.zeros((B, T, H, dv), dtype=np.float64)
    final = np.zeros((B, H, dk, dv), dtype=np.float64)
    rc = _load().oracle_forward(B, T, H, dk, dv, gate, _ptr(q), _ptr(k), _ptr(v),
                                _ptr(log_alpha), _ptr(beta), _ptr(init_state),
                                _ptr(out), _ptr(final),
                                nthreads or default_threads(), col_block)
    if rc != 0:
        raise RuntimeError(f"oracle_forward returned {rc}")
    return out, final


def step(q, k, v, log_alpha, beta, state, *, nthreads: int | None = None):
    """One decode step (the loop body once).

    q, k [B,H,dk]; v [B,H,dv]; beta [B,H]; log_alpha None, [B,H] or [B,H,dk];
    state [B,H,dk,dv].  Returns (out [B,H,dv], new_state [B,H,dk,dv]) as float64;
    the input state is not modified.
    """
    q, k, v, beta = to_f64(q), to_f64(k), to_f64(v), to_f64(beta)
    log_alpha = to_f64(log_alpha)
    st = to_f64(state).copy()
    B, H, dk = q.shape
    dv = v.shape[-1]
    if st.shape != (B, H, dk, dv):
        raise ValueError("state must be [B,H,dk,dv]")
    gate = _gate_of(log_alpha, (B, H), dk)
    out = np.zeros((B, H, dv), dtype=np.float64)
    rc = _load().oracle_step(B, H, dk, dv, gate, _ptr(q), _ptr(k), _ptr(v),
                             _ptr(log_alpha), _ptr(beta), _ptr(st), _ptr(out),
                             nthreads or default_threads())
    if rc != 0:
        raise RuntimeError(f"oracle_step returned {rc}")
    return out, st


# ---------------------------------------------------------------- neighbouring steps
# The steps either side of the recurrence, for the library's fused entry points: q and k
# L2-normalised per (b, t, h) vector (the workloads' recipe normalises them), beta taken as
# the sigmoid of logits, and the output gate of the page "linear-attention gated-deltanet
# guide" (section 4: a gate with a SiLU activation on what is read out), out = o * silu(z).
# The pages print no epsilon for the normalisation; the reading is x / sqrt(|x|^2 + eps)
# with eps = 1e-6.  Nor do they fix the precision of beta: the reading is that the sigmoid
# is stored in beta's own dtype, as a beta computed before the call would be (for bf16
# logits, the sigmoid rounded to nearest-even bf16).
L2NORM_EPS = 1e-6


def round_bf16(x) -> np.ndarray:
    """float64 values rounded to the nearest bfloat16 (8 significant bits), ties to even,
    for normal bf16 magnitudes (|x| >= 2^-126) and zero."""
    x = to_f64(x)
    m, e = np.frexp(x)                  # x = m 2^e, 0.5 <= |m| < 1
    return np.ldexp(np.round(m * 256.0) / 256.0, e)   # np.round: half to even


def _is_bf16(x) -> bool:
    try:
        import torch
        return isinstance(x, torch.Tensor) and x.dtype == torch.bfloat16
    except ImportError:
        return False


def l2_normalize(x) -> np.ndarray:
    """x / sqrt(|x|^2 + L2NORM_EPS) along the last axis, in float64."""
    x = to_f64(x)
    return x / np.sqrt((x * x).sum(axis=-1, keepdims=True) + L2NORM_EPS)


def sigmoid(x) -> np.ndarray:
    """1 / (1 + exp(-x)) in float64, without overflow for large |x|."""
    x = to_f64(x)
    e = np.exp(-np.abs(x))
    return np.where(x >= 0, 1.0 / (1.0 + e), e / (1.0 + e))


def silu(x) -> np.ndarray:
    """x * sigmoid(x) in float64."""
    x = to_f64(x)
    return x * sigmoid(x)


def forward_fused(q, k, v, log_alpha, beta, init_state=None, *, qk_l2norm=False,
                  beta_sigmoid=False, z=None, **kw):
    """``forward`` with the neighbouring steps: q, k normalised first (qk_l2norm), beta
    given as logits (beta_sigmoid; the sigmoid stored in the logits' dtype), and the output
    multiplied by silu(z) (z given, in the output's layout).  The final state is that of
    ``forward`` on the prepared inputs."""
    bf16_beta = _is_bf16(beta)
    q, k, beta = to_f64(q), to_f64(k), to_f64(beta)
    if qk_l2norm:
        q, k = l2_normalize(q), l2_normalize(k)
    if beta_sigmoid:
        beta = round_bf16(sigmoid(beta)) if bf16_beta else sigmoid(beta)
    out, final = forward(q, k, v, log_alpha, beta, init_state, **kw)
    if z is not None:
        out = out * silu(to_f64(z))
    return out, final


def step_fused(q, k, v, log_alpha, beta, state, *, qk_l2norm=False, beta_sigmoid=False,
               z=None, **kw):
    """``step`` with the same neighbouring steps as ``forward_fused``."""
    bf16_beta = _is_bf16(beta)
    q, k, beta = to_f64(q), to_f64(k), to_f64(beta)
    if qk_l2norm:
        q, k = l2_normalize(q), l2_normalize(k)
    if beta_sigmoid:
        beta = round_bf16(sigmoid(beta)) if bf16_beta else sigmoid(beta)
    out, st = step(q, k, v, log_alpha, beta, state, **kw)
    if z is not None:
        out = out * silu(to_f64(z))
    return out, st


# ---------------------------------------------------------------- backward
# Reverse mode of the token loop of ``forward`` (the recurrence of the page "NLP: linear
# attention summary", KDA section, in the order of the `gated_delta_rule` loop of the page
# "linear-attention gated-deltanet guide", section 4): with the loss
#     L = sum(d_out * out) + sum(d_final * final_state),
# the step S' = Diag(a_t) S_{t-1}, p = S'^T k_t, e = beta_t (v_t - p), S_t = S' + k_t e^T,
# o_t = S_t^T q_t is differentiated line by line, last token first.  States are recomputed
# from checkpoints every `block` tokens.  Pinned by central differences of ``forward``.
def backward(q, k, v, log_alpha, beta, init_state, d_out, d_final=None, *, block: int = 64):
    """Gradients of L with respect to every input, in float64:
    (dq [B,T,H,dk], dk [B,T,H,dk], dv [B,T,H,dv], dlog_alpha (shape of log_alpha, or None),
    dbeta [B,T,H], dinit [B,H,dk,dv])."""
    q, k, v, beta = to_f64(q), to_f64(k), to_f64(v), to_f64(beta)
    la, s0, do = to_f64(log_alpha), to_f64(init_state), to_f64(d_out)
    dfin = to_f64(d_final)
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    gate = _gate_of(la, (B, T, H), dk)
    # [B,H,T,...] views; a = alpha per key channel
    qt, kt, vt, dot = (np.moveaxis(x, 2, 1) for x in (q, k, v, do))
    bt = np.moveaxis(beta, 2, 1)
    if gate == GATE_NONE:
        a = np.ones((B, H, T, dk))
    elif gate == GATE_SCALAR:
        a = np.repeat(np.exp(np.moveaxis(la, 2, 1))[..., None], dk, axis=-1)
    else:
        a = np.exp(np.moveaxis(la, 2, 1))

    def step_fwd(S, t):
        Sd = a[:, :, t, :, None] * S
        p = np.einsum("bhij,bhi->bhj", Sd, kt[:, :, t])
        e = bt[:, :, t, None] * (vt[:, :, t] - p)
        return Sd, p, e, Sd + kt[:, :, t, :, None] * e[:, :, None, :]

    S = np.zeros((B, H, dk, dv)) if s0 is None else s0.copy()
    ckpt = {}
    for t in range(T):
        if t % block == 0:
            ckpt[t] = S.copy()
        S = step_fwd(S, t)[3]
    dS = np.zeros((B, H, dk, dv)) if dfin is None else dfin.copy()
    gq, gk, gv = np.zeros_like(qt), np.zeros_like(kt), np.zeros_like(vt)
    gb = np.zeros_like(bt)
    gla = np.zeros((B, H, T, dk))      # d log alpha per key channel
    for t0 in reversed(range(0, T, block)):
        t1 = min(T, t0 + block)
        prev = [ckpt[t0]]               # state before each step of the block
        for t in range(t0, t1 - 1):
            prev.append(step_fwd(prev[-1], t)[3])
        for t in reversed(range(t0, t1)):
            Sd, p, e, St = step_fwd(prev[t - t0], t)
            dS = dS + qt[:, :, t, :, None] * dot[:, :, t, None, :]        # o_t = S_t^T q_t
            gq[:, :, t] = np.einsum("bhij,bhj->bhi", St, dot[:, :, t])
            de = np.einsum("bhij,bhi->bhj", dS, kt[:, :, t])          # through S_t = S' + k e^T
            gk[:, :, t] = np.einsum("bhij,bhj->bhi", dS, e)
            dSd = dS.copy()
            gv[:, :, t] = bt[:, :, t, None] * de                       # e = beta (v - p)
            gb[:, :, t] = (de * (vt[:, :, t] - p)).sum(-1)
            dp = -bt[:, :, t, None] * de
            dSd = dSd + kt[:, :, t, :, None] * dp[:, :, None, :]       # p = S'^T k
            gk[:, :, t] += np.einsum("bhij,bhj->bhi", Sd, dp)
            gla[:, :, t] = (dSd * Sd).sum(-1)                          # S' = Diag(a) S
            dS = a[:, :, t, :, None] * dSd
    back = lambda x: np.ascontiguousarray(np.moveaxis(x, 1, 2))
    if gate == GATE_NONE:
        dla = None
    elif gate == GATE_SCALAR:
        dla = back(gla.sum(-1))
    else:
        dla = back(gla)
    return back(gq), back(gk), back(gv), dla, back(gb), dS
