"""Pins of the fp64 oracle to facts the pages and the mathematics fix (CPU only).

Each pin is a function of an implementation ``impl(q, k, v, log_alpha, beta, s0) ->
(out, final_state)`` (float64, shapes as in ``oracle.forward``).  The oracle must pass all
of them; deliberately broken token loops (planted mistakes, below) must each fail at least
one, which shows the pins are sensitive to the mistakes a loop like this can make.

Sources (page titles and sections):
  P1 = "NLP: linear attention summary": DeltaNet gradient-step equation, orthogonal-key
       capacity argument (linear attention, core limits), Gated DeltaNet equation, KDA
       equation and its unrolled product form (KDA design principle 3).
  P4 = "linear-attention gated-deltanet guide", section 4: order decay -> predict ->
       write -> read.
"""
from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.default_rng(12345)


# ---------------------------------------------------------------- helpers
def rand_problem(B, T, H, dk, dv, gate, *, unit=True, init=True, beta=None,
                 la_range=(0.0, 0.7), rng=RNG):
    q = rng.standard_normal((B, T, H, dk))
    k = rng.standard_normal((B, T, H, dk))
    if unit:
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, H, dv))
    b = rng.uniform(0, 1, (B, T, H)) if beta is None else np.full((B, T, H), beta, float)
    if gate == "none":
        la = None
    elif gate == "scalar":
        la = -rng.uniform(*la_range, (B, T, H))
    else:
        la = -rng.uniform(*la_range, (B, T, H, dk))
    s0 = rng.standard_normal((B, H, dk, dv)) * 0.3 if init else None
    return q, k, v, la, b, s0


def oracle_impl(q, k, v, la, b, s0):
    return oracle.forward(q, k, v, la, b, s0, nthreads=3, col_block=3)


def decay_vec(la, b, t, h, dk):
    """alpha_t as a d_k vector (1 without a gate)."""
    if la is None:
        return np.ones(dk)
    x = la[b, t, h]
    return np.exp(np.full(dk, x) if np.ndim(x) == 0 else x)


# ---------------------------------------------------------------- pins
def pin_a_zero_write(impl):
    """alpha = 1, beta = 0, S_0 = 0  =>  o = 0 and S_T = 0 exactly (P1 DeltaNet equation
    with beta = 0: nothing is ever written)."""
    q, k, v, _, _, _ = rand_problem(2, 9, 2, 5, 4, "none", init=False, beta=0.0)
    b = np.zeros(q.shape[:3])
    out, fin = impl(q, k, v, None, b, None)
    return max(np.abs(out).max(), np.abs(fin).max())


def pin_b_orthonormal_retrieval(impl):
    """alpha = 1, beta = 1, orthonormal keys k_1..k_T (T <= d_k), S_0 = 0  =>
    S_T^T k_j = v_j for every j (P1: retrieval without crosstalk needs orthogonal keys;
    the delta rule with beta = 1 overwrites exactly the slot of k_t)."""
    dk, dv, T = 8, 5, 7
    Qm, _ = np.linalg.qr(RNG.standard_normal((dk, dk)))
    k = Qm[:, :T].T.reshape(1, T, 1, dk)
    q = RNG.standard_normal((1, T, 1, dk))
    v = RNG.standard_normal((1, T, 1, dv))
    out, fin = impl(q, k, v, None, np.ones((1, T, 1)), None)
    S = fin[0, 0]
    return max(np.abs(S.T @ k[0, j, 0] - v[0, j, 0]).max() for j in range(T))


def pin_b2_exact_write(impl):
    """beta_t = 1 and |k_t| = 1  =>  right after step t, S_t^T k_t = v_t whatever the gate
    and the earlier state.  Read out through o_t with q_t = k_t (o_t = S_t^T q_t, read
    after the write)."""
    worst = 0.0
    for gate in ("none", "scalar", "channel"):
        q, k, v, la, _, s0 = rand_problem(2, 11, 2, 6, 5, gate, beta=1.0)
        b = np.ones(k.shape[:3])
        out, _ = impl(k.copy(), k, v, la, b, s0)
        worst = max(worst, np.abs(out - v).max())
    return worst


def closed_form(q, k, v, la, b, s0):
    """Unrolled product form, P1 KDA design principle 3, with the reading that fits the
    recurrence: M_j = (I - beta_j k_j k_j^T) Diag(alpha_j) and the write of token i is
    beta_i k_i v_i^T.  S_t = M_t..M_1 S_0 + sum_i M_t..M_{i+1} beta_i k_i v_i^T.  Every
    product of transition matrices is formed from scratch, densely."""
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    out = np.zeros((B, T, H, dv))
    fin = np.zeros((B, H, dk, dv))
    for bb in range(B):
        for h in range(H):
            M = [(np.eye(dk) - b[bb, j, h] * np.outer(k[bb, j, h], k[bb, j, h]))
                 @ np.diag(decay_vec(la, bb, j, h, dk)) for j in range(T)]

            def prod(hi, lo):   # M_hi M_{hi-1} ... M_lo  (identity if hi < lo)
                P = np.eye(dk)
                for j in range(lo, hi + 1):
                    P = M[j] @ P
                return P

            S0 = np.zeros((dk, dv)) if s0 is None else s0[bb, h]
            for t in range(T):
                St = prod(t, 0) @ S0
                for i in range(t + 1):
                    St = St + prod(t, i + 1) @ np.outer(b[bb, i, h] * k[bb, i, h],
                                                        v[bb, i, h])
                out[bb, t, h] = St.T @ q[bb, t, h]
                if t == T - 1:
                    fin[bb, h] = St
    return out, fin


def pin_c_closed_form(impl):
    """The unrolled product-of-matrices form equals the result for T <= 16, all gates."""
    worst = 0.0
    for gate in ("none", "scalar", "channel"):
        prob = rand_problem(2, 7, 2, 5, 4, gate)
        o1, f1 = impl(*prob)
        o2, f2 = closed_form(*prob)
        worst = max(worst, np.abs(o1 - o2).max(), np.abs(f1 - f2).max())
    return worst


def pin_d_gradient_step(impl):
    """One step equals one gradient step of lr beta_t on L(S) = 1/2 |S^T k_t - v_t|^2,
    taken at the decayed state Diag(alpha_t) S_{t-1} (P1 DeltaNet equation; P4 decays
    first).  The gradient is taken by central differences, which are exact for a
    quadratic up to rounding."""
    worst = 0.0
    for gate in ("none", "scalar", "channel"):
        q, k, v, la, b, s0 = rand_problem(1, 1, 1, 6, 4, gate)
        out, fin = impl(q, k, v, la, b, s0)
        kt, vt = k[0, 0, 0], v[0, 0, 0]
        Sd = np.diag(decay_vec(la, 0, 0, 0, 6)) @ s0[0, 0]

        def L(S):
            r = S.T @ kt - vt
            return 0.5 * float(r @ r)

        G = np.zeros_like(Sd)
        h = 1e-3
        for i in range(Sd.shape[0]):
            for j in range(Sd.shape[1]):
                E = np.zeros_like(Sd)
                E[i, j] = h
                G[i, j] = (L(Sd + E) - L(Sd - E)) / (2 * h)
        S_new = Sd - b[0, 0, 0] * G
        worst = max(worst, np.abs(fin[0, 0] - S_new).max(),
                    np.abs(out[0, 0, 0] - S_new.T @ q[0, 0, 0]).max())
    return worst


def pin_e_pure_decay(impl):
    """beta = 0  =>  S_t = Diag(prod_{u<=t} alpha_u) S_0 and o_t = S_t^T q_t (P1 KDA /
    Gated DeltaNet equations with the write switched off)."""
    worst = 0.0
    for gate in ("scalar", "channel"):
        q, k, v, la, _, s0 = rand_problem(2, 8, 3, 5, 4, gate, beta=0.0)
        b = np.zeros(q.shape[:3])
        out, fin = impl(q, k, v, la, b, s0)
        B, T, H, dk = q.shape
        for bb in range(B):
            for h in range(H):
                cum = np.zeros(dk)
                for t in range(T):
                    cum = cum + np.log(decay_vec(la, bb, t, h, dk))
                    St = np.exp(cum)[:, None] * s0[bb, h]
                    worst = max(worst, np.abs(out[bb, t, h] - St.T @ q[bb, t, h]).max())
                worst = max(worst, np.abs(fin[bb, h] - St).max())
    return worst


def pin_f_channel_equals_scalar(impl):
    """A per-channel gate whose d_k entries all equal the scalar gate gives the scalar
    result (P1: KDA generalises the Gated DeltaNet scalar to Diag(alpha_t))."""
    q, k, v, la, b, s0 = rand_problem(2, 10, 2, 6, 5, "scalar")
    o1, f1 = impl(q, k, v, la, b, s0)
    la_c = np.repeat(la[..., None], 6, axis=-1)
    o2, f2 = impl(q, k, v, la_c, b, s0)
    return max(np.abs(o1 - o2).max(), np.abs(f1 - f2).max())


def pin_h_carry_over(impl):
    """run(T1) then run(T2, init = its final state) equals run(T1 + T2)."""
    worst = 0.0
    for gate in ("none", "scalar", "channel"):
        q, k, v, la, b, s0 = rand_problem(2, 12, 2, 5, 6, gate)
        o, f = impl(q, k, v, la, b, s0)
        sl = lambda x, a, z: None if x is None else x[:, a:z]
        o1, f1 = impl(q[:, :5], k[:, :5], v[:, :5], sl(la, 0, 5), b[:, :5], s0)
        o2, f2 = impl(q[:, 5:], k[:, 5:], v[:, 5:], sl(la, 5, 12), b[:, 5:], f1)
        worst = max(worst, np.abs(np.concatenate([o1, o2], 1) - o).max(),
                    np.abs(f2 - f).max())
    return worst


PINS = {
    "a_zero_write": (pin_a_zero_write, 0.0),
    "b_orthonormal_retrieval": (pin_b_orthonormal_retrieval, 1e-12),
    "b2_exact_write": (pin_b2_exact_write, 1e-12),
    "c_closed_form": (pin_c_closed_form, 1e-12),
    "d_gradient_step": (pin_d_gradient_step, 1e-9),
    "e_pure_decay": (pin_e_pure_decay, 1e-12),
    "f_channel_equals_scalar": (pin_f_channel_equals_scalar, 0.0),
    "h_carry_over": (pin_h_carry_over, 0.0),
}


@pytest.mark.parametrize("name", sorted(PINS))
def test_oracle_pin(name):
    fn, tol = PINS[name]
    err = fn(oracle_impl)
    assert err <= tol, f"pin {name}: error {err} > {tol}"


# ---------------------------------------------------------------- worked example
def _parse_golden(path):
    rows = {}
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, val = line.split(":", 1)
            rows[key.strip()] = [[Fraction(x) for x in tok.split()]
                                 for tok in val.split("|")]
    return rows


def test_worked_example_by_hand():
    """The oracle reproduces the hand-derived d = 2, T = 3 example (tests/golden)."""
    g = _parse_golden(os.path.join(GOLDEN, "worked_example_d2_T3.txt"))
    T = len(g["k"])
    f = lambda key: np.array([[float(x) for x in r] for r in g[key]])
    k = f("k").reshape(1, T, 1, 2)
    v = f("v").reshape(1, T, 1, 2)
    q = f("q").reshape(1, T, 1, 2)
    b = f("beta").reshape(1, T, 1)
    la = np.log(f("alpha")).reshape(1, T, 1)
    out, fin = oracle.forward(q, k, v, la, b, None, nthreads=1)
    assert np.abs(out.reshape(T, 2) - f("out")).max() < 1e-15
    assert np.abs(fin.reshape(2, 2) - f("final_state")).max() < 1e-15


def test_exact_rational_matrix_form():
    """Random rational inputs: the oracle agrees with the page's matrix-form updates
    (erase matrix times the decayed state plus the write), evaluated exactly in rationals,
    for DeltaNet, Gated DeltaNet and KDA gates.  Gates are powers of 1/2 so that
    exp(log alpha) is exact in fp64."""
    rng = np.random.default_rng(7)
    dk, dv, T = 3, 2, 6
    for gate in ("none", "scalar", "channel"):
        Fr = lambda: Fraction(int(rng.integers(-8, 9)), int(rng.integers(1, 6)))
        k = [[Fr() for _ in range(dk)] for _ in range(T)]
        v = [[Fr() for _ in range(dv)] for _ in range(T)]
        q = [[Fr() for _ in range(dk)] for _ in range(T)]
        beta = [Fraction(int(rng.integers(0, 5)), 4) for _ in range(T)]
        if gate == "none":
            alpha = [[Fraction(1)] * dk for _ in range(T)]
        elif gate == "scalar":
            alpha = [[Fraction(1, 2 ** int(rng.integers(0, 3)))] * dk for _ in range(T)]
        else:
            alpha = [[Fraction(1, 2 ** int(rng.integers(0, 3))) for _ in range(dk)]
                     for _ in range(T)]
        S = [[Fraction(0)] * dv for _ in range(dk)]
        outs = []
        for t in range(T):
            # (I - beta k k^T) Diag(alpha) S + beta k v^T, element by element
            D = [[alpha[t][i] * S[i][j] for j in range(dv)] for i in range(dk)]
            E = [[(1 if i == m else 0) - beta[t] * k[t][i] * k[t][m] for m in range(dk)]
                 for i in range(dk)]
            S = [[sum(E[i][m] * D[m][j] for m in range(dk)) + beta[t] * k[t][i] * v[t][j]
                  for j in range(dv)] for i in range(dk)]
            outs.append([sum(S[i][j] * q[t][i] for i in range(dk)) for j in range(dv)])
        arr = lambda x: np.array([[float(y) for y in r] for r in x])
        qa, ka, va = (arr(x).reshape(1, T, 1, -1) for x in (q, k, v))
        ba = np.array([float(x) for x in beta]).reshape(1, T, 1)
        al = np.array([[math.log(float(x)) for x in r] for r in alpha])
        la = None if gate == "none" else (al[:, 0].reshape(1, T, 1) if gate == "scalar"
                                          else al.reshape(1, T, 1, dk))
        out, fin = oracle.forward(qa, ka, va, la, ba, None, nthreads=1)
        ref_o, ref_s = arr(outs), arr(S)
        scale = max(1.0, np.abs(ref_o).max(), np.abs(ref_s).max())
        assert np.abs(out.reshape(T, dv) - ref_o).max() <= 1e-13 * scale
        assert np.abs(fin.reshape(dk, dv) - ref_s).max() <= 1e-13 * scale


# ---------------------------------------------------------------- decode oracle
def test_step_matches_one_token_forward():
    """The decode oracle is the loop body once: a step from state S equals the forward
    over one token with init S, and 16 steps equal the forward over those 16 tokens."""
    for gate in ("none", "scalar", "channel"):
        q, k, v, la, b, s0 = rand_problem(3, 16, 2, 6, 5, gate)
        o_ref, f_ref = oracle.forward(q, k, v, la, b, s0)
        st = s0.copy()
        for t in range(16):
            o, st = oracle.step(q[:, t], k[:, t], v[:, t],
                                None if la is None else la[:, t], b[:, t], st)
            assert np.array_equal(o, o_ref[:, t])
        assert np.array_equal(st, f_ref)


def test_step_gradient_identity():
    """Pin (d) through the decode entry: new state = decayed state - beta * grad."""
    q, k, v, la, b, s0 = rand_problem(1, 1, 1, 6, 4, "channel")
    _, st = oracle.step(q[:, 0], k[:, 0], v[:, 0], la[:, 0], b[:, 0], s0)
    Sd = np.exp(la[0, 0, 0])[:, None] * s0[0, 0]
    kt, vt = k[0, 0, 0], v[0, 0, 0]
    grad = np.outer(kt, Sd.T @ kt - vt)   # d/dS of 1/2|S^T k - v|^2, by hand
    assert np.abs(st[0, 0] - (Sd - b[0, 0, 0] * grad)).max() < 1e-13


def test_threading_and_blocking_do_not_change_bits():
    """Task split over chains and state-column blocks leaves every result bit-identical
    (each column follows the same loop)."""
    prob = rand_problem(2, 20, 3, 7, 9, "channel")
    o1, f1 = oracle.forward(*prob, nthreads=1, col_block=0)
    o2, f2 = oracle.forward(*prob, nthreads=5, col_block=2)
    assert np.array_equal(o1, o2) and np.array_equal(f1, f2)


def test_final_state_may_alias_init():
    """The C entry allows final_state == init_state (in-place carry)."""
    q, k, v, la, b, s0 = rand_problem(1, 1, 2, 4, 4, "scalar")
    o1, f1 = oracle.forward(q, k, v, la, b, s0)
    st = s0.copy()
    o2, st2 = oracle.step(q[:, 0], k[:, 0], v[:, 0], la[:, 0], b[:, 0], st)
    assert np.array_equal(st2, f1) and np.array_equal(o2, o1[:, 0])


def test_bf16_inputs_convert_exactly():
    import torch
    x = torch.randn(1000).to(torch.bfloat16)
    y = oracle.to_f64(x)
    assert np.array_equal(y.astype(np.float32), x.float().numpy())
    assert np.array_equal(torch.from_numpy(y).to(torch.bfloat16).float().numpy(),
                          x.float().numpy())


# ---------------------------------------------------------------- planted mistakes
def _loop(q, k, v, la, b, s0, mistake):
    """Token loop with one planted mistake (test-only; never used as a reference)."""
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    out = np.zeros((B, T, H, dv))
    fin = np.zeros((B, H, dk, dv))
    for bb in range(B):
        for h in range(H):
            S = np.zeros((dk, dv)) if s0 is None else s0[bb, h].copy()
            for t in range(T):
                a = decay_vec(la, bb, t, h, dk)
                kt, vt, qt, bt = k[bb, t, h], v[bb, t, h], q[bb, t, h], b[bb, t, h]
                S_prev = S
                if mistake == "decay_after_write":
                    S = S + bt * np.outer(kt, vt - S.T @ kt)
                    S = a[:, None] * S
                elif mistake == "no_decay":
                    S = S + bt * np.outer(kt, vt - S.T @ kt)
                elif mistake == "beta_only_on_write":
                    S = a[:, None] * S
                    S = S - np.outer(kt, S.T @ kt) + bt * np.outer(kt, vt)
                elif mistake == "sign":
                    S = a[:, None] * S
                    S = S + bt * np.outer(kt, vt + S.T @ kt)
                elif mistake == "gate_on_columns":
                    S = S * a[None, :dv] if dk == dv else S
                    S = S + bt * np.outer(kt, vt - S.T @ kt)
                elif mistake == "predict_with_undecayed":
                    p = S.T @ kt
                    S = a[:, None] * S
                    S = S + bt * np.outer(kt, vt - p)
                else:
                    S = a[:, None] * S
                    S = S + bt * np.outer(kt, vt - S.T @ kt)
                if mistake == "read_before_write":
                    out[bb, t, h] = (a[:, None] * S_prev).T @ qt
                elif mistake == "transposed_read":
                    out[bb, t, h] = S @ qt
                else:
                    out[bb, t, h] = S.T @ qt
            fin[bb, h] = S
    return out, fin


MISTAKES = ["decay_after_write", "no_decay", "beta_only_on_write", "sign",
            "read_before_write", "transposed_read", "predict_with_undecayed"]


def _square_pins():
    """Pins rerun with d_k = d_v so that transposition mistakes type-check."""
    def c_square(impl):
        worst = 0.0
        for gate in ("scalar", "channel"):
            prob = rand_problem(1, 6, 1, 5, 5, gate)
            o1, f1 = impl(*prob)
            o2, f2 = closed_form(*prob)
            worst = max(worst, np.abs(o1 - o2).max(), np.abs(f1 - f2).max())
        return worst
    return {"c_square": (c_square, 1e-12)}


def test_loop_without_mistake_passes_pins():
    impl = lambda *a: _loop(*a, mistake=None)
    for name, (fn, tol) in {**PINS, **_square_pins()}.items():
        assert fn(impl) <= max(tol, 1e-12), name


@pytest.mark.parametrize("mistake", MISTAKES)
def test_planted_mistake_is_caught(mistake):
    impl = lambda *a: _loop(*a, mistake=mistake)
    failed = []
    for name, (fn, tol) in {**PINS, **_square_pins()}.items():
        try:
            err = fn(impl)
        except ValueError:
            err = math.inf
        if not err <= max(tol, 1e-12):
            failed.append(name)
    assert failed, f"no pin caught the planted mistake {mistake}"


# ------------------------------------------------------------ neighbouring steps
# Pins of the fused entry points' reference: each ties one neighbouring step to a fact
# that does not restate its formula.
def _raw_problem(seed, gate="scalar", T=20):
    rng = np.random.default_rng(seed)
    B, H, dk, dv = 1, 2, 8, 6
    q = rng.standard_normal((B, T, H, dk))
    k = rng.standard_normal((B, T, H, dk))
    v = rng.standard_normal((B, T, H, dv))
    b = rng.standard_normal((B, T, H))
    la = -rng.uniform(0.0, 0.3, (B, T, H) if gate == "scalar" else (B, T, H, dk))
    s0 = rng.standard_normal((B, H, dk, dv)) * 0.1
    z = rng.standard_normal((B, T, H, dv))
    return q, k, v, la, b, s0, z


@pytest.mark.parametrize("gate", ["scalar", "channel"])
def test_l2norm_scale_invariance(gate):
    """Normalised keys and queries do not depend on the scale of the raw vectors (up to the
    epsilon's relative effect, eps / (2 |x|^2) < 1e-6 here; a missing normalisation would
    move the results by O(1))."""
    q, k, v, la, b, s0, _ = _raw_problem(1, gate)
    rng = np.random.default_rng(2)
    cq = rng.uniform(0.5, 4.0, q.shape[:3] + (1,))
    ck = rng.uniform(0.5, 4.0, k.shape[:3] + (1,))
    o1, f1 = oracle.forward_fused(q, k, v, la, oracle.sigmoid(b), s0, qk_l2norm=True)
    o2, f2 = oracle.forward_fused(q * cq, k * ck, v, la, oracle.sigmoid(b), s0, qk_l2norm=True)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-5)
    np.testing.assert_allclose(f1, f2, rtol=0, atol=1e-5)


def test_l2norm_leaves_unit_vectors():
    """Unit vectors are (up to eps) left alone: normalised inputs give the plain forward."""
    q, k, v, la, b, s0, _ = _raw_problem(3)
    qu = q / np.linalg.norm(q, axis=-1, keepdims=True)
    ku = k / np.linalg.norm(k, axis=-1, keepdims=True)
    bb = oracle.sigmoid(b)
    o1, f1 = oracle.forward_fused(qu, ku, v, la, bb, s0, qk_l2norm=True)
    o2, f2 = oracle.forward(qu, ku, v, la, bb, s0)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-5)
    np.testing.assert_allclose(f1, f2, rtol=0, atol=1e-5)


def test_beta_logits_limits():
    """Logits of -40, 0, +40 act as beta = 0, 1/2, 1 (no write, half write, full write)."""
    q, k, v, la, _, s0, _ = _raw_problem(4)
    for logit, beta in [(-40.0, 0.0), (0.0, 0.5), (40.0, 1.0)]:
        bl = np.full(q.shape[:3], logit)
        o1, f1 = oracle.forward_fused(q, k, v, la, bl, s0, beta_sigmoid=True)
        o2, f2 = oracle.forward(q, k, v, la, np.full(q.shape[:3], beta), s0)
        np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
        np.testing.assert_allclose(f1, f2, rtol=0, atol=1e-12)


def test_output_gate_identities():
    """z = 0 closes the gate exactly; out(z) - out(-z) = o * z (an odd-part identity of
    x * sigmoid(x)); a large z passes o * z; the state is never gated."""
    q, k, v, la, b, s0, z = _raw_problem(5)
    bb = oracle.sigmoid(b)
    o, f = oracle.forward(q, k, v, la, bb, s0)
    o0, f0 = oracle.forward_fused(q, k, v, la, bb, s0, z=np.zeros_like(z))
    assert np.all(o0 == 0.0) and np.array_equal(f0, f)
    op, _ = oracle.forward_fused(q, k, v, la, bb, s0, z=z)
    om, _ = oracle.forward_fused(q, k, v, la, bb, s0, z=-z)
    np.testing.assert_allclose(op - om, o * z, rtol=0, atol=1e-12)
    ob, _ = oracle.forward_fused(q, k, v, la, bb, s0, z=np.full_like(z, 40.0))
    np.testing.assert_allclose(ob, o * 40.0, rtol=1e-12, atol=1e-12)


def test_step_fused_is_one_token_forward_fused():
    q, k, v, la, b, s0, z = _raw_problem(6, "channel", T=1)
    o1, f1 = oracle.forward_fused(q, k, v, la, b, s0, qk_l2norm=True, beta_sigmoid=True, z=z)
    o2, f2 = oracle.step_fused(q[:, 0], k[:, 0], v[:, 0], la[:, 0], b[:, 0], s0,
                               qk_l2norm=True, beta_sigmoid=True, z=z[:, 0])
    np.testing.assert_allclose(o1[:, 0], o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(f1, f2, rtol=0, atol=1e-13)


def _fused_with_mistake(mistake):
    """A copy of oracle.forward_fused with one plausible mistake planted."""
    def f(q, k, v, la, b, s0, *, qk_l2norm=False, beta_sigmoid=False, z=None):
        q, k, b = oracle.to_f64(q), oracle.to_f64(k), oracle.to_f64(b)
        if qk_l2norm:
            q = oracle.l2_normalize(q)
            if mistake != "normalise_q_only":
                k = oracle.l2_normalize(k)
        if beta_sigmoid:
            b = oracle.sigmoid(-b) if mistake == "sigmoid_sign" else oracle.sigmoid(b)
        out, fin = oracle.forward(q, k, v, la, b, s0)
        if z is not None:
            out = out * (oracle.sigmoid(z) if mistake == "gate_sigmoid" else oracle.silu(z))
        return out, fin
    return f


@pytest.mark.parametrize("mistake", ["normalise_q_only", "sigmoid_sign", "gate_sigmoid"])
def test_fused_pins_catch_planted_mistake(mistake, monkeypatch):
    monkeypatch.setattr(oracle, "forward_fused", _fused_with_mistake(mistake))
    pins = [lambda: test_l2norm_scale_invariance("scalar"), test_beta_logits_limits,
            test_output_gate_identities]
    failed = 0
    for pin in pins:
        try:
            pin()
        except AssertionError:
            failed += 1
    assert failed >= 1, f"no pin caught {mistake}"


def test_round_bf16_matches_torch_on_fp32_values():
    """On fp32 values (no double rounding) the oracle's bf16 rounding is torch's cast."""
    import torch
    x = (torch.randn(200000) * torch.exp(torch.randn(200000) * 5)).float()
    x = torch.cat([x, torch.tensor([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8)])])
    ref = x.to(torch.bfloat16).double().numpy()
    assert np.array_equal(oracle.round_bf16(x.double().numpy()), ref)


def test_sigmoid_of_bf16_logits_is_stored_in_bf16():
    """Reading: a beta computed from bf16 logits is the bf16-stored sigmoid (ties to even),
    and that rounding changes the result (it is not a no-op)."""
    import torch
    q, k, v, la, b, s0, _ = _raw_problem(5, "scalar")
    qn, kn = oracle.l2_normalize(q), oracle.l2_normalize(k)
    bl = torch.from_numpy(b).to(torch.bfloat16)
    o1, f1 = oracle.forward_fused(qn, kn, v, la, bl, s0, beta_sigmoid=True)
    br = oracle.round_bf16(oracle.sigmoid(bl))
    o2, f2 = oracle.forward(qn, kn, v, la, br, s0)
    assert np.array_equal(o1, o2) and np.array_equal(f1, f2)
    o3, _ = oracle.forward(qn, kn, v, la, oracle.sigmoid(bl), s0)
    assert np.abs(o3 - o1).max() > 1e-6
    # fp32 / fp64 logits keep the unrounded sigmoid
    o4, _ = oracle.forward_fused(qn, kn, v, la, b, s0, beta_sigmoid=True)
    o5, _ = oracle.forward(qn, kn, v, la, oracle.sigmoid(b), s0)
    assert np.array_equal(o4, o5)


def _bwd_problem(seed, gate, B=1, T=7, H=2, dk=5, dv=4):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, T, H, dk))
    k = rng.standard_normal((B, T, H, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, H, dv))
    b = rng.uniform(0.1, 0.9, (B, T, H))
    la = None if gate == "none" else -rng.uniform(0.0, 0.5, (B, T, H) if gate == "scalar"
                                                  else (B, T, H, dk))
    s0 = rng.standard_normal((B, H, dk, dv)) * 0.3
    do = rng.standard_normal((B, T, H, dv))
    dfin = rng.standard_normal((B, H, dk, dv))
    return q, k, v, la, b, s0, do, dfin


@pytest.mark.parametrize("gate", ["none", "scalar", "channel"])
def test_backward_matches_central_differences(gate):
    """Every gradient of L = <d_out, out> + <d_final, final> equals the central difference
    of the (pinned) forward, element by element, on a tiny problem."""
    q, k, v, la, b, s0, do, dfin = _bwd_problem(3, gate)
    grads = oracle.backward(q, k, v, la, b, s0, do, dfin)
    names = ["q", "k", "v", "la", "b", "s0"]
    args = [q, k, v, la, b, s0]

    def loss(a):
        o, f = oracle.forward(*a)
        return float((do * o).sum() + (dfin * f).sum())

    h = 1e-6
    for idx, (name, x, g) in enumerate(zip(names, args, grads)):
        if x is None:
            assert g is None
            continue
        assert g.shape == x.shape, name
        fd = np.zeros_like(x)
        for e in range(x.size):
            xp, xm = x.copy(), x.copy()
            xp.flat[e] += h
            xm.flat[e] -= h
            ap, am = list(args), list(args)
            ap[idx], am[idx] = xp, xm
            fd.flat[e] = (loss(ap) - loss(am)) / (2 * h)
        scale = max(1.0, np.abs(fd).max())
        np.testing.assert_allclose(g, fd, rtol=0, atol=1e-7 * scale, err_msg=name)


def test_backward_checkpoint_interval_is_invisible():
    """Recomputing states from checkpoints every 3 tokens gives the same gradients bit for
    bit as one checkpoint."""
    q, k, v, la, b, s0, do, dfin = _bwd_problem(4, "channel", T=11)
    g1 = oracle.backward(q, k, v, la, b, s0, do, dfin, block=3)
    g2 = oracle.backward(q, k, v, la, b, s0, do, dfin, block=64)
    for a, c in zip(g1, g2):
        assert np.array_equal(a, c)


def test_backward_without_final_gradient_or_state():
    """d_final = None is a zero final-state gradient, init_state = None a zero state."""
    q, k, v, la, b, s0, do, dfin = _bwd_problem(5, "scalar")
    g1 = oracle.backward(q, k, v, la, b, None, do, None)
    g2 = oracle.backward(q, k, v, la, b, np.zeros_like(s0), do, np.zeros_like(dfin))
    for a, c in zip(g1, g2):
        assert np.array_equal(a, c)
