"""GPU parity of dr_chunk_fwd against the fp64 oracle (through the C ABI)."""
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


def dev(d):
    return {k: (None if v is None else v.cuda()) for k, v in d.items()}


def run(dr, d, **kw):
    g = dev(d)
    out, fin = dr.chunk_fwd(g["q"], g["k"], g["v"], g["log_alpha"], g["beta"],
                            g["init_state"], **kw)
    torch.cuda.synchronize()
    assert dr.device_status() == 0
    return out, fin


def check(dr, d, dtype, chunk=64, out_dtype=None):
    out, fin = run(dr, d, chunk=chunk, out_dtype=out_dtype)
    o_ref, f_ref = oracle.forward(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"],
                                  d["init_state"])
    e1 = assert_close(out, o_ref, dtype, "out")
    e2 = assert_close(fin, f_ref, dtype, "final_state")
    return e1, e2


# fp32, single sequence, single head, d = 64, T = 256, zero initial state
@pytest.mark.parametrize("chunk", [16, 32, 64])
def test_f32_single_head(dr, chunk):
    w = inputs.WORKLOADS["gdn_f32_B1_H1_T256_d64"]
    check(dr, inputs.workload_inputs(w), "f32", chunk=chunk)


@pytest.mark.parametrize("gate", ["none", "scalar", "channel"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 128), (128, 64), (64, 64)])
def test_small_shapes(dr, gate, dtype, dk, dv):
    # T = 150: two full chunks and a ragged tail of 22 tokens; nonzero initial state.
    d = inputs.chunk_inputs(2, 150, 3, dk, dv, gate=gate, dtype=dtype, init_state=True,
                            seed=11)
    check(dr, d, dtype)


@pytest.mark.parametrize("T", [0, 1, 15, 63, 64, 65, 127, 129])
def test_edge_lengths(dr, T):
    d = inputs.chunk_inputs(1, T, 2, 128, 128, gate="channel", dtype="f32",
                            init_state=True, seed=T)
    out, fin = run(dr, d)
    o_ref, f_ref = oracle.forward(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"],
                                  d["init_state"])
    assert out.shape == (1, T, 2, 128)
    if T:
        assert_close(out, o_ref, "f32", "out")
    assert_close(fin, f_ref, "f32", "final_state")


@pytest.mark.parametrize("gate", ["scalar", "channel"])
def test_strong_decay(dr, gate):
    """log alpha ~ -U(0, 5): cumulative decays underflow inside a chunk."""
    d = inputs.chunk_inputs(1, 200, 2, 128, 128, gate=gate, dtype="f32", init_state=True,
                            seed=3, log_alpha_range=(0.0, 5.0))
    check(dr, d, "f32")


def test_beta_extremes_and_no_decay(dr):
    """beta in {0, 1} and alpha = 1 (DeltaNet) with unit keys."""
    d = inputs.chunk_inputs(1, 130, 2, 64, 64, gate="none", dtype="f32", init_state=True,
                            seed=5)
    d["beta"] = (torch.arange(130 * 2).reshape(1, 130, 2) % 3 == 0).float()
    check(dr, d, "f32")


@pytest.mark.parametrize("chunk", [16, 32, 64])
def test_chunk_size_invariance_bf16(dr, chunk):
    d = inputs.chunk_inputs(2, 256, 4, 128, 128, gate="channel", dtype="bf16", seed=21)
    check(dr, d, "bf16", chunk=chunk)


def test_fp32_output_for_bf16_inputs(dr):
    d = inputs.chunk_inputs(2, 256, 4, 128, 128, gate="scalar", dtype="bf16", seed=22)
    out, _ = run(dr, d, out_dtype=torch.float32)
    assert out.dtype == torch.float32
    o_ref, _ = oracle.forward(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], None)
    assert_close(out, o_ref, "bf16", "out")


def test_carry_over_split(dr):
    """chunk_fwd(x[:T1]) then chunk_fwd(x[T1:], init = its final state) equals the oracle
    over the whole sequence (T1 not a multiple of the chunk)."""
    d = inputs.chunk_inputs(2, 300, 2, 128, 128, gate="scalar", dtype="f32",
                            init_state=True, seed=9)
    g = dev(d)
    sl = lambda t, a, b: None if t is None else t[:, a:b].contiguous()
    o1, f1 = dr.chunk_fwd(sl(g["q"], 0, 100), sl(g["k"], 0, 100), sl(g["v"], 0, 100),
                          sl(g["log_alpha"], 0, 100), sl(g["beta"], 0, 100), g["init_state"])
    o2, f2 = dr.chunk_fwd(sl(g["q"], 100, 300), sl(g["k"], 100, 300), sl(g["v"], 100, 300),
                          sl(g["log_alpha"], 100, 300), sl(g["beta"], 100, 300), f1,
                          final_state=f1)   # in-place carry
    torch.cuda.synchronize()
    o_ref, f_ref = oracle.forward(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"],
                                  d["init_state"])
    assert_close(torch.cat([o1, o2], 1), o_ref, "f32", "out")
    assert_close(f2, f_ref, "f32", "final_state")


def test_deterministic(dr):
    d = inputs.chunk_inputs(2, 200, 2, 128, 128, gate="channel", dtype="bf16", seed=4)
    o1, f1 = run(dr, d)
    o2, f2 = run(dr, d)
    assert torch.equal(o1, o2) and torch.equal(f1, f2)


# ------------------------------------------------------------ full-size workloads
def sampled_chains(w, n, seed=0):
    rng = np.random.default_rng(seed)
    chains = rng.choice(w.B * w.H, size=n, replace=False)
    return [(int(c) // w.H, int(c) % w.H) for c in chains]


@pytest.mark.slow
@pytest.mark.parametrize("out_dtype", ["bf16", "f32"])
@pytest.mark.parametrize("name,nsample", [
    ("gdn_bf16_B8_H16_T4096_d128", 6),
    ("kda_bf16_B4_H32_T8192_d128", 4),
    ("gdn_bf16_B1_H16_T65536_d128_init", 2),
    ("kda_bf16_B1_H16_T65536_d128_init", 2)])
def test_full_size_sampled_chains(dr, name, nsample, out_dtype):
    """The workload at full size, in the launch configuration the benchmark times; the
    oracle recomputes a sample of whole (b, h) chains.  With an fp32-stored output the
    plain rule applies (max |gpu - oracle| <= 2e-2 RMS, no representation allowance); with
    the default bf16 output the allowance of half a bf16 ulp applies, and the plain error
    is recorded beside it."""
    w = inputs.WORKLOADS[name]
    d = inputs.workload_inputs(w)
    odt = torch.float32 if out_dtype == "f32" else None
    out, fin = run(dr, d, chunk=w.chunk, out_dtype=odt)
    out_h, fin_h = out.cpu(), fin.cpu()
    worst = {"out": 0.0, "out_plain": 0.0, "state": 0.0}
    for b, h in sampled_chains(w, nsample):
        pick = lambda t: None if t is None else t[b:b + 1, :, h:h + 1].contiguous()
        s0 = None if d["init_state"] is None else d["init_state"][b:b + 1, h:h + 1]
        o_ref, f_ref = oracle.forward(pick(d["q"]), pick(d["k"]), pick(d["v"]),
                                      pick(d["log_alpha"]), pick(d["beta"]), s0)
        o_gpu = out_h[b:b + 1, :, h:h + 1]
        worst["out"] = max(worst["out"], assert_close(o_gpu, o_ref, "bf16", f"out chain {(b, h)}"))
        worst["out_plain"] = max(worst["out_plain"], plain_err(o_gpu, o_ref))
        worst["state"] = max(worst["state"],
                             assert_close(fin_h[b:b + 1, h:h + 1], f_ref, "bf16", f"state chain {(b, h)}"))
    record(name, f"chunk_fwd out={out_dtype}", **worst)


# ------------------------------------------------------------ tensor-core path
# bf16 inputs, d_k = d_v = 128, C = 64, scalar gate or none run on the fused tcgen05 kernel.
@pytest.mark.parametrize("T", [1, 15, 63, 64, 65, 127, 129, 200])
def test_tc_edge_lengths(dr, T):
    d = inputs.chunk_inputs(2, T, 3, 128, 128, gate="scalar", dtype="bf16",
                            init_state=True, seed=100 + T)
    check(dr, d, "bf16")


@pytest.mark.parametrize("gate", ["none", "scalar"])
def test_tc_many_heads(dr, gate):
    d = inputs.chunk_inputs(3, 333, 5, 128, 128, gate=gate, dtype="bf16", init_state=True,
                            seed=7)
    check(dr, d, "bf16")


def test_tc_strong_decay(dr):
    d = inputs.chunk_inputs(2, 300, 2, 128, 128, gate="scalar", dtype="bf16",
                            init_state=True, seed=12, log_alpha_range=(0.0, 5.0))
    check(dr, d, "bf16")


def test_tc_fp32_output_strict(dr):
    d = inputs.chunk_inputs(2, 500, 4, 128, 128, gate="scalar", dtype="bf16",
                            init_state=True, seed=13)
    check(dr, d, "bf16", out_dtype=torch.float32)


def test_tc_deterministic(dr):
    d = inputs.chunk_inputs(2, 300, 3, 128, 128, gate="scalar", dtype="bf16", seed=14)
    o1, f1 = run(dr, d)
    o2, f2 = run(dr, d)
    assert torch.equal(o1, o2) and torch.equal(f1, f2)


def test_tc_workspace_sizes(dr):
    # many chains: the single kernel, no workspace
    desc = dr.chunk_desc(8, 4096, 16, 128, 128, dr.DR_BF16, dr.DR_BF16, dr.DR_GATE_SCALAR, 64)
    assert dr.workspace_bytes(desc) == 0 and dr.min_workspace_bytes(desc) == 0
    # few long chains: three segment-state slabs of 64 KB per (b, h, segment), plus, on the
    # fastest path, one 16 KB T-operand image and 512 B of row norms per (b, h, chunk): 9
    # segments of 114 chunks
    desc = dr.chunk_desc(1, 65536, 16, 128, 128, dr.DR_BF16, dr.DR_BF16, dr.DR_GATE_SCALAR, 64)
    seg = 3 * 16 * 9 * 65536
    assert dr.min_workspace_bytes(desc) == seg
    assert dr.workspace_bytes(desc) == seg + 16 * 1024 * (16384 + 512)


@pytest.mark.parametrize("gate", ["none", "scalar"])
def test_tc_single_kernel_path_without_workspace(dr, gate):
    """With less workspace than the T operands need, the single kernel solves inside each
    chain; its results equal the oracle's as well."""
    d = inputs.chunk_inputs(2, 333, 3, 128, 128, gate=gate, dtype="bf16", init_state=True,
                            seed=61)
    g = dev(d)
    out, fin = dr.chunk_fwd(g["q"], g["k"], g["v"], g["log_alpha"], g["beta"], g["init_state"],
                            workspace=torch.empty(16, dtype=torch.uint8, device="cuda"))
    torch.cuda.synchronize()
    assert dr.device_status() == 0
    o_ref, f_ref = oracle.forward(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"],
                                  d["init_state"])
    assert_close(out, o_ref, "bf16", "out")
    assert_close(fin, f_ref, "bf16", "final_state")


# ------------------------------------------------------------ segmented long sequences
# Few chains with many chunks are split into segments (end states, chaining, outputs).
@pytest.mark.parametrize("gate,T,la_range", [
    ("scalar", 4096, (0.001, 0.1)),     # 2 chains x 64 chunks -> 4 segments of 16 chunks
    ("none", 3000, (0.001, 0.1)),       # DeltaNet: transitions do not decay; ragged tail
    ("scalar", 2500, (0.0, 0.02)),      # weak decay: the carried state matters across segments
])
def test_tc_segmented_long(dr, gate, T, la_range):
    d = inputs.chunk_inputs(1, T, 2, 128, 128, gate=gate, dtype="bf16", init_state=True,
                            seed=31, log_alpha_range=la_range)
    desc = dr.chunk_desc(1, T, 2, 128, 128, dr.DR_BF16, dr.DR_BF16,
                         inputs.GATE_CODE[gate], 64)
    assert dr.workspace_bytes(desc) > 0          # the segmented path is taken
    check(dr, d, "bf16")


# The CUDA-core path (fp32 inputs, or head sizes the tensor-core kernels do not take) splits
# few long chains the same way: one CTA per 32 columns of each segment's end state and of its
# transition, the chaining, then one CTA per 32 output columns of each segment.
@pytest.mark.parametrize("B,T,H,dk,dv,gate,dtype,la_range", [
    (1, 4096, 1, 128, 128, "scalar", "f32", (0.001, 0.1)),   # 1 chain x 64 chunks -> 4 segments
    (1, 3000, 2, 64, 128, "channel", "f32", (0.0, 0.02)),    # dk != dv, weak decay, ragged: 2
    (1, 8192, 1, 64, 64, "channel", "bf16", (0.001, 0.1)),   # 128 chunks -> 8 segments
    (2, 2048, 1, 64, 64, "none", "f32", (0.001, 0.1)),       # DeltaNet: no decay at all
])
def test_simt_segmented_long(dr, B, T, H, dk, dv, gate, dtype, la_range):
    d = inputs.chunk_inputs(B, T, H, dk, dv, gate=gate, dtype=dtype, init_state=True,
                            seed=36 + T, log_alpha_range=la_range)
    it = dr.DR_F32 if dtype == "f32" else dr.DR_BF16
    desc = dr.chunk_desc(B, T, H, dk, dv, it, it, inputs.GATE_CODE[gate], 64)
    nch, C = B * H * -(-T // 64), 64
    base = 4 * nch * (C * dk * 3 + C * dv + C * C + dk)     # the per-chunk fp32 slabs
    assert dr.workspace_bytes(desc) > base                  # the segmented path is taken
    e1, e2 = check(dr, d, dtype)
    record(f"simt_segmented_B{B}_T{T}_H{H}_d{dk}x{dv}_{gate}_{dtype}", "out", err=e1, state=e2)


def test_simt_segmented_in_place_carry(dr):
    d = inputs.chunk_inputs(1, 2048, 1, 64, 64, gate="scalar", dtype="f32", init_state=True,
                            seed=37, log_alpha_range=(0.0, 0.02))
    g = dev(d)
    st = g["init_state"].clone()
    out, _ = dr.chunk_fwd(g["q"], g["k"], g["v"], g["log_alpha"], g["beta"], st,
                          final_state=st)
    torch.cuda.synchronize()
    assert dr.device_status() == 0
    o_ref, f_ref = oracle.forward(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"],
                                  d["init_state"])
    assert_close(out, o_ref, "f32", "out")
    assert_close(st, f_ref, "f32", "final_state")


def test_tc_segmented_in_place_carry(dr):
    """final_state == init_state on the segmented path."""
    d = inputs.chunk_inputs(1, 2048, 2, 128, 128, gate="scalar", dtype="bf16",
                            init_state=True, seed=32, log_alpha_range=(0.0, 0.02))
    g = dev(d)
    st = g["init_state"].clone()
    out, fin = dr.chunk_fwd(g["q"], g["k"], g["v"], g["log_alpha"], g["beta"], st,
                            final_state=st)
    torch.cuda.synchronize()
    o_ref, f_ref = oracle.forward(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"],
                                  d["init_state"])
    assert_close(out, o_ref, "bf16", "out")
    assert_close(st, f_ref, "bf16", "final_state")


# ------------------------------------------------------------ per-channel gate, tensor cores
# bf16 inputs, d_k = d_v = 128, C = 64, per-channel gate: the prep + state kernel pair.
@pytest.mark.parametrize("T", [1, 15, 16, 17, 63, 64, 65, 127, 129, 200])
def test_kda_tc_edge_lengths(dr, T):
    d = inputs.chunk_inputs(2, T, 3, 128, 128, gate="channel", dtype="bf16",
                            init_state=True, seed=200 + T)
    check(dr, d, "bf16")


def test_kda_tc_many_heads(dr):
    d = inputs.chunk_inputs(3, 333, 5, 128, 128, gate="channel", dtype="bf16",
                            init_state=True, seed=8)
    check(dr, d, "bf16")


@pytest.mark.parametrize("la_range", [(0.0, 1.0), (0.0, 3.0), (0.0, 5.0)])
def test_kda_tc_strong_decay(dr, la_range):
    """Per-token log decays up to -1, -3, -5 per channel.  Up to -1 a chunk decays by at
    most e^-64 and takes one product against its last token; beyond, chunks take four
    products against 16-token block ends, and at -5 a block can decay by e^-80 (exact
    diagonal blocks)."""
    d = inputs.chunk_inputs(2, 300, 2, 128, 128, gate="channel", dtype="bf16",
                            init_state=True, seed=15, log_alpha_range=la_range)
    check(dr, d, "bf16")


def test_kda_tc_extreme_decay_exact_diagonal(dr):
    """log alpha ~ -U(0, 20): every 16-token block decays past exp(-64) in some channel, so
    the diagonal blocks of the intra-chunk products are taken on the exact fallback."""
    d = inputs.chunk_inputs(1, 256, 2, 128, 128, gate="channel", dtype="bf16",
                            init_state=True, seed=16, log_alpha_range=(0.0, 20.0))
    check(dr, d, "bf16", out_dtype=torch.float32)


def test_kda_tc_mixed_decay(dr):
    """Half of the channels barely decay, half decay steeply: the exact fallback runs for
    the chunk while the slow channels still carry state across chunks."""
    d = inputs.chunk_inputs(1, 320, 2, 128, 128, gate="channel", dtype="bf16",
                            init_state=True, seed=17, log_alpha_range=(0.0, 0.01))
    d["log_alpha"][..., 64:] *= 2000.0      # -U(0, 20) on channels 64..127
    check(dr, d, "bf16", out_dtype=torch.float32)


def test_kda_tc_fp32_output_strict(dr):
    d = inputs.chunk_inputs(2, 500, 4, 128, 128, gate="channel", dtype="bf16",
                            init_state=True, seed=18)
    check(dr, d, "bf16", out_dtype=torch.float32)


def test_kda_tc_deterministic(dr):
    d = inputs.chunk_inputs(2, 300, 3, 128, 128, gate="channel", dtype="bf16", seed=19)
    o1, f1 = run(dr, d)
    o2, f2 = run(dr, d)
    assert torch.equal(o1, o2) and torch.equal(f1, f2)


def test_kda_tc_in_place_carry(dr):
    d = inputs.chunk_inputs(2, 190, 2, 128, 128, gate="channel", dtype="bf16",
                            init_state=True, seed=20)
    g = dev(d)
    st = g["init_state"].clone()
    out, _ = dr.chunk_fwd(g["q"], g["k"], g["v"], g["log_alpha"], g["beta"], st,
                          final_state=st)
    torch.cuda.synchronize()
    assert dr.device_status() == 0
    o_ref, f_ref = oracle.forward(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"],
                                  d["init_state"])
    assert_close(out, o_ref, "bf16", "out")
    assert_close(st, f_ref, "bf16", "final_state")


def test_kda_tc_workspace_bytes(dr):
    # per (b, h, chunk): W 16 KiB (bf16), U 32 KiB (fp32), P 16 KiB (fp32), the Q*G pair
    # 32 KiB, (K*G_C/G)^T 32 KiB (fp32), G_C 512 B
    desc = dr.chunk_desc(4, 8192, 32, 128, 128, dr.DR_BF16, dr.DR_BF16,
                         dr.DR_GATE_CHANNEL, 64)
    assert dr.workspace_bytes(desc) == 4 * 32 * 128 * 131584
    # few long chains add three segment-state slabs of 64 KiB per (b, h, segment): 16 chains
    # of 1024 chunks split into 9 segments of 114 chunks
    desc = dr.chunk_desc(1, 65536, 16, 128, 128, dr.DR_BF16, dr.DR_BF16,
                         dr.DR_GATE_CHANNEL, 64)
    seg = 3 * 16 * 9 * 65536
    assert dr.workspace_bytes(desc) == 16 * 1024 * 131584 + seg
    assert dr.min_workspace_bytes(desc) == dr.workspace_bytes(desc)


# Few long per-channel chains are split into segments too (end states of every segment from
# a zero start and from the identity, the chaining of the affine maps, then the outputs).
@pytest.mark.parametrize("B,T,H,la_range,out_dtype", [
    (1, 4096, 2, (0.001, 0.1), None),            # 2 chains x 64 chunks -> 4 segments of 16
    (1, 3000, 2, (0.0, 0.02), None),             # weak decay, ragged tail (47 chunks: 2 + 1)
    (1, 16384, 4, (0.001, 0.1), torch.float32),  # 4 chains x 256 chunks -> 16 segments
    (2, 2048, 3, (0.0, 0.005), torch.float32),   # very weak decay: the carry dominates
])
def test_kda_tc_segmented_long(dr, B, T, H, la_range, out_dtype):
    d = inputs.chunk_inputs(B, T, H, 128, 128, gate="channel", dtype="bf16", init_state=True,
                            seed=33 + T, log_alpha_range=la_range)
    desc = dr.chunk_desc(B, T, H, 128, 128, dr.DR_BF16, dr.DR_BF16, dr.DR_GATE_CHANNEL, 64)
    nch = B * H * -(-T // 64)
    assert dr.workspace_bytes(desc) > nch * 131584    # the segmented path is taken
    e1, e2 = check(dr, d, "bf16", out_dtype=out_dtype)
    record(f"kda_segmented_B{B}_T{T}_H{H}", "out" if out_dtype is None else "out_f32",
           err=e1, state=e2)


def test_kda_tc_segmented_mixed_decay(dr):
    """Half of the channels barely decay across the whole sequence, half decay steeply:
    the segments' transitions keep the slow channels' state and drop the others."""
    d = inputs.chunk_inputs(1, 4096, 2, 128, 128, gate="channel", dtype="bf16",
                            init_state=True, seed=34, log_alpha_range=(0.0, 0.001))
    d["log_alpha"][..., 64:] *= 1000.0      # -U(0, 1) on channels 64..127
    check(dr, d, "bf16", out_dtype=torch.float32)


def test_kda_tc_segmented_in_place_carry(dr):
    """final_state == init_state on the segmented per-channel path."""
    d = inputs.chunk_inputs(1, 2048, 2, 128, 128, gate="channel", dtype="bf16",
                            init_state=True, seed=35, log_alpha_range=(0.0, 0.02))
    g = dev(d)
    st = g["init_state"].clone()
    out, _ = dr.chunk_fwd(g["q"], g["k"], g["v"], g["log_alpha"], g["beta"], st,
                          final_state=st)
    torch.cuda.synchronize()
    assert dr.device_status() == 0
    o_ref, f_ref = oracle.forward(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"],
                                  d["init_state"])
    assert_close(out, o_ref, "bf16", "out")
    assert_close(st, f_ref, "bf16", "final_state")
