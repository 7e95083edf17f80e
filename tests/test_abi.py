"""The C ABI without a GPU: the library loads, exports every function include/dr.h
declares, and rejects bad arguments on the host before any CUDA call."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def dr():
    from gated_delta_rule_15_gb300 import build
    build.build()
    import gated_delta_rule_15_gb300.dr as m
    return m


def header_functions():
    names = set()
    for hdr in os.listdir(os.path.join(ROOT, "include")):
        if not hdr.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", hdr)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(dr_\w+)\s*\(", text, re.M))
    return names


def test_header_declares_the_binding_symbols(dr):
    assert header_functions() == set(dr.EXPORTED)


def test_every_declared_symbol_is_exported(dr):
    lib = dr.lib()
    for name in header_functions():
        assert hasattr(lib, name), name


def test_version_and_strerror(dr):
    assert dr.version() >= 1
    for st in (0, -1, -2, -3, -4, -5, 17):
        assert isinstance(dr.strerror(st), str) and dr.strerror(st)


def _desc(dr, **kw):
    # per-channel gate: a two-kernel path, which needs a workspace
    d = dict(B=2, T=100, H=3, dk=128, dv=128, in_dtype=dr.DR_BF16, out_dtype=dr.DR_BF16,
             gate=dr.DR_GATE_CHANNEL, chunk=64)
    d.update(kw)
    return dr.ChunkDesc(**d)


def test_workspace_query(dr):
    n = dr.workspace_bytes(_desc(dr))
    assert n > 0 and n % 16 == 0
    assert dr.workspace_bytes(_desc(dr, T=0)) == 0
    # the tensor-core path (bf16, d = 128, C = 64, scalar gate) with many short chains: none
    assert dr.workspace_bytes(_desc(dr, gate=dr.DR_GATE_SCALAR)) == 0
    assert dr.min_workspace_bytes(_desc(dr, gate=dr.DR_GATE_SCALAR)) == 0
    # few long chains (segments): the fastest path also holds 16 KB of T operands and 512 B
    # of row norms per chunk
    long = _desc(dr, B=1, T=64 * 64, H=2, gate=dr.DR_GATE_SCALAR)
    assert dr.workspace_bytes(long) == dr.min_workspace_bytes(long) + 2 * 64 * (16384 + 512)
    # the fused neighbours' fastest path (two kernels) takes them for many chains too; a fused
    # output gate with fp32 outputs stays on the single kernel
    many = _desc(dr, gate=dr.DR_GATE_SCALAR)
    assert dr.ex_workspace_bytes(many, 0) == 0
    for fl in (dr.DR_FUSE_QK_L2NORM, dr.DR_FUSE_BETA_SIGMOID, dr.DR_FUSE_OUT_SILU_GATE, 7):
        assert dr.ex_workspace_bytes(many, fl) == 2 * 3 * 2 * (16384 + 512)
    f32out = _desc(dr, gate=dr.DR_GATE_SCALAR, out_dtype=dr.DR_F32)
    assert dr.ex_workspace_bytes(f32out, dr.DR_FUSE_OUT_SILU_GATE) == 0
    assert dr.ex_workspace_bytes(f32out, dr.DR_FUSE_QK_L2NORM) == 2 * 3 * 2 * (16384 + 512)
    for d in (_desc(dr), _desc(dr, in_dtype=dr.DR_F32)):   # other paths: the plain answer
        assert dr.ex_workspace_bytes(d, 7) == dr.workspace_bytes(d)
    with pytest.raises(dr.DrError):
        dr.ex_workspace_bytes(many, 8)
    assert dr.workspace_bytes(_desc(dr, gate=dr.DR_GATE_SCALAR, in_dtype=dr.DR_F32)) > 0
    for d in (_desc(dr), _desc(dr, in_dtype=dr.DR_F32), _desc(dr, T=0)):   # other paths: equal
        assert dr.min_workspace_bytes(d) == dr.workspace_bytes(d)
    # few long chains on the per-channel tensor-core path: the segments' transitions,
    # zero-start end states and start states, 64 KB each per (b, h, segment): 2 chains of 64
    # chunks -> 4 segments
    kda = _desc(dr, B=1, T=64 * 64, H=2)
    assert dr.workspace_bytes(kda) == 2 * 64 * 131584 + 3 * 2 * 4 * 65536
    # ... and on the CUDA-core path (fp32 slabs per chunk: W, Q*G, K*G_C/G [C][dk], U [C][dv],
    # P [C][C], G_C [dk]; per segment Phi [dk][dk], S0 and the start [dk][dv]): 1 chain of 64
    # chunks, dk = 64, dv = 128 -> 4 segments
    simt = _desc(dr, B=1, T=64 * 64, H=1, dk=64, dv=128, in_dtype=dr.DR_F32, out_dtype=dr.DR_F32)
    slabs = 64 * (64 * 64 * 3 + 64 * 128 + 64 * 64 + 64)
    assert dr.workspace_bytes(simt) == 4 * (slabs + 4 * (64 * 64 + 2 * 64 * 128))


@pytest.mark.parametrize("bad,status", [
    (dict(dk=96), -2), (dict(dv=32), -2), (dict(chunk=48), -2), (dict(chunk=-1), -1),
    (dict(B=0), -1), (dict(H=0), -1), (dict(T=-1), -1), (dict(gate=3), -1),
    (dict(in_dtype=7), -1), (dict(out_dtype=-1), -1)])
def test_bad_descriptors_rejected(dr, bad, status):
    n = ctypes.c_size_t(0)
    rc = dr.lib().dr_chunk_fwd_workspace_bytes(ctypes.byref(_desc(dr, **bad)), ctypes.byref(n))
    assert rc == status


# The next two tests pass fake (never dereferenced) device addresses and expect host-side
# rejection.  They are kept off machines with a GPU, where a validation bug would turn
# them into a launch on unmapped memory.
no_gpu_only = pytest.mark.skipif(
    __import__("torch").cuda.is_available(), reason="fake-pointer checks run only without a GPU")


@no_gpu_only
def test_chunk_fwd_host_side_errors(dr):
    lib = dr.lib()
    d = _desc(dr)
    fake = ctypes.c_void_p(1 << 20)        # aligned, never dereferenced: rejected first
    mis = ctypes.c_void_p((1 << 20) + 8)   # misaligned
    null = None
    args = lambda **o: [o.get(n, fake) for n in
                        ("q", "k", "v", "la", "beta", "s0", "out", "fin", "ws")]
    call = lambda a, wb=1 << 40: lib.dr_chunk_fwd(ctypes.byref(d), *a, wb, None)
    assert lib.dr_chunk_fwd(None, *args(), 0, None) == dr.DR_ERR_INVALID
    assert call(args(q=null)) == dr.DR_ERR_INVALID
    assert call(args(la=null)) == dr.DR_ERR_INVALID          # a gate needs log_alpha
    assert call(args(out=mis)) == dr.DR_ERR_INVALID
    assert call(args(ws=null)) == dr.DR_ERR_WORKSPACE
    assert call(args(), wb=16) == dr.DR_ERR_WORKSPACE
    # final_state partially overlapping init_state
    assert call(args(s0=ctypes.c_void_p(1 << 20), fin=ctypes.c_void_p((1 << 20) + 1024))) \
        == dr.DR_ERR_INVALID


@no_gpu_only
def test_recurrent_step_host_side_errors(dr):
    lib = dr.lib()
    fake = ctypes.c_void_p(1 << 20)
    d = dr.StepDesc(4, 2, 128, 128, dr.DR_BF16, dr.DR_BF16, dr.DR_GATE_CHANNEL, 0)
    call = lambda desc, **o: lib.dr_recurrent_step(
        ctypes.byref(desc), *[o.get(n, fake) for n in ("q", "k", "v", "la", "beta")],
        o.get("state", ctypes.c_void_p(1 << 30)), o.get("out", ctypes.c_void_p(1 << 32)), None)
    assert call(d, la=None) == dr.DR_ERR_INVALID
    assert call(d, state=None) == dr.DR_ERR_INVALID
    assert call(d, out=ctypes.c_void_p((1 << 30) + 64)) == dr.DR_ERR_INVALID  # overlaps state
    d2 = dr.StepDesc(4, 2, 128, 80, dr.DR_BF16, dr.DR_BF16, dr.DR_GATE_CHANNEL, 0)
    assert call(d2) == dr.DR_ERR_UNSUPPORTED
    d3 = dr.StepDesc(4, 2, 128, 128, dr.DR_BF16, dr.DR_BF16, dr.DR_GATE_CHANNEL, 1)
    assert call(d3) == dr.DR_ERR_INVALID


@no_gpu_only
def test_fused_entry_points_host_side_errors(dr):
    lib = dr.lib()
    d = _desc(dr)
    fake = ctypes.c_void_p(1 << 20)
    far = lambda n: ctypes.c_void_p(n << 32)   # disjoint fake buffers, never dereferenced
    names = ("q", "k", "v", "la", "beta", "z", "s0", "out", "fin", "ws")
    args = lambda **o: [o.get(n, fake if n not in ("z", "out") else far(names.index(n)))
                        for n in names]
    call = lambda fuse, a: lib.dr_chunk_fwd_ex(ctypes.byref(d), fuse, *a, 1 << 40, None)
    assert call(8, args()) == dr.DR_ERR_INVALID                        # unknown bit
    assert call(dr.DR_FUSE_OUT_SILU_GATE, args(z=None)) == dr.DR_ERR_INVALID
    assert call(dr.DR_FUSE_OUT_SILU_GATE, args(z=ctypes.c_void_p((2 << 32) + 8))) \
        == dr.DR_ERR_INVALID                                           # misaligned z
    assert call(dr.DR_FUSE_OUT_SILU_GATE, args(z=far(7))) == dr.DR_ERR_INVALID  # z overlaps out
    assert call(dr.DR_FUSE_QK_L2NORM, args(q=None)) == dr.DR_ERR_INVALID
    sd = dr.StepDesc(4, 2, 128, 128, dr.DR_BF16, dr.DR_BF16, dr.DR_GATE_CHANNEL, 0)
    step = lambda fuse, **o: lib.dr_recurrent_step_ex(
        ctypes.byref(sd), fuse, *[o.get(n, fake) for n in ("q", "k", "v", "la", "beta")],
        o.get("z", far(3)), far(1), far(2), None)
    assert step(16) == dr.DR_ERR_INVALID
    assert step(dr.DR_FUSE_OUT_SILU_GATE, z=None) == dr.DR_ERR_INVALID
    assert step(dr.DR_FUSE_OUT_SILU_GATE, z=far(1)) == dr.DR_ERR_INVALID   # z overlaps state


def test_python_binding_rejects_host_tensors(dr):
    import torch
    x = torch.zeros(1, 4, 1, 64)
    with pytest.raises(ValueError):
        dr.chunk_fwd(x, x, x, None, torch.zeros(1, 4, 1))


@no_gpu_only
def test_chunk_bwd_host_side_errors(dr):
    lib = dr.lib()
    d = _desc(dr)   # per-channel gate
    names = ("q", "k", "v", "la", "beta", "s0", "do", "dfin", "dq", "dk", "dv", "dla", "db",
             "dinit", "ws")
    far = lambda n: ctypes.c_void_p((n + 1) << 32)
    args = lambda **o: [o.get(n, far(i)) for i, n in enumerate(names)]
    call = lambda a, wb=1 << 40: lib.dr_chunk_bwd(ctypes.byref(d), *a, wb, None)
    n = ctypes.c_size_t(0)
    assert lib.dr_chunk_bwd_workspace_bytes(ctypes.byref(d), ctypes.byref(n)) == 0
    assert n.value > dr.workspace_bytes(d)
    assert call(args(dq=None)) == dr.DR_ERR_INVALID
    assert call(args(dla=None)) == dr.DR_ERR_INVALID            # a gate needs d_log_alpha
    assert call(args(do=ctypes.c_void_p((3 << 32) + 8))) == dr.DR_ERR_INVALID
    assert call(args(ws=None)) == dr.DR_ERR_WORKSPACE
    assert call(args(), wb=n.value - 16) == dr.DR_ERR_WORKSPACE
    d0 = _desc(dr, gate=dr.DR_GATE_NONE)
    assert lib.dr_chunk_bwd(ctypes.byref(d0), *args(), 1 << 40, None) == dr.DR_ERR_INVALID


def test_selftest_budget_checked_on_host(dr):
    lib = dr.lib()
    assert lib.dr_selftest_bounded_wait(0, None) == dr.DR_ERR_INVALID
    assert lib.dr_selftest_bounded_wait(5_000_000_000, None) == dr.DR_ERR_INVALID


def test_host_entry_point_checks(dr):
    lib = dr.lib()
    d = _desc(dr)
    n = ctypes.c_size_t(0)
    assert lib.dr_chunk_fwd_host_dev_bytes(ctypes.byref(d), 4, ctypes.byref(n)) == 0
    staging = 2 * 100 * 3 * (3 * 128 * 2 + 2 + 128 * 4 + 128 * 2) + 2 * 3 * 128 * 128 * 4
    assert n.value >= staging + dr.workspace_bytes(d)
    assert lib.dr_chunk_fwd_host_dev_bytes(ctypes.byref(d), 0, ctypes.byref(n)) == dr.DR_ERR_INVALID
    fake = ctypes.c_void_p(1 << 20)
    call = lambda pieces, dev, nbytes: lib.dr_chunk_fwd_host(
        ctypes.byref(d), pieces, fake, fake, fake, fake, fake, None, fake, None, dev, nbytes, None)
    assert call(0, fake, 1 << 40) == dr.DR_ERR_INVALID
    assert call(2, None, 1 << 40) == dr.DR_ERR_WORKSPACE
    assert call(2, ctypes.c_void_p((1 << 20) + 16), 1 << 40) == dr.DR_ERR_WORKSPACE   # not 256-aligned
    assert call(2, fake, 16) == dr.DR_ERR_WORKSPACE
