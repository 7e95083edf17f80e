"""ctypes binding of libdr.so (include/dr.h).

Argument marshalling only: shapes and dtypes are read off torch tensors, pointers and the
current CUDA stream are passed to the C ABI, and every step of the computation runs in the
library's CUDA kernels.  There is no CPU path: importing this module loads libdr.so and
raises ImportError if it has not been built.

Host (CPU) tensors are accepted by the ``*_host`` helpers only, which copy inputs to the
device on the current stream, call the same entry point and copy the results back: that
is the end-to-end path a caller with host buffers takes.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libdr.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"libdr.so is not built ({LIB_PATH}); run "
                      "`python -c 'import __graft_entry__ as g; g.build()'`")
_lib = ctypes.CDLL(LIB_PATH)

DR_F32, DR_BF16 = 0, 1
DR_GATE_NONE, DR_GATE_SCALAR, DR_GATE_CHANNEL = 0, 1, 2
DR_OK, DR_ERR_INVALID, DR_ERR_UNSUPPORTED, DR_ERR_CUDA, DR_ERR_TIMEOUT, DR_ERR_WORKSPACE = \
    0, -1, -2, -3, -4, -5
# fused neighbours (flags of dr_chunk_fwd_ex / dr_recurrent_step_ex)
DR_FUSE_QK_L2NORM, DR_FUSE_BETA_SIGMOID, DR_FUSE_OUT_SILU_GATE = 1, 2, 4
DR_FUSE_ALL = 7
L2NORM_EPS = 1e-6   # DR_L2NORM_EPS

# Symbols of include/dr.h (checked by tests/test_abi.py against the header).
EXPORTED = ("dr_version", "dr_chunk_fwd_workspace_bytes", "dr_chunk_fwd_min_workspace_bytes",
            "dr_chunk_fwd_ex_workspace_bytes", "dr_chunk_fwd",
            "dr_recurrent_step", "dr_get_device_status", "dr_strerror",
            "dr_chunk_fwd_noalloc", "dr_chunk_fwd_ex", "dr_recurrent_step_ex",
            "dr_chunk_bwd_workspace_bytes", "dr_chunk_bwd", "dr_selftest_bounded_wait",
            "dr_chunk_fwd_host_dev_bytes", "dr_chunk_fwd_host")


class ChunkDesc(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("T", ctypes.c_int64), ("H", ctypes.c_int64),
                ("dk", ctypes.c_int64), ("dv", ctypes.c_int64),
                ("in_dtype", ctypes.c_int32), ("out_dtype", ctypes.c_int32),
                ("gate", ctypes.c_int32), ("chunk", ctypes.c_int32)]


class StepDesc(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("H", ctypes.c_int64), ("dk", ctypes.c_int64),
                ("dv", ctypes.c_int64), ("in_dtype", ctypes.c_int32),
                ("out_dtype", ctypes.c_int32), ("gate", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


_vp = ctypes.c_void_p
_lib.dr_version.argtypes = []
_lib.dr_version.restype = ctypes.c_int
_lib.dr_chunk_fwd_workspace_bytes.argtypes = [ctypes.POINTER(ChunkDesc),
                                              ctypes.POINTER(ctypes.c_size_t)]
_lib.dr_chunk_fwd_workspace_bytes.restype = ctypes.c_int
_lib.dr_chunk_fwd_min_workspace_bytes.argtypes = [ctypes.POINTER(ChunkDesc),
                                                  ctypes.POINTER(ctypes.c_size_t)]
_lib.dr_chunk_fwd_min_workspace_bytes.restype = ctypes.c_int
_lib.dr_chunk_fwd_ex_workspace_bytes.argtypes = [ctypes.POINTER(ChunkDesc), ctypes.c_uint32,
                                                 ctypes.POINTER(ctypes.c_size_t)]
_lib.dr_chunk_fwd_ex_workspace_bytes.restype = ctypes.c_int
_lib.dr_chunk_fwd.argtypes = [ctypes.POINTER(ChunkDesc), _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                              _vp, _vp, ctypes.c_size_t, _vp]
_lib.dr_chunk_fwd.restype = ctypes.c_int
_lib.dr_recurrent_step.argtypes = [ctypes.POINTER(StepDesc), _vp, _vp, _vp, _vp, _vp, _vp,
                                   _vp, _vp]
_lib.dr_recurrent_step.restype = ctypes.c_int
_lib.dr_chunk_fwd_ex.argtypes = [ctypes.POINTER(ChunkDesc), ctypes.c_uint32, _vp, _vp, _vp, _vp,
                                 _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]
_lib.dr_chunk_fwd_ex.restype = ctypes.c_int
_lib.dr_recurrent_step_ex.argtypes = [ctypes.POINTER(StepDesc), ctypes.c_uint32, _vp, _vp, _vp,
                                      _vp, _vp, _vp, _vp, _vp, _vp]
_lib.dr_recurrent_step_ex.restype = ctypes.c_int
_lib.dr_chunk_bwd_workspace_bytes.argtypes = [ctypes.POINTER(ChunkDesc),
                                              ctypes.POINTER(ctypes.c_size_t)]
_lib.dr_chunk_bwd_workspace_bytes.restype = ctypes.c_int
_lib.dr_chunk_bwd.argtypes = [ctypes.POINTER(ChunkDesc)] + [_vp] * 15 + [ctypes.c_size_t, _vp]
_lib.dr_chunk_bwd.restype = ctypes.c_int
_lib.dr_chunk_fwd_host_dev_bytes.argtypes = [ctypes.POINTER(ChunkDesc), ctypes.c_int,
                                             ctypes.POINTER(ctypes.c_size_t)]
_lib.dr_chunk_fwd_host_dev_bytes.restype = ctypes.c_int
_lib.dr_chunk_fwd_host.argtypes = [ctypes.POINTER(ChunkDesc), ctypes.c_int] + [_vp] * 9 + \
    [ctypes.c_size_t, _vp]
_lib.dr_chunk_fwd_host.restype = ctypes.c_int
_lib.dr_selftest_bounded_wait.argtypes = [ctypes.c_longlong, _vp]
_lib.dr_selftest_bounded_wait.restype = ctypes.c_int
_lib.dr_get_device_status.argtypes = [_vp]
_lib.dr_get_device_status.restype = ctypes.c_int
_lib.dr_strerror.argtypes = [ctypes.c_int]
_lib.dr_strerror.restype = ctypes.c_char_p
_lib.dr_chunk_fwd_noalloc.argtypes = [ctypes.POINTER(ChunkDesc), _vp, _vp, _vp, _vp, _vp, _vp,
                                      _vp, _vp, _vp]
_lib.dr_chunk_fwd_noalloc.restype = ctypes.c_int
NOALLOC_SCRATCH_BYTES = 64 << 20   # DR_NOALLOC_SCRATCH_BYTES of include/dr.h

_DT = {torch.float32: DR_F32, torch.bfloat16: DR_BF16}
_TORCH_DT = {DR_F32: torch.float32, DR_BF16: torch.bfloat16}


class DrError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {strerror(status)} (status {status})")
        self.status = status


def lib() -> ctypes.CDLL:
    return _lib


def version() -> int:
    return _lib.dr_version()


def strerror(status: int) -> str:
    return _lib.dr_strerror(status).decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _gate_of(log_alpha, bth_shape, dk):
    if log_alpha is None:
        return DR_GATE_NONE
    if tuple(log_alpha.shape) == tuple(bth_shape):
        return DR_GATE_SCALAR
    if tuple(log_alpha.shape) == tuple(bth_shape) + (dk,):
        return DR_GATE_CHANNEL
    raise ValueError(f"log_alpha shape {tuple(log_alpha.shape)} fits neither "
                     f"{tuple(bth_shape)} nor {tuple(bth_shape) + (dk,)}")


def _check_dev(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")


def fuse_flags(qk_l2norm: bool = False, beta_sigmoid: bool = False, z=None) -> int:
    """DR_FUSE_* bits for the fused neighbours requested."""
    return ((DR_FUSE_QK_L2NORM if qk_l2norm else 0) | (DR_FUSE_BETA_SIGMOID if beta_sigmoid else 0)
            | (DR_FUSE_OUT_SILU_GATE if z is not None else 0))


def chunk_desc(B, T, H, dk, dv, in_dtype, out_dtype, gate, chunk=64) -> ChunkDesc:
    return ChunkDesc(B, T, H, dk, dv, in_dtype, out_dtype, gate, chunk)


def workspace_bytes(desc: ChunkDesc) -> int:
    n = ctypes.c_size_t(0)
    rc = _lib.dr_chunk_fwd_workspace_bytes(ctypes.byref(desc), ctypes.byref(n))
    if rc != DR_OK:
        raise DrError(rc, "dr_chunk_fwd_workspace_bytes")
    return n.value


def min_workspace_bytes(desc: ChunkDesc) -> int:
    n = ctypes.c_size_t(0)
    rc = _lib.dr_chunk_fwd_min_workspace_bytes(ctypes.byref(desc), ctypes.byref(n))
    if rc != DR_OK:
        raise DrError(rc, "dr_chunk_fwd_min_workspace_bytes")
    return n.value


def ex_workspace_bytes(desc: ChunkDesc, fuse: int) -> int:
    n = ctypes.c_size_t(0)
    rc = _lib.dr_chunk_fwd_ex_workspace_bytes(ctypes.byref(desc), fuse, ctypes.byref(n))
    if rc != DR_OK:
        raise DrError(rc, "dr_chunk_fwd_ex_workspace_bytes")
    return n.value


def chunk_fwd(q, k, v, log_alpha, beta, init_state=None, *, chunk: int = 64,
              out_dtype=None, return_final_state: bool = True, out=None,
              final_state=None, workspace=None, stream=None, qk_l2norm: bool = False,
              beta_sigmoid: bool = False, z=None):
    """Chunkwise forward (dr_chunk_fwd, or dr_chunk_fwd_ex with fused neighbours) on
    device tensors.

    q, k [B,T,H,dk]; v [B,T,H,dv]; beta [B,T,H] (q's dtype); log_alpha None, fp32
    [B,T,H] or [B,T,H,dk]; init_state None or fp32 [B,H,dk,dv].  Returns
    (out [B,T,H,dv], final_state [B,H,dk,dv] fp32 or None).  ``final_state`` may be the
    ``init_state`` tensor for an in-place carry.  Fused neighbours: ``qk_l2norm`` divides
    q and k rows by their norms, ``beta_sigmoid`` reads beta as logits, ``z``
    ([B,T,H,dv], q's dtype) gates the output by silu(z).
    """
    _check_dev(q, k, v, log_alpha, beta, init_state, out, final_state, workspace, z)
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if q.dtype not in _DT or k.dtype != q.dtype or v.dtype != q.dtype or beta.dtype != q.dtype:
        raise ValueError("q, k, v, beta must share one dtype (float32 or bfloat16)")
    if tuple(k.shape) != (B, T, H, dk) or tuple(v.shape[:3]) != (B, T, H) \
            or tuple(beta.shape) != (B, T, H):
        raise ValueError("inconsistent shapes")
    if log_alpha is not None and log_alpha.dtype != torch.float32:
        raise ValueError("log_alpha must be float32")
    if init_state is not None and (init_state.dtype != torch.float32
                                   or tuple(init_state.shape) != (B, H, dk, dv)):
        raise ValueError("init_state must be float32 [B,H,dk,dv]")
    if z is not None and (z.dtype != q.dtype or tuple(z.shape) != (B, T, H, dv)):
        raise ValueError("z must have q's dtype and shape [B,T,H,dv]")
    fuse = fuse_flags(qk_l2norm, beta_sigmoid, z)
    gate = _gate_of(log_alpha, (B, T, H), dk)
    odt = _DT[out_dtype or q.dtype]
    desc = chunk_desc(B, T, H, dk, dv, _DT[q.dtype], odt, gate, chunk)
    if out is None:
        out = torch.empty((B, T, H, dv), dtype=_TORCH_DT[odt], device=q.device)
    if final_state is None and return_final_state:
        final_state = torch.empty((B, H, dk, dv), dtype=torch.float32, device=q.device)
    need = ex_workspace_bytes(desc, fuse) if fuse else workspace_bytes(desc)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if fuse:
        rc = _lib.dr_chunk_fwd_ex(ctypes.byref(desc), fuse, _ptr(q), _ptr(k), _ptr(v),
                                  _ptr(log_alpha), _ptr(beta), _ptr(z), _ptr(init_state),
                                  _ptr(out), _ptr(final_state), _ptr(workspace), wbytes,
                                  _stream_handle(stream))
        if rc != DR_OK:
            raise DrError(rc, "dr_chunk_fwd_ex")
        return out, final_state
    rc = _lib.dr_chunk_fwd(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha),
                           _ptr(beta), _ptr(init_state), _ptr(out), _ptr(final_state),
                           _ptr(workspace), wbytes, _stream_handle(stream))
    if rc != DR_OK:
        raise DrError(rc, "dr_chunk_fwd")
    return out, final_state


def bwd_workspace_bytes(desc: ChunkDesc) -> int:
    n = ctypes.c_size_t(0)
    rc = _lib.dr_chunk_bwd_workspace_bytes(ctypes.byref(desc), ctypes.byref(n))
    if rc != DR_OK:
        raise DrError(rc, "dr_chunk_bwd_workspace_bytes")
    return n.value


def chunk_bwd(q, k, v, log_alpha, beta, init_state, d_out, d_final_state=None, *,
              chunk: int = 64, return_d_init: bool = True, workspace=None, stream=None):
    """Backward of chunk_fwd (dr_chunk_bwd): gradients of <d_out, out> +
    <d_final_state, final_state>.  Inputs as for chunk_fwd; d_out [B,T,H,dv] in the
    forward output's dtype; d_final_state None or fp32 [B,H,dk,dv].  Returns (dq, dk, dv,
    d_log_alpha, d_beta, d_init_state): the first three and d_beta in the inputs' dtype,
    d_log_alpha fp32 with log_alpha's shape (None without a gate), d_init_state fp32
    [B,H,dk,dv] (None unless return_d_init)."""
    _check_dev(q, k, v, log_alpha, beta, init_state, d_out, d_final_state, workspace)
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if q.dtype not in _DT or k.dtype != q.dtype or v.dtype != q.dtype or beta.dtype != q.dtype:
        raise ValueError("q, k, v, beta must share one dtype (float32 or bfloat16)")
    if d_out.dtype not in _DT or tuple(d_out.shape) != (B, T, H, dv):
        raise ValueError("d_out must be float32 or bfloat16 [B,T,H,dv]")
    for t in (init_state, d_final_state):
        if t is not None and (t.dtype != torch.float32 or tuple(t.shape) != (B, H, dk, dv)):
            raise ValueError("states must be float32 [B,H,dk,dv]")
    gate = _gate_of(log_alpha, (B, T, H), dk)
    desc = chunk_desc(B, T, H, dk, dv, _DT[q.dtype], _DT[d_out.dtype], gate, chunk)
    dq, dk_, dv_ = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dla = None if log_alpha is None else torch.empty_like(log_alpha)
    dbeta = torch.empty_like(beta)
    dinit = (torch.empty((B, H, dk, dv), dtype=torch.float32, device=q.device)
             if return_d_init else None)
    need = bwd_workspace_bytes(desc)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = _lib.dr_chunk_bwd(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha),
                           _ptr(beta), _ptr(init_state), _ptr(d_out), _ptr(d_final_state),
                           _ptr(dq), _ptr(dk_), _ptr(dv_), _ptr(dla), _ptr(dbeta), _ptr(dinit),
                           _ptr(workspace), wbytes, _stream_handle(stream))
    if rc != DR_OK:
        raise DrError(rc, "dr_chunk_bwd")
    return dq, dk_, dv_, dla, dbeta, dinit


def chunk_fwd_noalloc(q, k, v, log_alpha, beta, init_state, out, final_state, *,
                      chunk: int = 64, stream=None):
    """dr_chunk_fwd_noalloc: the chunk forward for callers that cannot allocate device
    memory (a host framework that owns all memory through its own pool, a plugin whose
    execute callback must not allocate, a loop that cannot pay cudaMalloc's implicit
    synchronisation).  The caller passes preallocated ``out`` and ``final_state`` (or
    None); the library's static 64 MiB device scratch replaces the workspace.  Calls that
    overlap on the GPU race on that scratch; the first call on a device must precede any
    stream capture.  Returns the status code (0 on success)."""
    _check_dev(q, k, v, log_alpha, beta, init_state, out, final_state)
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    desc = chunk_desc(B, T, H, dk, dv, _DT[q.dtype], _DT[out.dtype],
                      _gate_of(log_alpha, (B, T, H), dk), chunk)
    return _lib.dr_chunk_fwd_noalloc(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v),
                                     _ptr(log_alpha), _ptr(beta), _ptr(init_state),
                                     _ptr(out), _ptr(final_state), _stream_handle(stream))


def recurrent_step(q, k, v, log_alpha, beta, state, *, out=None, out_dtype=None,
                   stream=None, qk_l2norm: bool = False, beta_sigmoid: bool = False, z=None):
    """One decode step (dr_recurrent_step, or dr_recurrent_step_ex with fused neighbours,
    flags as for chunk_fwd; z [B,H,dv]); ``state`` [B,H,dk,dv] fp32 is updated in
    place.  q, k [B,H,dk]; v [B,H,dv]; beta [B,H]; log_alpha None, [B,H] or [B,H,dk].
    Returns out [B,H,dv]."""
    _check_dev(q, k, v, log_alpha, beta, state, out, z)
    B, H, dk = q.shape
    dv = v.shape[-1]
    if q.dtype not in _DT or k.dtype != q.dtype or v.dtype != q.dtype or beta.dtype != q.dtype:
        raise ValueError("q, k, v, beta must share one dtype (float32 or bfloat16)")
    if state.dtype != torch.float32 or tuple(state.shape) != (B, H, dk, dv):
        raise ValueError("state must be float32 [B,H,dk,dv]")
    if log_alpha is not None and log_alpha.dtype != torch.float32:
        raise ValueError("log_alpha must be float32")
    if z is not None and (z.dtype != q.dtype or tuple(z.shape) != (B, H, dv)):
        raise ValueError("z must have q's dtype and shape [B,H,dv]")
    fuse = fuse_flags(qk_l2norm, beta_sigmoid, z)
    gate = _gate_of(log_alpha, (B, H), dk)
    odt = _DT[out_dtype or q.dtype]
    desc = StepDesc(B, H, dk, dv, _DT[q.dtype], odt, gate, 0)
    if out is None:
        out = torch.empty((B, H, dv), dtype=_TORCH_DT[odt], device=q.device)
    if fuse:
        rc = _lib.dr_recurrent_step_ex(ctypes.byref(desc), fuse, _ptr(q), _ptr(k), _ptr(v),
                                       _ptr(log_alpha), _ptr(beta), _ptr(z), _ptr(state),
                                       _ptr(out), _stream_handle(stream))
        if rc != DR_OK:
            raise DrError(rc, "dr_recurrent_step_ex")
        return out
    rc = _lib.dr_recurrent_step(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v),
                                _ptr(log_alpha), _ptr(beta), _ptr(state), _ptr(out),
                                _stream_handle(stream))
    if rc != DR_OK:
        raise DrError(rc, "dr_recurrent_step")
    return out


def selftest_bounded_wait(cycles: int = 2_000_000, stream=None) -> int:
    """dr_selftest_bounded_wait: a wait that runs out on purpose (no fault); the next
    device_status() returns DR_ERR_TIMEOUT.  Returns the enqueue status."""
    return _lib.dr_selftest_bounded_wait(int(cycles), _stream_handle(stream))


def device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the sticky device status word."""
    return _lib.dr_get_device_status(_stream_handle(stream))


class HostChunkRunner:
    """End-to-end chunk forward for callers holding HOST buffers, through dr_chunk_fwd_host.

    Owns the device staging buffer and pinned host result buffers for one problem shape.
    Each call enqueues, behind the current stream, the host -> device copies of the inputs,
    the forward and the device -> host copies of out and final_state, the sequence split
    into `pieces` time ranges so that copies and kernels overlap; with `sync` it waits for
    the stream.  Returns the pinned host result tensors (reused across calls).  The host
    inputs should be pinned."""

    def __init__(self, like: dict, *, chunk: int = 64, out_dtype=None, pieces: int = 4,
                 device="cuda"):
        q, v = like["q"], like["v"]
        B, T, H, dk = q.shape
        dv = v.shape[-1]
        odt = out_dtype or q.dtype
        self.pieces = pieces
        self.out_h = torch.empty((B, T, H, dv), dtype=odt, pin_memory=True)
        self.fin_h = torch.empty((B, H, dk, dv), dtype=torch.float32, pin_memory=True)
        gate = _gate_of(like["log_alpha"], (B, T, H), dk)
        self.desc = chunk_desc(B, T, H, dk, dv, _DT[q.dtype], _DT[odt], gate, chunk)
        self.with_init = like.get("init_state") is not None
        n = ctypes.c_size_t(0)
        rc = _lib.dr_chunk_fwd_host_dev_bytes(ctypes.byref(self.desc), pieces, ctypes.byref(n))
        if rc != DR_OK:
            raise DrError(rc, "dr_chunk_fwd_host_dev_bytes")
        self.dev = torch.empty(n.value + 256, dtype=torch.uint8, device=device)
        self.dev_off = (-self.dev.data_ptr()) % 256     # 256-byte aligned start
        self.dev_bytes = n.value
        self.h2d_bytes = sum(t.numel() * t.element_size() for t in like.values()
                             if t is not None)
        self.d2h_bytes = (self.out_h.numel() * self.out_h.element_size()
                          + self.fin_h.numel() * self.fin_h.element_size())

    def __call__(self, host: dict, sync: bool = True):
        for t in host.values():
            if t is not None and t.is_cuda:
                raise ValueError("HostChunkRunner takes host tensors")
        rc = _lib.dr_chunk_fwd_host(
            ctypes.byref(self.desc), self.pieces, _ptr(host["q"]), _ptr(host["k"]), _ptr(host["v"]),
            _ptr(host["log_alpha"]), _ptr(host["beta"]), _ptr(host.get("init_state")),
            _ptr(self.out_h), _ptr(self.fin_h),
            ctypes.c_void_p(self.dev.data_ptr() + self.dev_off), self.dev_bytes,
            _stream_handle(None))
        if rc != DR_OK:
            raise DrError(rc, "dr_chunk_fwd_host")
        if sync:
            torch.cuda.current_stream().synchronize()
        return self.out_h, self.fin_h


def chunk_fwd_host(q, k, v, log_alpha, beta, init_state=None, *, chunk: int = 64,
                   out_dtype=None, pieces: int = 4):
    """One-shot end-to-end call for host tensors (see HostChunkRunner)."""
    like = {"q": q, "k": k, "v": v, "log_alpha": log_alpha, "beta": beta,
            "init_state": init_state}
    return HostChunkRunner(like, chunk=chunk, out_dtype=out_dtype, pieces=pieces)(like)
