"""Seeded synthetic inputs for the gated delta rule.

This module holds none of the method's arithmetic: it only draws random tensors and
applies the input recipe (per-token L2 normalisation of q and k, beta = sigmoid of a
Gaussian logit, log alpha drawn directly, casts to the storage dtype).  Both the tests'
oracle side and the CUDA side take their inputs from here and nowhere else.

Recipe (one CPU torch.Generator seeded once per workload, draws in this order, fp32):
    q, k ~ N(0, 1) [B,T,H,dk];  v ~ N(0, 1) [B,T,H,dv];  beta-logits ~ N(0, 1) [B,T,H];
    log alpha = -Uniform(lo, hi)  ([B,T,H] scalar gate, [B,T,H,dk] per-channel gate,
    not drawn without a gate);  initial state ~ N(0, 0.02^2) [B,H,dk,dv] where used.
Then q <- q/|q|, k <- k/|k| per (b, t, h) in fp32, beta = sigmoid(logits), and q, k, v,
beta are cast to the storage dtype (round to nearest even); log alpha and the state stay
fp32.

Raw inputs for the fused neighbours (`raw=True`): the same draws, then z ~ N(0, 1)
[B,T,H,dv]; q, k are stored unnormalised (scaled by a per-token factor ~ U(0.25, 4), drawn
after z, so that the norms vary), beta keeps its logits, and z is stored in the storage
dtype.  The normalisation, the sigmoid and the output gate are then the library's work.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

GATES = ("none", "scalar", "channel")
GATE_CODE = {"none": 0, "scalar": 1, "channel": 2}
DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class ChunkWorkload:
    """One chunk-forward workload: sizes, gate kind, storage dtype, initial state."""
    name: str
    B: int
    T: int
    H: int
    dk: int
    dv: int
    gate: str = "scalar"
    dtype: str = "bf16"
    init_state: bool = False
    chunk: int = 64
    log_alpha_range: tuple = (0.001, 0.1)

    def head_tokens(self) -> int:
        return self.B * self.T * self.H


@dataclass(frozen=True)
class DecodeWorkload:
    """A run of single-token decode steps against a resident fp32 state."""
    name: str
    B: int
    H: int
    dk: int
    dv: int
    gate: str = "scalar"
    dtype: str = "bf16"
    steps: int = 64
    log_alpha_range: tuple = (0.001, 0.1)


# The workloads the method is measured on (single sequence fp32; Gated DeltaNet at
# T = 4096; KDA per-channel gate at T = 8192; long-context Gated DeltaNet with a carried
# state at T = 65536; batched decode against a 512 MiB state), and the long-context shape
# with the per-channel gate, which exercises that gate's segment-parallel form.
WORKLOADS = {
    "gdn_f32_B1_H1_T256_d64": ChunkWorkload(
        "gdn_f32_B1_H1_T256_d64", B=1, T=256, H=1, dk=64, dv=64, gate="scalar",
        dtype="f32"),
    "gdn_bf16_B8_H16_T4096_d128": ChunkWorkload(
        "gdn_bf16_B8_H16_T4096_d128", B=8, T=4096, H=16, dk=128, dv=128,
        gate="scalar", dtype="bf16"),
    "kda_bf16_B4_H32_T8192_d128": ChunkWorkload(
        "kda_bf16_B4_H32_T8192_d128", B=4, T=8192, H=32, dk=128, dv=128,
        gate="channel", dtype="bf16"),
    "gdn_bf16_B1_H16_T65536_d128_init": ChunkWorkload(
        "gdn_bf16_B1_H16_T65536_d128_init", B=1, T=65536, H=16, dk=128, dv=128,
        gate="scalar", dtype="bf16", init_state=True),
    "kda_bf16_B1_H16_T65536_d128_init": ChunkWorkload(
        "kda_bf16_B1_H16_T65536_d128_init", B=1, T=65536, H=16, dk=128, dv=128,
        gate="channel", dtype="bf16", init_state=True),
}
DECODE_WORKLOADS = {
    "decode_scalar_B256_H32_d128": DecodeWorkload(
        "decode_scalar_B256_H32_d128", B=256, H=32, dk=128, dv=128, gate="scalar"),
    "decode_channel_B256_H32_d128": DecodeWorkload(
        "decode_channel_B256_H32_d128", B=256, H=32, dk=128, dv=128, gate="channel"),
}


def _log_alpha(g, shape, lo, hi):
    return -(lo + (hi - lo) * torch.rand(shape, generator=g))


def chunk_inputs(B, T, H, dk, dv, *, gate="scalar", dtype="bf16", init_state=False,
                 seed=0, log_alpha_range=(0.001, 0.1), unit_keys=True, raw=False):
    """Draw one chunk-forward problem on the CPU.  Returns a dict with q, k, v
    ([B,T,H,d], storage dtype), beta ([B,T,H], storage dtype), log_alpha (fp32 or
    None) and init_state (fp32 [B,H,dk,dv] or None); with `raw`, also z ([B,T,H,dv],
    storage dtype), and q, k, beta as described in the module's recipe."""
    if gate not in GATES:
        raise ValueError(gate)
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((B, T, H, dk), generator=g)
    k = torch.randn((B, T, H, dk), generator=g)
    v = torch.randn((B, T, H, dv), generator=g)
    bl = torch.randn((B, T, H), generator=g)
    lo, hi = log_alpha_range
    if gate == "scalar":
        la = _log_alpha(g, (B, T, H), lo, hi)
    elif gate == "channel":
        la = _log_alpha(g, (B, T, H, dk), lo, hi)
    else:
        la = None
    s0 = 0.02 * torch.randn((B, H, dk, dv), generator=g) if init_state else None
    dt = DTYPES[dtype]
    if raw:
        z = torch.randn((B, T, H, dv), generator=g)
        q = q * (0.25 + 3.75 * torch.rand((B, T, H, 1), generator=g))
        k = k * (0.25 + 3.75 * torch.rand((B, T, H, 1), generator=g))
        return {"q": q.to(dt).contiguous(), "k": k.to(dt).contiguous(),
                "v": v.to(dt).contiguous(), "beta": bl.to(dt).contiguous(),
                "log_alpha": None if la is None else la.contiguous(),
                "init_state": None if s0 is None else s0.contiguous(),
                "z": z.to(dt).contiguous()}
    if unit_keys:
        q = q / q.norm(dim=-1, keepdim=True)
        k = k / k.norm(dim=-1, keepdim=True)
    beta = torch.sigmoid(bl)
    return {"q": q.to(dt).contiguous(), "k": k.to(dt).contiguous(),
            "v": v.to(dt).contiguous(), "beta": beta.to(dt).contiguous(),
            "log_alpha": None if la is None else la.contiguous(),
            "init_state": None if s0 is None else s0.contiguous()}


def workload_inputs(w: ChunkWorkload, seed=0):
    return chunk_inputs(w.B, w.T, w.H, w.dk, w.dv, gate=w.gate, dtype=w.dtype,
                        init_state=w.init_state, seed=seed,
                        log_alpha_range=w.log_alpha_range)


def decode_inputs(B, H, dk, dv, steps, *, gate="scalar", dtype="bf16", seed=0,
                  log_alpha_range=(0.001, 0.1), raw=False):
    """Draw `steps` single-token decode inputs and the initial state.  q, k [steps,B,H,dk],
    v [steps,B,H,dv], beta [steps,B,H], log_alpha [steps,B,H] or [steps,B,H,dk] (None
    without a gate), state [B,H,dk,dv] fp32 ~ N(0, 0.02^2); with `raw`, z [steps,B,H,dv]
    and raw q, k, beta as for chunk_inputs."""
    d = chunk_inputs(steps, B, H, dk, dv, gate=gate, dtype=dtype, init_state=False,
                     seed=seed, log_alpha_range=log_alpha_range, raw=raw)
    g = torch.Generator().manual_seed(seed + 1)
    state = 0.02 * torch.randn((B, H, dk, dv), generator=g)
    d["state"] = state.contiguous()
    del d["init_state"]
    return d


def decode_workload_inputs(w: DecodeWorkload, seed=0, steps=None):
    return decode_inputs(w.B, w.H, w.dk, w.dv, steps or w.steps, gate=w.gate,
                         dtype=w.dtype, seed=seed, log_alpha_range=w.log_alpha_range)
