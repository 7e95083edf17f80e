"""Benchmark of the gated delta rule chunk forward and decode step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]

One step = one dr_chunk_fwd call over the Gated DeltaNet workload B=8, H=16, T=4096,
d_k=d_v=128 (bf16 q/k/v/beta, fp32 scalar log alpha, zero initial state, output and final
state returned), inputs resident in HBM.  `value` is whole-job tokens/s (B*T tokens per
call per GPU, summed over GPUs; every rank runs its own independent batch: weak scaling,
no collective on the data path).  The decode step (B=256, H=32, 512 MiB fp32 state, 64
consecutive steps, scalar and per-channel gate) is timed in the same run and reported in
GB/s against the HBM roofline, as are the KDA and long-context chunk workloads.

`--impl reference` times the fp64 CPU oracle instead (on a bounded sample of the same
workload, on this host's cores) and prints the same line with "impl": "reference".
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "tokens/s gated-delta chunk fwd (T=4096,H=16,d=128) & decode GB/s; % roofline"
HEADLINE = "gdn_bf16_B8_H16_T4096_d128"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# GB300 HBM3e datasheet bandwidth (GB/s): reported beside the measured-copy fraction, since
# a streaming in-place kernel can move bytes slightly faster than the copy that measured
# the peak.
HBM_NOMINAL_GBS = 7900.0

# DRAM traffic per launch (read + write bytes) of the dominant kernel, from one ncu capture
# of the headline's launch shape (128 chains) at half its head-tokens (B8 H16 T2048); the
# kernel's traffic is proportional to head-tokens, so the figure is twice the captured one.  Valid only while the kernel
# sources hash to `src` (moved only for edits that leave the compiled kernel byte-identical); otherwise the bench
# reports null.
TRAFFIC = {"chunk_fwd": {"bytes": 2 * (203137280 + 49185280), "src": "c4ff1e6ef8947858"}}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return PEAKS_FALLBACK, "fallback"


# Sources of the headline kernel (chunk_tc_kernel): the traffic figure below was captured
# from these; it is reported only while they are unchanged.
HEADLINE_SOURCES = ("chunk_tc.cu", "tc_common.cuh", "umma.cuh", "common.cuh", "chunk_layout.h")


def csrc_hash():
    h = hashlib.sha256()
    d = os.path.join(ROOT, "gated_delta_rule_15_gb300", "csrc")
    for name in HEADLINE_SOURCES:
        with open(os.path.join(d, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def tc_path(w):
    """The fused tensor-core kernel serves bf16, d_k = d_v = 128, C = 64, scalar or no gate."""
    return (w.dtype == "bf16" and w.dk == 128 and w.dv == 128 and w.chunk == 64
            and w.gate in ("none", "scalar") and w.T > 0)


def kda_path(w):
    """The prep + state tensor-core pair serves the same shapes with the per-channel gate."""
    return (w.dtype == "bf16" and w.dk == 128 and w.dv == 128 and w.chunk == 64
            and w.gate == "channel" and w.T > 0)


def path_kernels(w):
    """Kernels one dr_chunk_fwd call launches for workload w, in launch order (the segment
    rule mirrors the library's: chains <= 76 with >= 32 chunks are split for 152 SMs)."""
    if tc_path(w):
        nc, bh = -(-w.T // w.chunk), w.B * w.H
        if bh <= 76 and nc >= 32 and min(nc // 16, 152 // bh) >= 2:
            return ["gdn_prep_kernel", "gdn_chain_kernel (segment end states)", "seg_combine_kernel",
                    "gdn_chain_kernel (segment outputs)"]
        return ["chunk_tc_kernel"]
    if kda_path(w):
        nc, bh = -(-w.T // w.chunk), w.B * w.H
        if bh <= 76 and nc >= 32 and min(nc // 16, 152 // bh) >= 2:
            return ["kda_prep_kernel", "kda_state_kernel (segment end states)", "seg_combine_kernel",
                    "kda_state_kernel (segment outputs)"]
        return ["kda_prep_kernel", "kda_state_kernel"]
    return ["chunk_prep_kernel", "chunk_state_kernel"]


# ------------------------------------------------------------------ algorithmic counts
def chunk_bytes(w):
    """Each input read once, each output written once; a zero initial state is not read."""
    e = 2 if w.dtype == "bf16" else 4
    ht = w.B * w.T * w.H
    b = ht * (2 * w.dk + w.dv) * e + ht * e + ht * w.dv * e   # q, k, v, beta, out
    b += ht * 4 * (w.dk if w.gate == "channel" else (1 if w.gate == "scalar" else 0))
    st = w.B * w.H * w.dk * w.dv * 4
    return b + st + (st if w.init_state else 0)


def chunk_flops(w):
    """GEMM flops as issued by the chunk form: per chunk C^2 (6 dk + 4 dv) + 6 C dk dv."""
    C = w.chunk
    nchunks = w.B * w.H * ((w.T + C - 1) // C)
    return nchunks * (C * C * (6 * w.dk + 4 * w.dv) + 6 * C * w.dk * w.dv)


def decode_bytes(w):
    e = 2 if w.dtype == "bf16" else 4
    bh = w.B * w.H
    b = 2 * bh * w.dk * w.dv * 4                       # state read + write
    b += bh * (2 * w.dk + w.dv) * e + bh * e + bh * w.dv * e   # q, k, v, beta, out
    b += bh * 4 * (w.dk if w.gate == "channel" else (1 if w.gate == "scalar" else 0))
    return b


# ------------------------------------------------------------------ clocks sampler
class ClockSampler:
    """nvidia-smi samples every 20 ms around the soak and the timed region."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index, self.rows, self.proc = index, [], None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([x.strip() for x in line.split(",")])

    def __exit__(self, *exc):
        time.sleep(0.25)
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[0]) for r in self.rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4)
                          if len(r) > 3 + i and r[3 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(self.rows)}


# ------------------------------------------------------------------ distributed
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x, world):
    """The largest of every rank's x (a time: the slowest rank sets the job's)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_seed(rank):
    """Each rank draws its own batch (weak scaling over independent batches)."""
    return 1000 * rank


def job_throughput(units_per_rank, ms_max, world):
    """Units all ranks processed per second, over the slowest rank's time."""
    return world * units_per_rank / (ms_max * 1e-3)


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ native arm
def time_calls(fn, steps, warmup, world, sampler_index=None, soak_s=1.0):
    """CUDA-event time of `steps` calls on the current stream after `warmup` calls.

    With a sampler, nvidia-smi records clocks every 20 ms from before a ~`soak_s` second
    back-to-back run of the same call (untimed) through the end of the timed calls, so the
    samples describe the GPU under this load; the timed calls follow the soak directly."""
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    barrier(world)
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(sampler_index) if sampler_index is not None else None
    if sampler:
        sampler.__enter__()
        # soak: repeat the call until ~soak_s seconds of device time are queued and done
        e0.record(s)
        fn()
        e1.record(s)
        torch.cuda.synchronize()
        per = max(e0.elapsed_time(e1), 1e-3)
        for _ in range(max(1, int(soak_s * 1e3 / per))):
            fn()
    else:
        torch.cuda.synchronize()
    e0.record(s)
    for _ in range(steps):
        fn()
    e1.record(s)
    torch.cuda.synchronize()
    if sampler:
        sampler.__exit__(None, None, None)
    barrier(world)
    ms = e0.elapsed_time(e1) / steps
    return max_over_ranks(ms, world), (sampler.summary() if sampler else None)


def bench_chunk(w, steps, warmup, world, sample_clocks=None, seed=0):
    import torch
    from gated_delta_rule_15_gb300 import dr, inputs
    d = inputs.workload_inputs(w, seed=seed)
    g = {k: (None if t is None else t.cuda()) for k, t in d.items()}
    B, T, H = w.B, w.T, w.H
    out = torch.empty((B, T, H, w.dv), dtype=g["q"].dtype, device="cuda")
    fin = torch.empty((B, H, w.dk, w.dv), dtype=torch.float32, device="cuda")
    desc = dr.chunk_desc(B, T, H, w.dk, w.dv, dr._DT[g["q"].dtype], dr._DT[out.dtype],
                         inputs.GATE_CODE[w.gate], w.chunk)
    nws = dr.workspace_bytes(desc)
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda") if nws else None

    def call():
        dr.chunk_fwd(g["q"], g["k"], g["v"], g["log_alpha"], g["beta"], g["init_state"],
                     chunk=w.chunk, out=out, final_state=fin, workspace=ws)

    ms, clocks = time_calls(call, steps, warmup, world, sample_clocks)
    return {"ms": ms, "clocks": clocks, "host_inputs": d, "workspace_bytes": nws}


def bench_chunk_e2e(w, d, steps, warmup, world):
    """Same metric through the C-ABI call for host buffers (dr_chunk_fwd_host): per step
    the H2D copies of the inputs from pinned memory, the forward and the D2H copies of out
    and final_state, the sequence in 4 time pieces so that copies and kernels overlap."""
    import torch
    from gated_delta_rule_15_gb300 import dr
    host = {k: (None if t is None else t.pin_memory()) for k, t in d.items()}
    runner = dr.HostChunkRunner(host, chunk=w.chunk)
    ms, _ = time_calls(lambda: runner(host, sync=False), steps, warmup, world)
    return ms, runner.h2d_bytes, runner.d2h_bytes


def bench_bwd(w, steps, warmup, world):
    """dr_chunk_bwd on the workload (d_out ~ N(0, 1) in the output dtype, no final-state
    gradient): ms per call."""
    import torch
    from gated_delta_rule_15_gb300 import dr, inputs
    d = inputs.workload_inputs(w)
    g = {k: (None if t is None else t.cuda()) for k, t in d.items()}
    gen = torch.Generator().manual_seed(1)
    dout = torch.randn((w.B, w.T, w.H, w.dv), generator=gen).to(g["q"].dtype).cuda()
    desc = dr.chunk_desc(w.B, w.T, w.H, w.dk, w.dv, dr._DT[g["q"].dtype], dr._DT[dout.dtype],
                         inputs.GATE_CODE[w.gate], w.chunk)
    ws = torch.empty(dr.bwd_workspace_bytes(desc), dtype=torch.uint8, device="cuda")
    call = lambda: dr.chunk_bwd(g["q"], g["k"], g["v"], g["log_alpha"], g["beta"],
                                g["init_state"], dout, None, chunk=w.chunk, workspace=ws)
    ms, _ = time_calls(call, steps, warmup, world)
    return ms


def bench_fused(w, steps, warmup, world):
    """dr_chunk_fwd_ex with every fused neighbour (raw q, k, beta logits, SiLU gate z):
    ms per call."""
    import torch
    from gated_delta_rule_15_gb300 import dr, inputs
    d = inputs.chunk_inputs(w.B, w.T, w.H, w.dk, w.dv, gate=w.gate, dtype=w.dtype,
                            init_state=w.init_state, log_alpha_range=w.log_alpha_range, raw=True)
    g = {k: (None if t is None else t.cuda()) for k, t in d.items()}
    out = torch.empty((w.B, w.T, w.H, w.dv), dtype=g["q"].dtype, device="cuda")
    fin = torch.empty((w.B, w.H, w.dk, w.dv), dtype=torch.float32, device="cuda")
    desc = dr.chunk_desc(w.B, w.T, w.H, w.dk, w.dv, dr._DT[g["q"].dtype], dr._DT[out.dtype],
                         inputs.GATE_CODE[w.gate], w.chunk)
    ws = torch.empty(max(16, dr.ex_workspace_bytes(desc, dr.DR_FUSE_ALL)), dtype=torch.uint8, device="cuda")
    call = lambda: dr.chunk_fwd(g["q"], g["k"], g["v"], g["log_alpha"], g["beta"],
                                g["init_state"], chunk=w.chunk, out=out, final_state=fin,
                                workspace=ws, qk_l2norm=True, beta_sigmoid=True, z=g["z"])
    ms, _ = time_calls(call, steps, warmup, world)
    return ms


def bench_decode(w, steps, warmup, world):
    import torch
    from gated_delta_rule_15_gb300 import dr, inputs
    s = inputs.decode_workload_inputs(w)
    st = s["state"].cuda()
    g = {k: (None if t is None else t.cuda()) for k, t in s.items() if k != "state"}
    out = torch.empty((w.B, w.H, w.dv), dtype=g["q"].dtype, device="cuda")
    n = g["q"].shape[0]
    i = [0]

    def call():
        t = i[0] % n
        i[0] += 1
        dr.recurrent_step(g["q"][t], g["k"][t], g["v"][t],
                          None if g["log_alpha"] is None else g["log_alpha"][t],
                          g["beta"][t], st, out=out)

    ms, _ = time_calls(call, steps, warmup, world)
    return ms


def cpu_baseline_chunk(w, d, budget_s=20.0):
    """The fp64 oracle, as it stands, on whole chains of the same workload, on this host's
    cores; runs chains until about `budget_s` seconds have passed."""
    import oracle
    cores = oracle.default_threads()
    done_ht, t0 = 0, time.perf_counter()
    chains = 0
    # batches of 16 chains (one batch row at a time) until the budget is used
    for b in range(w.B):
        pick = lambda t: None if t is None else t[b:b + 1]
        s0 = None if d["init_state"] is None else d["init_state"][b:b + 1]
        oracle.forward(pick(d["q"]), pick(d["k"]), pick(d["v"]), pick(d["log_alpha"]),
                       pick(d["beta"]), s0, nthreads=cores)
        done_ht += w.T * w.H
        chains += w.H
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return {"value": done_ht / w.H / dt, "unit": "tokens/s", "cores": cores,
            "kind": "oracle",
            "sample": f"{chains} of {w.B * w.H} (b,h) chains x T={w.T} tokens of {w.name} "
                      f"(fp64 token loop, {dt:.1f} s)"}


def run_native(args):
    import torch
    from gated_delta_rule_15_gb300 import inputs
    world, rank, local = dist_setup()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    pk, pk_kind = peaks()
    hbm, tc = pk["hbm_gbs"], pk["bf16_tflops"]

    w = inputs.WORKLOADS[HEADLINE]
    r = bench_chunk(w, args.steps, args.warmup, world, sample_clocks=local, seed=rank_seed(rank))
    ms = r["ms"]
    tokens = w.B * w.T
    value = job_throughput(tokens, ms, world)
    byts, flops = chunk_bytes(w), chunk_flops(w)
    ach_gbs = byts / (ms * 1e-3) / 1e9
    e2e_ms, h2d, d2h = bench_chunk_e2e(w, r["host_inputs"], max(2, args.steps // 2),
                                       max(3, args.warmup), world)
    kernels = path_kernels(w)
    launches_per_call = len(kernels)

    extra = {}
    if not args.quick:
        fms = bench_fused(w, max(2, args.steps // 3), 3, world)
        extra["fused_neighbours_" + w.name] = {
            "what": "dr_chunk_fwd_ex: q/k L2 norm, beta = sigmoid(logit), SiLU output gate",
            "ms_per_call": round(fms, 4), "tokens_per_s": w.B * w.T / (fms * 1e-3),
            "vs_plain": round(fms / ms, 3)}
        bms = bench_bwd(w, 2, 3, world)
        extra["backward_" + w.name] = {
            "what": "dr_chunk_bwd (fp32 sums, TF32 tensor-core tiles): every input gradient",
            "ms_per_call": round(bms, 3), "tokens_per_s": w.B * w.T / (bms * 1e-3),
            "vs_forward": round(bms / ms, 1)}
        for name in ("kda_bf16_B4_H32_T8192_d128", "gdn_bf16_B1_H16_T65536_d128_init",
                     "kda_bf16_B1_H16_T65536_d128_init"):
            wx = inputs.WORKLOADS[name]
            rx = bench_chunk(wx, max(2, args.steps // 3), 3, world)
            bx, fx = chunk_bytes(wx), chunk_flops(wx)
            extra[name] = {
                "ms_per_call": round(rx["ms"], 4),
                "tokens_per_s": wx.B * wx.T / (rx["ms"] * 1e-3),
                "gbs": bx / (rx["ms"] * 1e-3) / 1e9,
                "hbm_frac": bx / (rx["ms"] * 1e-3) / 1e9 / hbm,
                "tflops": fx / (rx["ms"] * 1e-3) / 1e12,
                "tensor_frac": fx / (rx["ms"] * 1e-3) / 1e12 / tc,
                "kernels": path_kernels(wx)}
            del rx
    decode = {}
    for name in ("decode_scalar_B256_H32_d128", "decode_channel_B256_H32_d128"):
        wd = inputs.DECODE_WORKLOADS[name]
        dms = bench_decode(wd, wd.steps, 3, world)
        db = decode_bytes(wd)
        decode[name] = {"ms_per_step": round(dms, 5), "steps": wd.steps,
                        "gbs": db / (dms * 1e-3) / 1e9,
                        "hbm_frac": db / (dms * 1e-3) / 1e9 / hbm,
                        "hbm_frac_nominal": db / (dms * 1e-3) / 1e9 / HBM_NOMINAL_GBS,
                        "tokens_per_s": wd.B / (dms * 1e-3),
                        "bytes_per_step": db}

    if rank != 0:
        return
    cpu = cpu_baseline_chunk(w, r["host_inputs"], budget_s=args.cpu_budget)
    src = csrc_hash()
    tr = TRAFFIC.get("chunk_fwd")
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded; q,k L2-normalised, beta=sigmoid(N(0,1)), "
                                 "log alpha=-U(0.001,0.1))",
        "config": {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "dk": w.dk, "dv": w.dv,
                   "gate": w.gate, "chunk": w.chunk, "init_state": w.init_state,
                   "parallelism": f"dp{world} (independent batches)",
                   "l2": f"inputs larger than L2 ({byts / 1e6:.0f} MB per call); no flush"},
        "roofline": {"bound": "hbm", "achieved": ach_gbs, "peak": hbm, "unit": "GB/s",
                     "frac": ach_gbs / hbm, "peak_source": pk_kind,
                     "traffic": (tr["bytes"] if tr and tr["src"] == src else None),
                     "kernel": " + ".join(kernels),
                     "algorithmic_bytes": byts,
                     "tensor_tflops": flops / (ms * 1e-3) / 1e12,
                     "tensor_frac": flops / (ms * 1e-3) / 1e12 / tc},
        "cpu_baseline": cpu,
        "e2e": {"value": job_throughput(tokens, e2e_ms, world), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms},
        "gpu_launches": launches_per_call * args.steps,
        "clocks": r["clocks"],
        "decode": decode,
        "other_workloads": extra,
        "csrc": src,
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ reference arm
def run_reference(args):
    """The oracle as it stands, timed on this host's cores, on the native arm's workload,
    metric and unit.  Each step is a bounded sample: one batch row of the workload (H whole
    (b, h) chains x T tokens), the rows taken in turn, so that the oracle's tasks (one per
    chain) cover the host's cores."""
    world, rank, _ = dist_setup()
    if rank != 0:
        return
    import oracle
    from gated_delta_rule_15_gb300 import inputs
    w = inputs.WORKLOADS[HEADLINE]
    d = inputs.workload_inputs(w)
    cores = oracle.default_threads()
    rows = [0]

    def run():
        b = rows[0] % w.B
        rows[0] += 1
        pick = lambda t: None if t is None else t[b:b + 1]
        s0 = None if d["init_state"] is None else d["init_state"][b:b + 1]
        oracle.forward(pick(d["q"]), pick(d["k"]), pick(d["v"]), pick(d["log_alpha"]),
                       pick(d["beta"]), s0, nthreads=cores)

    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    dt = (time.perf_counter() - t0) / args.steps
    value = w.T / dt          # tokens (of H heads each) per second
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (same recipe as the native arm)",
        "config": {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "dk": w.dk, "dv": w.dv,
                   "gate": w.gate, "sample_per_step": f"1 batch row = {w.H} (b,h) chains x {w.T} tokens"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"one batch row ({w.H} whole (b,h) chains x T={w.T}) of {w.name} per step"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--quick", action="store_true", help="headline workload and decode only")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)   # at least 3 untimed warm-up calls, always
    if args.impl == "reference":
        run_reference(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
