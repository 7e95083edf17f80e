"""Run one kernel of the library a few times on a chosen workload, for profilers.

    python profile_case.py --what decode --B 128 --iters 3
    python profile_case.py --what chunk \
        --workload gdn_bf16_B8_H16_T4096_d128 --B 2 --iters 3

Sizes default to the named workload; --B / --T / --H shrink it (keep inputs larger than
L2 for meaningful DRAM counters).  Prints the CUDA-event time per launch (a number taken
under a profiler is not a benchmark result).
"""
from __future__ import annotations

import argparse
import dataclasses
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))


def with_raw(make, fl):
    """Prepared inputs, with the raw q, k / beta logits / z of the same draw for the
    fused neighbours in `fl`."""
    d = make(False)
    if fl:
        raw = make(True)
        if "l2" in fl:
            d["q"], d["k"] = raw["q"], raw["k"]
        if "sigmoid" in fl:
            d["beta"] = raw["beta"]
        d["z"] = raw["z"]
    return d


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--what", choices=["chunk", "bwd", "decode"], required=True)
    ap.add_argument("--workload", default=None)
    ap.add_argument("--B", type=int, default=None)
    ap.add_argument("--T", type=int, default=None)
    ap.add_argument("--H", type=int, default=None)
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--fused", nargs="?", const="l2,sigmoid,silu", default="",
                    help="raw inputs with the fused neighbours listed (default: all of "
                         "l2, sigmoid, silu)")
    args = ap.parse_args()

    import torch
    from gated_delta_rule_15_gb300 import dr, inputs

    torch.cuda.set_device(0)
    fl = set(filter(None, args.fused.split(",")))
    if fl - {"l2", "sigmoid", "silu"}:
        ap.error(f"unknown fused neighbours {fl}")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if args.what == "bwd":
        w = inputs.WORKLOADS[args.workload or "gdn_bf16_B8_H16_T4096_d128"]
        w = dataclasses.replace(w, **{k: getattr(args, k) for k in ("B", "T", "H")
                                      if getattr(args, k) is not None})
        d = inputs.workload_inputs(w)
        g = {k: (None if t is None else t.cuda()) for k, t in d.items()}
        gen = torch.Generator().manual_seed(1)
        dout = torch.randn((w.B, w.T, w.H, w.dv), generator=gen).to(g["q"].dtype).cuda()
        dB = dr.chunk_desc(w.B, w.T, w.H, w.dk, w.dv, dr._DT[g["q"].dtype], dr._DT[dout.dtype],
                           inputs.GATE_CODE[w.gate], w.chunk)
        ws = torch.empty(dr.bwd_workspace_bytes(dB), dtype=torch.uint8, device="cuda")
        run = lambda: dr.chunk_bwd(g["q"], g["k"], g["v"], g["log_alpha"], g["beta"],
                                   g["init_state"], dout, None, chunk=w.chunk, workspace=ws)
    elif args.what == "chunk":
        w = inputs.WORKLOADS[args.workload or "gdn_bf16_B8_H16_T4096_d128"]
        w = dataclasses.replace(w, **{k: getattr(args, k) for k in ("B", "T", "H")
                                      if getattr(args, k) is not None})
        mk = lambda raw: inputs.chunk_inputs(w.B, w.T, w.H, w.dk, w.dv, gate=w.gate,
                                             dtype=w.dtype, init_state=w.init_state,
                                             log_alpha_range=w.log_alpha_range, raw=raw)
        d = with_raw(mk, fl)
        g = {k: (None if t is None else t.cuda()) for k, t in d.items()}
        fz = dict(qk_l2norm="l2" in fl, beta_sigmoid="sigmoid" in fl,
                  z=g["z"] if "silu" in fl else None) if fl else {}
        run = lambda: dr.chunk_fwd(g["q"], g["k"], g["v"], g["log_alpha"], g["beta"],
                                   g["init_state"], chunk=w.chunk, **fz)
    else:
        w = inputs.DECODE_WORKLOADS[args.workload or "decode_scalar_B256_H32_d128"]
        w = dataclasses.replace(w, **({"B": args.B} if args.B else {}))
        s = with_raw(lambda raw: inputs.decode_inputs(
            w.B, w.H, w.dk, w.dv, max(1, args.iters), gate=w.gate, dtype=w.dtype,
            log_alpha_range=w.log_alpha_range, raw=raw), fl)
        st = s["state"].cuda()
        g = {k: (None if t is None else t.cuda()) for k, t in s.items() if k != "state"}
        i = [0]

        def run():
            t = i[0] % g["q"].shape[0]
            i[0] += 1
            la = None if g["log_alpha"] is None else g["log_alpha"][t]
            fz = dict(qk_l2norm="l2" in fl, beta_sigmoid="sigmoid" in fl,
                      z=g["z"][t] if "silu" in fl else None) if fl else {}
            dr.recurrent_step(g["q"][t], g["k"][t], g["v"][t], la, g["beta"][t], st, **fz)
    run()
    torch.cuda.synchronize()
    e0.record()
    for _ in range(args.iters):
        run()
    e1.record()
    torch.cuda.synchronize()
    tag = f" fused[{args.fused}]" if fl else ""
    print(f"{w.name}{tag} {dataclasses.asdict(w)}: {e0.elapsed_time(e1) / args.iters:.4f} ms/launch")


if __name__ == "__main__":
    main()
