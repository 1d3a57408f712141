"""Benchmark: PaTH forward TFLOP/s (B8 H12 L4096 d128 bf16) and decode us/step at a 32K cache.

One step = one PaTH forward over the 760M-shaped workload (B8 H12 L4096 d128
bf16, inputs resident in HBM) followed by a 256-token decode sequence over the
32K-token cache (B64 H12 d128 bf16), i.e. the whole hot path once.  ``value``
is the forward's attention-equivalent TFLOP/s (4 B H d L^2 / 2 FLOP per call);
decode is reported alongside in us/step.  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun every rank runs its own replica of the workload (the path
shards by (batch, head) with no exchange, so there is no collective on the
data path); the barrier and max-over-ranks timing use torch.distributed.
``--impl reference`` times the fp64 CPU oracle on a bounded sample instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

FWD_NAME = "path760m_bf16"
DEC_NAME = "decode32k_bf16"
METRIC = "PaTH fwd TFLOP/s (L=4096,d=128,bf16) & decode µs/step @32K cache, % roofline"


def _traffic(kernel: str, units: float):
    """DRAM bytes per launch from the committed ncu capture (profiles/traffic.json), scaled
    to `units`; None when the kernel's source changed since the capture."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        t = json.load(open(p))[kernel]
        src = open(os.path.join(ROOT, t["source"]), "rb").read()
    except (OSError, KeyError, ValueError):
        return None
    if hashlib.sha256(src).hexdigest()[:16] != t["sha256_16"]:
        return None
    return t["captured_bytes"] * units / t["captured_units"]


# GB300 nominal figures, reported beside the measured peaks: dense bf16 tensor
# throughput and the ~8 TB/s HBM3e bandwidth the targets are stated against
SPEC_BF16_TFLOPS = 2250.0
SPEC_HBM_GBS = 8000.0


def fwd_tensor_flops(B, H, L, d, visited=None):
    """Executed tensor-core FLOPs of one bf16 forward scan: per (query tile, earlier key block) pair
    the fused product [S | q~] += bf16(q~) [khat ; P - I]^T (2*128*(128+d)*d) and O += P V
    (2*128*128*d); per diagonal tile S = Q K^T + Y (-Z)^T (2*128*128*(d+128)) and P V.  `visited`:
    (tile, block) pairs visited including the diagonal (default: the full causal triangle)."""
    nt = -(-L // 128)
    tiles = B * H * nt
    pairs = B * H * nt * (nt + 1) // 2 if visited is None else visited
    blk = 2 * 128 * (128 + d) * d + 2 * 128 * 128 * d
    diag = 2 * 128 * 128 * (d + 128) + 2 * 128 * 128 * d
    return float((pairs - tiles) * blk + tiles * diag)


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), d.get("bf16_tflops_sustained"), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        load = [s for s in sm if s > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(load), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- CPU oracle leg
def oracle_sample(n_heads: int, seed_heads: int = 0):
    """Time the fp64 oracle on n_heads full heads of the forward workload; returns
    (attention-equivalent TFLOP/s, seconds, threads, description)."""
    import numpy as np
    from attention_causal_attn_fwd_gb300 import inputs
    from oracle import oracle as orc
    cfg = inputs.FWD_CONFIGS[FWD_NAME]
    x = cfg.make()
    f = inputs.f64
    rng = np.random.default_rng(seed_heads)
    picks = [(int(rng.integers(0, cfg.B)), int(rng.integers(0, cfg.H))) for _ in range(n_heads)]
    sel = lambda t: np.stack([t[b, h] for b, h in picks])
    args = [sel(f(t)) for t in (x.q, x.k, x.v, x.w, x.beta)]
    orc.build()
    t0 = time.perf_counter()
    orc.path_attn(*args, scale=x.scale)
    dt = time.perf_counter() - t0
    flops = 4.0 * cfg.d * cfg.L * cfg.L / 2.0 * n_heads
    desc = "fp64 oracle, %d full head(s) of %d (B%d H%d L%d d%d), attention-equivalent FLOPs of those heads" % (
        n_heads, cfg.B * cfg.H, cfg.B, cfg.H, cfg.L, cfg.d)
    return flops / dt / 1e12, dt, orc.threads(), desc


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    for _ in range(args.warmup):
        oracle_sample(1)
    times = []
    vals = []
    for s in range(args.steps):
        v, dt, cores, desc = oracle_sample(1, seed_heads=s)
        times.append(dt)
        vals.append(v)
    value = 4.0 * 128 * 4096 * 4096 / 2.0 * args.steps / sum(times) / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sum(times) / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded CPU generator)",
            "config": {"workload": "PaTH forward B8 H12 L4096 d128 (one head per step on the CPU oracle)",
                       "B": 8, "H": 12, "L": 4096, "d": 128},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ----------------------------------------------------------------------------- GPU leg
def run_ours(args, rank, world, local):
    import attention_causal_attn_fwd_gb300 as P
    from attention_causal_attn_fwd_gb300 import inputs

    dev = torch.device("cuda", local)
    hbm_gbs, bf16_tf, bf16_sust, peak_src = _peaks()
    import dataclasses
    fc = inputs.FWD_CONFIGS[FWD_NAME]
    dc = inputs.DECODE_CONFIGS[DEC_NAME]
    if args.fwd_B != fc.B:  # smaller batch, only for profiling captures
        fc = dataclasses.replace(fc, B=args.fwd_B)
    if args.decode_B != dc.B:
        dc = dataclasses.replace(dc, B=args.decode_B)
    x = fc.make()
    q, k, v, w, beta = (t.to(dev) for t in (x.q, x.k, x.v, x.w, x.beta))
    o = torch.empty_like(q)
    ws_f = P.alloc_workspace(P.path_attn_workspace_bytes(fc.B, fc.H, fc.L, fc.d, q.dtype), dev)

    Td = args.decode_steps
    n_max = dc.n0 + Td
    if Td > 0:
        kc, vc = inputs.make_decode_cache(dc.B, dc.H, dc.n0, dc.d, n_max, dc.dtype, dc.seed)
        kc, vc = kc.to(dev), vc.to(dev)
        dq, dk, dv, dw, db = (t.to(dev) for t in inputs.make_decode_steps(dc.B, dc.H, dc.d, Td, dc.dtype, dc.seed))
        od = torch.empty((Td, dc.B, dc.H, dc.d), dtype=kc.dtype, device=dev)
        ws_d = P.alloc_workspace(P.path_decode_workspace_bytes(dc.B, dc.H, n_max, dc.d), dev)

    def mk():
        e = torch.cuda.Event(enable_timing=True)
        e.record()
        return e

    def one_step(rec, s=0):
        # rec: dict of per-step event lists (timed steps), or None (warm-up)
        if rec is not None:
            P.path_debug_set_timing_events(rec["fk0"][s], rec["fk1"][s])
            rec["f0"][s].record()
        P.path_attn_fwd(q, k, v, w, beta, scale=x.scale, out=o, workspace=ws_f)
        if rec is not None:
            rec["f1"][s].record()
        for t in range(Td):
            if rec is not None:
                P.path_debug_set_timing_events(rec["dk0"][s][t], rec["dk1"][s][t])
            P.path_decode_step(dq[t], dk[t], dv[t], dw[t], db[t], kc, vc, dc.n0 + t, scale=dc.d ** -0.5,
                               out=od[t], workspace=ws_d)
        if rec is not None:
            P.path_debug_set_timing_events(None, None)
            rec["d1"][s].record()

    P.path_debug_set_timing_events(None, None)
    for _ in range(args.warmup):
        one_step(None)
    torch.cuda.synchronize()
    rec = {kk: [] for kk in ("f0", "f1", "fk0", "fk1", "d1", "dk0", "dk1")}
    for _ in range(args.steps):
        for kk in ("f0", "f1", "fk0", "fk1", "d1"):
            rec[kk].append(mk())
        rec["dk0"].append([mk() for _ in range(Td)])
        rec["dk1"].append([mk() for _ in range(Td)])
    torch.cuda.synchronize()

    clocks = Clocks(torch.cuda.current_device())
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record()
    for s in range(args.steps):
        one_step(rec, s)
    t_end.record()
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    total_ms = max_over_ranks(t_start.elapsed_time(t_end), world)
    fwd_ms = [a.elapsed_time(b) for a, b in zip(rec["f0"], rec["f1"])]
    fwd_kernel_ms = [a.elapsed_time(b) for a, b in zip(rec["fk0"], rec["fk1"])]
    dec_ms = [a.elapsed_time(b) for a, b in zip(rec["f1"], rec["d1"])] if Td else [0.0]
    dec_kernel_ms = [a.elapsed_time(b) for s in range(args.steps) for a, b in zip(rec["dk0"][s], rec["dk1"][s])]
    fwd_ms_max = max_over_ranks(sum(fwd_ms), world)
    dec_ms_max = max_over_ranks(sum(dec_ms), world)

    attn_flops = fc.attn_flops
    value = attn_flops * world * args.steps / (fwd_ms_max * 1e-3) / 1e12
    fk = statistics.mean(fwd_kernel_ms)
    achieved = attn_flops / (fk * 1e-3) / 1e12
    lines = {}
    lines["roofline"] = {"kernel": "path_fwd_tc (right-to-left scan; the UT prep is in whole_call below)",
                         "bound": "tensor", "achieved": achieved, "peak": bf16_tf, "unit": "TFLOP/s",
                         "frac": achieved / bf16_tf, "peak_source": peak_src + " bf16 burst",
                         "frac_of_spec": achieved / SPEC_BF16_TFLOPS, "spec_peak": SPEC_BF16_TFLOPS,
                         "traffic": _traffic("path_fwd_tc", fc.B * fc.H),
                         "flops_per_launch": attn_flops, "flops_kind": "attention-equivalent 4*B*H*d*L^2/2",
                         "kernel_ms": fk}
    # the scan's executed tensor-core work, for context (1.5x the attention-equivalent FLOPs off the diagonal)
    tensor_flops = fwd_tensor_flops(fc.B, fc.H, fc.L, fc.d)
    lines["roofline"]["tensor_flops_per_launch"] = tensor_flops
    lines["roofline"]["tensor_frac"] = tensor_flops / (fk * 1e-3) / 1e12 / bf16_tf
    # the whole path_attn_fwd call (UT prep + scan), which the 40 % target is stated on
    fwd_call_ms = fwd_ms_max / args.steps
    whole = attn_flops / (fwd_call_ms * 1e-3) / 1e12
    lines["whole_call"] = {"kernels": "ut_prep_tc + path_fwd_tc", "achieved": whole, "peak": bf16_tf,
                           "unit": "TFLOP/s", "frac": whole / bf16_tf, "frac_of_spec": whole / SPEC_BF16_TFLOPS,
                           "peak_source": peak_src + " bf16 burst", "call_ms": fwd_call_ms,
                           "ut_prep_ms": fwd_call_ms - fk, "ut_prep_ms_kind": "call minus scan kernel (CUDA events)"}
    dec_obj = None
    if Td:
        # algorithmic bytes per decode step: K read + K write + V read of every cached row
        bytes_steps = [3.0 * dc.B * dc.H * (dc.n0 + t) * dc.d * 2 for t in range(Td)]
        avg_bytes = sum(bytes_steps) / Td
        dk_mean = statistics.mean(dec_kernel_ms)
        dec_gbs = avg_bytes / (dk_mean * 1e-3) / 1e9
        us_per_step = dec_ms_max * 1e3 / (args.steps * Td)
        dec_obj = {"us_per_step": us_per_step, "steps_per_sequence": Td, "cache_tokens": dc.n0,
                   "B": dc.B, "H": dc.H, "d": dc.d,
                   "roofline": {"kernel": "decode_update_score", "bound": "hbm", "achieved": dec_gbs,
                                "peak": hbm_gbs, "unit": "GB/s", "frac": dec_gbs / hbm_gbs,
                                "peak_source": peak_src, "frac_of_spec": dec_gbs / SPEC_HBM_GBS,
                                "spec_peak": SPEC_HBM_GBS,
                                "traffic": _traffic("decode_update_score", dc.B * dc.H),
                                "bytes_per_launch": avg_bytes},
                   "step_gbs": avg_bytes / (us_per_step * 1e-6) / 1e9}

    # decode end to end through the public API: every step copies that step's q_t, k_t, v_t, w_t and
    # beta_t from pinned host memory to the device, runs path_decode_step, and copies o_t back to the
    # host.  Copies in run on a side stream into double-buffered device inputs (step t+1's inputs cross
    # while step t computes); the copy out runs on a third stream.
    if Td and args.decode_e2e_steps > 0:
        Te = min(args.decode_e2e_steps, Td)
        hin = [t.cpu().pin_memory() for t in (dq, dk, dv, dw, db)]  # [Td, B, H, d] / [Td, B, H]
        hout = torch.empty((Te,) + tuple(od.shape[1:]), dtype=od.dtype).pin_memory()
        dbuf = [[torch.empty_like(t[0]) for t in (dq, dk, dv, dw, db)] for _ in range(2)]
        obuf = [torch.empty_like(od[0]) for _ in range(2)]
        comp = torch.cuda.current_stream()
        cin, cout = torch.cuda.Stream(), torch.cuda.Stream()
        e_free = [torch.cuda.Event(), torch.cuda.Event()]
        e_in = [torch.cuda.Event(), torch.cuda.Event()]
        e_done = [torch.cuda.Event(), torch.cuda.Event()]
        e_read = [torch.cuda.Event(), torch.cuda.Event()]

        def run_dec_e2e():
            for t in range(Te):
                i = t % 2
                cin.wait_event(e_free[i])
                with torch.cuda.stream(cin):
                    for dst, src in zip(dbuf[i], hin):
                        dst.copy_(src[t], non_blocking=True)
                e_in[i].record(cin)
                comp.wait_event(e_in[i])
                comp.wait_event(e_read[i])
                P.path_decode_step(*dbuf[i], kc, vc, dc.n0 + t, scale=dc.d ** -0.5, out=obuf[i], workspace=ws_d)
                e_free[i].record(comp)
                e_done[i].record(comp)
                cout.wait_event(e_done[i])
                with torch.cuda.stream(cout):
                    hout[t].copy_(obuf[i], non_blocking=True)
                e_read[i].record(cout)
            comp.wait_stream(cout)

        for ev in e_free + e_read:
            ev.record(comp)
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(comp)
        cin.wait_event(a)
        cout.wait_event(a)
        run_dec_e2e()
        b.record(comp)
        torch.cuda.synchronize()
        ems = max_over_ranks(a.elapsed_time(b), world)
        h2d = sum(t[0].numel() * t.element_size() for t in hin)
        d2h = hout[0].numel() * hout.element_size()
        dec_obj["e2e"] = {"value": ems * 1e3 / Te, "unit": "us/step", "steps": Te, "h2d_bytes_per_step": h2d,
                          "d2h_bytes_per_step": d2h,
                          "overlap": "inputs copied on a side stream, double-buffered; o_t copied out on a third"}
        del hin, hout, dbuf, obuf

    # value-side transport (the route transport applied to the values as well): the decode step that
    # transports both caches in place, on the decode workload, and the CUDA-core forward on one batch
    # of the forward workload's heads.  Timed separately, not part of the step.
    vt = None
    if Td and args.vt_steps > 0:
        Tv = min(args.vt_steps, Td)
        ev = [(mk(), mk()) for _ in range(Tv)]
        for t in range(2):
            P.path_decode_step(dq[t], dk[t], dv[t], dw[t], db[t], kc, vc, dc.n0 + t, scale=dc.d ** -0.5,
                               out=od[t], workspace=ws_d, value_transport=True)
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        for t in range(Tv):
            P.path_debug_set_timing_events(ev[t][0], ev[t][1])
            P.path_decode_step(dq[t], dk[t], dv[t], dw[t], db[t], kc, vc, dc.n0 + t, scale=dc.d ** -0.5,
                               out=od[t], workspace=ws_d, value_transport=True)
        P.path_debug_set_timing_events(None, None)
        b.record()
        torch.cuda.synchronize()
        # algorithmic bytes: K and V each read and written once per cached row
        vbytes = statistics.mean(4.0 * dc.B * dc.H * (dc.n0 + t) * dc.d * 2 for t in range(Tv))
        vk = statistics.mean(e0.elapsed_time(e1) for e0, e1 in ev)
        vgbs = vbytes / (vk * 1e-3) / 1e9
        vt = {"decode": {"us_per_step": a.elapsed_time(b) * 1e3 / Tv, "steps": Tv, "cache_tokens": dc.n0,
                         "roofline": {"kernel": "decode_update_score (value transport)", "bound": "hbm",
                                      "achieved": vgbs, "peak": hbm_gbs, "unit": "GB/s", "frac": vgbs / hbm_gbs,
                                      "peak_source": peak_src, "frac_of_spec": vgbs / SPEC_HBM_GBS,
                                      "bytes_per_launch": vbytes, "kernel_ms": vk},
                         "workload": "decode B%d H%d d%d bf16 at a %d-token cache; K and V transported in place"
                                     % (dc.B, dc.H, dc.d, dc.n0)}}
        if args.vt_fwd_steps > 0:
            vq, vk_, vv, vw, vb = q, k, v, w, beta  # the forward's workload
            vo = torch.empty_like(vq)
            vws = P.alloc_workspace(P.load().path_attn_fwd_vt_workspace_bytes(fc.B, fc.H, fc.L, fc.d,
                                                                              P._DT[vq.dtype]), dev)
            P.path_attn_fwd_vt(vq, vk_, vv, vw, vb, scale=x.scale, out=vo, workspace=vws)
            torch.cuda.synchronize()
            a.record()
            for _ in range(args.vt_fwd_steps):
                P.path_attn_fwd_vt(vq, vk_, vv, vw, vb, scale=x.scale, out=vo, workspace=vws)
            b.record()
            torch.cuda.synchronize()
            fms_vt = a.elapsed_time(b) / args.vt_fwd_steps
            vflops = fc.attn_flops
            vt["forward"] = {"ms": fms_vt, "steps": args.vt_fwd_steps,
                             "attn_equiv_tflops": vflops / (fms_vt * 1e-3) / 1e12,
                             "workload": "value-transport forward B%d H%d L%d d%d bf16 (blockwise: UT prep of "
                                         "keys and values, value chains, tensor-core scan over the carried value "
                                         "blocks, diagonal walks)" % (fc.B, fc.H, fc.L, fc.d)}
            del vo, vws

    # end to end through the public API with host buffers: pinned inputs -> device, forward, o -> host,
    # every step.  Copies run on their own stream into double-buffered device inputs, so the next
    # step's inputs cross while this step computes (the order per step is still copy in -> forward
    # -> copy out, enforced with events).
    e2e = None
    if args.e2e_steps > 0:
        hq, hk, hv, hw = (t.pin_memory() for t in (x.q, x.k, x.v, x.w))
        hb = x.beta.pin_memory()
        hos = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for _ in range(2)]
        dins = [[torch.empty_like(t) for t in (q, k, v, w, beta)] for _ in range(2)]
        douts = [torch.empty_like(o) for _ in range(2)]
        h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hw, hb))
        d2h = hos[0].numel() * hos[0].element_size()
        comp = torch.cuda.current_stream()
        # one stream per input tensor (the copy engines run in parallel; beta rides with w) and
        # one for the result
        cps = [torch.cuda.Stream() for _ in range(4)]
        out_s = torch.cuda.Stream()
        freed = [torch.cuda.Event(), torch.cuda.Event()]   # forward done with buffer i
        done = [torch.cuda.Event(), torch.cuda.Event()]    # output of buffer i written
        read = [torch.cuda.Event(), torch.cuda.Event()]    # output of buffer i copied to the host
        srcs = (hq, hk, hv, hw, hb)

        def run_e2e(nsteps):
            for sidx in range(nsteps):
                i = sidx % 2
                for j, dst in enumerate(dins[i]):
                    cs = cps[min(j, 3)]
                    cs.wait_event(freed[i])
                    with torch.cuda.stream(cs):
                        dst.copy_(srcs[j], non_blocking=True)
                for cs in cps:
                    comp.wait_stream(cs)
                comp.wait_event(read[i])  # the previous copy-out of this output buffer has finished
                P.path_attn_fwd(*dins[i], scale=x.scale, out=douts[i], workspace=ws_f)
                freed[i].record(comp)
                done[i].record(comp)
                out_s.wait_event(done[i])
                with torch.cuda.stream(out_s):
                    hos[i].copy_(douts[i], non_blocking=True)
                read[i].record(out_s)
            comp.wait_stream(out_s)

        for ev in freed + read:
            ev.record(comp)
        run_e2e(2)
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(comp)
        for cs in cps + [out_s]:
            cs.wait_event(a)
        run_e2e(args.e2e_steps)
        b.record(comp)
        torch.cuda.synchronize()
        ms = max_over_ranks(a.elapsed_time(b), world)
        e2e = {"value": attn_flops * world * args.e2e_steps / (ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": args.e2e_steps,
               "overlap": "input copies on four streams and the result copy on a fifth, double-buffered: "
                          "step s+1's inputs cross during step s"}

    # PaTH-FoX forwards at L=16384 and L=65536 (far blocks skipped exactly), timed separately,
    # not part of the step
    fox = {}
    for key, cname in (("fox16k", "fox16k_bf16"), ("fox64k", "fox64k_bf16")):
        if args.fox_steps <= 0:
            break
        fxc = inputs.FWD_CONFIGS[cname]
        fx = fxc.make()
        fargs = [t.to(dev) for t in (fx.q, fx.k, fx.v, fx.w, fx.beta, fx.log_f)]
        fscale = fx.scale
        del fx
        fo = torch.empty_like(fargs[0])
        fws = P.alloc_workspace(P.path_attn_workspace_bytes(fxc.B, fxc.H, fxc.L, fxc.d, fargs[0].dtype), dev)
        for _ in range(2):
            P.path_attn_fwd_fox(*fargs, scale=fscale, out=fo, workspace=fws)
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(args.fox_steps):
            P.path_attn_fwd_fox(*fargs, scale=fscale, out=fo, workspace=fws)
        b.record()
        torch.cuda.synchronize()
        fms = a.elapsed_time(b) / args.fox_steps
        visited = P.path_fwd_visited_blocks(fws)
        ntf = -(-fxc.L // 128)
        total = fxc.B * fxc.H * ntf * (ntf + 1) // 2
        executed = fwd_tensor_flops(fxc.B, fxc.H, fxc.L, fxc.d, visited)
        fox[key] = {"ms": fms, "steps": args.fox_steps,
                    "visited_blocks": visited, "total_blocks": total, "visited_frac": visited / total,
                    "executed_tflops": executed / (fms * 1e-3) / 1e12,
                    "executed_frac": executed / (fms * 1e-3) / 1e12 / bf16_tf,
                    "attn_equiv_tflops_full_triangle": fxc.attn_flops / (fms * 1e-3) / 1e12,
                    "workload": "PaTH-FoX forward B%d H%d L%d d%d bf16, log f = logsigmoid(N(3,1)); the far-block "
                                "stop visits visited_blocks of total_blocks (query tile, key block) pairs; "
                                "executed_tflops counts the tensor work of the visited pairs, "
                                "attn_equiv_tflops_full_triangle the full causal triangle (not a throughput)"
                                % (fxc.B, fxc.H, fxc.L, fxc.d)}
        del fargs, fo, fws

    # PaTH + GGD-BAM relative-position prior on the forward workload (side measurement)
    relb = None
    if args.fox_steps > 0:
        rel = inputs.ggd_bam_bias(fc.H, fc.L, seed=fc.seed).to(dev)
        ws_r = P.alloc_workspace(P.path_attn_workspace_bytes(fc.B, fc.H, fc.L, fc.d, q.dtype), dev)
        o_r = torch.empty_like(q)
        for _ in range(2):
            P.path_attn_fwd_relbias(q, k, v, w, beta, rel, scale=x.scale, out=o_r, workspace=ws_r)
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(args.fox_steps):
            P.path_attn_fwd_relbias(q, k, v, w, beta, rel, scale=x.scale, out=o_r, workspace=ws_r)
        b.record()
        torch.cuda.synchronize()
        rms = a.elapsed_time(b) / args.fox_steps
        rvis = P.path_fwd_visited_blocks(ws_r)
        rexec = fwd_tensor_flops(fc.B, fc.H, fc.L, fc.d, rvis)
        relb = {"ms": rms, "attn_equiv_tflops": fc.attn_flops / (rms * 1e-3) / 1e12, "steps": args.fox_steps,
                "visited_blocks": rvis, "executed_tflops": rexec / (rms * 1e-3) / 1e12,
                "workload": "PaTH + GGD-BAM relative-position bias, B%d H%d L%d d%d bf16 (every block visited)"
                            % (fc.B, fc.H, fc.L, fc.d)}
        del rel, ws_r, o_r

    # prefill -> decode hand-off on the forward workload (timed separately, not part of the step)
    prefill = None
    if args.prefill_steps > 0:
        kc_p = torch.empty((fc.B, fc.H, fc.L, fc.d), dtype=q.dtype, device=dev)
        ws_p = P.alloc_workspace(P.path_prefill_workspace_bytes(fc.B, fc.H, fc.L, fc.d, q.dtype), dev)
        P.path_prefill_kcache(k, w, beta, kcache=kc_p, workspace=ws_p)
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(args.prefill_steps):
            P.path_prefill_kcache(k, w, beta, kcache=kc_p, workspace=ws_p)
        b.record()
        torch.cuda.synchronize()
        prefill = {"ms": a.elapsed_time(b) / args.prefill_steps, "steps": args.prefill_steps,
                   "workload": "transported key cache of a B%d H%d L%d d%d bf16 prompt" % (fc.B, fc.H, fc.L, fc.d)}
        del kc_p, ws_p

    # backward pass on the forward workload (timed separately, not part of the step): gradients of
    # every input for a seeded dO, from the forward's own o and lse
    bwd = None
    if args.bwd_steps > 0:
        o_b, lse_b = P.path_attn_fwd(q, k, v, w, beta, scale=x.scale, lse=True)
        gen = torch.Generator(device=dev).manual_seed(1002)
        dO_b = torch.randn(q.shape, generator=gen, device=dev).to(q.dtype)
        ws_b = P.alloc_workspace(P.path_attn_bwd_workspace_bytes(fc.B, fc.H, fc.L, fc.d, q.dtype), dev)
        P.path_attn_bwd(q, k, v, w, beta, o_b, lse_b, dO_b, scale=x.scale, workspace=ws_b)
        torch.cuda.synchronize()
        ev = [[mk() for _ in range(4)] for _ in range(args.bwd_steps)]
        for e in ev:
            P.path_debug_set_timing_events(e[2], e[3])
            e[0].record()
            P.path_attn_bwd(q, k, v, w, beta, o_b, lse_b, dO_b, scale=x.scale, workspace=ws_b)
            e[1].record()
        P.path_debug_set_timing_events(None, None)
        torch.cuda.synchronize()
        bms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
        kms = statistics.mean(e[2].elapsed_time(e[3]) for e in ev)
        # tensor-core FLOPs of the chunk chains (bwd_chain_tc; two 64-row query chunks per 128-row
        # tile, nA = the longer chain): per step down S = U khat^T and dO v^T (M 128, N 64, K 128)
        # and, past key chunk 0, U P^T as three hi/lo products (M 128, N 128, K 128); per step up
        # dS khat (M 128, N 128, K 64) and, past key chunk 0, G P as three products
        nc = -(-fc.L // 64)
        chain_flops = 0
        for kk in range(nc // 2):
            nA = nc - 1 - 2 * kk
            chain_flops += nA * (2 * 2 * 128 * 64 * 128 + 2 * 128 * 128 * 64) + (nA - 1) * 2 * 3 * 2 * 128 ** 3
        chain_flops *= fc.B * fc.H
        ach = chain_flops / (kms * 1e-3) / 1e12
        bwd_traffic = _traffic("bwd_chain_tc", fc.B * fc.H)
        bwd = {"ms": bms, "attn_equiv_tflops": 2.5 * fc.attn_flops / (bms * 1e-3) / 1e12, "steps": args.bwd_steps,
               "workload": "PaTH backward B%d H%d L%d d%d bf16 (dq, dk, dv, dw, dbeta for a seeded dO); "
                           "attention-equivalent FLOPs 2.5 x the forward's" % (fc.B, fc.H, fc.L, fc.d),
               "workspace_gb": ws_b.numel() / 1e9,
               "roofline": {"kernel": "bwd_chain_tc (query-side chunk chains, tcgen05)", "bound": "tensor",
                            "achieved": ach, "peak": bf16_tf, "unit": "TFLOP/s", "frac": ach / bf16_tf,
                            "peak_source": peak_src + " bf16 burst", "traffic": bwd_traffic,
                            "flops_per_launch": float(chain_flops), "flops_kind": "executed MMA FLOPs",
                            "kernel_ms": kms}}
        del o_b, lse_b, dO_b, ws_b

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        v_cpu, dt, cores, desc = oracle_sample(args.cpu_heads)
        cpu = {"value": v_cpu, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": desc,
               "seconds": dt}

    launches_per_step = 2 + 2 * Td  # UT prep + scan; decode: update/score + combine
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded CPU generator; no dataset or trained weights)",
            "config": {"workload": "PaTH forward B%d H12 L4096 d128 bf16 (760M-shaped) + decode B%d H12 d128 "
                                   "bf16 at a 32768-token cache, %d steps" % (fc.B, dc.B, Td),
                       "B": fc.B, "H": fc.H, "L": fc.L, "d": fc.d, "global_batch": fc.B * world,
                       "seq_len": fc.L, "parallelism": "replicas (b,h)-independent" if world > 1 else "single GPU",
                       "l2": "inputs larger than L2 (forward 384 MiB of q,k,v,w; decode caches 13 GB)"},
            "fwd_ms": fwd_ms_max / args.steps, "fwd_kernel_ms": fk, "whole_call": lines["whole_call"],
            "decode": dec_obj, "value_transport": vt, "prefill_kcache": prefill, "fox16k": fox.get("fox16k"), "fox64k": fox.get("fox64k"), "relbias_ggd": relb, "backward": bwd, "roofline": lines["roofline"], "clocks": clk, "e2e": e2e, "cpu_baseline": cpu,
            "gpu_launches": launches_per_step * args.steps}
    if rank == 0:
        print(json.dumps(line))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--decode-steps", type=int, default=256)
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--decode-e2e-steps", type=int, default=64)
    ap.add_argument("--prefill-steps", type=int, default=2)
    ap.add_argument("--vt-steps", type=int, default=16, help="value-transport decode steps (0 = skip)")
    ap.add_argument("--vt-fwd-steps", type=int, default=2, help="value-transport forward calls (0 = skip)")
    ap.add_argument("--fox-steps", type=int, default=3)
    ap.add_argument("--bwd-steps", type=int, default=2)
    ap.add_argument("--cpu-heads", type=int, default=96)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--fwd-B", type=int, default=8, help="forward batch (8 = the timed workload)")
    ap.add_argument("--decode-B", type=int, default=64, help="decode batch (64 = the timed workload)")
    args = ap.parse_args()
    if args.warmup < 3:
        sys.stderr.write("note: warm-up raised to 3 steps\n")
        args.warmup = 3
    rank, world, local = dist_setup()
    if args.impl == "reference":
        rc = run_reference(args, rank, world)
    else:
        rc = run_ours(args, rank, world, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return rc


if __name__ == "__main__":
    sys.exit(main())
