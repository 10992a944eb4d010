#!/usr/bin/env python3
"""Benchmark of the fused mHC boundary (n_hc = 4) on GB300.

A step is one shifted fused boundary call (residual update, sums of squares,
mixer contraction, coefficients, collapse and layer RMSNorm) over the
prefill workload: 8192 tokens, hidden 7168, with every input resident in HBM
when the timed region starts. Per step the inputs (1.18 GB) are far larger
than L2 (129 MB), so no flush is needed; the prepared mixer (2.75 MB) stays
L2-resident as it does in a serving loop.

Prints one JSON line (rank 0). --impl reference times the CPU oracle instead
(there is no other reference implementation), on a bounded sample of the
same workload.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "mHC boundary tokens/s and achieved HBM GB/s (% of GB300 peak), hidden 7168"
WORKLOAD = "prefill_t8192_h7168"


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def alg_bytes_call(T: int, H: int) -> int:
    """Algorithmic bytes of one shifted fused boundary call: residual read and
    write (8H each), x read and layer input write (2H each), 96 B of
    coefficients in and 96 B out per token; the prepared mixer (384H) and the
    fp32 norm weight (4H) once."""
    return T * (20 * H + 192) + 388 * H


# The shifted call is one kernel (the streaming kernel also forms the
# coefficients), so its algorithmic bytes are those of the whole call.
alg_bytes_stream_kernel = alg_bytes_call


def alg_bytes_form(form: str, T: int, H: int) -> int:
    """Algorithmic bytes of one call of each form (one pass over each tensor,
    the byte convention of the FlashInfer page's SOL figures): shifted as
    alg_bytes_call; unshifted fused: no lagged pre in (80 B of coefficients
    in per token); pre-only: residual in, layer input and 96 B of
    coefficients out per token. The prepared mixer and the fp32 norm
    weight once in every form."""
    per_tok = {"shifted": 20 * H + 192, "unshifted": 20 * H + 176, "pre": 10 * H + 96}[form]
    return T * per_tok + 388 * H


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one
# streaming-kernel launch, by (tokens, hidden), from one-pass ncu captures
# of the full-size workload, each with the hash of the kernel sources it was
# taken on (source_hash()). A figure whose hash no longer matches the
# sources being run is not reported: the kernel has changed since.
STREAM_KERNEL_TRAFFIC = {(8192, 7168): (598.66e6 + 540.80e6, "52a3435832430bf3")}
KERNEL_SOURCES = ("stream_kernel.cu", "ptx.cuh", "coef.cuh", "elementwise.cuh", "mhc_internal.h")


def source_hash() -> str:
    """First 16 hex digits of the SHA-256 of the streaming kernel's sources."""
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "manifold_constrained_hyper_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def stream_kernel_traffic(T: int, H: int):
    """(bytes per launch or None, note)."""
    rec = STREAM_KERNEL_TRAFFIC.get((T, H))
    if rec is None:
        return None, "no capture of this size"
    if rec[1] != source_hash():
        print(f"bench: the DRAM traffic figure for {T}x{H} was captured on other kernel "
              f"sources ({rec[1]} != {source_hash()}); reporting traffic null", file=sys.stderr)
        return None, "kernel changed since the capture"
    return rec[0], f"one-pass ncu capture of this workload, sources {rec[1]}"


# ---------------------------------------------------------------- clocks


class ClockSampler:
    """Samples SM clock and clock-event reasons through NVML (read-only)
    every few milliseconds while running."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, torch_dev: int):
        self.samples, self.reasons, self.max_mhz, self.ok = [], set(), None, False
        self._stop = threading.Event()
        try:
            import torch
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return
            props = torch.cuda.get_device_properties(torch_dev)
            bus = f"{props.pci_domain_id:08X}:{props.pci_bus_id:02X}:{props.pci_device_id:02X}.0"
            h = ctypes.c_void_p()
            if nv.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) != 0:
                return
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = mx.value
            self.nv, self.h, self.ok = nv, h, True
        except Exception:
            self.ok = False

    def _run(self):
        mhz, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop.is_set():
            if self.nv.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(mhz)) == 0:
                self.samples.append(mhz.value)
            if self.nv.nvmlDeviceGetCurrentClocksEventReasons(self.h, ctypes.byref(rs)) == 0:
                for bit, name in self.REASONS.items():
                    if rs.value & bit:
                        self.reasons.add(name)
            time.sleep(0.002)

    def __enter__(self):
        if self.ok:
            self._t = threading.Thread(target=self._run, daemon=True)
            self._t.start()
        return self

    def __exit__(self, *a):
        if self.ok:
            self._stop.set()
            self._t.join()

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": sorted(self.reasons),
                    "samples": 0}
        return {"sm_mhz": float(statistics.median(self.samples)), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(self.reasons), "samples": len(self.samples)}


# ---------------------------------------------------------------- oracle timing


def time_oracle(T_sample: int, H: int, seed: int, budget_s: float, chunk: int = 32):
    """The oracle as it stands, on fresh seeded tokens of the workload's
    distribution, single-threaded; stops after `budget_s` or `T_sample`
    tokens. Returns (tokens, seconds)."""
    import oracle as orc
    from manifold_constrained_hyper_gb300 import synth
    d = synth.make_inputs(min(chunk, T_sample), H, seed)
    done, t0 = 0, time.perf_counter()
    while done < T_sample and time.perf_counter() - t0 < budget_s:
        orc.boundary(orc.MODE_FUSED_SHIFTED, d["residual"], d["fn"], d["scale"], d["base"],
                     d["norm_w"], x=d["x"], post_mix=d["post"], comb=d["comb"],
                     pre_lag=d["pre_lag"])
        done += d["residual"].shape[0]
    return done, time.perf_counter() - t0


def time_oracle_threads(T_sample: int, H: int, seed: int, budget_s: float, threads: int,
                        chunk: int = 32):
    """The same oracle, token-parallel: `threads` host threads each run it on
    chunks of the seeded tokens (the C oracle releases the interpreter while
    it computes), until `T_sample` tokens or `budget_s` seconds. Returns
    (tokens, seconds)."""
    import oracle as orc
    from concurrent.futures import ThreadPoolExecutor
    from manifold_constrained_hyper_gb300 import synth
    d = synth.make_inputs(min(chunk, T_sample), H, seed)
    n_chunk = d["residual"].shape[0]
    lock = threading.Lock()
    issued = [0]
    t0 = time.perf_counter()

    def worker(_):
        n = 0
        while True:
            with lock:
                if issued[0] >= T_sample or time.perf_counter() - t0 >= budget_s:
                    return n
                issued[0] += n_chunk
            orc.boundary(orc.MODE_FUSED_SHIFTED, d["residual"], d["fn"], d["scale"], d["base"],
                         d["norm_w"], x=d["x"], post_mix=d["post"], comb=d["comb"],
                         pre_lag=d["pre_lag"])
            n += n_chunk

    with ThreadPoolExecutor(threads) as ex:
        done = sum(ex.map(worker, range(threads)))
    return done, time.perf_counter() - t0


def host_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ---------------------------------------------------------------- arms


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


def rank_seed(base_seed: int, rank: int) -> int:
    """Each rank draws its own shard of tokens (independent inputs)."""
    return base_seed + 7919 * rank


def max_over_ranks(x: float, world: int, device) -> float:
    """The job's time is its slowest rank's."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world: int, tokens_per_rank: int, steps: int, ms: float) -> float:
    """Tokens per second over all ranks (weak scaling: every rank has its own tokens)."""
    return world * tokens_per_rank * steps / (ms / 1e3)


def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return
    if args.form != "shifted":
        raise SystemExit("bench: --impl reference times the shifted call only")
    from manifold_constrained_hyper_gb300 import synth
    import oracle as orc
    orc.build_oracle()
    cfg = synth.WORKLOADS[args.workload]
    H = cfg["H"]
    threads = host_threads()
    chunk = 16
    per_step = max(args.reference_tokens, chunk * threads)
    for _ in range(args.warmup):
        time_oracle_threads(chunk * threads, H, cfg["seed"], 1e9, threads, chunk=chunk)
    total_tok, total_s = 0, 0.0
    for _ in range(args.steps):
        n, s = time_oracle_threads(per_step, H, cfg["seed"], 1e9, threads, chunk=chunk)
        total_tok += n
        total_s += s
    v = total_tok / total_s
    sample = (f"{per_step} tokens per step of the {args.workload} workload (H={H}), "
              f"C oracle token-parallel on {threads} host threads")
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total_s / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": args.workload, "tokens": cfg["T"], "hidden": H, "n_hc": 4,
                   "variant": "shifted fused boundary"},
        "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _graph_us(call, n: int, dev) -> float:
    """Per-call device time of `call` from one replay of a CUDA graph of n calls."""
    import torch
    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for _ in range(n):
                call(s)
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    g.replay()
    b.record()
    torch.cuda.synchronize()
    del g
    return a.elapsed_time(b) * 1e3 / n


def _boundary_call(form, ins, outs, ws, params=None):
    """A call of one form on prepared device tensors: (stream -> None)."""
    from manifold_constrained_hyper_gb300 import ops
    if form == "pre":
        o = {k: outs[k] for k in ("layer_input", "pre_out", "post_out", "comb_out")}
        return lambda st=None: ops.mhc_pre(ins["res"], ins["w"], ins["scale"], ins["base"],
                                           ins["nw"], params, workspace=ws, stream=st, **o)
    pl = ins["pl"] if form == "shifted" else None
    return lambda st=None: ops.mhc_boundary_fused(ins["x"], ins["res"], ins["post"], ins["comb"],
                                                  ins["w"], ins["scale"], ins["base"], ins["nw"],
                                                  pl, params, workspace=ws, stream=st, **outs)


def _device_inputs(d, dev):
    import torch
    from manifold_constrained_hyper_gb300 import ops
    f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(dev)
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a)).view(torch.bfloat16).to(dev)
    res = d["residual_dev"] if "residual_dev" in d else bf(d["residual"])
    x = d["x_dev"] if "x_dev" in d else bf(d["x"])
    return dict(res=res, x=x, post=f32(d["post"]), comb=f32(d["comb"]), pl=f32(d["pre_lag"]),
                scale=f32(d["scale"]), base=f32(d["base"]), nw=f32(d["norm_w"]),
                w=ops.mhc_prepare_weight(f32(d["fn"])))


def _device_outputs(T, H, res, dev):
    import torch
    return dict(residual_out=torch.empty_like(res),
                layer_input=torch.empty(T, H, dtype=torch.bfloat16, device=dev),
                pre_out=torch.empty(T, 4, device=dev), post_out=torch.empty(T, 4, device=dev),
                comb_out=torch.empty(T, 4, 4, device=dev))


def measure_decode(dev, token_counts=None):
    """Latency of one call at the decode batch sizes, hidden 7168 (the seeded
    decode workload, seed 1000 + T):
    * graph / graph_unshifted / graph_pre: per call from a CUDA graph of 100
      calls of the shifted, unshifted fused and pre-only forms (launch cost
      amortised, L2 warm as in a decode loop);
    * eager_warm: device time of one eager shifted call with L2 warm, its
      events and the call enqueued behind a short GPU sleep so that they run
      back to back (the host's enqueue time is not counted); the mean over
      60 calls (one call's event pair reads on a coarse grid, in steps of
      about 2 us, so a median would be a grid value);
    * eager_cold_l2: the same after a 256 MB buffer was written (L2 cold),
      mean over 30 calls;
    * host_us_per_call: host time of one eager shifted call through the
      Python binding, through ctypes with its arguments prebuilt, and of the
      C entry point alone (the ctypes time less that of a 0-token call, which
      returns after its first checks), mean over 200 calls;
    * pair_pdl / pair_no_pdl (1 and 64 tokens): a copy kernel producing x
      followed by the call, per pair from a CUDA graph of 50 pairs, with the
      boundary launched as a programmatic dependent of the producer or not.
    The decode path of each size is the default one (cluster_ctas > 0: one
    thread-block cluster; else the slice-parallel streaming kernel)."""
    import ctypes as ct
    import torch
    from manifold_constrained_hyper_gb300 import ops, synth
    token_counts = token_counts or synth.DECODE_TOKENS
    H = synth.DECODE_HIDDEN
    scrub = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    out = {"hidden": H, "unit": "us/call", "graph": {}, "graph_unshifted": {}, "graph_pre": {},
           "eager_warm": {}, "eager_cold_l2": {}, "host_us_per_call": {}, "pair_pdl": {},
           "pair_no_pdl": {}, "slices": {}, "cluster_ctas": {}, "waves": {}}
    sms = min(152, torch.cuda.get_device_properties(dev).multi_processor_count)
    for T in token_counts:
        cfg = synth.decode_workload(T)
        d = synth.make_inputs(cfg["T"], cfg["H"], seed=cfg["seed"])
        ins = _device_inputs(d, dev)
        outs = _device_outputs(T, H, ins["res"], dev)
        ws = torch.empty(ops.workspace_bytes(T, H), dtype=torch.uint8, device=dev)
        call = _boundary_call("shifted", ins, outs, ws)
        for _ in range(5):
            call()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(90)]
        for a, b in ev:
            a.record()
            b.record()
        torch.cuda.synchronize()
        warm, cold = [], []
        for i, (a, b) in enumerate(ev):
            if i < 30:
                scrub.add_(1)
            torch.cuda._sleep(100_000)               # the GPU waits while the host enqueues
            a.record()
            call()
            b.record()
            torch.cuda.synchronize()
            (cold if i < 30 else warm).append(a.elapsed_time(b) * 1e3)
        # host time per call: Python binding, then the C entry point alone
        lib = ops.load()
        p = ops.Params().c()
        cst = ops._stream(None, ins["res"].device)
        args = [ins["x"].data_ptr(), ins["res"].data_ptr(), ins["post"].data_ptr(),
                ins["comb"].data_ptr(), ins["pl"].data_ptr(), ins["w"].data_ptr(),
                ins["scale"].data_ptr(), ins["base"].data_ptr(), ins["nw"].data_ptr(), 0,
                ct.byref(p), T, H, outs["residual_out"].data_ptr(), outs["layer_input"].data_ptr(),
                outs["pre_out"].data_ptr(), outs["post_out"].data_ptr(), outs["comb_out"].data_ptr(),
                ws.data_ptr(), ws.numel(), cst]
        # the same call with 0 tokens returns right after its first checks:
        # its time is the ctypes marshalling of the 21 arguments alone
        args0 = list(args)
        args0[11] = 0
        host = {}
        for kind in ("python", "c_entry_via_ctypes", "ctypes_only"):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            for _ in range(200):
                if kind == "python":
                    call()
                elif kind == "c_entry_via_ctypes":
                    lib.mhc_boundary_fused(*args)
                else:
                    lib.mhc_boundary_fused(*args0)
            host[kind] = (time.perf_counter() - t0) / 200 * 1e6
            torch.cuda.synchronize()
        host["c_entry"] = host["c_entry_via_ctypes"] - host["ctypes_only"]
        out["host_us_per_call"][str(T)] = host
        # a producer of x (a copy kernel) and the boundary, replayed from a
        # graph of 50 pairs, with the boundary a programmatic dependent of
        # the producer (its set-up overlapping the producer's end) or not
        if T in (1, 64):
            x_src = ins["x"].clone()
            pair_call = lambda st=None: (ops.mhc_debug_delayed_copy(x_src, ins["x"], 0, stream=st),
                                         call(st))
            for pdl in (1, 0):
                ops.mhc_debug_set_pdl(pdl)
                out["pair_pdl" if pdl else "pair_no_pdl"][str(T)] = _graph_us(pair_call, 50, dev)
            ops.mhc_debug_set_pdl(1)
        key = str(T)
        out["graph"][key] = _graph_us(call, 100, dev)
        for form in ("unshifted", "pre"):
            out["graph_" + form][key] = _graph_us(_boundary_call(form, ins, outs, ws), 100, dev)
        out["eager_warm"][key] = statistics.fmean(warm)
        out["eager_cold_l2"][key] = statistics.fmean(cold)
        S, _ = ops.plan(T, H)
        out["slices"][key] = S
        out["cluster_ctas"][key] = ops.plan_cluster(T, H)
        out["waves"][key] = -(-((T + 127) // 128 * S) // sms)
    if ops.mhc_get_device_status() != 0:
        raise RuntimeError("device-side wait timed out during the decode sweep")
    return out


def measure_forms(dev):
    """Every form of the boundary at the mid-batch (512 x 7168) and prefill
    (8192 x 7168) sizes, and the stress workload (1024 x 4096, residual ~
    N(0, 8) with outliers, base ~ N(0, 4), 20 Sinkhorn iterations): per call
    from a CUDA graph of calls (inputs larger than L2 at 8192 tokens; at the
    smaller sizes the inputs stay L2-resident between calls, as in a layer
    loop that reuses its buffers), GB/s over each form's algorithmic bytes
    (alg_bytes_form) and its fraction of the measured copy bandwidth."""
    import torch
    from manifold_constrained_hyper_gb300 import ops, synth
    peak, _ = measured_peaks()
    res_out = {"unit": "us/call", "peak_gbs": peak, "cases": {}}
    cases = [("mid_t512_h7168", 50), ("prefill_t8192_h7168", 10), ("stress_t1024_h4096", 20)]
    for name, n in cases:
        cfg = dict(synth.WORKLOADS[name])
        T, H, seed = cfg.pop("T"), cfg.pop("H"), cfg.pop("seed")
        d = synth.make_inputs_device(T, H, seed, dev, **cfg)
        ins = _device_inputs(d, dev)
        outs = _device_outputs(T, H, ins["res"], dev)
        ws = torch.empty(ops.workspace_bytes(T, H), dtype=torch.uint8, device=dev)
        for form in ("shifted", "unshifted", "pre"):
            us = _graph_us(_boundary_call(form, ins, outs, ws), n, dev)
            gbs = alg_bytes_form(form, T, H) / us / 1e3
            res_out["cases"][f"{name}/{form}"] = {
                "tokens": T, "hidden": H, "us": us, "tokens_per_s": T / us * 1e6, "gbps": gbs,
                "frac_of_peak": gbs / peak, "graph_calls": n}
        del d, ins, outs, ws
        torch.cuda.empty_cache()
    if ops.mhc_get_device_status() != 0:
        raise RuntimeError("device-side wait timed out while timing the forms")
    return res_out


def measure_split_k(dev):
    """Per-call time of the split-K pre at the shapes the FlashInfer page
    times its pure path on (tokens x hidden: 4096 x 4096, 4096 x 7168,
    128 x 7168; one split), from a CUDA graph of 20 calls. Inputs are seeded
    on the device; the 4096-token cases exceed L2."""
    import torch
    from manifold_constrained_hyper_gb300 import ops, synth
    out = {"unit": "us/call", "splits": 1, "cases": {}}
    for T, H in ((4096, 4096), (4096, 7168), (128, 7168)):
        d = synth.make_inputs_device(T, H, 3, dev)
        f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(dev)
        g = torch.Generator(dev).manual_seed(5)
        dm = torch.randn(1, T, 24, device=dev, generator=g)
        sq = 4.0 * H * (0.8 + 0.4 * torch.rand(1, T, device=dev, generator=g))
        scale, base, nw = f32(d["scale"]), f32(d["base"]), f32(d["norm_w"])
        o = dict(layer_input=torch.empty(T, H, dtype=torch.bfloat16, device=dev),
                 pre_out=torch.empty(T, 4, device=dev), post_out=torch.empty(T, 4, device=dev),
                 comb_out=torch.empty(T, 4, 4, device=dev))
        res = d["residual_dev"]

        def call(s=None):
            ops.mhc_pre_split_k(res, dm, sq, scale, base, nw, stream=s, **o)

        for _ in range(3):
            call()
        torch.cuda.synchronize()
        st = torch.cuda.Stream(device=dev)
        st.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(st):
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=st):
                for _ in range(20):
                    call(st)
        torch.cuda.synchronize()
        gr.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        gr.replay()
        b.record()
        torch.cuda.synchronize()
        us = a.elapsed_time(b) * 1e3 / 20
        byts = T * (8 * H + 2 * H + 196) + 4 * H
        peak, _ = measured_peaks()
        out["cases"][f"{T}x{H}"] = {"us": us, "gbps": byts / us / 1e3,
                                    "frac_of_peak": byts / us / 1e3 / peak}
        del gr
    return out


def run_ours(args):
    import torch
    import torch.distributed as dist
    from manifold_constrained_hyper_gb300 import build as mbuild
    from manifold_constrained_hyper_gb300 import ops, synth

    rank, local, world = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")
    if rank == 0 or not os.path.exists(ops.lib_path()):
        mbuild.build()
    if world > 1:
        dist.barrier()
    ops.load()
    dev = torch.device("cuda", local)
    cfg = dict(synth.WORKLOADS[args.workload])
    if args.tokens:
        cfg["T"] = args.tokens
    if args.hidden:
        cfg["H"] = args.hidden
    T, H = cfg["T"], cfg["H"]
    extra = {k: v for k, v in cfg.items() if k not in ("T", "H", "seed")}
    d = synth.make_inputs_device(T, H, rank_seed(cfg["seed"], rank), dev, **extra)
    f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(dev)
    res, x = d["residual_dev"], d["x_dev"]
    post, comb, pre_lag = f32(d["post"]), f32(d["comb"]), f32(d["pre_lag"])
    scale, base, nw = f32(d["scale"]), f32(d["base"]), f32(d["norm_w"])
    w = ops.mhc_prepare_weight(f32(d["fn"]))
    params = ops.Params(sinkhorn_iters=20)
    ro = torch.empty_like(res)
    li = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    pr = torch.empty(T, 4, device=dev)
    po = torch.empty(T, 4, device=dev)
    cb = torch.empty(T, 4, 4, device=dev)
    ws = torch.empty(max(ops.workspace_bytes(T, H), 16), dtype=torch.uint8, device=dev)

    form = args.form

    def step():
        if form == "pre":
            ops.mhc_pre(res, w, scale, base, nw, params, layer_input=li, pre_out=pr, post_out=po,
                        comb_out=cb, workspace=ws)
        else:
            ops.mhc_boundary_fused(x, res, post, comb, w, scale, base, nw,
                                   pre_lag if form == "shifted" else None, params,
                                   residual_out=ro, layer_input=li, pre_out=pr, post_out=po,
                                   comb_out=cb, workspace=ws)

    for _ in range(max(args.warmup, 0)):
        step()
    torch.cuda.synchronize()
    if ops.mhc_get_device_status() != 0:
        raise RuntimeError("device-side wait timed out during warm-up")

    # A step is one kernel launch (the shifted call's streaming kernel also
    # forms the coefficients) and nothing else runs on the stream, so two
    # events bracketing K back-to-back steps time that kernel: its average
    # duration is the region over K, as a layer loop runs it (each launch a
    # programmatic dependent of the previous one, its set-up overlapping that
    # one's end). An event between launches would cut that overlap and add
    # its own time: the same kernel with events around each launch is timed
    # apart, after the timed region (kernel_ms.stream_isolated).
    K = args.steps
    t_begin, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # torch creates CUDA events lazily: record each once so that no creation
    # lands in the timed region
    for e in (t_begin, t_end):
        e.record()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    launches0 = ops.mhc_debug_launch_count()
    with ClockSampler(local) as clk:
        t_begin.record()
        for i in range(K):
            step()
        t_end.record()
        torch.cuda.synchronize()
    # this library's kernels launched in the timed region (counted by the library)
    gpu_launches = ops.mhc_debug_launch_count() - launches0
    if world > 1:
        dist.barrier()
    status = ops.mhc_get_device_status()
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed region")
    total_ms = max_over_ranks(t_begin.elapsed_time(t_end), world, dev)
    stream_ms = t_begin.elapsed_time(t_end) / K
    ms_per_step = total_ms / K
    value = whole_job_rate(world, T, K, total_ms)
    peak, peak_kind = measured_peaks()
    gbps_call = alg_bytes_form(form, T, H) / (ms_per_step / 1e3) / 1e9
    # the shifted call is the streaming kernel alone; the other forms are
    # timed as whole calls (past a single wave: streaming, coefficients and
    # collapse kernels)
    ach = alg_bytes_form(form, T, H) / (stream_ms / 1e3) / 1e9
    # the same kernel with events on both sides of each launch (50 launches)
    n_iso = min(K, 50)
    ev_s = [torch.cuda.Event(enable_timing=True) for _ in range(n_iso)]
    ev_e = [torch.cuda.Event(enable_timing=True) for _ in range(n_iso)]
    for e in ev_s + ev_e:
        e.record()
    torch.cuda.synchronize()
    for i in range(n_iso):
        ev_s[i].record()
        step()
        ev_e[i].record()
    torch.cuda.synchronize()
    stream_iso_ms = statistics.mean(ev_s[i].elapsed_time(ev_e[i]) for i in range(n_iso))

    # ---------------- end to end: host buffers through the public API
    # Every step copies its inputs in from pinned host memory and its outputs
    # back out. Device buffers are double-buffered and the copies run on
    # their own streams, so that step k's copy-out overlaps step k + 1's
    # copy-in (the host link carries both directions at once).
    e2e = None
    if not args.no_e2e and form == "shifted":
        K2 = max(1, min(K, args.e2e_steps))
        dev_in = [(torch.empty_like(res), torch.empty_like(x), [torch.empty_like(t) for t in (post, comb, pre_lag)])
                  for _ in range(2)]
        dev_out = [[torch.empty_like(t) for t in (ro, li, pr, po, cb)] for _ in range(2)]
        h_in = [(torch.empty(res.shape, dtype=res.dtype, pin_memory=True).copy_(res),
                 torch.empty(x.shape, dtype=x.dtype, pin_memory=True).copy_(x),
                 [torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t)
                  for t in (post, comb, pre_lag)]) for _ in range(2)]
        h_out = [[torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (ro, li, pr, po, cb)]
                 for _ in range(2)]
        h2d = sum(t.numel() * t.element_size() for t in [h_in[0][0], h_in[0][1]] + h_in[0][2])
        d2h = sum(t.numel() * t.element_size() for t in h_out[0])
        s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        s_comp = torch.cuda.current_stream()

        def e2e_run(n):
            comp_done = [None, None]
            out_done = [None, None]
            for k in range(n):
                b = k % 2
                (dres, dx, dsm), (hres, hx, hsm) = dev_in[b], h_in[b]
                with torch.cuda.stream(s_in):
                    if comp_done[b] is not None:          # step k - 2 has read these inputs
                        s_in.wait_event(comp_done[b])
                    dres.copy_(hres, non_blocking=True)
                    dx.copy_(hx, non_blocking=True)
                    for dd, hh in zip(dsm, hsm):
                        dd.copy_(hh, non_blocking=True)
                    in_done = torch.cuda.Event()
                    in_done.record(s_in)
                s_comp.wait_event(in_done)
                if out_done[b] is not None:               # step k - 2's outputs are on the host
                    s_comp.wait_event(out_done[b])
                o = dev_out[b]
                ops.mhc_boundary_fused(dx, dres, dsm[0], dsm[1], w, scale, base, nw, dsm[2], params,
                                       residual_out=o[0], layer_input=o[1], pre_out=o[2],
                                       post_out=o[3], comb_out=o[4], workspace=ws, stream=s_comp)
                comp_done[b] = torch.cuda.Event()
                comp_done[b].record(s_comp)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(comp_done[b])
                    for hh, dd in zip(h_out[b], o):
                        hh.copy_(dd, non_blocking=True)
                    out_done[b] = torch.cuda.Event()
                    out_done[b].record(s_out)
            torch.cuda.synchronize()

        e2e_run(2)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        e2e_run(K2)
        e_ms = max_over_ranks((time.perf_counter() - t0) * 1e3, world, dev)
        e2e = {"value": whole_job_rate(world, T, K2, e_ms), "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": K2,
               "overlap": "double-buffered; copy-in and copy-out on their own streams"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        threads = host_threads()
        n1, s1 = time_oracle(T, H, cfg["seed"], args.cpu_seconds / 4)
        n, s = time_oracle_threads(T * 8, H, cfg["seed"], args.cpu_seconds, threads)
        cpu = {"value": n / s, "unit": "tokens/s", "cores": threads, "kind": "oracle",
               "sample": f"{n} tokens of the {args.workload} distribution in {s:.1f} s, "
                         f"C oracle token-parallel on {threads} host threads, chunks of 32",
               "single_thread": {"value": n1 / s1, "cores": 1,
                                 "sample": f"{n1} tokens in {s1:.1f} s"}}

    decode = forms = split_k = None
    if not args.no_decode:
        decode = measure_decode(dev)
        forms = measure_forms(dev)
        split_k = measure_split_k(dev)

    S, sw = ops.plan(T, H)
    traffic, traffic_note = (stream_kernel_traffic(T, H) if form == "shifted"
                             else (None, "no capture of this form"))
    variant = {"shifted": "shifted fused boundary", "unshifted": "unshifted fused boundary",
               "pre": "unshifted pre-only boundary"}[form]
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; residual/x ~ N(0,1) bf16, doubly stochastic comb)",
        "config": {"workload": args.workload, "tokens": T, "hidden": H, "n_hc": 4,
                   "variant": variant, "sinkhorn_iters": 20,
                   "decode_path": "cluster" if ops.plan_cluster(T, H) else "slice-parallel",
                   "norm_w": "fp32", "hidden_slices": S, "slice_width": sw,
                   "l2": "inputs larger than L2 (no flush); prepared mixer L2-resident",
                   "parallelism": f"replicas x{world} (token-sharded, no collective)"},
        "achieved_gbps": gbps_call,
        "achieved_frac_of_peak": gbps_call / peak,
        "kernel_ms": {"stream": stream_ms, "stream_isolated": stream_iso_ms},
        "roofline": {"bound": "hbm",
                     "kernel": "stream_kernel" if form == "shifted" else "whole call",
                     "achieved": ach, "peak": peak,
                     "unit": "GB/s", "frac": ach / peak, "traffic": traffic,
                     "traffic_source": traffic_note, "peak_source": peak_kind},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": gpu_launches,
        "decode": decode,
        "forms": forms,
        "pre_split_k": split_k,
        "clocks": clk.summary(),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--form", choices=["shifted", "unshifted", "pre"], default="shifted",
                    help="the form timed on the workload (the headline is the shifted call; "
                         "the others for their own roofline and launch lists)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode", action="store_true",
                    help="skip the decode-latency sweep (1-64 tokens), the other forms and "
                         "workloads, and the split-K pre timings")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--reference-tokens", type=int, default=256)
    ap.add_argument("--tokens", type=int, default=0,
                    help="override the workload's token count (profiling a smaller case)")
    ap.add_argument("--hidden", type=int, default=0,
                    help="override the workload's hidden size (profiling another kernel: a "
                         "shifted call of up to 16 tokens at hidden 512 takes the cluster kernel)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
